// expert_args.cuh -- what the two grouped expert GEMM kernels (tensor memory, expert_tc.cu;
// register MMA for small groups, expert_mma.cu) share: the launch arguments, the mapping of a
// persistent CTA's work item to (group, m-tile), and the addresses of an item's operands.
//
// Work items: for the gate/up GEMM an item is 128 interleaved gate/up weight rows (64
// outputs) of one group's expert; for the down GEMM, 128 output rows.  Shared-expert groups
// come first, then routed groups, each group's m-tiles consecutive.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.cuh"
#include "tc.cuh"

namespace moe {

struct TcArgs {
  const uint8_t *routed;
  uint64_t routed_stride;
  const uint8_t *shared;
  ExpertLayout LR, LS;
  int H, E, k, T, Imax, P;
  const Group *groups;
  Ctrl *ctrl;
  int ns;
  const uint8_t *xg;  // gate/up B tiles (bf16)
  uint8_t *hg;        // gate/up output = down B tiles (fp16)
  float *y;           // down output [rows][H]
  int ra, rb;         // chunks per code run / per activation-tile run
  long wait_limit;    // nanoseconds a single wait may take before it gives up
  long long *trace;   // MOE_TRACE builds only: per-chunk event clocks of CTA 0
};

template <int BITS>
struct ATile {
  static constexpr int row_bytes = 64 * BITS / 8;
  static constexpr int bytes = 128 * row_bytes;  // one chunk of 128 weight rows
};

struct Item {
  Group g;
  int mt, K, KC, rowsB, rows8, Npad;
  bool sh;
  const uint8_t *ebase;
};

template <bool DOWN>
__device__ __forceinline__ bool tc_item(const TcArgs &a, int item, Item &it) {
  const int n_groups = a.ctrl->n_groups;
  const int mt_s = DOWN ? a.H / 128 : a.LS.inter / 64;
  const int mt_r = DOWN ? a.H / 128 : a.LR.inter / 64;
  const int shi = a.ns * mt_s;
  if (item >= shi + (n_groups - a.ns) * mt_r) return false;
  int gi;
  if (item < shi) { gi = item / mt_s; it.mt = item % mt_s; it.sh = true; }
  else { int i2 = item - shi; gi = a.ns + i2 / mt_r; it.mt = i2 % mt_r; it.sh = false; }
  it.g = a.groups[gi];
  const ExpertLayout &L = it.sh ? a.LS : a.LR;
  it.ebase = it.sh ? a.shared : a.routed + a.routed_stride * it.g.e;
  it.K = DOWN ? L.inter : a.H;
  it.KC = it.K / kKChunk;
  it.rowsB = DOWN ? it.g.n : a.P * it.g.n;
  it.rows8 = round8(it.rowsB);
  it.Npad = round16(it.rowsB);
  return true;
}

// codes of chunk kc of the item's matrix (consecutive chunks are contiguous)
template <int BITS, bool DOWN>
__device__ __forceinline__ const uint8_t *a_src(const TcArgs &a, const Item &it, int kc) {
  const ExpertLayout &L = it.sh ? a.LS : a.LR;
  return it.ebase + (DOWN ? L.down_off : L.gu_off) +
         ((size_t)it.mt * it.KC + kc) * ATile<BITS>::bytes;
}

// the item's activation tile of chunk kc (consecutive chunks are contiguous)
template <bool DOWN>
__device__ __forceinline__ const uint8_t *b_src(const TcArgs &a, const Item &it, int kc) {
  const uint8_t *base = DOWN ? a.hg + (size_t)it.g.hrow0 * a.Imax * 2
                             : a.xg + (size_t)it.g.xrow0 * a.H * 2;
  return base + (size_t)kc * it.rows8 * 128;
}

// bounded wait that ignores the abort flag (used to drain after an abort)
__device__ __forceinline__ bool wait_nofail(uint64_t *bar, uint32_t parity, long limit_ns) {
  const uint64_t t0 = tc::global_ns();
  while (!tc::mbar_try_wait_sleep(bar, parity, 20000))
    if ((long)(tc::global_ns() - t0) > limit_ns) return false;
  return true;
}

// Small-group expert GEMMs (every group's B rows <= kMmaMaxRows): register-MMA kernel.
constexpr int kMmaMaxRows = 16;
int launch_experts_mma(int bits, bool down, TcArgs a, int rows_max, int kc_gcd, int bound,
                       int sms, cudaStream_t st);
size_t mma_smem_bytes(int bits);

}  // namespace moe

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
  const uint8_t *xg;  // gate/up B tiles (fp16, x_t * tscale[t])
  const uint8_t *xt;    // decode-sized forwards: per-token fp16 rows [T][P][H] (register MMA)
  const float *tscale;  // per token: the power-of-two activation scale
  const int32_t *perm;  // slot of every permuted row (token = slot / k)
  float *rscale;      // per xg row: 1 / tscale of the row's token
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
  int mt, nmt, K, KC, rowsB, rows8, Npad;  // first m-tile, m-tiles of the item (1 or MT)
  bool sh;
  const uint8_t *ebase;
};

// Work item `item` of a launch whose items are MT consecutive m-tiles of one group (the
// last item of a group takes fewer when MT does not divide the group's m-tiles).
template <bool DOWN, int MT = 1>
__device__ __forceinline__ bool tc_item(const TcArgs &a, int item, Item &it) {
  // through L2 (every role reads the work list, written by earlier launches, after the
  // kernel's griddepcontrol.wait)
  const int n_groups = __ldcg(&a.ctrl->n_groups);
  const int nm_s = DOWN ? a.H / 128 : a.LS.inter / 64;  // m-tiles of a shared-expert group
  const int nm_r = DOWN ? a.H / 128 : a.LR.inter / 64;
  const int mt_s = (nm_s + MT - 1) / MT, mt_r = (nm_r + MT - 1) / MT;  // items per group
  const int shi = a.ns * mt_s;
  if (item >= shi + (n_groups - a.ns) * mt_r) return false;
  int gi, nm;
  if (item < shi) { gi = item / mt_s; it.mt = (item % mt_s) * MT; it.sh = true; nm = nm_s; }
  else {
    int i2 = item - shi;
    gi = a.ns + i2 / mt_r;
    it.mt = (i2 % mt_r) * MT;
    it.sh = false;
    nm = nm_r;
  }
  it.nmt = nm - it.mt < MT ? nm - it.mt : MT;
  {
    const int4 *gp = (const int4 *)(a.groups + gi);
    const int4 g0 = __ldcg(gp), g1 = __ldcg(gp + 1);
    it.g = Group{g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  }
  const ExpertLayout &L = it.sh ? a.LS : a.LR;
  it.ebase = it.sh ? a.shared : a.routed + a.routed_stride * it.g.e;
  it.K = DOWN ? L.inter : a.H;
  it.KC = it.K / kKChunk;
  it.rowsB = DOWN ? it.g.n : a.P * it.g.n;
  it.rows8 = round8(it.rowsB);
  it.Npad = round16(it.rowsB);
  return true;
}

// codes of chunk kc of m-tile it.mt + m of the item's matrix (consecutive chunks are
// contiguous)
template <int BITS, bool DOWN>
__device__ __forceinline__ const uint8_t *a_src(const TcArgs &a, const Item &it, int kc,
                                                int m = 0) {
  const ExpertLayout &L = it.sh ? a.LS : a.LR;
  return it.ebase + (DOWN ? L.down_off : L.gu_off) +
         ((size_t)(it.mt + m) * it.KC + kc) * ATile<BITS>::bytes;
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

// ---------------------------------------------------------------- codes -> fp16 pairs
// Dequantisation to exact small integers in fp16 (the codes' per-row scale is applied to
// the fp32 accumulator).  A biased code c placed in the low mantissa bits of 1024.0
// (0x6400) reads as 1024 + c; placed 4 (or 2, 6) bits higher it reads as 1024 + 16c
// (4c, 64c), and one fused multiply-add by 1/16 (1/4, 1/64) removes both the magic and
// the bias.  Every intermediate is an integer below 2048 or its exact power-of-two
// multiple, so each step is exact.  The pair of a word's two 16-bit halves is one (lo, hi)
// fragment register of a 16-bit MMA operand.
__device__ __forceinline__ uint32_t h2_sub(uint32_t v, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t v, uint32_t m, uint32_t a) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(m), "r"(a));
  return r;
}
__device__ __forceinline__ uint32_t lop_and_or(uint32_t v, uint32_t mask, uint32_t magic) {
  uint32_t r;  // (v & mask) | magic in one logic op: truth table (a & b) | c = 0xEA
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "r"(mask), "r"(magic));
  return r;
}

// int4 word (pair p in nibbles p and p+4) -> pairs 0..3
__device__ __forceinline__ void dq_word_i4(uint32_t w, uint32_t *o) {
  const uint32_t M = 0x64006400u;
  const uint32_t w8 = w >> 8;
  o[0] = h2_sub(lop_and_or(w, 0x000F000Fu, M), 0x64086408u);               // 1024+c - 1032
  o[1] = h2_fma(lop_and_or(w, 0x00F000F0u, M), 0x2C002C00u, 0xD480D480u);  // /16 - 72
  o[2] = h2_sub(lop_and_or(w8, 0x000F000Fu, M), 0x64086408u);
  o[3] = h2_fma(lop_and_or(w8, 0x00F000F0u, M), 0x2C002C00u, 0xD480D480u);
}

// int2 word (pair p in 2-bit fields p and p+8) -> pairs 0..7
__device__ __forceinline__ void dq_word_i2(uint32_t w, uint32_t *o) {
  const uint32_t M = 0x64006400u;
#pragma unroll
  for (int half = 0; half < 2; half++) {
    const uint32_t v = half ? w >> 8 : w;
    uint32_t *q = o + 4 * half;
    q[0] = h2_sub(lop_and_or(v, 0x00030003u, M), 0x64026402u);               // 1024+c - 1026
    q[1] = h2_fma(lop_and_or(v, 0x000C000Cu, M), 0x34003400u, 0xDC08DC08u);  // /4 - 258
    q[2] = h2_fma(lop_and_or(v, 0x00300030u, M), 0x2C002C00u, 0xD420D420u);  // /16 - 66
    q[3] = h2_fma(lop_and_or(v, 0x00C000C0u, M), 0x24002400u, 0xCC80CC80u);  // /64 - 18
  }
}

// int8 word (two's complement bytes 0..3) -> pairs 0..1: b ^ 0x80 = b + 128 in [0, 255]
// goes under 0x64 (1024 + b + 128), minus 1152
__device__ __forceinline__ void dq_word_i8(uint32_t w, uint32_t *o) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  o[0] = h2_sub(a, 0x64806480u);
  o[1] = h2_sub(b, 0x64806480u);
}

// Small-group expert GEMMs (every group's B rows <= kMmaMaxRows): register-MMA kernel.
// Down launches split each item's contraction into ks parts (ks must divide every item's
// count of code runs), part sp > 0 writing y plane sp at ysplit + (sp - 1) * yplane floats.
int launch_experts_mma(int bits, bool down, TcArgs a, int rows_max, int kc_gcd, int bound,
                       int sms, cudaStream_t st, int ks = 1, float *ysplit = nullptr,
                       long yplane = 0);
size_t mma_smem_bytes(int bits);

}  // namespace moe

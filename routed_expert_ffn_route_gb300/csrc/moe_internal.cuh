// moe_internal.cuh -- private layouts and helpers of the GB300 MoE-layer library.
//
// Packed weight blob (device memory, caller-owned; private layout, versioned header):
//   [header 256 B][router_w fp32 E*H][router_bias fp32 E][router tiles]
//   [expert 0]...[expert E-1][shared]
// Router tiles: the fp32 router matrix as three bf16 pieces (w = hi + mid + lo exactly),
// the tensor-core router's A operand: [piece][E/128 m-tiles][H/64 k-chunks] blocks of
// [128 rows][64 bf16], 128-byte swizzled (16-byte chunk c of row r at c ^ (r & 7)); rows
// past E are zero.
// Every expert block is 4096-byte aligned and holds
//   gate/up codes : (I/64 m-tiles) x (H/64 k-chunks) blocks of [128 rows][CB bytes]
//                   rows interleaved: row 2j = gate row (64*mt + j), row 2j+1 = up row
//   down codes    : (H/128 m-tiles) x (I/64 k-chunks) blocks of [128 rows][CB bytes]
//   gate/up scales: fp32 [I/64][128], same interleave as the rows
//   down scales   : fp32 [H]
// CB = 64 * bits / 8 bytes: one row's 64 contraction elements of one k-chunk.
// Code order inside a row chunk (biased codes, b = q + 2^(bits-1)):
//   int4: 8 words of 32 bits; word w holds elements 8w..8w+7, element 8w+2p+s in
//         nibble p+4s  (so (word >> 4p) & 0x000F000F yields the pair (2p, 2p+1)).
//   int2: 4 words; word w holds elements 16w..16w+15, element 16w+2p+s in 2-bit
//         field p+8s  (so (word >> 2p) & 0x00030003 yields the pair (2p, 2p+1)).
//   int8: 16 words; element 4w+i in byte i of word w, plain two's complement.
// The [128 rows][CB] blocks stream as contiguous 4 KB (int4) units; a row's pair
// layout feeds both the fp32 FMA path and a 16-bit tensor-core operand directly.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr uint32_t kMagic = 0x50454F4Du;  // "MOEP"
constexpr uint32_t kVersion = 2;
constexpr int kHeaderBytes = 256;
constexpr int kKChunk = 64;     // contraction elements per chunk
constexpr int kTileRows = 128;  // weight rows per block

struct PackHeader {
  uint32_t magic, version;
  int32_t hidden, inter, inter_shared, n_experts, n_shared, weight_bits;
  int32_t act_q8_0, router, n_group, topk_group;
};

struct ExpertLayout {
  int inter;                 // I of this expert
  uint64_t gu_off, down_off, sgu_off, sd_off;  // relative to the expert base
  uint64_t bytes;            // stride of the expert block (aligned)
};

struct PackLayout {
  uint64_t router_w_off, router_b_off, router_t_off, experts_off, shared_off, total;
  ExpertLayout routed, shared;
};

constexpr int kRouterTileBytes = 128 * 64 * 2;  // one router tile: 128 rows x 64 bf16
static inline int router_mtiles(const moe_layer_config &c) { return (c.n_experts + 127) / 128; }

static inline uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

static inline ExpertLayout expert_layout(int H, int I, int bits) {
  ExpertLayout L;
  L.inter = I;
  uint64_t cb = (uint64_t)kKChunk * bits / 8;
  uint64_t gu = (uint64_t)(I / 64) * (H / kKChunk) * kTileRows * cb;
  uint64_t dn = (uint64_t)(H / kTileRows) * (I / kKChunk) * kTileRows * cb;
  L.gu_off = 0;
  L.down_off = align_up(gu, 256);
  L.sgu_off = align_up(L.down_off + dn, 256);
  L.sd_off = align_up(L.sgu_off + (uint64_t)2 * I * 4, 256);
  L.bytes = align_up(L.sd_off + (uint64_t)H * 4, 4096);
  return L;
}

static inline PackLayout pack_layout(const moe_layer_config &c) {
  PackLayout P;
  int Is = c.inter_shared ? c.inter_shared : c.inter;
  P.router_w_off = kHeaderBytes;
  P.router_b_off = align_up(P.router_w_off + (uint64_t)c.n_experts * c.hidden * 4, 256);
  P.router_t_off = align_up(P.router_b_off + (uint64_t)c.n_experts * 4, 1024);
  P.experts_off = align_up(P.router_t_off + (uint64_t)3 * router_mtiles(c) * (c.hidden / 64) *
                                                kRouterTileBytes,
                           4096);
  P.routed = expert_layout(c.hidden, c.inter, c.weight_bits);
  P.shared = expert_layout(c.hidden, Is, c.weight_bits);
  P.shared_off = P.experts_off + P.routed.bytes * (uint64_t)c.n_experts;
  P.total = P.shared_off + (c.n_shared ? P.shared.bytes : 0);
  return P;
}

// ---------------------------------------------------------------- workspace
// [ctrl 256 B][router partials fp32 HS*T*E][offsets E+1][perm T*k][slot_pos T*k]
// [groups max_groups][xq int8 T*H][xd fp32 T*H/32]
// tensor-core path: [tscale fp32 T][rscale fp32 xg rows][xg fp16 tiles][hg fp16 tiles]
// CUDA-core path: [h fp32 R*Imax]
// [y fp32 R*H], with R = T*k + n_shared*T rows (routed slots in permuted order, then the
// shared expert's tokens).  xg / hg hold each group's activation rows as 128-byte-swizzled
// tiles [k-chunk][rows rounded up to 8][64 elements], the B operand layout of the
// tensor-core GEMMs (1024-byte aligned chunk tiles).  xg holds x_t * tscale[t]: tscale is
// a power of two per token that brings max |x_t| into [2^14, 2^15), so that the fp16
// operand keeps every bf16 value exactly; rscale[row] = 1 / tscale of the row's token.
struct Ctrl {
  int status;      // moe_status recorded on the device (0 = OK)
  int detail;      // where it was recorded (kernel id)
  int n_groups;    // groups written by the permute kernel (shared groups included)
  int front_done;  // fused decode front: expert blocks of the router GEMV finished
  int pad[60];
};

constexpr int kRouterHS = 8;   // H splits of the small-T router GEMV
constexpr int kMmaMaxRows = 16;  // largest group (activation rows) of the register-MMA kernels
constexpr int kTcMaxRows = 128;  // B-operand rows (tokens x pieces) of one tensor-core group

// Expert kernels: tcgen05 tensor-core GEMMs for float activations; the CUDA-core dp4a
// kernels for Q8_0 activations (per-32-block integer dots with per-block scales).
static inline bool use_tc(const moe_layer_config &c) { return !c.act_q8_0; }

struct WsLayout {
  uint64_t ctrl, partials, offsets, perm, slot_pos, groups, xq, xd, tscale, rscale, xg, hg, h,
      y, ysplit, total;
  int max_groups, group_n, rows, pieces;
  int ks;  // contraction parts of the decode down launch (y planes: y, then ks - 1 at ysplit)
  bool tc;
  // The experts this call computes: routed experts [e0, e1) and, when `shared` is set, the
  // shared expert (an expert-parallel share of the layer; the whole layer by default).
  // The routing and the permutation always cover every expert.
  int e0, e1;
  bool shared;
};

int choose_group_n(const moe_layer_config &c, int T);
size_t permute_smem(int T, int E);

static inline int gcd_int(int x, int y) { return y ? gcd_int(y, x % y) : x; }

// The decode down launch (the register-MMA kernel: T <= kMmaMaxRows) has one work item per
// (expert, 128-row m-tile of H).  When the batch's experts give fewer items than about
// kDownSplitItems (a few experts with a long contraction, e.g. a Mixtral-shaped layer at
// T = 1: 2 experts x 32 m-tiles against ~300 CTAs), each item's contraction is split into
// ks contiguous parts (a power of two dividing every item's count of code runs), each part
// writing its own y plane, which the combine adds in plane order.  The item count is
// estimated from the config (the experts a batch of T tokens can reach), so ks only falls
// as T grows; the DeepSeek-V3-shaped layer (>= 9 experts x 48 m-tiles) never splits.
constexpr int kDownSplitItems = 512;  // Mixtral T = 4: 2 parts, down 53 -> 45 us
constexpr int kDownSplitMax = 8;
static inline int down_splits(const moe_layer_config &c, int T) {
  if (c.act_q8_0 || T < 1 || T > kMmaMaxRows) return 1;
  const int Is = c.inter_shared ? c.inter_shared : c.inter;
  const int kc = gcd_int(c.inter / 64, Is / 64);  // as the launch computes it
  const int ra = kc % 4 == 0 ? 4 : (kc % 2 == 0 ? 2 : 1);  // chunks per code run
  const int runs = kc / ra;
  const long items = (long)((c.n_experts < T * c.top_k ? c.n_experts : T * c.top_k) +
                            (c.n_shared ? 1 : 0)) * (c.hidden / 128);
  int s = 1;
  while (s < kDownSplitMax && items * 2 * s <= kDownSplitItems && runs % (2 * s) == 0) s *= 2;
  return s;
}

// `pieces`: fp16 rows per token in the tensor-core B operand (1 for bf16 x, 2 for fp32 x
// split as hi + lo).  Region offsets and the total do not depend on it.
static inline WsLayout ws_layout(const moe_layer_config &c, int T, int pieces = 1) {
  WsLayout W;
  int Is = c.inter_shared ? c.inter_shared : c.inter;
  int Imax = c.inter > Is ? c.inter : Is;
  int k = c.top_k;
  W.tc = use_tc(c);
  W.pieces = pieces;
  int gn_min = W.tc ? kTcMaxRows / 2 : choose_group_n(c, T);
  // Tensor-core groups of at most 128 B rows, or 64 when the batch gives an expert few
  // tokens on average (T k <= 16 E): launches of <= 64-row groups take two m-tiles per work
  // item, which saves more than the few large groups lose by reading their codes twice
  // (DSV3 T = 128 / 256: gate/up + down 987 -> 812, 1110 -> 949 us; at T = 1024 the cap
  // costs 20%).  The work list is sized for 64-row groups either way.
  const int gcap = (long)T * k <= 16L * c.n_experts ? kTcMaxRows / 2 : kTcMaxRows;
  W.group_n = W.tc ? gcap / pieces : gn_min;
  W.rows = T * k + (c.n_shared ? T : 0);
  W.e0 = 0;
  W.e1 = c.n_experts;
  W.shared = c.n_shared != 0;
  int tk = T * k;
  W.max_groups = (tk + gn_min - 1) / gn_min + (c.n_experts < tk ? c.n_experts : tk) +
                 (c.n_shared ? (T + gn_min - 1) / gn_min : 0) + 1;
  // tile rows per group are padded to a multiple of 8: up to 7 extra rows per group
  uint64_t xg_rows = W.tc ? (uint64_t)2 * W.rows + 7ull * W.max_groups : 0;
  uint64_t hg_rows = W.tc ? (uint64_t)W.rows + 7ull * W.max_groups : 0;
  uint64_t o = 0;
  W.ctrl = o; o += 256;
  // router partial logits [HS][T][E], then per-slice max |x| [HS][T]
  W.partials = o; o = align_up(o + (uint64_t)kRouterHS * T * (c.n_experts + 1) * 4, 256);
  W.offsets = o; o = align_up(o + (uint64_t)(c.n_experts + 1) * 4, 256);
  W.perm = o; o = align_up(o + (uint64_t)tk * 4, 256);
  W.slot_pos = o; o = align_up(o + (uint64_t)tk * 4, 256);
  W.groups = o; o = align_up(o + (uint64_t)W.max_groups * 32, 256);
  W.xq = o; o = align_up(o + (c.act_q8_0 ? (uint64_t)T * c.hidden : 0), 256);
  W.xd = o; o = align_up(o + (c.act_q8_0 ? (uint64_t)T * (c.hidden / 32) * 4 : 0), 256);
  W.tscale = o; o = align_up(o + (W.tc ? (uint64_t)T * 4 : 0), 256);
  W.rscale = o; o = align_up(o + xg_rows * 4, 1024);
  W.xg = o; o = align_up(o + xg_rows * c.hidden * 2, 1024);
  W.hg = o; o = align_up(o + hg_rows * Imax * 2, 256);
  W.h = o; o = align_up(o + (W.tc ? 0 : (uint64_t)W.rows * Imax * 4), 256);
  W.y = o; o = align_up(o + (uint64_t)W.rows * c.hidden * 4, 256);
  // planes 1.. of a split decode down launch: sized for the most parts any T' <= T takes
  // (T' = 1) times the rows of min(T, kMmaMaxRows) tokens, so a workspace sized for T
  // holds every smaller call's planes
  W.ks = down_splits(c, T);
  {
    const int t16 = T < kMmaMaxRows ? T : kMmaMaxRows;
    const uint64_t rows16 = (uint64_t)t16 * k + (c.n_shared ? t16 : 0);
    W.ysplit = o;
    o = align_up(o + (uint64_t)(down_splits(c, 1) - 1) * rows16 * c.hidden * 4, 256);
  }
  W.total = o;
  return W;
}

// The router takes the GEMV path (logits split over H slices) for small batches.
static inline bool router_gemv(const moe_layer_config &c, int T) {
  return T <= 16 && (size_t)T * (c.hidden / kRouterHS) * 4 <= 96 * 1024;
}

// Decode-sized forwards: every gate/up group fits the register-MMA kernel (pieces x tokens
// <= 16 rows).  Those kernels read each token's fp16 activation row (xt, at the start of
// the xg region) instead of per-group tiles; with the GEMV router, the GEMV's last CTA
// also selects, permutes and writes those rows (one launch in front of the expert GEMMs).
static inline bool decode_rows(const moe_layer_config &c, int T, int pieces) {
  return use_tc(c) && T <= kTcMaxRows / pieces && pieces * T <= kMmaMaxRows;
}
static inline bool fused_front(const moe_layer_config &c, int T, int pieces) {
  return decode_rows(c, T, pieces) && router_gemv(c, T);
}

// ---------------------------------------------------------------- device helpers
enum KernelId { kKRouter = 1, kKTopk = 2, kKPermute = 3, kKGateUp = 4, kKDown = 5,
                kKCombine = 6, kKQuant = 7, kKDebugWait = 8 };

__device__ __forceinline__ void record_status(Ctrl *ctrl, int status, int where) {
  if (atomicCAS(&ctrl->status, 0, status) == 0) ctrl->detail = where;
}

// The packed blob's header against the layer config (checked once per router launch).
__device__ __forceinline__ void check_header(const uint8_t *packed, const moe_layer_config &c,
                                             Ctrl *ctrl) {
  const PackHeader *h = (const PackHeader *)packed;
  int Is = c.inter_shared ? c.inter_shared : c.inter;
  if (h->magic != kMagic || h->version != kVersion || h->hidden != c.hidden ||
      h->inter != c.inter || h->inter_shared != Is || h->n_experts != c.n_experts ||
      h->n_shared != c.n_shared || h->weight_bits != c.weight_bits)
    record_status(ctrl, MOE_ERR_PACKED, kKRouter);
}

// A group: `n` permuted rows starting at `pos0` that all use expert `e`.  For the shared
// expert (e == E), rows are tokens pos0 .. pos0+n-1.  xrow0 / hrow0: the group's first
// row in the xg / hg tile buffers (tensor-core path).
struct Group {
  int e, pos0, n, xrow0, hrow0, pad0, pad1, pad2;
};

__host__ __device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }
__host__ __device__ __forceinline__ int round8(int v) { return (v + 7) & ~7; }

// ---------------------------------------------------------------- launch helpers
// Record a caller's timing event on `st`.  While `st` is being captured into a CUDA graph
// the record becomes a graph node (replays record it), so stage timings also work for
// graph-launched forwards.
static inline cudaError_t record_stage_event(void *ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cudaErrorUnknown;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags((cudaEvent_t)ev, st, cudaEventRecordExternal)
             : cudaEventRecord((cudaEvent_t)ev, st);
}

// Launch `k` on `st` with programmatic stream serialisation: the kernel may begin while
// its predecessor finishes, and calls pdl_wait() before it touches the predecessor's output.
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

struct DevInfo {
  int sms;
  int smem_optin;
};
DevInfo dev_info();
// Per (kernel, device) host-side caches: the dynamic shared-memory limit is raised once;
// occupancy answers are computed once per launch shape.
void set_dyn_smem(const void *func, int bytes);
int cached_blocks_per_sm(const void *func, int threads, size_t smem);

// kernels (one translation unit each)
// fused: the decode front (selection, permutation and activation rows in the GEMV launch)
int launch_router(const moe_layer_config &c, const uint8_t *packed, const void *x, moe_dtype dt,
                  int T, int32_t *ids, float *w, uint8_t *ws, const WsLayout &W,
                  cudaStream_t st, bool fused = false);
int launch_permute(const moe_layer_config &c, int T, const int32_t *ids, uint8_t *ws,
                   const WsLayout &W, cudaStream_t st);
int launch_quant_x(const moe_layer_config &c, const void *x, moe_dtype dt, int T, uint8_t *ws,
                   const WsLayout &W, cudaStream_t st);
int launch_experts_tc(const moe_layer_config &c, const uint8_t *packed, const void *x,
                      moe_dtype dt, int T, uint8_t *ws, const WsLayout &W, cudaStream_t st,
                      void *act, void *mid, bool front_rows);
// act_event / mid_event (cudaEvent_t or null) are recorded after the activation encoding
// (tensor-core path: the fp16 tile gather or token rows) and between the gate/up and down
// launches; front_rows: the fused decode front already wrote the token rows
int launch_experts(const moe_layer_config &c, const uint8_t *packed, const void *x,
                   moe_dtype dt, int T, uint8_t *ws, const WsLayout &W, cudaStream_t st,
                   void *act_event, void *mid_event, bool front_rows = false);
// pf, pf_bytes: an optional region (16-byte aligned, a multiple of 16 bytes) the combine starts
// loading into L2, for the launch that follows
int launch_combine(const moe_layer_config &c, int T, const float *w, float *out, uint8_t *ws,
                   const WsLayout &W, cudaStream_t st, const uint8_t *pf = nullptr,
                   uint64_t pf_bytes = 0);
int launch_pack_expert(const moe_layer_config &c, const ExpertLayout &L, const int8_t *gate,
                       const int8_t *up, const int8_t *down, const float *sg, const float *su,
                       const float *sd, uint8_t *base, cudaStream_t st);
int launch_unpack_expert(const moe_layer_config &c, const ExpertLayout &L, const uint8_t *base,
                         int8_t *gate, int8_t *up, int8_t *down, float *sg, float *su, float *sd,
                         cudaStream_t st);
int launch_write_header(const moe_layer_config &c, uint8_t *packed, cudaStream_t st);
int launch_router_tiles(const moe_layer_config &c, const float *router_w, uint8_t *tiles,
                        cudaStream_t st);
// router logits of large bf16 batches on the tensor cores: partials[hs][t][e] for hsplits
// H slices (the selection adds them in slice order); false when the launch does not apply
bool router_tc_applies(const moe_layer_config &c, moe_dtype dt, int T);
int launch_router_tc(const moe_layer_config &c, const uint8_t *packed, const void *x, int T,
                     float *partials, int hsplits, Ctrl *ctrl, cudaStream_t st);
int launch_quantize_rows(const void *w, moe_dtype dt, int rows, int cols, int bits, int8_t *q,
                         float *scale, cudaStream_t st);
int launch_q8_quantize(const void *x, moe_dtype dt, int T, int n, int8_t *q, float *d,
                       cudaStream_t st);
int launch_block_dots(const moe_layer_config &c, const uint8_t *mat, int K, int mat_rows,
                      int which, const int32_t *rows, int n_rows, const int8_t *qa, int n_tok,
                      int32_t *dots, cudaStream_t st);
int launch_debug_wait(uint8_t *ws, int iterations, cudaStream_t st);

}  // namespace moe

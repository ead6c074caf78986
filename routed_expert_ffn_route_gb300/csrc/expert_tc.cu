// expert_tc.cu -- the grouped SwiGLU expert GEMMs on the 5th-generation tensor cores.
//
// Expert FFN ("企业官网建设流程全解析", §3.1 激活内存池化: SwiGLU gate_proj; "Show HN: 如何在我的
// 低配置电脑上运行 GLM-5.2", 已实现的功能: routed-expert SwiGLU, 量化内核 int8/int4/int2 逐行缩放,
// 使用时反量化; "colibrì 深度拆解", §5.1 per-row scaled int4):
//   g = s_g * (Q_g x),  u = s_u * (Q_u x),  h = silu(g) * u,  y = s_d * (Q_d h)
//
// Tensor-core formulation (one CTA per SM, persistent over work items of one group and
// one or two m-tiles of 128 weight rows):
//   D[128 weight rows][N] (fp32, TMEM) += A[128][K] * B[N][K]^T, per m-tile
//   A = codes of 128 weight rows, dequantised to exact small integers in fp16 (against
//       fp16 activation tiles: scaled x, or h) and written to TMEM, so the weight
//       operand costs no shared-memory read bandwidth (tcgen05.mma with A in TMEM);
//   B = the group's activation rows (<= 128 tokens x pieces, padded to a multiple of 8), a
//       128-byte-swizzled K-major tile produced in that exact layout in global memory; the
//       MMA's N is the row count rounded up to 16, and the extra rows it reads only feed
//       accumulator columns the epilogue never reads; one tile serves both m-tiles of a
//       two-m-tile item;
//   the fp32 per-row scale factors out of each dot and is applied in the epilogue.
//
// The K dimension streams in 64-element chunks.  Operands move in runs of several chunks
// per bulk copy (codes: RA chunks of each of the item's m-tiles, RA x 4 KB at int4;
// activation tiles: RB chunks), so the hand-off latency of a copy (its stage must first be
// released by the consumers) is paid once per run.  A unit of two chunks (of every m-tile
// of the item) of dequantised codes lives in one of the TMEM stages next to the
// accumulators; the unit's stage hand-off between dequantisers and MMA issuer costs about
// the same whether it carries 8 MMAs or 16, so narrow launches (groups of <= 64 rows,
// where TMEM has room) take two m-tiles per item.
//
// Warp roles: 20 code producer and 21 activation-tile producer (bulk copies, one thread
// each), 0 MMA issuer (the warp runs the loop, one elected thread issues; items alternate
// between two TMEM accumulator buffers), 8-19 dequantisers in three sets that take turns
// by unit (one weight row of each m-tile per thread, smem -> registers -> TMEM; no more
// sets than stages), 4-7 epilogue (TMEM -> registers, scale, SwiGLU, stores; overlaps the
// next item's MMAs).  Every wait is bounded: a wait that gives up records MOE_ERR_TIMEOUT,
// all roles stop, in-flight copies and MMAs are drained and TMEM is freed before exit.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dev.cuh"
#include "expert_args.cuh"
#include "rows.cuh"
#include "moe_internal.cuh"
#include "tc.cuh"

namespace moe {

// Pipeline tracing for development builds (-DMOE_TRACE): the SM clock at each hand-off of
// the first kTraceChunks chunks of CTA 0, one row of kTraceChunks per event.
#ifdef MOE_TRACE
constexpr int kTraceChunks = 256;
#define MOE_TC_TRACE(ev, c)                                               \
  do {                                                                    \
    if (blockIdx.x == 0 && a.trace && (c) < kTraceChunks)                 \
      a.trace[(ev) * kTraceChunks + (c)] = (long long)clock64();          \
  } while (0)
static long long *g_trace = nullptr;
long long *g_router_trace = nullptr;  // router selection phases (row 16 of the buffer)
extern "C" void moe_trace_set(void *buf) {
  g_trace = (long long *)buf;
  g_router_trace = buf ? (long long *)buf + 16 * kTraceChunks : nullptr;
}
#define MOE_TC_TRACE_R(ev, c) \
  do {                         \
    if (r == 0) MOE_TC_TRACE(ev, c); \
  } while (0)
#else
#define MOE_TC_TRACE_R(ev, c) \
  do {                        \
  } while (0)
#define MOE_TC_TRACE(ev, c) \
  do {                      \
  } while (0)
#endif

// warps: 0-3 MMA issuers (0 also owns TMEM), 4-7 epilogue, 8-19 dequantiser sets (4 warps
// each: one per TMEM lane quarter), 20 code producer, 21 activation-tile producer
constexpr int kDqSets = 3;
constexpr int kDqWarp0 = 8;
constexpr int kProdWarp0 = kDqWarp0 + 4 * kDqSets;
constexpr int kWarps = kProdWarp0 + 2;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxIssuers = 4;
// Chunks per hand-off between the dequantisers and the MMA issuer (one TMEM stage): a
// barrier round trip costs a few hundred cycles on a busy SM, so each one covers 8 MMAs.
// Every K is a multiple of 128, so every item has a whole number of units.
constexpr int kUnit = 2;
constexpr int kMaxStages = 16;
constexpr int kMaxRuns = 24;

// One MMA issuer warp (issuing from converged code costs about one MMA's math time at
// N = 128).  The accumulator (NMAX columns, NMAX = the launch's largest B row count) is
// double-buffered by item parity, so that the epilogue of one item overlaps the MMAs of
// the next.  TMEM (512 columns) holds the two accumulators and up to 15 chunk stages of
// dequantised codes (32 columns each).  Shared memory holds the code-run ring and the
// activation-tile ring.
// MT: m-tiles per work item (1 or 2).  With two, one unit hands the issuer both m-tiles'
// chunks (16 MMAs against one activation tile): the stage hand-off, not the MMAs, bounds
// the pipeline at small group sizes, so a unit costs about the same with twice the work.
// A stage holds MT x kUnit chunks; each accumulator buffer holds MT accumulators of NMAX
// columns; ACCB: accumulator buffers (2: the epilogue overlaps the next item's MMAs).
template <int NMAX, int MT = 1, int ACCB = 2>
struct Plan {
  static constexpr int issuers = 1;
  static constexpr int acc_bufs = ACCB;
  static constexpr int buf_cols = MT * NMAX;  // one accumulator buffer
  static constexpr int stage_cols = 32 * kUnit * MT;
  static constexpr int stages_fit = (512 - acc_bufs * buf_cols) / stage_cols;
  static constexpr int stages = stages_fit < kMaxStages ? stages_fit : kMaxStages;
  static constexpr int acc_col = stages * stage_cols;
};

// Shared-memory rings.  Each code run (16 KB at int4) covers several chunks, so three runs
// (two at int8) give ample lookahead; everything else goes to the activation-tile ring,
// whose copies wait on the most latency (tiles read by many CTAs, across both dies' L2).
template <int NMAX, int BITS>
struct Rings {
  static constexpr int a_ring = BITS == 8 ? 64 * 1024 : 48 * 1024;
  static constexpr int b_ring = 220 * 1024 - a_ring;
};

struct TcBars {
  uint64_t a_full[kMaxRuns], a_empty[kMaxRuns];  // code runs (smem)
  uint64_t b_full[kMaxRuns], b_empty[kMaxRuns];  // activation-tile runs (smem)
  uint64_t t_full[kMaxStages];                   // codes dequantised into a TMEM stage
  uint64_t done[kMaxStages];                     // the chunk's MMAs completed
  uint64_t acc_full[2], acc_empty[2];  // per accumulator buffer
  uint64_t drain[kMaxIssuers];
  uint32_t tmem_base;
  int abort_flag;
  float escale[4][kTcMaxRows];  // gate/up epilogue, per warp: the item's per-row act. scales
};

template <int NMAX, int BITS>
constexpr size_t tc_smem() {
  return 1024 + (size_t)Rings<NMAX, BITS>::a_ring + Rings<NMAX, BITS>::b_ring + sizeof(TcBars);
}

// One weight row's 64 codes (one k-chunk) -> 32 pairs of exact fp16 integers (element 2c
// in the low half of column c).  Rows are 32 B apart at int4: lanes read the two 16-byte
// halves in an order that puts the 8 lanes of each shared-memory phase on distinct banks.
template <int BITS>
__device__ __forceinline__ void dequant_row(const uint8_t *src, int lane, uint32_t (&o)[32]) {
  if (BITS == 4) {
    const int h0 = (lane >> 2) & 1;
    const uint4 ua = ((const uint4 *)src)[h0], ub = ((const uint4 *)src)[h0 ^ 1];
    const uint4 u0 = h0 ? ub : ua, u1 = h0 ? ua : ub;
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int i = 0; i < 8; i++) dq_word_i4(w[i], o + 4 * i);
  } else if (BITS == 2) {
    const uint4 u = ((const uint4 *)src)[0];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) dq_word_i2(w[i], o + 8 * i);
  } else {
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const uint4 u = ((const uint4 *)src)[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; i++) dq_word_i8(w[i], o + 8 * q + 2 * i);
    }
  }
}

// Position in a ring of S stages (stage, phase parity), advanced one step at a time: the
// ring sizes and run lengths are launch parameters, and stepping avoids integer division.
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int S) {
    if (++s == S) { s = 0; ph ^= 1; }
  }
};
// A chunk's place in runs of R chunks that occupy a ring of S stages.
struct RunPos {
  int j = 0;  // chunk within its run
  Ring r;     // the run's stage
  __device__ __forceinline__ void next(int R, int S) {
    if (++j == R) { j = 0; r.next(S); }
  }
};

// Consecutive CTAs take adjacent m-tiles of a group, which read the same activation tiles:
// each CTA loads its own copy of them (the group's first reader brings them into L2).
template <int BITS, bool DOWN, int NMAX, int MT, int ACCB>
__global__ void __launch_bounds__(kThreads, 1) tc_expert_kernel(TcArgs a, int item_bound) {
  using PL = Plan<NMAX, MT, ACCB>;
  using RG = Rings<NMAX, BITS>;
  constexpr int NI = PL::issuers;
  constexpr int AB = ATile<BITS>::bytes, RB = ATile<BITS>::row_bytes;
  extern __shared__ uint8_t smraw[];
  uint8_t *base = tc::align_smem_1024(smraw);
  uint8_t *bring = base;
  uint8_t *aring = base + RG::b_ring;
  TcBars *bars = (TcBars *)(aring + RG::a_ring);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int where = DOWN ? kKDown : kKGateUp;
  // ring geometry of this launch
  const int ra = a.ra, rb = a.rb;
  const int a_run = MT * ra * AB;  // bytes of a code run: [m-tile][ra chunks]
  const int b_stride = (rb + (rb > 1 ? 1 : 0)) * NMAX * 128;  // run + the MMA's over-read
  const int SA = min(kMaxRuns, RG::a_ring / a_run), SB = min(kMaxRuns, RG::b_ring / b_stride);
  // TMEM stages in use.  A dequantiser set waits only on the ring runs of its own units, so
  // it may poll a ring stage for run r while run r - (ring size), one lap back, is still in
  // flight; a parity wait cannot tell those two phases apart.  A set works at most ST units
  // ahead of the oldest unit whose MMAs are unfinished, and every chunk before that window
  // has landed, so the early pass cannot happen while the stages hold no more chunks than
  // either ring: kUnit * ST <= SA * ra and <= SB * rb.
  const int ST = min(PL::stages, min(SA * ra, SB * rb) / kUnit);
  // Dequantiser sets in use.  A set waits on a stage's `done` barrier for the stage's
  // previous unit, which another set may have taken; its own last unit on that stage is
  // `sets` units back in the rotation, so with more sets than stages the stage can turn
  // over twice between its waits and the parity test passes a lap early.  No more sets
  // than stages, then (the others idle).
  const int nsets = min(kDqSets, ST);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; s++) {
      tc::mbar_init(&bars->a_full[s], 1);
      tc::mbar_init(&bars->a_empty[s], 4 * ra);  // every dequantiser warp of every chunk
    }
    for (int s = 0; s < SB; s++) {
      tc::mbar_init(&bars->b_full[s], 1);
      tc::mbar_init(&bars->b_empty[s], rb < NI ? rb : NI);  // the issuers
    }
    for (int s = 0; s < ST; s++) {
      tc::mbar_init(&bars->t_full[s], 4);  // the set's 4 warps
      tc::mbar_init(&bars->done[s], 1);
    }
    for (int b = 0; b < 2; b++) {
      tc::mbar_init(&bars->acc_full[b], NI);
      tc::mbar_init(&bars->acc_empty[b], 4);  // the 4 epilogue warps
    }
    for (int i = 0; i < NI; i++) tc::mbar_init(&bars->drain[i], 1);
    bars->abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc<512>(&bars->tmem_base);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  pdl_wait();  // the set-up above overlaps the previous launch; the work list is its output
  pdl_trigger();
  const uint32_t tbase = bars->tmem_base;
  volatile int *abort = &bars->abort_flag;
  const long lim = a.wait_limit;
  auto give_up = [&]() {
    if (!*abort) { *abort = 1; record_status(a.ctrl, MOE_ERR_TIMEOUT, where); }
  };

  if (warp >= kProdWarp0) {
    // ------------------------------------------------ producers: one bulk copy per run
    if (lane == 0) {
      const bool isA = warp == kProdWarp0;
      const int R = isA ? ra : rb, S = isA ? SA : SB;
      uint64_t *full = isA ? bars->a_full : bars->b_full;
      uint64_t *empty = isA ? bars->a_empty : bars->b_empty;
      uint32_t armed = 0, last_ph = 0;
      int run = 0;
      Ring pos;
      bool ok = true;
      Item it;
      for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x) {
        if (!tc_item<DOWN, MT>(a, item, it)) break;
        // the item's activation tiles are one contiguous range, read again by the group's
        // other m-tiles: start it towards L2 now, so that the ring's copies hit L2
        if (!isA)
          tc::bulk_prefetch_l2(b_src<DOWN>(a, it, 0), (uint32_t)it.KC * it.rows8 * 128);
        for (int kc = 0; kc < it.KC; kc += R, run++, pos.next(S)) {
          const int s = pos.s;
          const uint32_t ph = pos.ph;
          if (!tc::mbar_wait_backoff(&empty[s], ph ^ 1, abort, lim, 64)) { ok = false; break; }
          if (isA) {
            // one copy per m-tile of the item: [m-tile][ra chunks] in the run's stage
            const int nmt = MT == 1 ? 1 : it.nmt;
            tc::mbar_arrive_expect_tx(&full[s], (uint32_t)(nmt * ra * AB));
            for (int m = 0; m < nmt; m++)
              tc::bulk_g2s(aring + s * a_run + m * ra * AB, a_src<BITS, DOWN>(a, it, kc, m),
                           ra * AB, &full[s]);
            MOE_TC_TRACE(0, run * R);
          } else {
            const uint32_t bytes = (uint32_t)R * it.rows8 * 128;
            tc::mbar_arrive_expect_tx(&full[s], bytes);  // every run lands here
            tc::bulk_g2s(bring + s * b_stride, b_src<DOWN>(a, it, kc), bytes, &full[s]);
            MOE_TC_TRACE(1, run * R);
          }
          armed |= 1u << s;
          last_ph = (last_ph & ~(1u << s)) | (ph << s);
        }
      }
      if (!ok) {
        give_up();
        // let every copy this thread started land before the CTA exits
        for (int q = 0; q < S; q++)
          if ((armed >> q) & 1) wait_nofail(&full[q], (last_ph >> q) & 1, lim);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------ MMA issuer
    // The whole warp runs the loop (uniform control flow and operands); one elected lane
    // waits and issues the tcgen05 instructions.  A unit of kUnit chunks needs one wait: its
    // dequantiser set publishes the TMEM stage only once the chunks' activation tiles landed.
    static_assert(NI == 1, "one issuer");
    if (warp == 0) {
      const bool leader = tc::elect_one();
      int c = 0, n = 0;
      Ring tpos;    // TMEM stage of the unit
      RunPos bpos;  // activation-tile run of chunk c
      bool ok = true, issued = false;
      Item it;
      for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x, n++) {
        if (!tc_item<DOWN, MT>(a, item, it)) break;
        // accumulator buffer ab, used for the au-th time
        const int ab = n % PL::acc_bufs, au = n / PL::acc_bufs;
        int got = 1;
        if (leader) got = tc::mbar_wait(&bars->acc_empty[ab], (au & 1) ^ 1, abort, lim);
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t idesc = tc::idesc_f16(0, it.Npad);  // fp16 x fp16 -> fp32
        // m-tile m of the item accumulates at dcol + m * NMAX
        const uint32_t dcol = tbase + PL::acc_col + ab * PL::buf_cols;
        for (int ku = 0; ku < it.KC; ku += kUnit, tpos.next(ST)) {
          got = 1;
          if (leader) MOE_TC_TRACE(10, c);
          if (leader) got = tc::mbar_wait_spin(&bars->t_full[tpos.s], tpos.ph, abort, lim);
          if (leader) MOE_TC_TRACE(11, c);
          ok = __all_sync(0xffffffffu, got);
          if (!ok) break;
          tc::fence_after_sync();
          if (leader) MOE_TC_TRACE(5, c);
#pragma unroll
          for (int j = 0; j < kUnit; j++, c++, bpos.next(rb, SB)) {
            const uint32_t bsm =
                tc::smem_u32(bring + bpos.r.s * b_stride) + bpos.j * it.rows8 * 128;
            // chunk j of m-tile m sits at stage column m * 32 * kUnit + j * 32
            const uint32_t acol = tbase + tpos.s * PL::stage_cols + j * 32;
            const bool last_of_run = bpos.j + 1 >= rb || ku + j + 1 >= it.KC;
            if (leader) {
#pragma unroll
              for (int m = 0; m < MT; m++) {
                if (MT == 1 || m < it.nmt) {
#pragma unroll
                  for (int kk = 0; kk < 4; kk++)
                    tc::mma_ts(dcol + m * NMAX, acol + m * 32 * kUnit + kk * 8,
                               tc::sdesc_sw128(bsm + kk * 32), idesc, ku + j + kk > 0);
                }
              }
              if (last_of_run) tc::mma_commit(&bars->b_empty[bpos.r.s]);  // release the stage
            }
          }
          if (leader) {
            MOE_TC_TRACE(3, c - 1);
            tc::mma_commit(&bars->done[tpos.s]);
            MOE_TC_TRACE(6, c - 1);
          }
          __syncwarp();
          issued = true;
        }
        if (!ok) break;
        if (leader) tc::mma_commit(&bars->acc_full[ab]);
        __syncwarp();
      }
      if (!ok && leader) {
        give_up();
        if (issued) {  // all MMAs issued so far complete before TMEM is freed
          tc::mma_commit(&bars->drain[0]);
          wait_nofail(&bars->drain[0], 0, lim);
        }
      }
    }
  } else if (warp >= kDqWarp0) {
    // ------------------------------------------------ dequantisers: one weight row a thread
    // The sets take units of kUnit chunks in turn; a unit's chunks go to one TMEM stage.
    const int q = warp & 3, r = 32 * q + lane, set = (warp - kDqWarp0) >> 2;
    const uint32_t tlane = (uint32_t)(32 * q) << 16;
    int c = 0;     // running chunk index over all items of this CTA (all roles count alike)
    int turn = 0;  // the set that takes the current unit
    Ring tpos;     // TMEM stage of the unit
    RunPos apos;   // code run of chunk c
    RunPos bpos;   // activation-tile run of chunk c
    bool ok = true;
    Item it;
    // sets beyond nsets idle
    for (int item = blockIdx.x; ok && set < nsets && item < item_bound; item += gridDim.x) {
      if (!tc_item<DOWN, MT>(a, item, it)) break;
      for (int ku = 0; ku < it.KC; ku += kUnit, turn = turn + 1 == nsets ? 0 : turn + 1,
               tpos.next(ST)) {
        if (turn != set) {
#pragma unroll
          for (int j = 0; j < kUnit; j++, c++) apos.next(ra, SA), bpos.next(rb, SB);
          continue;
        }
        // the stage's previous unit has been multiplied
        ok = __all_sync(0xffffffffu,
                        tc::mbar_wait_backoff(&bars->done[tpos.s], tpos.ph ^ 1, abort, lim, 32));
        if (!ok) break;
        MOE_TC_TRACE_R(7, c);
        tc::fence_after_sync();
#pragma unroll 1
        for (int j = 0; j < kUnit; j++, c++, apos.next(ra, SA), bpos.next(rb, SB)) {
          ok = __all_sync(0xffffffffu, tc::mbar_wait_backoff(&bars->a_full[apos.r.s], apos.r.ph,
                                                             abort, lim, 32));
          if (!ok) break;
          MOE_TC_TRACE_R(2, c);
#pragma unroll
          for (int m = 0; m < MT; m++) {
            if (MT == 1 || m < it.nmt) {  // row r of m-tile m: [m-tile][ra chunks] in the stage
              uint32_t v[32];
              dequant_row<BITS>(aring + apos.r.s * a_run + (m * ra + apos.j) * AB + r * RB,
                                lane, v);
              tc::tmem_st32(tbase + tlane + tpos.s * PL::stage_cols + m * 32 * kUnit + j * 32,
                            v);
            }
          }
          __syncwarp();  // the warp's shared-memory reads are done: one arrival per warp
          if (lane == 0) tc::mbar_arrive(&bars->a_empty[apos.r.s]);
          if (q == 0) {
            // the chunk's activation tile has landed: the published stage then stands for
            // both MMA operands (the tile's ring stage cannot be reused before this chunk's
            // MMAs: the ring holds at least as many chunks as TMEM has stages)
            ok = __all_sync(0xffffffffu, tc::mbar_wait_backoff(&bars->b_full[bpos.r.s],
                                                               bpos.r.ph, abort, lim, 32));
            if (!ok) break;
          }
        }
        if (!ok) break;
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars->t_full[tpos.s]);
        MOE_TC_TRACE_R(4, c - 1);
        if (lane == 0) MOE_TC_TRACE(12 + q, c - 1);
      }
    }
    if (!ok && lane == 0) give_up();
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------ epilogue: one output row a thread
    const int q = warp & 3, r = 32 * q + lane;
    const uint32_t tlane = (uint32_t)(32 * q) << 16;
    uint32_t d0 = tbase + tlane + PL::acc_col;  // + the item's buffer
    // 16 accumulator columns from c0 of the accumulator at column d (summed over the
    // issuers' copies, NMAX columns apart; one issuer here)
    auto load_sum = [&](uint32_t d, int c0, float (&v)[16]) {
#pragma unroll
      for (int i = 0; i < NI; i++) {
        uint32_t t[16];
        tc::tmem_ld16(d + i * NMAX + c0, t);
        tc::tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 16; jj++) v[jj] = (i ? v[jj] : 0.f) + __uint_as_float(t[jj]);
      }
    };
    int n = 0;
    bool ok = true;
    Item it;
    for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x, n++) {
      if (!tc_item<DOWN, MT>(a, item, it)) break;
      const int ab = n % PL::acc_bufs, au = n / PL::acc_bufs;
      ok = __all_sync(0xffffffffu,
                      tc::mbar_wait_backoff(&bars->acc_full[ab], au & 1, abort, lim, 256));
      d0 = tbase + tlane + PL::acc_col + ab * PL::buf_cols;  // m-tile m at d0 + m * NMAX
      if (!ok) break;
      MOE_TC_TRACE_R(8, n);
      tc::fence_after_sync();
      const ExpertLayout &L = it.sh ? a.LS : a.LR;
      const int gn = it.g.n;
      if (!DOWN) {
        // 1 / the token's activation scale, per B row: loaded once per item into this warp's
        // slice of shared memory (no load waits behind the stores of the loop below)
        float *rsc = bars->escale[q];
        __syncwarp();
        for (int i = lane; i < it.Npad; i += 32)
          rsc[i] = i < it.rowsB ? a.rscale[it.g.xrow0 + i] : 0.f;
        __syncwarp();
        const int j = r >> 1;  // output index within the m-tile (64 outputs)
        const bool odd = r & 1;  // rows 2j (gate) and 2j + 1 (up) sit in adjacent lanes
        bool bad = false;
        const int nmt = MT == 1 ? 1 : it.nmt;
        for (int m = 0; m < nmt; m++) {
          const int mt = it.mt + m;
          const float s = ((const float *)(it.ebase + L.sgu_off))[mt * 128 + r];
          uint8_t *hbase =
              a.hg + (size_t)it.g.hrow0 * a.Imax * 2 + (size_t)mt * round8(gn) * 128;
          // tokens in pairs (i, i + 1): the gate lane computes h for token i, the up lane
          // for token i + 1; one exchange gives each lane the other operand it needs
          auto pair = [&](int i, float w0, float w1) {
            const float other = __shfl_xor_sync(0xffffffffu, odd ? w0 : w1, 1);
            const int tok = odd ? i + 1 : i;
            const float g = odd ? other : w0, u = odd ? w1 : other;
            if (tok < gn) {
              const __half hv = __float2half_rn(silu_fast(g) * u);
              bad |= __hisinf(hv) || __hisnan(hv);
              *(__half *)(hbase + (size_t)tok * 128 + (((j >> 3) ^ (tok & 7)) << 4) +
                          (j & 7) * 2) = hv;
            }
          };
          for (int c0 = 0; c0 < it.Npad; c0 += 16) {
            float acc[16];
            load_sum(d0 + m * NMAX, c0, acc);
            if (a.P == 1) {
#pragma unroll
              for (int jj = 0; jj < 16; jj += 2)
                pair(c0 + jj, acc[jj] * s * rsc[c0 + jj], acc[jj + 1] * s * rsc[c0 + jj + 1]);
            } else {  // columns 2i, 2i + 1: the hi and lo pieces of token i
#pragma unroll
              for (int jj = 0; jj < 16; jj += 4)
                pair((c0 + jj) >> 1, (acc[jj] + acc[jj + 1]) * s * rsc[c0 + jj],
                     (acc[jj + 2] + acc[jj + 3]) * s * rsc[c0 + jj + 2]);
            }
          }
        }
        if (bad) record_status(a.ctrl, MOE_ERR_NUMERIC, where);
      } else {
        const long yrow0 = it.sh ? (long)a.T * a.k + it.g.pos0 : (long)it.g.pos0;
        const int nmt = MT == 1 ? 1 : it.nmt;
        for (int m = 0; m < nmt; m++) {
          const int mt = it.mt + m;
          const float s = ((const float *)(it.ebase + L.sd_off))[mt * 128 + r];
          float *ycol = a.y + yrow0 * a.H + mt * 128 + r;
          for (int c0 = 0; c0 < it.Npad; c0 += 16) {
            float acc[16];
            load_sum(d0 + m * NMAX, c0, acc);
#pragma unroll
            for (int jj = 0; jj < 16; jj++)
              if (c0 + jj < gn) ycol[(size_t)(c0 + jj) * a.H] = acc[jj] * s;
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      MOE_TC_TRACE_R(9, n);
      if (lane == 0) tc::mbar_arrive(&bars->acc_empty[ab]);
    }
    if (!ok && lane == 0) give_up();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc<512>(tbase);
}

// x -> the gate/up B tiles: per group, [k-chunk][rows rounded up to 8][128-byte swizzled
// row] of fp16 x_t * tscale[t], row = token * P + piece (fp32 x is split into fp16 hi + lo
// pieces); the padding rows are zero.  Also rscale[row] = 1 / tscale of the row's token.
// One warp per tile row: it reads the token's x row front to back and, for each k-chunk,
// eight lanes write the chunk's 128-byte line (16 bytes each, at its swizzled slot).  The
// tokens and scales of a warp's rows are looked up together first (a lane per row), so the
// x loads of consecutive rows do not each wait behind two dependent lookups.
// blockIdx.x: group; the warps of blockIdx.y stride over the group's rows.
__global__ void __launch_bounds__(256, 5) gather_x_kernel(TcArgs a, const void *x, int is_bf16,
                                                          const int32_t *perm, const float *tscale) {
  pdl_wait();
  pdl_trigger();
  const int gi = blockIdx.x;
  if (gi >= a.ctrl->n_groups) return;
  const Group g = a.groups[gi];
  const bool sh = g.e == a.E;
  const int rows = a.P * g.n, rows8 = round8(rows), KC = a.H / kKChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *base = const_cast<uint8_t *>(a.xg) + (size_t)g.xrow0 * a.H * 2;
  // W warps per group; when the group has fewer rows than that, wpr warps share a row,
  // each taking every wpr-th group of four k-chunks
  const int W = gridDim.y * 8, wid = blockIdx.y * 8 + warp;
  const int wpr = W > rows8 ? W / rows8 : 1, part = wid % wpr;
  const int r0 = wid / wpr, rstep = W / wpr;
  const int nr = rows8 > r0 ? (rows8 - r0 + rstep - 1) / rstep : 0;  // this warp's rows
  const int c = lane & 7;  // the lane's 16-byte slot of a 128-byte line
  for (int jb = 0; jb < nr; jb += 32) {
    int ltok = 0;
    float lsc = 0.f;
    {
      const int j = jb + lane, row = r0 + j * rstep;
      if (j < nr && row < rows) {
        const int i = row / a.P;
        ltok = sh ? g.pos0 + i : perm[g.pos0 + i] / a.k;
        lsc = tscale[ltok];
        if (part == 0) a.rscale[g.xrow0 + row] = 1.0f / lsc;
      } else if (j < nr && part == 0) {
        a.rscale[g.xrow0 + row] = 0.f;
      }
    }
    const int nj = min(32, nr - jb);
    for (int jj = 0; jj < nj; jj++) {
      const int row = r0 + (jb + jj) * rstep;
      const int tok = __shfl_sync(0xffffffffu, ltok, jj);
      const float sc = __shfl_sync(0xffffffffu, lsc, jj);
      if (row >= rows) {
        for (int kc = 4 * part + (lane >> 3); kc < KC; kc += 4 * wpr)
          *(uint4 *)(base + ((size_t)kc * rows8 + row) * 128 + ((c ^ (row & 7)) << 4)) =
              make_uint4(0, 0, 0, 0);
        continue;
      }
      const int piece = row - (row / a.P) * a.P;
#pragma unroll 8
      for (int kc = 4 * part + (lane >> 3); kc < KC; kc += 4 * wpr) {
        const size_t col = (size_t)kc * kKChunk + c * 8;
        float f[8];
        if (is_bf16) {
          const uint4 u = *(const uint4 *)((const uint16_t *)x + (size_t)tok * a.H + col);
          const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int m = 0; m < 4; m++) {
            f[2 * m] = __uint_as_float(q[m] << 16);
            f[2 * m + 1] = __uint_as_float(q[m] & 0xFFFF0000u);
          }
        } else {
          const float4 *src = (const float4 *)((const float *)x + (size_t)tok * a.H + col);
          const float4 f0 = src[0], f1 = src[1];
          f[0] = f0.x; f[1] = f0.y; f[2] = f0.z; f[3] = f0.w;
          f[4] = f1.x; f[5] = f1.y; f[6] = f1.z; f[7] = f1.w;
        }
        uint32_t o[4];
#pragma unroll
        for (int m = 0; m < 4; m++) {
          const float v0 = f[2 * m] * sc, v1 = f[2 * m + 1] * sc;  // exact: sc is a power of two
          __half2 hv = __floats2half2_rn(v0, v1);
          if (piece) hv = __floats2half2_rn(v0 - __low2float(hv), v1 - __high2float(hv));
          o[m] = *(uint32_t *)&hv;
        }
        *(uint4 *)(base + ((size_t)kc * rows8 + row) * 128 + ((c ^ (row & 7)) << 4)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

// Decode-sized forwards whose router did not write them: the per-token fp16 rows of the
// register-MMA gate/up kernel (every block but the last) and every group row's 1 / scale
// (the last block).
__global__ void __launch_bounds__(256) token_rows_kernel(TcArgs a, const void *x, int is_bf16) {
  pdl_wait();
  pdl_trigger();
  const int nb = gridDim.x - 1;
  if ((int)blockIdx.x < nb) {
    convert_token_rows(x, is_bf16, a.T, a.H, a.P, a.tscale, const_cast<uint8_t *>(a.xt),
                       blockIdx.x * blockDim.x + threadIdx.x, nb * blockDim.x);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ng = a.ctrl->n_groups;
  for (int gi = warp; gi < ng; gi += 8)
    write_group_row_scales(a.groups[gi], a.E, a.k, a.P, a.perm, a.tscale, a.rscale, lane);
}

template <int BITS, bool DOWN, int NMAX, int MT, int ACCB>
static int launch_tc(const TcArgs &a, int bound, int sms, cudaStream_t st) {
  constexpr size_t smem = tc_smem<NMAX, BITS>();
  auto k = tc_expert_kernel<BITS, DOWN, NMAX, MT, ACCB>;
  set_dyn_smem((const void *)k, (int)smem);
  if (launch_pdl(k, dim3(bound < sms ? bound : sms), dim3(kThreads), smem, st, a, bound) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Launches of groups of up to 128 rows: one m-tile per work item, a double-buffered
// accumulator and 4 stages (1 here).  Two m-tiles would leave TMEM room for a single
// accumulator buffer and 2 stages, hence 2 dequantiser sets: slower at DSV3 T = 2048
// (gate/up 1.40 vs 1.26 ms), while at <= 64 rows (T = 20..64) two m-tiles with a double
// buffer take 12-20% less time than one.
constexpr int kMt128 = 1;

// NMAX: the smallest supported width >= the largest B row count of any group in the launch
// (`bound`: an upper bound of the launch's items counted as single m-tiles)
template <int BITS, bool DOWN>
static int launch_tc_n(TcArgs a, int rows_max, int kc_gcd, int bound, int sms, cudaStream_t st) {
  // chunks per copy: code runs of 4 chunks (16 KB at int4) where every K allows it, 2
  // chunks of each of two m-tiles for two-m-tile items; activation tiles in runs too when
  // they are small (decode), else one chunk per copy
  const int ra1 = kc_gcd % 4 == 0 ? 4 : (kc_gcd % 2 == 0 ? 2 : 1);
  const int ra2 = kc_gcd % 2 == 0 ? 2 : 1;
  const bool two = rows_max <= 64 || kMt128 == 2;
  a.ra = two ? ra2 : ra1;
  a.rb = rows_max <= 32 ? a.ra : 1;
  if (rows_max <= 32) return launch_tc<BITS, DOWN, 32, 2, 2>(a, bound, sms, st);
  // 64 rows: one accumulator buffer leaves room for 3 stages, hence 3 sets (6-8% faster at
  // DSV3 T = 48..256 than two buffers with 2 stages and 2 sets)
  if (rows_max <= 64) return launch_tc<BITS, DOWN, 64, 2, 1>(a, bound, sms, st);
  if constexpr (kMt128 == 2) return launch_tc<BITS, DOWN, 128, 2, 1>(a, bound, sms, st);
  else return launch_tc<BITS, DOWN, 128, 1, 2>(a, bound, sms, st);
}

static int gcd_i(int x, int y) { return y ? gcd_i(y, x % y) : x; }

template <int BITS>
static int run_tc(const TcArgs &a, const WsLayout &W, const void *x, int is_bf16,
                  const int32_t *perm, const float *tscale, cudaStream_t st, void *act,
                  void *mid, bool front_rows, float *ysplit) {
  DevInfo d = dev_info();
  if ((long)tc_smem<128, BITS>() > d.smem_optin || (long)tc_smem<32, BITS>() > d.smem_optin ||
      (long)mma_smem_bytes(BITS) > d.smem_optin)
    return MOE_ERR_UNSUPPORTED;
  // 8 warps per CTA, each with about eight 4-line steps of work; no more CTAs per group
  // than it takes to cover the SMs a few times over
  // a group holds at most min(group_n, T) tokens (a token takes an expert at most once)
  const int grows = W.group_n < a.T ? W.group_n : a.T;
  // groups of at most 16 B rows (decode) take the register-MMA kernel, which reads
  // per-token activation rows; larger ones the tensor-memory kernel and per-group tiles
  const int rows_gu = a.P * grows;
  if (rows_gu <= kMmaMaxRows) {
    // about eight chunks of 8 elements per converting thread
    const int nb = std::max(1, std::min(2 * d.sms, (a.T * (a.H / 8) + 2047) / 2048));
    if (!front_rows && launch_pdl(token_rows_kernel, dim3(nb + 1), dim3(256), 0, st, a, x,
                                  is_bf16) != cudaSuccess)
      return MOE_ERR_CUDA;
  } else {
    // enough CTAs per group to cover the SMs about 8 times over, counted on the groups a
    // batch usually has (the shared expert's, one per expert in use) rather than the
    // bound the work list is sized for: most of the grid's rows find no group and exit
    const int rows8_max = round8(a.P * std::min(W.group_n, a.T));
    const int groups_est = std::min(W.max_groups, a.ns + std::min(a.E, a.T * a.k));
    const int gy = std::max(1, std::min((rows8_max * (a.H / kKChunk / 4) + 63) / 64,
                                        (8 * d.sms + groups_est - 1) / groups_est));
    if (launch_pdl(gather_x_kernel, dim3(W.max_groups, gy), dim3(256), 0, st, a, x, is_bf16,
                   perm, tscale) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (act && record_stage_event(act, st) != cudaSuccess) return MOE_ERR_CUDA;
  const int mt_s = a.LS.inter / 64, mt_r = a.LR.inter / 64, mt_d = a.H / 128;
  const int bound_gu = a.ns * mt_s + (W.max_groups - a.ns) * mt_r;
  const int bound_dn = W.max_groups * mt_d;
  int r = rows_gu <= kMmaMaxRows
              ? launch_experts_mma(BITS, false, a, rows_gu, a.H / kKChunk, bound_gu, d.sms, st)
              : launch_tc_n<BITS, false>(a, rows_gu, a.H / kKChunk, bound_gu, d.sms, st);
  if (r) return r;
  if (mid && record_stage_event(mid, st) != cudaSuccess) return MOE_ERR_CUDA;
  TcArgs ad = a;
  ad.trace = nullptr;  // traces (development builds) cover the gate/up kernel
  const int kc_dn = gcd_i(a.LR.inter / kKChunk, a.LS.inter / kKChunk);
  // only the register-MMA down launch splits its contraction (the combine adds W.ks planes)
  if (W.ks > 1 && grows > kMmaMaxRows) return MOE_ERR_UNSUPPORTED;
  return grows <= kMmaMaxRows
             ? launch_experts_mma(BITS, true, ad, grows, kc_dn, bound_dn, d.sms, st, W.ks,
                                  W.ks > 1 ? ysplit : nullptr, (long)W.rows * a.H)
             : launch_tc_n<BITS, true>(ad, grows, kc_dn, bound_dn, d.sms, st);
}

int launch_experts_tc(const moe_layer_config &c, const uint8_t *packed, const void *x,
                      moe_dtype dt, int T, uint8_t *ws, const WsLayout &W, cudaStream_t st,
                      void *act, void *mid, bool front_rows) {
  PackLayout P = pack_layout(c);
  TcArgs a{};
  a.routed = packed + P.experts_off;
  a.routed_stride = P.routed.bytes;
  a.shared = c.n_shared && W.shared ? packed + P.shared_off : nullptr;
  a.LR = P.routed;
  a.LS = P.shared;
  a.H = c.hidden;
  a.E = c.n_experts;
  a.k = c.top_k;
  a.T = T;
  int Is = c.inter_shared ? c.inter_shared : c.inter;
  a.Imax = c.inter > Is ? c.inter : Is;
  a.P = W.pieces;
  a.groups = (const Group *)(ws + W.groups);
  a.ctrl = (Ctrl *)(ws + W.ctrl);
  a.ns = c.n_shared && W.shared ? (T + W.group_n - 1) / W.group_n : 0;
  a.xg = ws + W.xg;
  a.xt = ws + W.xg;  // decode-sized forwards use the region for token rows instead
  a.tscale = (const float *)(ws + W.tscale);
  a.rscale = (float *)(ws + W.rscale);
  const float *tscale = (const float *)(ws + W.tscale);
  a.hg = ws + W.hg;
  a.y = (float *)(ws + W.y);
  a.wait_limit = 2000000000L;  // 2 s: a wait this long means the pipeline is stuck
#ifdef MOE_TRACE
  a.trace = g_trace;
#endif
  const int32_t *perm = (const int32_t *)(ws + W.perm);
  a.perm = perm;
  const int is_bf16 = dt == MOE_DT_BF16;
  float *ysplit = (float *)(ws + W.ysplit);  // y planes 1.. of a split down launch
  switch (c.weight_bits) {
    case 4: return run_tc<4>(a, W, x, is_bf16, perm, tscale, st, act, mid, front_rows, ysplit);
    case 2: return run_tc<2>(a, W, x, is_bf16, perm, tscale, st, act, mid, front_rows, ysplit);
    case 8: return run_tc<8>(a, W, x, is_bf16, perm, tscale, st, act, mid, front_rows, ysplit);
    default: return MOE_ERR_UNSUPPORTED;
  }
}

}  // namespace moe

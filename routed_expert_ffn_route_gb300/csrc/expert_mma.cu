// expert_mma.cu -- the grouped SwiGLU expert GEMMs for small token groups (decode).
//
// Same computation as expert_tc.cu ("企业官网建设流程全解析", §3.1 SwiGLU; "Show HN: 如何在我的
// 低配置电脑上运行 GLM-5.2", 已实现的功能: 量化内核 逐行缩放 使用时反量化; "colibrì 深度拆解",
// §5.1), for launches whose groups hold at most 16 activation rows.  There each weight is
// used by a few tokens only, the layer is bound by streaming the codes from HBM, and the
// work per byte is small: the kernel keeps HBM busy with the fewest hand-offs.
//
//  - One producer warp per CTA streams runs of up to 4 code chunks (16 KB at int4, one
//    bulk copy) into a ring of stages, with the run's activations: for gate/up one bulk
//    copy per group row from the per-token fp16 rows written in front of the launch (rows
//    padded by 16 bytes in the stage against bank conflicts), for down the run's chunks
//    of the group's h tile.  Launched as programmatic dependents, the gate/up kernel
//    prefetches the shared expert's codes into L2 while the router still selects, and the
//    down kernel issues its first code copies before the gate/up grid has finished.
//  - Eight compute warps each own 16 of the item's 128 weight rows for the whole K loop:
//    codes go from shared memory to registers, are dequantised (exact small integers in
//    fp16) straight into the A fragments of mma.sync m16n8k16, the fp16 activations give
//    the B fragments, and the fp32 accumulators stay in registers (two chains per
//    8-token tile, even and odd k-steps, to halve the MMA dependency chain).
//  - A run's chunk count is a template constant, so the chunk loop unrolls and the
//    compiler overlaps one chunk's loads and dequantisation with the previous MMAs.
//  - The epilogue is per warp: per-row scale, SwiGLU across the interleaved gate/up rows
//    (adjacent rows sit 4 lanes apart in the accumulator fragment), and the same outputs
//    as the tensor-memory kernel (fp16 h tiles for the down projection, fp32 y rows).
//  - A down launch with few work items (see down_splits) splits each item's contraction
//    into `ks` contiguous parts: work item i is part i % ks of item i / ks, and part sp
//    writes y plane sp (plane 0 is y, planes 1.. follow at ysplit, yplane floats apart).
//
// K order inside a 64-element chunk.  A dot product does not depend on the order of its
// terms, so the MMA's k slots may take the chunk's elements in any order, as long as A and
// B use the same one.  Element pairs are numbered pi = 0..31 (elements 2pi, 2pi+1); lane
// (g, t) of the fragment layout feeds k-step ks, half h (k slots 2t+8h, 2t+8h+1) with pair
// pi = 8t + 2ks + h.  Then a lane's pairs are one contiguous quarter of each code row (8
// bytes at int4, whole words, no cross-lane shuffles) and two whole 16-byte chunks of each
// activation row (chunks 2t and 2t+1: k-steps 0-1 and 2-3).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dev.cuh"
#include "expert_args.cuh"
#include "moe_internal.cuh"
#include "tc.cuh"

namespace moe {

constexpr int kMmaWarps = 8;  // compute warps, 16 weight rows each
constexpr int kMmaThreads = (kMmaWarps + 1) * 32;
constexpr int kMmaRun = 4;               // chunks per run, where the item's K allows
// activation stage: gate/up holds up to 16 token rows of a run (4 x 128 B, padded by 16 B
// so that the fragment loads of 8 rows hit distinct banks); down holds the run's chunks of
// the group's 128-byte-swizzled h tile (4 x 16 rows x 128 B)
constexpr int kMmaBStage = 16 * (kMmaRun * 128 + 16);
constexpr int kMmaMaxStages = 8;

// ring geometry per code width: about 100 KB of stages, so two CTAs share an SM
template <int BITS>
struct MmaPlan {
  static constexpr int a_stage = kMmaRun * ATile<BITS>::bytes;
  static constexpr int fit = (100 * 1024) / (a_stage + kMmaBStage);
  static constexpr int stages = fit < kMmaMaxStages ? fit : kMmaMaxStages;
  static constexpr size_t smem = 1024 + (size_t)stages * (a_stage + kMmaBStage) + 256;
};

struct MmaBars {
  uint64_t full[kMmaMaxStages], empty[kMmaMaxStages];
  int abort_flag;
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A lane's quarter of one code row (pairs 8t..8t+7 of the chunk; `q` points at it) -> 8
// fp16 pairs, o[l] = pair 8t + l.  The quarter is 8 bytes at int4 (two words of four
// pairs), 4 bytes at int2 (one word of eight pairs), 16 bytes at int8 (four words of two).
template <int BITS>
__device__ __forceinline__ void dequant_quarter(const uint8_t *q, uint32_t (&o)[8]) {
  if (BITS == 4) {
    const uint2 w = *(const uint2 *)q;
    dq_word_i4(w.x, o);
    dq_word_i4(w.y, o + 4);
  } else if (BITS == 2) {
    dq_word_i2(*(const uint32_t *)q, o);
  } else {
    const uint4 u = *(const uint4 *)q;
    dq_word_i8(u.x, o);
    dq_word_i8(u.y, o + 2);
    dq_word_i8(u.z, o + 4);
    dq_word_i8(u.w, o + 6);
  }
}

template <int BITS, bool DOWN, int NT, int RA>
__global__ void __launch_bounds__(kMmaThreads, 2) mma_expert_kernel(TcArgs a, int item_bound,
                                                                     int ks, float *ysplit,
                                                                     long yplane) {
  using PL = MmaPlan<BITS>;
  constexpr int S = PL::stages, AB = ATile<BITS>::bytes, RB = ATile<BITS>::row_bytes;
  constexpr int RS = RA * 128 + 16;  // gate/up: bytes of one activation row in a stage
  extern __shared__ uint8_t smraw[];
  uint8_t *base = tc::align_smem_1024(smraw);
  uint8_t *bring = base;                   // S x kMmaBStage
  uint8_t *aring = base + S * kMmaBStage;  // S x a_stage
  MmaBars *bars = (MmaBars *)(aring + S * PL::a_stage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int where = DOWN ? kKDown : kKGateUp;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], kMmaWarps);
    }
    bars->abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  volatile int *abort = &bars->abort_flag;
  const long lim = a.wait_limit;
  auto give_up = [&]() {
    if (!*abort) { *abort = 1; record_status(a.ctrl, MOE_ERR_TIMEOUT, where); }
  };

  if (warp == kMmaWarps) {
    // ------------------------------------------------ producer warp
    uint32_t armed = 0, last_ph = 0;  // lane 0: stages with copies in flight, their phase
    int run = 0;
    bool ok = true;
    if constexpr (DOWN) {
      // Lane 0 copies each run of codes and the run's h tile.  The first S runs' code
      // copies go out while the gate/up grid may still run; their h tiles (its output)
      // only after pdl_wait.
      bool waited = false;
      const uint8_t *pend_src[S];
      uint32_t pend_bytes[S];
      auto release = [&](int n) {  // wait for the predecessor, then the deferred tiles
        pdl_wait();
        pdl_trigger();
        if (lane == 0)
          for (int q = 0; q < n; q++)
            tc::bulk_g2s(bring + q * kMmaBStage, pend_src[q], pend_bytes[q], &bars->full[q]);
        waited = true;
      };
      Item it;
      for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x) {
        const int base = item / ks, sp = item - base * ks;
        if (!tc_item<DOWN>(a, base, it)) break;
        const int kpart = it.KC / ks;
        for (int kc = sp * kpart; kc < (sp + 1) * kpart; kc += RA, run++) {
          if (!waited && run == S) release(S);
          const int s = run % S;
          const uint32_t ph = (run / S) & 1;
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars->empty[s], ph ^ 1, abort, lim));
          if (!ok) break;
          if (lane == 0) {
            const uint32_t bbytes = (uint32_t)RA * it.rows8 * 128;
            tc::mbar_arrive_expect_tx(&bars->full[s], RA * AB + bbytes);
            tc::bulk_g2s(aring + s * PL::a_stage, a_src<BITS, DOWN>(a, it, kc), RA * AB,
                         &bars->full[s]);
            if (waited) {
              tc::bulk_g2s(bring + s * kMmaBStage, b_src<DOWN>(a, it, kc), bbytes,
                           &bars->full[s]);
            } else {  // run < S: stage s == run
              pend_src[s] = b_src<DOWN>(a, it, kc);
              pend_bytes[s] = bbytes;
            }
            armed |= 1u << s;
            last_ph = (last_ph & ~(1u << s)) | (ph << s);
          }
        }
      }
      if (!waited) release(run < S ? run : S);
    } else {
      // Gate/up: lane 0 copies each run of codes, lane r the run's slice of group row r
      // (its token's fp16 row, or row piece, written in front of this launch).  The shared
      // expert's items do not depend on the routing, so before waiting for the router, lane
      // 0 of a CTA that will take one warms L2 with the item's codes: the router's selection
      // runs in a single CTA and leaves HBM idle meanwhile.
      if (lane == 0 && a.ns) {
        const int mt_s = a.LS.inter / 64, kc = a.H / kKChunk;
        for (int item = blockIdx.x; item < a.ns * mt_s && item < item_bound; item += gridDim.x)
          tc::bulk_prefetch_l2(a.shared + a.LS.gu_off + (size_t)(item % mt_s) * kc * AB,
                               (uint32_t)kc * AB);
      }
      pdl_wait();
      pdl_trigger();
      Item it;
      for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x) {
        if (!tc_item<DOWN>(a, item, it)) break;
        const uint8_t *rsrc = nullptr;  // this lane's row
        if (lane < it.rowsB) {
          const int i = lane / a.P, piece = lane - i * a.P;
          const int tok = it.sh ? it.g.pos0 + i : __ldcg(a.perm + it.g.pos0 + i) / a.k;
          rsrc = a.xt + ((size_t)tok * a.P + piece) * a.H * 2;
        }
        for (int kc = 0; kc < it.KC; kc += RA, run++) {
          const int s = run % S;
          const uint32_t ph = (run / S) & 1;
          ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars->empty[s], ph ^ 1, abort, lim));
          if (!ok) break;
          if (lane == 0) {
            tc::mbar_arrive_expect_tx(&bars->full[s], RA * AB + (uint32_t)it.rowsB * RA * 128);
            tc::bulk_g2s(aring + s * PL::a_stage, a_src<BITS, DOWN>(a, it, kc), RA * AB,
                         &bars->full[s]);
            armed |= 1u << s;
            last_ph = (last_ph & ~(1u << s)) | (ph << s);
          }
          __syncwarp();  // the stage's byte count is set before its row copies start
          if (lane < it.rowsB)
            tc::bulk_g2s(bring + s * kMmaBStage + lane * RS, rsrc + (size_t)kc * 128, RA * 128,
                         &bars->full[s]);
        }
      }
    }
    if (lane == 0) {
      if (!ok) give_up();
      // every copy this warp started lands before the CTA exits (already true when the
      // compute warps consumed them all)
      for (int q = 0; q < S; q++)
        if ((armed >> q) & 1) wait_nofail(&bars->full[q], (last_ph >> q) & 1, lim);
    }
  } else {
    // ------------------------------------------------ compute warp: weight rows 16w..16w+15
    pdl_wait();
    pdl_trigger();
    const int g = lane >> 2, t = lane & 3;
    const int r0 = 16 * warp + g, r1 = r0 + 8;  // the two rows of this lane's A fragments
    const int aoff0 = r0 * RB + (RB / 4) * t, aoff1 = aoff0 + 8 * RB;
    // activation row g of an 8-row tile: its 16-byte chunks 2t (k-steps 0, 1) and 2t+1
    // (k-steps 2, 3); down tiles store chunk c of row r at c ^ (r & 7), gate/up rows are
    // plain and RS bytes apart
    const int boff0 = DOWN ? g * 128 + (((2 * t) ^ g) << 4) : g * RS + 32 * t;
    const int boff1 = DOWN ? g * 128 + (((2 * t + 1) ^ g) << 4) : g * RS + 32 * t + 16;
    constexpr int tile_step = DOWN ? 1024 : 8 * RS;  // bytes between 8-row tiles
    int run = 0;
    bool ok = true;
    Item it;
    for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x) {
      const int base = DOWN ? item / ks : item, sp = DOWN ? item - base * ks : 0;
      if (!tc_item<DOWN>(a, base, it)) break;
      const int kpart = it.KC / (DOWN ? ks : 1);
      const int nt = it.rows8 >> 3;  // 8-row activation tiles of this group (<= NT)
      const int bstride = it.rows8 * 128;
      float acc[NT][2][4];
#pragma unroll
      for (int n = 0; n < NT; n++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[n][0][i] = acc[n][1][i] = 0.f;
      for (int kc0 = sp * kpart; kc0 < (sp + 1) * kpart; kc0 += RA, run++) {
        const int s = run % S;
        const uint32_t ph = (run / S) & 1;
        ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars->full[s], ph, abort, lim));
        if (!ok) break;
        const uint8_t *as = aring + s * PL::a_stage;
        const uint8_t *bs = bring + s * kMmaBStage;
#pragma unroll
        for (int j = 0; j < RA; j++) {
          uint32_t q0[8], q1[8];  // rows r0 and r1: pairs 8t..8t+7
          dequant_quarter<BITS>(as + j * AB + aoff0, q0);
          dequant_quarter<BITS>(as + j * AB + aoff1, q1);
          const uint8_t *bt = bs + (DOWN ? j * bstride : j * 128);
#pragma unroll
          for (int n = 0; n < NT; n++) {
            if (n < nt) {
              const uint4 c0 = *(const uint4 *)(bt + n * tile_step + boff0);
              const uint4 c1 = *(const uint4 *)(bt + n * tile_step + boff1);
              const uint32_t a0[4] = {q0[0], q1[0], q0[1], q1[1]};
              const uint32_t a1[4] = {q0[2], q1[2], q0[3], q1[3]};
              const uint32_t a2[4] = {q0[4], q1[4], q0[5], q1[5]};
              const uint32_t a3[4] = {q0[6], q1[6], q0[7], q1[7]};
              mma_16816(acc[n][0], a0, c0.x, c0.y);
              mma_16816(acc[n][1], a1, c0.z, c0.w);
              mma_16816(acc[n][0], a2, c1.x, c1.y);
              mma_16816(acc[n][1], a3, c1.z, c1.w);
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bars->empty[s]);
      }
      if (!ok) break;
      // ---------------------------------------------- epilogue of this warp's 16 rows
      const ExpertLayout &L = it.sh ? a.LS : a.LR;
      const int gn = it.g.n;
      if (!DOWN) {
        const float *sg = (const float *)(it.ebase + L.sgu_off) + it.mt * 128;
        const float s0 = sg[r0], s1 = sg[r1];
        const float *rsc = a.rscale + it.g.xrow0;  // 1 / the token's activation scale, per B row
        // the down GEMM's B tile of this m-tile: round8(gn) token rows of 64 fp16 values
        uint8_t *hbase = a.hg + (size_t)it.g.hrow0 * a.Imax * 2 + (size_t)it.mt * round8(gn) * 128;
        bool bad = false;
#pragma unroll
        for (int n = 0; n < NT; n++) {
          if (n >= nt) break;
          float c[4];
#pragma unroll
          for (int i = 0; i < 4; i++) c[i] = acc[n][0][i] + acc[n][1][i];
          int tok[2];
          float v[2][2];  // [fragment row r0 / r1][token]
          if (a.P == 2) {  // columns 2t, 2t+1 are the hi and lo pieces of one token
            tok[0] = 4 * n + t;
            tok[1] = 1 << 30;
            const float inv = rsc[2 * tok[0]];
            v[0][0] = (c[0] + c[1]) * s0 * inv;
            v[1][0] = (c[2] + c[3]) * s1 * inv;
            v[0][1] = v[1][1] = 0.f;
          } else {
            tok[0] = 8 * n + 2 * t;
            tok[1] = tok[0] + 1;
            const float i0 = rsc[tok[0]], i1 = rsc[tok[1]];
            v[0][0] = c[0] * s0 * i0;
            v[0][1] = c[1] * s0 * i1;
            v[1][0] = c[2] * s1 * i0;
            v[1][1] = c[3] * s1 * i1;
          }
#pragma unroll
          for (int hh = 0; hh < 2; hh++)
#pragma unroll
            for (int q = 0; q < 2; q++) {
              const float up = __shfl_xor_sync(0xffffffffu, v[hh][q], 4);  // row r + 1: lane + 4
              const int i = tok[q], jo = (hh ? r1 : r0) >> 1;  // token; output within the m-tile
              if ((g & 1) == 0 && i < gn) {
                const __half hv = __float2half_rn(silu_fast(v[hh][q]) * up);
                bad |= __hisinf(hv) || __hisnan(hv);
                *(__half *)(hbase + (size_t)i * 128 + (((jo >> 3) ^ (i & 7)) << 4) + (jo & 7) * 2) =
                    hv;
              }
            }
        }
        if (bad) record_status(a.ctrl, MOE_ERR_NUMERIC, where);
      } else {
        const float *sd = (const float *)(it.ebase + L.sd_off) + it.mt * 128;
        const float s0 = sd[r0], s1 = sd[r1];
        const long yrow0 = it.sh ? (long)a.T * a.k + it.g.pos0 : (long)it.g.pos0;
        float *ybase = (sp ? ysplit + (sp - 1) * yplane : a.y) + yrow0 * a.H + it.mt * 128;
#pragma unroll
        for (int n = 0; n < NT; n++) {
          if (n >= nt) break;
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const int i = 8 * n + 2 * t + (q & 1);
            const float c = acc[n][0][q] + acc[n][1][q];
            if (i < gn) ybase[(size_t)i * a.H + ((q & 2) ? r1 : r0)] = c * ((q & 2) ? s1 : s0);
          }
        }
      }
    }
    if (!ok && lane == 0) give_up();
  }
  __syncthreads();
}

template <int BITS, bool DOWN, int NT, int RA>
static int launch_mma(const TcArgs &a, int bound, int sms, cudaStream_t st, int ks,
                      float *ysplit, long yplane) {
  auto k = mma_expert_kernel<BITS, DOWN, NT, RA>;
  constexpr size_t smem = MmaPlan<BITS>::smem;
  set_dyn_smem((const void *)k, (int)smem);
  const int grid = 2 * sms < bound ? 2 * sms : bound;  // two CTAs per SM
  if (launch_pdl(k, dim3(grid), dim3(kMmaThreads), smem, st, a, bound, ks, ysplit, yplane) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int BITS, bool DOWN, int NT>
static int launch_mma_ra(const TcArgs &a, int kc_gcd, int bound, int sms, cudaStream_t st,
                         int ks, float *ysplit, long yplane) {
  if (kc_gcd % 4 == 0) return launch_mma<BITS, DOWN, NT, 4>(a, bound, sms, st, ks, ysplit, yplane);
  if (kc_gcd % 2 == 0) return launch_mma<BITS, DOWN, NT, 2>(a, bound, sms, st, ks, ysplit, yplane);
  return launch_mma<BITS, DOWN, NT, 1>(a, bound, sms, st, ks, ysplit, yplane);
}

template <int BITS>
static int launch_mma_bits(bool down, const TcArgs &a, bool two, int kc_gcd, int bound, int sms,
                           cudaStream_t st, int ks, float *ysplit, long yplane) {
  if (down)
    return two ? launch_mma_ra<BITS, true, 2>(a, kc_gcd, bound, sms, st, ks, ysplit, yplane)
               : launch_mma_ra<BITS, true, 1>(a, kc_gcd, bound, sms, st, ks, ysplit, yplane);
  return two ? launch_mma_ra<BITS, false, 2>(a, kc_gcd, bound, sms, st, 1, nullptr, 0)
             : launch_mma_ra<BITS, false, 1>(a, kc_gcd, bound, sms, st, 1, nullptr, 0);
}

int launch_experts_mma(int bits, bool down, TcArgs a, int rows_max, int kc_gcd, int bound,
                       int sms, cudaStream_t st, int ks, float *ysplit, long yplane) {
  if (rows_max > kMmaMaxRows) return MOE_ERR_UNSUPPORTED;
  // every item's code runs split evenly: ks divides kc_gcd / (chunks per run)
  const int ra = kc_gcd % 4 == 0 ? 4 : (kc_gcd % 2 == 0 ? 2 : 1);
  if (!down) ks = 1;
  if (ks < 1 || (kc_gcd / ra) % ks || (ks > 1 && !ysplit)) return MOE_ERR_INVALID_ARG;
  const int items = (long)bound * ks > 0x7fffffff ? 0x7fffffff : bound * ks;
  const bool two = rows_max > 8;
  switch (bits) {
    case 4: return launch_mma_bits<4>(down, a, two, kc_gcd, items, sms, st, ks, ysplit, yplane);
    case 2: return launch_mma_bits<2>(down, a, two, kc_gcd, items, sms, st, ks, ysplit, yplane);
    case 8: return launch_mma_bits<8>(down, a, two, kc_gcd, items, sms, st, ks, ysplit, yplane);
    default: return MOE_ERR_UNSUPPORTED;
  }
}

size_t mma_smem_bytes(int bits) {
  return bits == 4 ? MmaPlan<4>::smem : bits == 2 ? MmaPlan<2>::smem : MmaPlan<8>::smem;
}

}  // namespace moe

// expert_mma.cu -- the grouped SwiGLU expert GEMMs for small token groups (decode).
//
// Same computation as expert_tc.cu ("企业官网建设流程全解析", §3.1 SwiGLU; "Show HN: 如何在我的
// 低配置电脑上运行 GLM-5.2", 已实现的功能: 量化内核 逐行缩放 使用时反量化; "colibrì 深度拆解",
// §5.1), for launches whose groups hold at most 16 activation rows.  There each weight is
// used by a few tokens only, the layer is bound by streaming the codes from HBM, and the
// work per byte is small: the kernel keeps HBM busy with the fewest hand-offs.
//
//  - One producer thread per CTA streams runs of up to 4 code chunks (16 KB at int4) and
//    the matching activation-tile chunks, one bulk copy each, into a ring of stages.
//  - Eight compute warps each own 16 of the item's 128 weight rows for the whole K loop:
//    codes go from shared memory to registers, are dequantised (exact small integers in
//    bf16 / fp16) straight into the A fragments of mma.sync m16n8k16, the activation tile
//    gives the B fragments, and the fp32 accumulators stay in registers.
//  - The epilogue is per warp: per-row scale, SwiGLU across the interleaved gate/up rows
//    (adjacent rows sit 4 lanes apart in the accumulator fragment), and the same outputs
//    as the tensor-memory kernel (fp16 h tiles for the down projection, fp32 y rows).
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
constexpr int kMmaBStage = kMmaRun * 16 * 128;  // 4 chunks x 16 activation rows x 128 B
constexpr int kMmaMaxStages = 8;

// ring geometry per code width: about 96 KB of stages, so two CTAs share an SM
template <int BITS>
struct MmaPlan {
  static constexpr int a_stage = kMmaRun * ATile<BITS>::bytes;
  static constexpr int fit = (96 * 1024) / (a_stage + kMmaBStage);
  static constexpr int stages = fit < kMmaMaxStages ? fit : kMmaMaxStages;
  static constexpr size_t smem = 1024 + (size_t)stages * (a_stage + kMmaBStage) + 256;
};

struct MmaBars {
  uint64_t full[kMmaMaxStages], empty[kMmaMaxStages];
  int abort_flag;
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, bool f16) {
  if (f16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t sub16x2(uint32_t v, uint32_t b, bool f16) {
  uint32_t r;
  if (f16) asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(b));
  else asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(b));
  return r;
}

// A lane's quarter of one code row (pairs 8t..8t+7 of the chunk) -> 8 pairs of exact 16-bit
// integers, o[l] = pair 8t + l.  The quarter is 8 bytes at int4 (two words, four pairs each
// at nibbles p and p+4), 4 bytes at int2 (one word, eight pairs at 2-bit fields p and p+8),
// 16 bytes at int8 (four words, two pairs each).  F16: fp16 pairs (down), else bf16.
template <int BITS, bool F16>
__device__ __forceinline__ void dequant_quarter(const uint8_t *row, int t, uint32_t (&o)[8]) {
  const uint32_t magic = F16 ? 0x64006400u : 0x43004300u;  // 1024 (fp16) / 128 (bf16)
  if (BITS == 4) {
    const uint2 w = *(const uint2 *)(row + 8 * t);
    const uint32_t bias = magic + 0x00080008u;  // codes are stored biased by 8
#pragma unroll
    for (int l = 0; l < 8; l++) {
      const uint32_t word = l < 4 ? w.x : w.y;
      o[l] = sub16x2(((word >> (4 * (l & 3))) & 0x000F000Fu) | magic, bias, F16);
    }
  } else if (BITS == 2) {
    const uint32_t word = *(const uint32_t *)(row + 4 * t);
    const uint32_t bias = magic + 0x00020002u;  // codes are stored biased by 2
#pragma unroll
    for (int l = 0; l < 8; l++)
      o[l] = sub16x2(((word >> (2 * l)) & 0x00030003u) | magic, bias, F16);
  } else {
    const uint4 u = *(const uint4 *)(row + 16 * t);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int l = 0; l < 8; l++) {
      const uint32_t word = w[l >> 1];
      const int sh = 16 * (l & 1);
      const float f0 = (float)(int8_t)((word >> sh) & 0xFF);
      const float f1 = (float)(int8_t)((word >> (sh + 8)) & 0xFF);
      if (F16) {
        __half2 h = __floats2half2_rn(f0, f1);
        o[l] = *(uint32_t *)&h;
      } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
        o[l] = *(uint32_t *)&h;
      }
    }
  }
}

template <int BITS, bool DOWN, int NT>
__global__ void __launch_bounds__(kMmaThreads, 2) mma_expert_kernel(TcArgs a, int item_bound) {
  using PL = MmaPlan<BITS>;
  constexpr int S = PL::stages, AB = ATile<BITS>::bytes, RB = ATile<BITS>::row_bytes;
  extern __shared__ uint8_t smraw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  uint8_t *bring = base;                          // S x kMmaBStage
  uint8_t *aring = base + S * kMmaBStage;         // S x a_stage
  MmaBars *bars = (MmaBars *)(aring + S * PL::a_stage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int where = DOWN ? kKDown : kKGateUp;
  const int ra = a.ra;

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
    // ------------------------------------------------ producer: codes + tiles, a copy per run
    if (lane == 0) {
      uint32_t armed = 0, last_ph = 0;
      int run = 0;
      bool ok = true;
      Item it;
      for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x) {
        if (!tc_item<DOWN>(a, item, it)) break;
        for (int kc = 0; kc < it.KC; kc += ra, run++) {
          const int s = run % S;
          const uint32_t ph = (run / S) & 1;
          if (!tc::mbar_wait(&bars->empty[s], ph ^ 1, abort, lim)) { ok = false; break; }
          const uint32_t abytes = (uint32_t)ra * AB, bbytes = (uint32_t)ra * it.rows8 * 128;
          tc::mbar_arrive_expect_tx(&bars->full[s], abytes + bbytes);
          tc::bulk_g2s(aring + s * PL::a_stage, a_src<BITS, DOWN>(a, it, kc), abytes,
                       &bars->full[s]);
          tc::bulk_g2s(bring + s * kMmaBStage, b_src<DOWN>(a, it, kc), bbytes, &bars->full[s]);
          armed |= 1u << s;
          last_ph = (last_ph & ~(1u << s)) | (ph << s);
        }
      }
      if (!ok) give_up();
      // every copy this thread started lands before the CTA exits (already true when the
      // compute warps consumed them all)
      for (int q = 0; q < S; q++)
        if ((armed >> q) & 1) wait_nofail(&bars->full[q], (last_ph >> q) & 1, lim);
    }
  } else {
    // ------------------------------------------------ compute warp: weight rows 16w..16w+15
    const int g = lane >> 2, t = lane & 3;
    const int r0 = 16 * warp + g, r1 = r0 + 8;  // the two rows of this lane's A fragments
    int run = 0;
    bool ok = true;
    Item it;
    for (int item = blockIdx.x; ok && item < item_bound; item += gridDim.x) {
      if (!tc_item<DOWN>(a, item, it)) break;
      const int nt = it.rows8 >> 3;  // 8-row activation tiles of this group (<= NT)
      float acc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; n++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[n][i] = 0.f;
      for (int kc0 = 0; kc0 < it.KC; kc0 += ra, run++) {
        const int s = run % S;
        const uint32_t ph = (run / S) & 1;
        ok = __all_sync(0xffffffffu, tc::mbar_wait(&bars->full[s], ph, abort, lim));
        if (!ok) break;
        const uint8_t *astage = aring + s * PL::a_stage;
        const uint8_t *bstage = bring + s * kMmaBStage;
        for (int j = 0; j < ra; j++) {
          uint32_t q0[8], q1[8];  // rows r0 and r1: pairs 8t..8t+7
          dequant_quarter<BITS, DOWN>(astage + j * AB + r0 * RB, t, q0);
          dequant_quarter<BITS, DOWN>(astage + j * AB + r1 * RB, t, q1);
          const uint8_t *btile = bstage + j * it.rows8 * 128;
#pragma unroll
          for (int n = 0; n < NT; n++) {
            if (n >= nt) break;
            // activation row 8n + g: 16-byte chunks 2t (k-steps 0, 1) and 2t+1 (k-steps 2, 3),
            // stored at chunk ^ (row & 7)
            const uint8_t *brow = btile + (8 * n + g) * 128;
            const uint4 c0 = *(const uint4 *)(brow + (((2 * t) ^ g) << 4));
            const uint4 c1 = *(const uint4 *)(brow + (((2 * t + 1) ^ g) << 4));
            const uint32_t b[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int ks = 0; ks < 4; ks++) {
              const uint32_t af[4] = {q0[2 * ks], q1[2 * ks], q0[2 * ks + 1], q1[2 * ks + 1]};
              mma_16816(acc[n], af, b[2 * ks], b[2 * ks + 1], DOWN);
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
        // the down GEMM's B tile of this m-tile: round8(gn) token rows of 64 fp16 values
        uint8_t *hbase = a.hg + (size_t)it.g.hrow0 * a.Imax * 2 + (size_t)it.mt * round8(gn) * 128;
        bool bad = false;
#pragma unroll
        for (int n = 0; n < NT; n++) {
          if (n >= nt) break;
#pragma unroll
          for (int hh = 0; hh < 2; hh++) {  // fragment row r0 (c0, c1) or r1 (c2, c3)
            const int r = hh ? r1 : r0;
            const float s = hh ? s1 : s0;
            float v[2];
            int tok[2];
            if (a.P == 2) {  // columns 2t, 2t+1 are the hi and lo pieces of one token
              v[0] = (acc[n][2 * hh] + acc[n][2 * hh + 1]) * s;
              v[1] = 0.f;
              tok[0] = 4 * n + t;
              tok[1] = 1 << 30;
            } else {
              v[0] = acc[n][2 * hh] * s;
              v[1] = acc[n][2 * hh + 1] * s;
              tok[0] = 8 * n + 2 * t;
              tok[1] = tok[0] + 1;
            }
#pragma unroll
            for (int q = 0; q < 2; q++) {
              const float up = __shfl_xor_sync(0xffffffffu, v[q], 4);  // row r + 1: lane + 4
              const int i = tok[q], jo = r >> 1;  // token; output index within the m-tile
              if ((g & 1) == 0 && i < gn) {
                const __half hv = __float2half_rn(silu_f(v[q]) * up);
                bad |= __hisinf(hv) || __hisnan(hv);
                *(__half *)(hbase + (size_t)i * 128 + (((jo >> 3) ^ (i & 7)) << 4) + (jo & 7) * 2) =
                    hv;
              }
            }
          }
        }
        if (bad) record_status(a.ctrl, MOE_ERR_NUMERIC, where);
      } else {
        const float *sd = (const float *)(it.ebase + L.sd_off) + it.mt * 128;
        const float s0 = sd[r0], s1 = sd[r1];
        const long yrow0 = it.sh ? (long)a.T * a.k + it.g.pos0 : (long)it.g.pos0;
        float *ybase = a.y + yrow0 * a.H + it.mt * 128;
#pragma unroll
        for (int n = 0; n < NT; n++) {
          if (n >= nt) break;
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const int i = 8 * n + 2 * t + (q & 1);
            if (i < gn) ybase[(size_t)i * a.H + ((q & 2) ? r1 : r0)] = acc[n][q] * ((q & 2) ? s1 : s0);
          }
        }
      }
    }
    if (!ok && lane == 0) give_up();
  }
  __syncthreads();
}

template <int BITS, bool DOWN, int NT>
static int launch_mma_nt(const TcArgs &a, int bound, int sms, cudaStream_t st) {
  auto k = mma_expert_kernel<BITS, DOWN, NT>;
  constexpr size_t smem = MmaPlan<BITS>::smem;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const int grid = 2 * sms < bound ? 2 * sms : bound;  // two CTAs per SM
  k<<<grid, kMmaThreads, smem, st>>>(a, bound);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int BITS>
static int launch_mma_bits(bool down, const TcArgs &a, bool two, int bound, int sms,
                           cudaStream_t st) {
  if (down) return two ? launch_mma_nt<BITS, true, 2>(a, bound, sms, st)
                       : launch_mma_nt<BITS, true, 1>(a, bound, sms, st);
  return two ? launch_mma_nt<BITS, false, 2>(a, bound, sms, st)
             : launch_mma_nt<BITS, false, 1>(a, bound, sms, st);
}

int launch_experts_mma(int bits, bool down, TcArgs a, int rows_max, int kc_gcd, int bound,
                       int sms, cudaStream_t st) {
  if (rows_max > 16) return MOE_ERR_UNSUPPORTED;
  a.ra = kc_gcd % kMmaRun == 0 ? kMmaRun : (kc_gcd % 2 == 0 ? 2 : 1);
  const bool two = rows_max > 8;
  switch (bits) {
    case 4: return launch_mma_bits<4>(down, a, two, bound, sms, st);
    case 2: return launch_mma_bits<2>(down, a, two, bound, sms, st);
    case 8: return launch_mma_bits<8>(down, a, two, bound, sms, st);
    default: return MOE_ERR_UNSUPPORTED;
  }
}

size_t mma_smem_bytes(int bits) {
  return bits == 4 ? MmaPlan<4>::smem : bits == 2 ? MmaPlan<2>::smem : MmaPlan<8>::smem;
}

}  // namespace moe

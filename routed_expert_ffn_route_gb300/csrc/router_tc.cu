// router_tc.cu -- router logits of large bf16 batches on the tensor cores
// (logits[t][e] = sum_h x[t][h] * Wr[e][h]: "Colibri——面向前沿大模型推理的轻量级MoE引擎", §3.2
// Step 1 gate projection; "colibrì 深度拆解", §4.3 router_forward).
//
// The fp32 router matrix is packed as three bf16 pieces (w = hi + mid + lo exactly) and x is
// bf16, so each product of a piece element and an activation is exact in fp32; the tensor
// cores sum the 3 H products of a logit in fp32 (in their own order; the CUDA-core kernels
// use another one, both within fp32 rounding of the exact sum).
//
// A CTA computes 128 experts x 256 tokens over one H slice.  Per 64-element k-chunk the
// three piece tiles (pre-swizzled in the packed blob, one bulk copy each) and the tokens'
// tile (read straight from x by a TMA tensor map with 128-byte swizzle; rows past T read
// as zero) land in a two-stage ring; one thread issues 3 pieces x 4 k-steps of
// tcgen05.mma (M = 128, N = 256, K = 16) into a 256-column fp32 accumulator in tensor
// memory; the four warps then store the slice's partial logits, which the selection adds
// in slice order.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "dev.cuh"
#include "expert_args.cuh"
#include "moe_internal.cuh"
#include "tc.cuh"

namespace moe {

constexpr int kRtN = 256;  // tokens per CTA (MMA N)
constexpr int kRtStageBytes = 3 * kRouterTileBytes + kRtN * 128;  // 3 piece tiles + x tile

struct RtBars {
  uint64_t full[2], empty[2], acc, drain;
  uint32_t tmem;
  int abort_flag;
};

constexpr size_t kRtSmem = 1024 + 2 * (size_t)kRtStageBytes + sizeof(RtBars);

__global__ void __launch_bounds__(128, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap xmap, moe_layer_config c,
                     const uint8_t *packed, const uint8_t *tiles, int T, int KC, int kc_split,
                     float *partials, Ctrl *ctrl, long lim) {
  extern __shared__ uint8_t smraw[];
  uint8_t *base = tc::align_smem_1024(smraw);
  RtBars *bars = (RtBars *)(base + 2 * kRtStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x, nt = blockIdx.y, hs = blockIdx.z, MT = gridDim.x;
  const int kc0 = hs * kc_split;
  const int E = c.n_experts;
  pdl_trigger();  // the selection kernel only prepares until this grid has completed
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
    check_header(packed, c, ctrl);
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; s++) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    tc::mbar_init(&bars->acc, 1);
    tc::mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc<256>(&bars->tmem);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = bars->tmem;
  volatile int *abort = &bars->abort_flag;
  auto give_up = [&]() {
    if (!*abort) { *abort = 1; record_status(ctrl, MOE_ERR_TIMEOUT, kKRouter); }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- producer: a stage per k-chunk
      bool ok = true;
      uint32_t armed = 0, last_ph = 0;
      for (int i = 0; i < kc_split; i++) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!tc::mbar_wait(&bars->empty[s], ph ^ 1, abort, lim)) { ok = false; break; }
        uint8_t *st = base + s * kRtStageBytes;
        const int kc = kc0 + i;
        tc::mbar_arrive_expect_tx(&bars->full[s], kRtStageBytes);
        for (int p = 0; p < 3; p++)
          tc::bulk_g2s(st + p * kRouterTileBytes,
                       tiles + (((long)p * MT + mt) * KC + kc) * kRouterTileBytes,
                       kRouterTileBytes, &bars->full[s]);
        tc::tma_load_2d(st + 3 * kRouterTileBytes, &xmap, kc * 64, nt * kRtN, &bars->full[s]);
        armed |= 1u << s;
        last_ph = (last_ph & ~(1u << s)) | (ph << s);
      }
      if (!ok) {
        give_up();
        for (int q = 0; q < 2; q++)  // every copy started lands before the CTA exits
          if ((armed >> q) & 1) wait_nofail(&bars->full[q], (last_ph >> q) & 1, lim);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (one elected lane)
    const bool leader = tc::elect_one();
    const uint32_t idesc = tc::idesc_f16(1, kRtN);  // bf16 x bf16 -> fp32
    bool ok = true, issued = false;
    for (int i = 0; i < kc_split; i++) {
      const int s = i & 1;
      int got = 1;
      if (leader) got = tc::mbar_wait(&bars->full[s], (i >> 1) & 1, abort, lim);
      ok = __all_sync(0xffffffffu, got);
      if (!ok) break;
      tc::fence_after_sync();
      if (leader) {
        const uint32_t sa = tc::smem_u32(base + s * kRtStageBytes);
        const uint32_t sb = sa + 3 * kRouterTileBytes;
#pragma unroll
        for (int p = 0; p < 3; p++)
#pragma unroll
          for (int kk = 0; kk < 4; kk++)
            tc::mma_ss(tbase, tc::sdesc_sw128(sa + p * kRouterTileBytes + kk * 32),
                       tc::sdesc_sw128(sb + kk * 32), idesc, (i | p | kk) != 0);
        tc::mma_commit(&bars->empty[s]);  // the stage is free once these MMAs are done
      }
      __syncwarp();
      issued = true;
    }
    if (leader) {
      if (ok) {
        tc::mma_commit(&bars->acc);
      } else {
        give_up();
        if (issued) {  // every MMA issued completes before the tensor memory is freed
          tc::mma_commit(&bars->drain);
          wait_nofail(&bars->drain, 0, lim);
        }
      }
    }
  }
  // -------------------------------------------------- epilogue: warp q, experts 32q..32q+31
  {
    const bool ok = __all_sync(0xffffffffu, tc::mbar_wait_backoff(&bars->acc, 0, abort, lim, 256));
    if (ok) {
      tc::fence_after_sync();
      const int e = mt * 128 + 32 * warp + lane;
      const uint32_t taddr = tbase + ((uint32_t)(32 * warp) << 16);
      for (int c0 = 0; c0 < kRtN; c0 += 16) {
        const int t0 = nt * kRtN + c0;
        if (t0 >= T) break;
        uint32_t v[16];
        tc::tmem_ld16(taddr + c0, v);
        tc::tmem_wait_ld();
        if (e < E) {
#pragma unroll
          for (int j = 0; j < 16; j++)
            if (t0 + j < T) partials[((long)hs * T + t0 + j) * E + e] = __uint_as_float(v[j]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc<256>(tbase);
}

bool router_tc_applies(const moe_layer_config &c, moe_dtype dt, int T) {
  return dt == MOE_DT_BF16 && !router_gemv(c, T) && c.n_experts <= 256 && c.hidden % 64 == 0;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to libcuda)
static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

int launch_router_tc(const moe_layer_config &c, const uint8_t *packed, const void *x, int T,
                     float *partials, int hsplits, Ctrl *ctrl, cudaStream_t st) {
  const PackLayout P = pack_layout(c);
  const int KC = c.hidden / 64, MT = router_mtiles(c), NT = (T + kRtN - 1) / kRtN;
  if (KC % hsplits) return MOE_ERR_UNSUPPORTED;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
  if (!enc) return MOE_ERR_CUDA;
  // x as a [T][H] bf16 tensor; a box is 64 elements (128 B, the swizzle span) x 256 rows
  CUtensorMap xmap;
  const cuuint64_t dims[2] = {(cuuint64_t)c.hidden, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)c.hidden * 2};
  const cuuint32_t box[2] = {64, kRtN};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MOE_ERR_CUDA;
  set_dyn_smem((const void *)router_tc_kernel, (int)kRtSmem);
  router_tc_kernel<<<dim3(MT, NT, hsplits), 128, kRtSmem, st>>>(
      xmap, c, packed, packed + P.router_t_off, T, KC, KC / hsplits, partials, ctrl,
      2000000000L);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

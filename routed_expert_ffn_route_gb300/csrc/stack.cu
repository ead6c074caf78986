// stack.cu -- the step between two stacked MoE layers.
//
// A layer's merged output feeds the next layer ("colibrì 深度拆解", §4.3).  The pages leave
// the stacking arithmetic open; the reading used here keeps a residual stream r and
// normalises each layer's input: r <- r + out, x = bf16(r / sqrt(mean(r^2) + eps))
// (unweighted RMSNorm), x being the next layer's bf16 hidden states.
#include <cuda_bf16.h>

#include "dev.cuh"
#include "moe_internal.cuh"

namespace moe {

// One CTA per token, 256 threads, 8 elements a thread per step (H a multiple of 8).
__global__ void __launch_bounds__(256) residual_rmsnorm_kernel(int H, float *r, const float *add,
                                                               const uint16_t *x0, float eps,
                                                               uint16_t *xn) {
  pdl_wait();  // the layer's combine (its predecessor) has written `add`
  pdl_trigger();
  const int t = blockIdx.x;
  float *rt = r + (size_t)t * H;
  const float *at = add ? add + (size_t)t * H : nullptr;
  float ss = 0.f;
  for (int i = 8 * threadIdx.x; i < H; i += 8 * blockDim.x) {
    float4 v0, v1;
    if (x0) {  // the stack's first residual: the bf16 input itself
      const uint4 u = *(const uint4 *)(x0 + (size_t)t * H + i);
      v0 = make_float4(bf16_to_f32(u.x & 0xFFFF), bf16_to_f32(u.x >> 16),
                       bf16_to_f32(u.y & 0xFFFF), bf16_to_f32(u.y >> 16));
      v1 = make_float4(bf16_to_f32(u.z & 0xFFFF), bf16_to_f32(u.z >> 16),
                       bf16_to_f32(u.w & 0xFFFF), bf16_to_f32(u.w >> 16));
      *(float4 *)(rt + i) = v0;
      *(float4 *)(rt + i + 4) = v1;
    } else {
      v0 = *(float4 *)(rt + i);
      v1 = *(float4 *)(rt + i + 4);
    }
    if (at && !x0) {
      const float4 a0 = *(const float4 *)(at + i), a1 = *(const float4 *)(at + i + 4);
      v0.x += a0.x; v0.y += a0.y; v0.z += a0.z; v0.w += a0.w;
      v1.x += a1.x; v1.y += a1.y; v1.z += a1.z; v1.w += a1.w;
      *(float4 *)(rt + i) = v0;
      *(float4 *)(rt + i + 4) = v1;
    }
    ss += v0.x * v0.x + v0.y * v0.y + v0.z * v0.z + v0.w * v0.w + v1.x * v1.x + v1.y * v1.y +
          v1.z * v1.z + v1.w * v1.w;
  }
  __shared__ float part[8];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; w++) tot += part[w];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  for (int i = 8 * threadIdx.x; i < H; i += 8 * blockDim.x) {
    const float4 v0 = *(const float4 *)(rt + i), v1 = *(const float4 *)(rt + i + 4);
    const float f[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t o[4];
#pragma unroll
    for (int m = 0; m < 4; m++) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * m] * inv, f[2 * m + 1] * inv);
      o[m] = *(uint32_t *)&b;
    }
    *(uint4 *)(xn + (size_t)t * H + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace moe

extern "C" int moe_residual_rmsnorm(int T, int H, float *resid, const float *add,
                                    const uint16_t *x0, float eps, uint16_t *x_next,
                                    void *stream) {
  if (T < 0 || H <= 0 || H % 8 || !(eps >= 0.f)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!resid || !x_next || ((uintptr_t)resid % 16) || ((uintptr_t)x_next % 16) ||
      (add && ((uintptr_t)add % 16)) || (x0 && ((uintptr_t)x0 % 16)))
    return MOE_ERR_INVALID_ARG;
  if (moe::launch_pdl(moe::residual_rmsnorm_kernel, dim3(T), dim3(256), 0, (cudaStream_t)stream,
                      H, resid, add, x0, eps, x_next) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// dev.cuh -- small device helpers shared by the kernels of this library.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// silu(z) = z / (1 + exp(-z))
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// silu with the hardware exponential and an approximate divide (relative error near 1e-6),
// for results that are rounded to fp16 (11 significant bits) right after: a large positive
// z gives z, a large negative z gives 0 (-0), a NaN stays NaN.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// Q8_0 encoding of one block of 32 values held one per lane of a full warp
// ("Show HN: 如何在我的低配置电脑上运行 GLM-5.2", 已实现的功能: Q8_0 风格 int8 激活):
// d = amax / 127 (IEEE fp32 division), q = round-half-away-from-zero(v / d) clamped to
// [-127, 127], and d == 0 gives q = 0.  Returns q; d in `d_out` (same on every lane).
__device__ __forceinline__ int q8_encode_lane(float v, float &d_out) {
  float amax = warp_max(fabsf(v));
  float d = __fdiv_rn(amax, 127.0f);
  d_out = d;
  if (d == 0.0f) return 0;
  float r = roundf(__fdiv_rn(v, d));
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return (int)r;
}

// int32 dot product of 32 int8 weights (8 words) with 32 int8 activations (8 words)
__device__ __forceinline__ int dot32_s8(const uint32_t w[8], const int a[8]) {
  int acc = 0;
#pragma unroll
  for (int j = 0; j < 8; j++) acc = __dp4a((int)w[j], a[j], acc);
  return acc;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while its predecessor in the stream is still running:
// pdl_wait() blocks the calling thread until the predecessor grid has completed and its
// memory is visible (a no-op without a programmatic predecessor), and pdl_trigger() lets
// the successor grid start launching once every CTA of this grid has called it or exited.
// Every kernel of the forward calls pdl_trigger() only after its own pdl_wait(), so when
// a kernel starts, everything two launches back has completed; before its own pdl_wait()
// a kernel reads only constant data (weights) or, through L2 (ld.global.cg), data of
// kernels two or more launches back.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Poll *flag until it is >= want, at most `iterations` times (with a short sleep between
// polls).  Returns false when the wait gave up; callers record MOE_ERR_TIMEOUT and return.
__device__ __forceinline__ bool bounded_wait_ge(volatile int *flag, int want, long iterations) {
  for (long i = 0; i < iterations; i++) {
    if (*flag >= want) return true;
    __nanosleep(64);
  }
  return *flag >= want;
}

}  // namespace moe

// rows.cuh -- per-token fp16 activation rows of decode-sized forwards.
//
// When every gate/up group fits the register-MMA kernel (pieces x tokens <= 16 rows), its
// producer copies each group row straight from a per-token row buffer instead of a
// per-group tile: xt[t][piece][H] (fp16, at the start of the workspace's xg region) holds
// x_t * sc_t, sc_t the token's power-of-two scale (max |x_t| * sc_t in [2^14, 2^15)), as one
// piece for bf16 x (exact) or two for fp32 x (hi = fp16(v), lo = fp16(v - hi)).  rscale
// keeps 1 / sc_t for every B row of every group, in the same places as the tile gather
// writes it, so the gate/up epilogue is the same for both sources.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_internal.cuh"

namespace moe {

// The token rows of a batch of T tokens, 8 elements (a chunk) per thread and step: chunk
// c (c = i0, i0 + step, ...) is elements 8c .. 8c+7 of the flattened [T][H] input.  Eight
// chunks are loaded before any is converted, so each thread keeps eight loads in flight.
__device__ __forceinline__ void convert_token_rows(const void *__restrict__ x, int is_bf16, int T,
                                                   int H, int P, const float *tscale,
                                                   uint8_t *__restrict__ xt, int i0, int step) {
  constexpr int U = 8;
  const int per = H / 8, n = T * per;
  for (int c0 = i0; c0 < n; c0 += U * step) {
    float f[U][8];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int c = c0 + u * step;
      if (c >= n) break;
      if (is_bf16) {
        const uint4 q = *(const uint4 *)((const uint16_t *)x + (size_t)c * 8);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int m = 0; m < 4; m++) {
          f[u][2 * m] = __uint_as_float(w[m] << 16);
          f[u][2 * m + 1] = __uint_as_float(w[m] & 0xFFFF0000u);
        }
      } else {
        const float4 *src = (const float4 *)((const float *)x + (size_t)c * 8);
        const float4 f0 = src[0], f1 = src[1];
        f[u][0] = f0.x; f[u][1] = f0.y; f[u][2] = f0.z; f[u][3] = f0.w;
        f[u][4] = f1.x; f[u][5] = f1.y; f[u][6] = f1.z; f[u][7] = f1.w;
      }
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int c = c0 + u * step;
      if (c >= n) break;
      const int t = c / per, i = (c - t * per) * 8;
      const float sc = tscale[t];
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int m = 0; m < 4; m++) {
        const float v0 = f[u][2 * m] * sc, v1 = f[u][2 * m + 1] * sc;  // exact: 2^e scale
        const __half2 h = __floats2half2_rn(v0, v1);
        const __half2 l = __floats2half2_rn(v0 - __low2float(h), v1 - __high2float(h));
        hi[m] = *(const uint32_t *)&h;
        lo[m] = *(const uint32_t *)&l;
      }
      uint8_t *row = xt + ((size_t)t * P * H + i) * 2;
      *(uint4 *)row = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      if (P == 2) *(uint4 *)(row + (size_t)H * 2) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
}

// 1 / sc of every B row of group g (rows padded to a multiple of 8 get 0), by the lanes of
// one warp.
__device__ __forceinline__ void write_group_row_scales(const Group &g, int E, int k, int P,
                                                       const int32_t *perm, const float *tscale,
                                                       float *rscale, int lane) {
  const int rows = P * g.n, rows8 = round8(rows);
  for (int r = lane; r < rows8; r += 32) {
    float v = 0.f;
    if (r < rows) {
      const int i = r / P;
      const int tok = g.e == E ? g.pos0 + i : __ldcg(perm + g.pos0 + i) / k;
      v = 1.0f / __ldcg(tscale + tok);
    }
    rscale[g.xrow0 + r] = v;
  }
}

}  // namespace moe

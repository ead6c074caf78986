// pack.cu -- packing int8 containers into the private GPU layout and back, the Q8_0
// activation encoder, the int8 block-dot debug kernel and the bounded-wait debug kernel.
//
// Packing follows the pages' quantised format: per-row fp32 scales and codes of 4, 8 or
// 2 bits that must round-trip bit for bit to the int8 container ("Show HN: 如何在我的低配置
// 电脑上运行 GLM-5.2", 已实现的功能: 量化内核 ... 打包已验证与 int8 容器逐位一致; "colibrì
// 深度拆解", §5.1 量化).  The in-word order of the codes is this library's own: it is chosen
// so that one shift-and-mask yields two adjacent contraction elements (see moe_internal.cuh).
#include "moe_internal.cuh"
#include <cuda_bf16.h>

#include "dev.cuh"

namespace moe {

template <int BITS>
__device__ __forceinline__ uint32_t pack_word(const int8_t *src /* 64 elements of the chunk */,
                                              int w) {
  uint32_t v = 0;
  if (BITS == 4) {
#pragma unroll
    for (int e = 0; e < 8; e++) {
      int p = (e >> 1), s = e & 1;
      uint32_t b = ((uint32_t)src[8 * w + e] & 0xF) ^ 0x8;
      v |= b << (4 * (p + 4 * s));
    }
  } else if (BITS == 2) {
#pragma unroll
    for (int e = 0; e < 16; e++) {
      int p = (e >> 1), s = e & 1;
      uint32_t b = ((uint32_t)src[16 * w + e] & 0x3) ^ 0x2;
      v |= b << (2 * (p + 8 * s));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; e++) v |= ((uint32_t)(uint8_t)src[4 * w + e]) << (8 * e);
  }
  return v;
}

template <int BITS>
__device__ __forceinline__ void unpack_word(uint32_t v, int8_t *dst /* 64 elements */, int w) {
  if (BITS == 4) {
#pragma unroll
    for (int e = 0; e < 8; e++) {
      int p = (e >> 1), s = e & 1;
      int b = (v >> (4 * (p + 4 * s))) & 0xF;
      dst[8 * w + e] = (int8_t)(b - 8);
    }
  } else if (BITS == 2) {
#pragma unroll
    for (int e = 0; e < 16; e++) {
      int p = (e >> 1), s = e & 1;
      int b = (v >> (2 * (p + 8 * s))) & 0x3;
      dst[16 * w + e] = (int8_t)(b - 2);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; e++) dst[4 * w + e] = (int8_t)((v >> (8 * e)) & 0xFF);
  }
}

// One thread per packed 32-bit word.  section 0 = gate/up (interleaved rows), 1 = down.
template <int BITS, bool UNPACK>
__global__ void pack_kernel(int section, int H, int I, const int8_t *gate, const int8_t *up,
                            const int8_t *down, int8_t *ogate, int8_t *oup, int8_t *odown,
                            uint32_t *words, long n_words) {
  constexpr int WPR = 64 * BITS / 8 / 4;  // words per row chunk
  long wi = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (wi >= n_words) return;
  int w = (int)(wi % WPR);
  long rb = wi / WPR;
  int r = (int)(rb % kTileRows);
  long blk = rb / kTileRows;
  int K = section == 0 ? H : I;
  int kchunks = K / kKChunk;
  int kc = (int)(blk % kchunks);
  int mt = (int)(blk / kchunks);
  long row;
  const int8_t *src;
  int8_t *dst;
  if (section == 0) {
    row = 64L * mt + (r >> 1);
    src = (r & 1) ? up : gate;
    dst = (r & 1) ? oup : ogate;
  } else {
    row = (long)kTileRows * mt + r;
    src = down;
    dst = odown;
  }
  long off = row * K + (long)kc * kKChunk;
  if (!UNPACK) {
    words[wi] = pack_word<BITS>(src + off, w);
  } else if (dst) {
    unpack_word<BITS>(words[wi], dst + off, w);
  }
}

// scales: gate/up interleaved [I/64][128]; down [H]
template <bool UNPACK>
__global__ void scales_kernel(int H, int I, const float *sg, const float *su, const float *sd,
                              float *osg, float *osu, float *osd, float *sgu, float *sdn) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < 2 * I) {
    int mt = i / 128, r = i % 128;
    int row = 64 * mt + (r >> 1);
    if (!UNPACK) {
      sgu[i] = (r & 1) ? su[row] : sg[row];
    } else {
      float *d = (r & 1) ? osu : osg;
      if (d) d[row] = sgu[i];
    }
  }
  if (i < H) {
    if (!UNPACK) sdn[i] = sd[i];
    else if (osd) osd[i] = sdn[i];
  }
}

template <int BITS, bool UNPACK>
static int run_pack(const moe_layer_config &c, const ExpertLayout &L, const int8_t *g,
                    const int8_t *u, const int8_t *d, int8_t *og, int8_t *ou, int8_t *od,
                    uint8_t *base, cudaStream_t st) {
  const int H = c.hidden, I = L.inter;
  constexpr int WPR = 64 * BITS / 8 / 4;
  long n_gu = (long)(I / 64) * (H / 64) * kTileRows * WPR;
  long n_dn = (long)(H / 128) * (I / 64) * kTileRows * WPR;
  const int tb = 256;
  pack_kernel<BITS, UNPACK><<<(unsigned)((n_gu + tb - 1) / tb), tb, 0, st>>>(
      0, H, I, g, u, d, og, ou, od, (uint32_t *)(base + L.gu_off), n_gu);
  pack_kernel<BITS, UNPACK><<<(unsigned)((n_dn + tb - 1) / tb), tb, 0, st>>>(
      1, H, I, g, u, d, og, ou, od, (uint32_t *)(base + L.down_off), n_dn);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_pack_expert(const moe_layer_config &c, const ExpertLayout &L, const int8_t *gate,
                       const int8_t *up, const int8_t *down, const float *sg, const float *su,
                       const float *sd, uint8_t *base, cudaStream_t st) {
  int r;
  switch (c.weight_bits) {
    case 4: r = run_pack<4, false>(c, L, gate, up, down, nullptr, nullptr, nullptr, base, st); break;
    case 8: r = run_pack<8, false>(c, L, gate, up, down, nullptr, nullptr, nullptr, base, st); break;
    case 2: r = run_pack<2, false>(c, L, gate, up, down, nullptr, nullptr, nullptr, base, st); break;
    default: return MOE_ERR_UNSUPPORTED;
  }
  if (r) return r;
  int n = 2 * L.inter > c.hidden ? 2 * L.inter : c.hidden;
  scales_kernel<false><<<(n + 255) / 256, 256, 0, st>>>(
      c.hidden, L.inter, sg, su, sd, nullptr, nullptr, nullptr, (float *)(base + L.sgu_off),
      (float *)(base + L.sd_off));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_unpack_expert(const moe_layer_config &c, const ExpertLayout &L, const uint8_t *base,
                         int8_t *gate, int8_t *up, int8_t *down, float *sg, float *su, float *sd,
                         cudaStream_t st) {
  uint8_t *b = const_cast<uint8_t *>(base);  // read-only in the unpack direction
  int r;
  switch (c.weight_bits) {
    case 4: r = run_pack<4, true>(c, L, nullptr, nullptr, nullptr, gate, up, down, b, st); break;
    case 8: r = run_pack<8, true>(c, L, nullptr, nullptr, nullptr, gate, up, down, b, st); break;
    case 2: r = run_pack<2, true>(c, L, nullptr, nullptr, nullptr, gate, up, down, b, st); break;
    default: return MOE_ERR_UNSUPPORTED;
  }
  if (r) return r;
  int n = 2 * L.inter > c.hidden ? 2 * L.inter : c.hidden;
  scales_kernel<true><<<(n + 255) / 256, 256, 0, st>>>(
      c.hidden, L.inter, nullptr, nullptr, nullptr, sg, su, sd, (float *)(b + L.sgu_off),
      (float *)(b + L.sd_off));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// The router matrix as three bf16 pieces in tensor-core tiles: hi = bf16(w),
// mid = bf16(w - hi), lo = bf16(w - hi - mid); each difference is exact in fp32 and lo
// holds the last 8 of the 24 significant bits, so hi + mid + lo == w exactly.  A thread
// writes one 16-byte chunk (8 elements) of one row of one piece's tile.
__global__ void router_tiles_kernel(int E, int H, int MT, const float *w, uint8_t *tiles) {
  const int KC = H / 64;
  const long n = 3L * MT * KC * 128 * 8;
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int c = (int)(i & 7), r = (int)((i >> 3) & 127);
  long q = i >> 10;
  const int kc = (int)(q % KC);
  q /= KC;
  const int mt = (int)(q % MT), piece = (int)(q / MT);
  const int e = mt * 128 + r;
  uint16_t out[8];
#pragma unroll
  for (int j = 0; j < 8; j++) {
    const float v = e < E ? w[(long)e * H + kc * 64 + c * 8 + j] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    const __nv_bfloat16 pv = piece == 0 ? hi : (piece == 1 ? mid : lo);
    out[j] = *(const uint16_t *)&pv;
  }
  uint8_t *dst = tiles + (((long)piece * MT + mt) * KC + kc) * kRouterTileBytes + r * 128 +
                 ((c ^ (r & 7)) << 4);
  *(uint4 *)dst = *(const uint4 *)out;
}

int launch_router_tiles(const moe_layer_config &c, const float *router_w, uint8_t *tiles,
                        cudaStream_t st) {
  const int MT = router_mtiles(c);
  const long n = 3L * MT * (c.hidden / 64) * 128 * 8;
  router_tiles_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(c.n_experts, c.hidden, MT,
                                                                  router_w, tiles);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

__global__ void header_kernel(PackHeader h, PackHeader *dst) { *dst = h; }

int launch_write_header(const moe_layer_config &c, uint8_t *packed, cudaStream_t st) {
  PackHeader h{};
  h.magic = kMagic;
  h.version = kVersion;
  h.hidden = c.hidden;
  h.inter = c.inter;
  h.inter_shared = c.inter_shared ? c.inter_shared : c.inter;
  h.n_experts = c.n_experts;
  h.n_shared = c.n_shared;
  h.weight_bits = c.weight_bits;
  h.act_q8_0 = c.act_q8_0;
  h.router = c.router;
  h.n_group = c.n_group;
  h.topk_group = c.topk_group;
  header_kernel<<<1, 1, 0, st>>>(h, (PackHeader *)packed);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- Q8_0 encoder
// One warp per block of 32 values: lane i encodes element i.
__global__ void q8_quantize_kernel(const void *x, int is_bf16, long n_blocks, int n, int8_t *q,
                                   float *d) {
  long gw = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= n_blocks) return;
  long idx = gw * 32 + lane;
  float v = is_bf16 ? bf16_to_f32(((const uint16_t *)x)[idx]) : ((const float *)x)[idx];
  float db;
  int qi = q8_encode_lane(v, db);
  q[idx] = (int8_t)qi;
  if (lane == 0) d[gw] = db;
}

int launch_q8_quantize(const void *x, moe_dtype dt, int T, int n, int8_t *q, float *d,
                       cudaStream_t st) {
  long nb = (long)T * n / 32;
  long threads = nb * 32;
  q8_quantize_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(x, dt == MOE_DT_BF16, nb,
                                                                          n, q, d);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- per-row weight quantiser
// "colibrì 深度拆解" §5.1 quantize_row, generalised by its own pattern: s = amax / qmax
// (fp32 IEEE division), q = roundf(w / s) (fp32 IEEE division, half away from zero)
// clamped to [-2^(bits-1), qmax]; amax == 0 gives s = 0 and q = 0; a NaN ratio gives 0.
// One CTA per row.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const void *w, int is_bf16, int cols,
                                                            int bits, int8_t *q, float *scale) {
  const int r = blockIdx.x;
  const size_t base = (size_t)r * cols;
  auto at = [&](int c) {
    return is_bf16 ? bf16_to_f32(((const uint16_t *)w)[base + c]) : ((const float *)w)[base + c];
  };
  float amax = 0.f;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(at(c)));
  __shared__ float part[8];
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i++) amax = fmaxf(amax, part[i]);
  const int qmax = (1 << (bits - 1)) - 1, qmin = -(1 << (bits - 1));
  const float s = __fdiv_rn(amax, (float)qmax);
  if (threadIdx.x == 0) scale[r] = s;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) {
    int v = 0;
    if (s != 0.f) {
      const float ratio = __fdiv_rn(at(c), s);
      if (ratio == ratio) {
        const float rr = roundf(ratio);
        v = rr < (float)qmin ? qmin : (rr > (float)qmax ? qmax : (int)rr);
      }
    }
    q[base + c] = (int8_t)v;
  }
}

int launch_quantize_rows(const void *w, moe_dtype dt, int rows, int cols, int bits, int8_t *q,
                         float *scale, cudaStream_t st) {
  quantize_rows_kernel<<<rows, 256, 0, st>>>(w, dt == MOE_DT_BF16, cols, bits, q, scale);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- int8 block dots (debug)
// dots[r][t][b] for matrix rows rows[r]; same device routine as the Q8_0 expert kernels.
__global__ void block_dots_kernel(const uint8_t *mat, int K, int mat_rows, int which,
                                  const int32_t *rows, int n_rows, const int8_t *qa, int n_tok,
                                  int32_t *dots) {
  int nb = K / 32;
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  long total = (long)n_rows * n_tok * nb;
  if (i >= total) return;
  int b = (int)(i % nb);
  int t = (int)((i / nb) % n_tok);
  int ri = (int)(i / ((long)nb * n_tok));
  int row = rows[ri];
  if (row < 0 || row >= mat_rows) { dots[i] = 0; return; }
  int mt, r;
  if (which == 2) { mt = row / kTileRows; r = row % kTileRows; }
  else { mt = row / 64; r = 2 * (row % 64) + which; }
  int kc = b >> 1, half = b & 1;
  const uint32_t *wp = (const uint32_t *)(mat + (((long)mt * (K / kKChunk) + kc) * kTileRows + r) * 64 +
                                          half * 32);
  const int *ap = (const int *)(qa + (long)t * K + (long)b * 32);
  uint32_t wv[8];
  int av[8];
#pragma unroll
  for (int j = 0; j < 8; j++) { wv[j] = wp[j]; av[j] = ap[j]; }
  dots[i] = dot32_s8(wv, av);
}

int launch_block_dots(const moe_layer_config &c, const uint8_t *mat, int K, int mat_rows,
                      int which, const int32_t *rows, int n_rows, const int8_t *qa, int n_tok,
                      int32_t *dots, cudaStream_t st) {
  long total = (long)n_rows * n_tok * (K / 32);
  block_dots_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(mat, K, mat_rows, which, rows,
                                                                       n_rows, qa, n_tok, dots);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- bounded wait (debug)
__global__ void debug_wait_kernel(Ctrl *ctrl, int iterations) {
  if (threadIdx.x != 0) return;
  // ctrl->pad[0] is a flag nothing ever sets: the wait must give up by itself
  if (!bounded_wait_ge((volatile int *)&ctrl->pad[0], 1, iterations))
    record_status(ctrl, MOE_ERR_TIMEOUT, kKDebugWait);
}

int launch_debug_wait(uint8_t *ws, int iterations, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>((Ctrl *)ws, iterations);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// expert_simt.cu -- grouped SwiGLU expert kernels on the CUDA cores, and the combine.
//
// Expert FFN ("企业官网建设流程全解析", §3.1 激活内存池化: SwiGLU gate_proj output; "Show HN:
// 如何在我的低配置电脑上运行 GLM-5.2", 已实现的功能: routed-expert SwiGLU, 量化内核 int8/int4/int2
// 逐行缩放 使用时反量化, 整数点积内核 Q8_0; "colibrì 深度拆解", §5.1-5.2 per-row scaled int4 and
// the int4 x fp32 matmul):
//   g = s_g * (Q_g x),  u = s_u * (Q_u x),  h = silu(g) * u,  y = s_d * (Q_d h)
// The per-row scale factors out of each dot product, so codes are dequantised to exact
// small floats (or used as int8 in dp4a block dots) and the scale is applied once.
//
// Work items are (group of <= GN rows of one expert) x (m-tile of 128 weight rows), with
// the m-tile fastest so neighbouring CTAs share a group's activations through L2.  A
// persistent grid walks the item list the permute kernel wrote; every weight byte of a
// selected expert is streamed once per group.  Each warp owns 16 rows of the tile; each
// lane owns one half (32 elements) of the row's 64-element chunk: the warp reads 512
// contiguous bytes (int4) per chunk.
//
// Combine ("colibrì 深度拆解", §4.3): out[t] = shared(x_t) + sum_j w[t][j] * y(t, j), summed in
// slot order; one thread per 4 outputs, no atomics, so results are bit-reproducible.  Slots
// without an output row (dropped by top-p, or outside an expert-parallel share) are skipped.
#include "dev.cuh"
#include "moe_internal.cuh"
#include "tc.cuh"

namespace moe {

struct ExpertArgs {
  const uint8_t *routed;   // base of expert 0
  uint64_t routed_stride;  // bytes between experts
  const uint8_t *shared;   // base of the shared expert (or null)
  ExpertLayout LR, LS;
  int H, E, k, T, Imax;
  const void *x;
  int is_bf16;
  const int32_t *perm;
  const Group *groups;
  const Ctrl *ctrl;
  int ns;                  // shared groups (listed first)
  float *h, *y;
  const int8_t *xq;        // Q8_0 codes of x [T][H]
  const float *xd;         // Q8_0 scales of x [T][H/32]
};

__device__ __forceinline__ bool decode_item(const ExpertArgs &a, int item, int mt_s, int mt_r,
                                            Group &g, int &mt, bool &shared) {
  int n_groups = a.ctrl->n_groups;
  int sh_items = a.ns * mt_s;
  int total = sh_items + (n_groups - a.ns) * mt_r;
  if (item >= total) return false;
  int gi;
  if (item < sh_items) { gi = item / mt_s; mt = item % mt_s; shared = true; }
  else { int i2 = item - sh_items; gi = a.ns + i2 / mt_r; mt = i2 % mt_r; shared = false; }
  g = a.groups[gi];
  return true;
}

__device__ __forceinline__ float magic_f(uint32_t v) {  // exact float of a small integer v < 2^16
  return __uint_as_float(0x4B000000u | v) - 8388608.0f;
}

// 32 contraction elements of one row (this lane's half chunk) times GN activation rows.
template <int BITS, int GN>
__device__ __forceinline__ void fma_half_chunk(const uint8_t *wp, const float *xs, int xstride,
                                               int col0, int n, float acc[GN]) {
  if (BITS == 4) {
    uint4 q = __ldg((const uint4 *)wp);
    uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int wl = 0; wl < 4; wl++) {
#pragma unroll
      for (int p = 0; p < 4; p++) {
        uint32_t v = (wd[wl] >> (4 * p)) & 0x000F000Fu;
        float lo = magic_f(v & 0xFFFF) - 8.0f, hi = magic_f(v >> 16) - 8.0f;
        int c = col0 + 8 * wl + 2 * p;
#pragma unroll
        for (int i = 0; i < GN; i++) {
          if (i < n) {
            float2 xv = *(const float2 *)(xs + i * xstride + c);
            acc[i] = fmaf(lo, xv.x, acc[i]);
            acc[i] = fmaf(hi, xv.y, acc[i]);
          }
        }
      }
    }
  } else if (BITS == 2) {
    uint2 q = __ldg((const uint2 *)wp);
    uint32_t wd[2] = {q.x, q.y};
#pragma unroll
    for (int wl = 0; wl < 2; wl++) {
#pragma unroll
      for (int p = 0; p < 8; p++) {
        uint32_t v = (wd[wl] >> (2 * p)) & 0x00030003u;
        float lo = magic_f(v & 0xFFFF) - 2.0f, hi = magic_f(v >> 16) - 2.0f;
        int c = col0 + 16 * wl + 2 * p;
#pragma unroll
        for (int i = 0; i < GN; i++) {
          if (i < n) {
            float2 xv = *(const float2 *)(xs + i * xstride + c);
            acc[i] = fmaf(lo, xv.x, acc[i]);
            acc[i] = fmaf(hi, xv.y, acc[i]);
          }
        }
      }
    }
  } else {
    uint4 q0 = __ldg((const uint4 *)wp), q1 = __ldg((const uint4 *)wp + 1);
    uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int wl = 0; wl < 8; wl++) {
#pragma unroll
      for (int b = 0; b < 4; b++) {
        float qv = (float)(int)(int8_t)(wd[wl] >> (8 * b));
        int c = col0 + 4 * wl + b;
#pragma unroll
        for (int i = 0; i < GN; i++)
          if (i < n) acc[i] = fmaf(qv, xs[i * xstride + c], acc[i]);
      }
    }
  }
}

// Q8_0 half chunk: 32 int8 weights = one Q8_0 block b of the activations
template <int GN>
__device__ __forceinline__ void q8_half_chunk(const uint8_t *wp, const int8_t *xq, const float *xd,
                                              int K, int b, int n, float acc[GN]) {
  uint4 q0 = __ldg((const uint4 *)wp), q1 = __ldg((const uint4 *)wp + 1);
  uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int i = 0; i < GN; i++) {
    if (i < n) {
      const int4 *ap = (const int4 *)(xq + (long)i * K + b * 32);
      int4 a0 = ap[0], a1 = ap[1];
      int av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      int d = dot32_s8(wd, av);
      acc[i] = fmaf(xd[i * (K / 32) + b], (float)d, acc[i]);
    }
  }
}

// ---------------------------------------------------------------- gate/up + SwiGLU
template <int BITS, int GN, bool Q8>
__global__ void __launch_bounds__(256) gate_up_kernel(ExpertArgs a, int item_bound) {
  extern __shared__ __align__(16) uint8_t smraw[];
  const int H = a.H;
  const int mt_s = a.LS.inter / 64, mt_r = a.LR.inter / 64;
  constexpr int CB = 64 * BITS / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp * 16 + (lane >> 1), half = lane & 1;
  float *xs = (float *)smraw;                       // [GN][H] fp32
  int8_t *xqs = (int8_t *)smraw;                    // Q8: [GN][H] int8
  float *xds = (float *)(smraw + (size_t)GN * H);   // Q8: [GN][H/32]
  for (int item = blockIdx.x; item < item_bound; item += gridDim.x) {
    Group g;
    int mt;
    bool sh;
    if (!decode_item(a, item, mt_s, mt_r, g, mt, sh)) break;
    const uint8_t *ebase = sh ? a.shared : a.routed + a.routed_stride * g.e;
    const ExpertLayout &L = sh ? a.LS : a.LR;
    __syncthreads();
    // stage the group's activation rows
    for (int i = 0; i < g.n; i++) {
      int tok = sh ? g.pos0 + i : a.perm[g.pos0 + i] / a.k;
      if (!Q8) {
        for (int cc = threadIdx.x; cc < H; cc += blockDim.x) {
          long src = (long)tok * H + cc;
          xs[i * H + cc] = a.is_bf16 ? bf16_to_f32(((const uint16_t *)a.x)[src])
                                     : ((const float *)a.x)[src];
        }
      } else {
        for (int cc = threadIdx.x * 16; cc < H; cc += blockDim.x * 16)
          *(int4 *)(xqs + i * H + cc) = *(const int4 *)(a.xq + (long)tok * H + cc);
        for (int b = threadIdx.x; b < H / 32; b += blockDim.x)
          xds[i * (H / 32) + b] = a.xd[(long)tok * (H / 32) + b];
      }
    }
    __syncthreads();
    float acc[GN];
#pragma unroll
    for (int i = 0; i < GN; i++) acc[i] = 0.f;
    const int kchunks = H / kKChunk;
    const uint8_t *wrow = ebase + L.gu_off + ((long)mt * kchunks * kTileRows + row) * CB + half * (CB / 2);
#pragma unroll 2
    for (int kc = 0; kc < kchunks; kc++) {
      const uint8_t *wp = wrow + (long)kc * kTileRows * CB;
      if (Q8) q8_half_chunk<GN>(wp, xqs, xds, H, 2 * kc + half, g.n, acc);
      else fma_half_chunk<BITS, GN>(wp, xs, H, kc * kKChunk + half * 32, g.n, acc);
    }
    const float s = ((const float *)(ebase + L.sgu_off))[mt * kTileRows + row];
#pragma unroll
    for (int i = 0; i < GN; i++) {
      float v = acc[i] + __shfl_xor_sync(0xffffffffu, acc[i], 1);
      v *= s;
      float partner = __shfl_xor_sync(0xffffffffu, v, 2);  // the up row of this output
      if (i < g.n && (row & 1) == 0 && half == 0) {
        float hv = silu_f(v) * partner;
        long hrow = sh ? (long)a.T * a.k + g.pos0 + i : (long)g.pos0 + i;
        a.h[hrow * a.Imax + mt * 64 + (row >> 1)] = hv;
      }
    }
  }
}

// ---------------------------------------------------------------- down projection
template <int BITS, int GN, bool Q8>
__global__ void __launch_bounds__(256) down_kernel(ExpertArgs a, int item_bound) {
  extern __shared__ __align__(16) uint8_t smraw[];
  const int H = a.H;
  const int mt_n = H / kTileRows;
  constexpr int CB = 64 * BITS / 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp * 16 + (lane >> 1), half = lane & 1;
  for (int item = blockIdx.x; item < item_bound; item += gridDim.x) {
    Group g;
    int mt;
    bool sh;
    if (!decode_item(a, item, mt_n, mt_n, g, mt, sh)) break;
    const uint8_t *ebase = sh ? a.shared : a.routed + a.routed_stride * g.e;
    const ExpertLayout &L = sh ? a.LS : a.LR;
    const int K = L.inter;
    float *hs = (float *)smraw;                      // [GN][K] fp32
    int8_t *hq = (int8_t *)smraw;                    // Q8: [GN][K] int8
    float *hd = (float *)(smraw + (size_t)GN * K);   // Q8: [GN][K/32]
    __syncthreads();
    for (int i = 0; i < g.n; i++) {
      long hrow = sh ? (long)a.T * a.k + g.pos0 + i : (long)g.pos0 + i;
      const float *src = a.h + hrow * a.Imax;
      if (!Q8) {
        for (int cc = threadIdx.x; cc < K; cc += blockDim.x) hs[i * K + cc] = src[cc];
      } else {
        // Q8_0 re-encoding of h, one warp per block of 32
        for (int b = warp; b < K / 32; b += 8) {
          float dv;
          int q = q8_encode_lane(src[b * 32 + lane], dv);
          hq[i * K + b * 32 + lane] = (int8_t)q;
          if (lane == 0) hd[i * (K / 32) + b] = dv;
        }
      }
    }
    __syncthreads();
    float acc[GN];
#pragma unroll
    for (int i = 0; i < GN; i++) acc[i] = 0.f;
    const int kchunks = K / kKChunk;
    const uint8_t *wrow = ebase + L.down_off + ((long)mt * kchunks * kTileRows + row) * CB + half * (CB / 2);
#pragma unroll 2
    for (int kc = 0; kc < kchunks; kc++) {
      const uint8_t *wp = wrow + (long)kc * kTileRows * CB;
      if (Q8) q8_half_chunk<GN>(wp, hq, hd, K, 2 * kc + half, g.n, acc);
      else fma_half_chunk<BITS, GN>(wp, hs, K, kc * kKChunk + half * 32, g.n, acc);
    }
    const float s = ((const float *)(ebase + L.sd_off))[mt * kTileRows + row];
#pragma unroll
    for (int i = 0; i < GN; i++) {
      float v = acc[i] + __shfl_xor_sync(0xffffffffu, acc[i], 1);
      if (i < g.n && half == 0) {
        long yrow = sh ? (long)a.T * a.k + g.pos0 + i : (long)g.pos0 + i;
        a.y[yrow * H + mt * kTileRows + row] = v * s;
      }
    }
  }
}

// ---------------------------------------------------------------- combine
// pf, pf_bytes (may be null / 0): a region to start loading into L2 (the next stacked layer's
// router weights), 32 KB slices spread over the threads of the first warp of every block;
// issued before the wait, it depends on nothing this launch reads.
__global__ void combine_kernel(int T, int H, int k, int n_shared, const float *w,
                               const int32_t *slot_pos, const float *y, float *out,
                               const uint8_t *pf, uint64_t pf_bytes, int ks,
                               const float *ysplit, long yplane) {
  if (pf && threadIdx.x < 32) {
    constexpr uint64_t kSlice = 32 * 1024;
    for (uint64_t off = ((uint64_t)blockIdx.x * 32 + threadIdx.x) * kSlice; off < pf_bytes;
         off += (uint64_t)gridDim.x * 32 * kSlice) {
      const uint64_t n = pf_bytes - off < kSlice ? pf_bytes - off : kSlice;
      tc::bulk_prefetch_l2(pf + off, (uint32_t)n);
    }
  }
  pdl_wait();
  pdl_trigger();
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  long per_t = H / 4;
  if (i >= (long)T * per_t) return;
  int t = (int)(i / per_t);
  int c4 = (int)(i % per_t);
  // a y row: plane 0, plus planes 1.. in order when the down launch split its contraction
  auto yrow = [&](long r) {
    float4 v = ((const float4 *)(y + r * H))[c4];
    for (int p = 1; p < ks; p++) {
      const float4 u = ((const float4 *)(ysplit + (p - 1) * yplane + r * H))[c4];
      v.x += u.x;
      v.y += u.y;
      v.z += u.z;
      v.w += u.w;
    }
    return v;
  };
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (n_shared) acc = yrow((long)T * k + t);
  for (int j = 0; j < k; j++) {
    const int sp = slot_pos[t * k + j];
    if (sp < 0) continue;  // dropped by top-p, or an expert outside the call's share
    float wj = w[t * k + j];
    float4 v = yrow(sp);
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  ((float4 *)(out + (long)t * H))[c4] = acc;
}

// ---------------------------------------------------------------- launches
static ExpertArgs make_args(const moe_layer_config &c, const uint8_t *packed, const void *x,
                            moe_dtype dt, int T, uint8_t *ws, const WsLayout &W) {
  PackLayout P = pack_layout(c);
  ExpertArgs a{};
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
  a.x = x;
  a.is_bf16 = dt == MOE_DT_BF16;
  a.perm = (const int32_t *)(ws + W.perm);
  a.groups = (const Group *)(ws + W.groups);
  a.ctrl = (const Ctrl *)(ws + W.ctrl);
  a.ns = c.n_shared && W.shared ? (T + W.group_n - 1) / W.group_n : 0;
  a.h = (float *)(ws + W.h);
  a.y = (float *)(ws + W.y);
  a.xq = (const int8_t *)(ws + W.xq);
  a.xd = (const float *)(ws + W.xd);
  return a;
}

template <class K>
static int launch_persistent(K kern, size_t smem, int item_bound, const ExpertArgs &a,
                             cudaStream_t st) {
  if (item_bound <= 0) return MOE_OK;
  DevInfo d = dev_info();
  if ((long)smem > d.smem_optin) return MOE_ERR_UNSUPPORTED;
  set_dyn_smem((const void *)kern, (int)smem);
  int per_sm = cached_blocks_per_sm((const void *)kern, 256, smem);
  if (per_sm < 1) per_sm = 1;
  int grid = d.sms * per_sm;
  if (grid > item_bound) grid = item_bound;
  kern<<<grid, 256, smem, st>>>(a, item_bound);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int BITS, int GN, bool Q8>
static int run_experts(const moe_layer_config &c, const ExpertArgs &a, const WsLayout &W, void *mid,
                       cudaStream_t st) {
  const int mt_s = a.LS.inter / 64, mt_r = a.LR.inter / 64, mt_n = a.H / kTileRows;
  const int max_routed = W.max_groups - a.ns;
  int bound_gu = a.ns * mt_s + max_routed * mt_r;
  int bound_dn = (a.ns + max_routed) * mt_n;
  size_t smem_gu = Q8 ? (size_t)GN * a.H + (size_t)GN * (a.H / 32) * 4 : (size_t)GN * a.H * 4;
  size_t smem_dn = Q8 ? (size_t)GN * a.Imax + (size_t)GN * (a.Imax / 32) * 4
                      : (size_t)GN * a.Imax * 4;
  int r = launch_persistent(gate_up_kernel<BITS, GN, Q8>, smem_gu, bound_gu, a, st);
  if (r) return r;
  if (mid && record_stage_event(mid, st) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_persistent(down_kernel<BITS, GN, Q8>, smem_dn, bound_dn, a, st);
}

template <int BITS, bool Q8>
static int run_gn(const moe_layer_config &c, const ExpertArgs &a, const WsLayout &W, void *mid,
                  cudaStream_t st) {
  switch (W.group_n) {
    case 1: return run_experts<BITS, 1, Q8>(c, a, W, mid, st);
    case 2: return run_experts<BITS, 2, Q8>(c, a, W, mid, st);
    case 4: return run_experts<BITS, 4, Q8>(c, a, W, mid, st);
    default: return run_experts<BITS, 8, Q8>(c, a, W, mid, st);
  }
}

int launch_experts(const moe_layer_config &c, const uint8_t *packed, const void *x,
                   moe_dtype dt, int T, uint8_t *ws, const WsLayout &W, cudaStream_t st,
                   void *act, void *mid, bool front_rows) {
  if (W.tc) return launch_experts_tc(c, packed, x, dt, T, ws, W, st, act, mid, front_rows);
  if (act && record_stage_event(act, st) != cudaSuccess) return MOE_ERR_CUDA;
  ExpertArgs a = make_args(c, packed, x, dt, T, ws, W);
  if (c.act_q8_0) return run_gn<8, true>(c, a, W, mid, st);
  switch (c.weight_bits) {
    case 4: return run_gn<4, false>(c, a, W, mid, st);
    case 2: return run_gn<2, false>(c, a, W, mid, st);
    default: return run_gn<8, false>(c, a, W, mid, st);
  }
}

int launch_quant_x(const moe_layer_config &c, const void *x, moe_dtype dt, int T, uint8_t *ws,
                   const WsLayout &W, cudaStream_t st) {
  return launch_q8_quantize(x, dt, T, c.hidden, (int8_t *)(ws + W.xq), (float *)(ws + W.xd), st);
}

int launch_combine(const moe_layer_config &c, int T, const float *w, float *out, uint8_t *ws,
                   const WsLayout &W, cudaStream_t st, const uint8_t *pf, uint64_t pf_bytes) {
  long n = (long)T * (c.hidden / 4);
  if (launch_pdl(combine_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, T, c.hidden,
                 c.top_k, c.n_shared && W.shared ? 1 : 0, w, (const int32_t *)(ws + W.slot_pos),
                 (const float *)(ws + W.y), out, pf, pf_bytes, W.ks,
                 (const float *)(ws + W.ysplit), (long)W.rows * c.hidden) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// router.cu -- router logits and top-k selection.
//
// Logits: logits[t][e] = sum_h x[t][h] * Wr[e][h] in fp32 ("Colibri——面向前沿大模型推理的轻量级
// MoE引擎", §3.2 Step 1 gate projection; "colibrì 深度拆解", §4.3 router_forward).
//  - T <= 16: a GEMV split over (8 experts) x (H/8 slices) per CTA so that all SMs stream the
//    fp32 router matrix at once; the 8 partial sums are added in a fixed order afterwards.
//  - T > 16: a tiled CUDA-core GEMM (128 x 128 or 64 x 64 tiles, 8 x 8 or 4 x 4 outputs a
//    thread), the H dimension split across CTAs as for the GEMV.
// Selection, one warp per token:
//  - softmax router: softmax with the maximum subtracted, the k largest, renormalised
//    (§3.2 Steps 2-3 of the same page);
//  - sigmoid grouped router ("Show HN: 如何在我的低配置电脑上运行 GLM-5.2", 已实现的功能:
//    DeepSeek-V3 风格 sigmoid 路由器 noaux_tc, routed_scaling_factor): s = sigmoid(logit),
//    c = s + bias; group score = sum of the two largest c of the group; the topk_group best
//    groups are kept; the k largest c of the kept groups are selected; weights are
//    s / sum(selected s) * routed_scaling_factor.
// Ties go to the lower index everywhere; slots are in descending selection score.
// The selection kernel also writes each token's activation scale for the expert GEMMs
// (a power of two taking max |x_t| into [2^14, 2^15), see token_scale).
#include "dev.cuh"
#include "moe_internal.cuh"

namespace moe {

#ifdef MOE_TRACE
extern long long *g_router_trace;
#define MOE_RT_TRACE(i)                                      \
  do {                                                       \
    if (t == 0 && lane == 0 && rtrace) rtrace[i] = clock64(); \
  } while (0)
#else
#define MOE_RT_TRACE(i) \
  do {                  \
  } while (0)
#endif

__device__ __forceinline__ void check_header(const uint8_t *packed, const moe_layer_config &c,
                                             Ctrl *ctrl) {
  const PackHeader *h = (const PackHeader *)packed;
  int Is = c.inter_shared ? c.inter_shared : c.inter;
  if (h->magic != kMagic || h->version != kVersion || h->hidden != c.hidden ||
      h->inter != c.inter || h->inter_shared != Is || h->n_experts != c.n_experts ||
      h->n_shared != c.n_shared || h->weight_bits != c.weight_bits)
    record_status(ctrl, MOE_ERR_PACKED, kKRouter);
}

template <int TM>
__global__ void __launch_bounds__(256) router_gemv_kernel(moe_layer_config c, const uint8_t *packed,
                                                          const float *wr, const void *x,
                                                          int is_bf16, int T, float *partials,
                                                          Ctrl *ctrl, float *xmax) {
  extern __shared__ float xs[];  // [T][HL]
  const int H = c.hidden, E = c.n_experts;
  const int HL = H / kRouterHS;
  const int hs = blockIdx.y;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) check_header(packed, c, ctrl);
  // 8 elements per thread and step (HL is a multiple of 16), unrolled so the loads overlap
#pragma unroll 4
  for (int i = 8 * threadIdx.x; i < T * HL; i += 8 * blockDim.x) {
    const int t = i / HL, cc = i - t * HL;
    const long src = (long)t * H + (long)hs * HL + cc;
    if (is_bf16) {
      const uint4 u = *(const uint4 *)((const uint16_t *)x + src);
      const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int m = 0; m < 4; m++) {
        xs[i + 2 * m] = __uint_as_float(q[m] << 16);
        xs[i + 2 * m + 1] = __uint_as_float(q[m] & 0xFFFF0000u);
      }
    } else {
      const float4 f0 = *(const float4 *)((const float *)x + src);
      const float4 f1 = *(const float4 *)((const float *)x + src + 4);
      *(float4 *)(xs + i) = f0;
      *(float4 *)(xs + i + 4) = f1;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the first expert block also reduces max |x| over its H slice, per token: the
  // selection kernel combines the slices into the token's activation scale
  if (xmax && blockIdx.x == 0)
    for (int t = warp; t < T; t += 8) {
      float m = 0.f;
      for (int i = lane; i < HL; i += 32) m = fmaxf(m, fabsf(xs[t * HL + i]));
      m = warp_max(m);
      if (lane == 0) xmax[hs * T + t] = m;
    }
  const int e = blockIdx.x * 8 + warp;
  const bool live = e < E;  // no early return: the block synchronises below
  const float4 *wrow = (const float4 *)(wr + (long)(live ? e : 0) * H + (long)hs * HL);
  float acc[TM];
#pragma unroll
  for (int t = 0; t < TM; t++) acc[t] = 0.f;
#pragma unroll 8
  for (int q = lane; live && q < HL / 4; q += 32) {  // unrolled: the row's loads in flight
    float4 wv = __ldg(wrow + q);
#pragma unroll
    for (int t = 0; t < TM; t++) {
      if (t < T) {
        float4 xv = *(const float4 *)(xs + t * HL + 4 * q);
        acc[t] = fmaf(wv.x, xv.x, acc[t]);
        acc[t] = fmaf(wv.y, xv.y, acc[t]);
        acc[t] = fmaf(wv.z, xv.z, acc[t]);
        acc[t] = fmaf(wv.w, xv.w, acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TM; t++) {
    if (t < T) {
      float s = warp_sum(acc[t]);
      if (lane == 0 && live) partials[((long)hs * T + t) * E + e] = s;
    }
  }
  // The last of the kRouterHS H-slice blocks of this expert block adds the slices' partial
  // logits in slice order into slice 0, so the selection kernel reads one value per logit.
  __shared__ int last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this block's partials are visible before it is counted
    last = atomicAdd(&ctrl->gemv_done[blockIdx.x], 1) == kRouterHS - 1;
  }
  __syncthreads();
  if (last) {
    __threadfence();
    for (int i = threadIdx.x; i < 8 * T; i += blockDim.x) {
      const int t = i >> 3, ee = blockIdx.x * 8 + (i & 7);
      if (ee >= E) continue;
      float v[kRouterHS];
#pragma unroll
      for (int h = 0; h < kRouterHS; h++) v[h] = __ldcg(partials + ((long)h * T + t) * E + ee);
      float sum = 0.f;
#pragma unroll
      for (int h = 0; h < kRouterHS; h++) sum += v[h];
      partials[(long)t * E + ee] = sum;
    }
  }
}

// Tiled fp32 GEMM over one H slice: partials[hs][t][e] = sum over h in slice hs of
// x[t][h] * Wr[e][h].  A CTA computes BM tokens x BN experts in k-steps of 8; each thread
// a TM x TN block from float4 shared-memory reads (tokens and experts stored k-major in
// shared memory).  The next k-step's tiles are loaded into registers while the current
// one is multiplied, and shared memory is double-buffered, so one barrier per k-step.
template <int BM, int BN, int TM, int TN>
__global__ void __launch_bounds__((BM / TM) * (BN / TN))
    router_gemm_kernel(moe_layer_config c, const uint8_t *packed, const float *wr, const void *x,
                       int is_bf16, int T, int hslice, float *partials, Ctrl *ctrl) {
  constexpr int NT = (BM / TM) * (BN / TN), BK = 8;
  constexpr int LA = BM * BK / NT, LB = BN * BK / NT;  // elements a thread loads per k-step
  static_assert(LA == 2 || LA == 4, "A loads of 2 or 4 elements");
  static_assert(LB == 2 || LB == 4, "B loads of 2 or 4 elements");
  __shared__ __align__(16) float As[2][BK][BM];
  __shared__ __align__(16) float Bs[2][BK][BN];
  const int H = c.hidden, E = c.n_experts;
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
    check_header(packed, c, ctrl);
  const int t0 = blockIdx.y * BM, e0 = blockIdx.x * BN, hs = blockIdx.z;
  const int tid = threadIdx.x;
  // loader mapping: row, first k of the thread's LA (LB) consecutive elements
  const int am = tid / (BK / LA), ak = (tid % (BK / LA)) * LA;
  const int bn = tid / (BK / LB), bk = (tid % (BK / LB)) * LB;
  const int ta = t0 + am, eb = e0 + bn;
  const long xrow = (long)(ta < T ? ta : 0) * H + (long)hs * hslice + ak;
  const long wrow = (long)(eb < E ? eb : 0) * H + (long)hs * hslice + bk;
  float ra[LA], rb[LB];
  auto load = [&](int k0) {
    if (ta < T) {
      if (is_bf16) {
        const uint16_t *p = (const uint16_t *)x + xrow + k0;
        if (LA == 4) {
          const uint2 u = *(const uint2 *)p;
          ra[0] = __uint_as_float(u.x << 16);
          ra[1] = __uint_as_float(u.x & 0xFFFF0000u);
          ra[LA > 2 ? 2 : 0] = __uint_as_float(u.y << 16);
          ra[LA > 2 ? 3 : 1] = __uint_as_float(u.y & 0xFFFF0000u);
        } else {
          const uint32_t u = *(const uint32_t *)p;
          ra[0] = __uint_as_float(u << 16);
          ra[1] = __uint_as_float(u & 0xFFFF0000u);
        }
      } else {
        const float *p = (const float *)x + xrow + k0;
        if (LA == 4) {
          const float4 f = *(const float4 *)p;
          ra[0] = f.x; ra[1] = f.y; ra[LA > 2 ? 2 : 0] = f.z; ra[LA > 2 ? 3 : 1] = f.w;
        } else {
          const float2 f = *(const float2 *)p;
          ra[0] = f.x; ra[1] = f.y;
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < LA; i++) ra[i] = 0.f;
    }
    if (eb < E) {
      const float *p = wr + wrow + k0;
      if (LB == 4) {
        const float4 f = __ldg((const float4 *)p);
        rb[0] = f.x; rb[1] = f.y; rb[LB > 2 ? 2 : 0] = f.z; rb[LB > 2 ? 3 : 1] = f.w;
      } else {
        const float2 f = __ldg((const float2 *)p);
        rb[0] = f.x; rb[1] = f.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < LB; i++) rb[i] = 0.f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int i = 0; i < LA; i++) As[buf][ak + i][am] = ra[i];
#pragma unroll
    for (int i = 0; i < LB; i++) Bs[buf][bk + i][bn] = rb[i];
  };
  const int tx = tid % (BN / TN), ty = tid / (BN / TN);
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; i++)
#pragma unroll
    for (int j = 0; j < TN; j++) acc[i][j] = 0.f;
  const int nks = hslice / BK;
  load(0);
  store(0);
  __syncthreads();
  for (int ks = 0; ks < nks; ks++) {
    const int buf = ks & 1;
    if (ks + 1 < nks) load((ks + 1) * BK);
#pragma unroll
    for (int k = 0; k < BK; k++) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; i += 4) {
        const float4 v = *(const float4 *)&As[buf][k][ty * TM + i];
        a[i] = v.x; a[i + 1] = v.y; a[i + 2] = v.z; a[i + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < TN; j += 4) {
        const float4 v = *(const float4 *)&Bs[buf][k][tx * TN + j];
        b[j] = v.x; b[j + 1] = v.y; b[j + 2] = v.z; b[j + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < TM; i++)
#pragma unroll
        for (int j = 0; j < TN; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (ks + 1 < nks) store(buf ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < TM; i++) {
    const int t = t0 + ty * TM + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < TN; j++) {
      const int e = e0 + tx * TN + j;
      if (e < E) partials[((long)hs * T + t) * E + e] = acc[i][j];
    }
  }
}

struct Cand {
  float s;  // selection score
  int e;    // expert index (large = none)
  float w;  // weight source value
};

__device__ __forceinline__ bool better(const Cand &a, const Cand &b) {
  return a.s > b.s || (a.s == b.s && a.e < b.e);
}

__device__ __forceinline__ Cand warp_best(Cand c) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    Cand d;
    d.s = __shfl_xor_sync(0xffffffffu, c.s, o);
    d.e = __shfl_xor_sync(0xffffffffu, c.e, o);
    d.w = __shfl_xor_sync(0xffffffffu, c.w, o);
    if (better(d, c)) c = d;
  }
  return c;
}

constexpr int kMaxV = 8;  // experts per lane (E <= 256)

// Order-preserving map of a float (not NaN) to an unsigned key: a > b iff key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The warp's best (score, index) pair: the largest score, ties to the lowest index, using
// two hardware warp reductions (index < 65536; lanes without a candidate pass key 0).
__device__ __forceinline__ int warp_argmax(uint32_t key, int idx) {
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
  const uint32_t inv = __reduce_max_sync(0xffffffffu, key == kmax ? 0xFFFFu - (uint32_t)idx : 0u);
  return (int)(0xFFFFu - inv);
}

// 2^e with max_abs * 2^e in [2^14, 2^15): x_t * 2^e converts to fp16 without loss for every
// element that bf16 holds within 2^-24 of the token's largest (fp16 keeps 11 significant
// bits over that range).  A zero or non-finite maximum gets 1.
__device__ __forceinline__ float token_scale(float max_abs) {
  if (!(max_abs > 0.f) || isinf(max_abs)) return 1.f;
  const int e = (int)((__float_as_uint(max_abs) >> 23) & 0xFF);  // biased exponent
  int se = 268 - e;  // biased exponent of 2^(141 - e): max_abs in [2^(e-127), 2^(e-126))
  se = se < 1 ? 1 : (se > 254 ? 254 : se);
  return __uint_as_float((uint32_t)se << 23);
}

__global__ void __launch_bounds__(256) router_topk_kernel(moe_layer_config c, const float *bias,
                                                          const float *partials, int hsplits,
                                                          int T, int32_t *ids, float *w,
                                                          Ctrl *ctrl, const void *x, int is_bf16,
                                                          float *tscale, const float *xmax,
                                                          long long *rtrace) {
  __shared__ float csm[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  MOE_RT_TRACE(0);
  const int E = c.n_experts, k = c.top_k;
  const bool grouped = c.router == MOE_ROUTER_SIGMOID_GROUPED;
  if (tscale && xmax) {  // max |x_t| from the router GEMV's kRouterHS H slices
    float m = lane < kRouterHS ? xmax[lane * T + t] : 0.f;
    m = warp_max(m);
    if (lane == 0) tscale[t] = token_scale(m);
  } else if (tscale) {
    const int H = c.hidden;
    float m = 0.f;
#pragma unroll 8
    for (int i = 8 * lane; i < H; i += 256) {  // unrolled: the row's loads in flight together
      if (is_bf16) {
        const uint4 u = *(const uint4 *)((const uint16_t *)x + (long)t * H + i);
        const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; j++)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(q[j] << 16)),
                             fabsf(__uint_as_float(q[j] & 0xFFFF0000u))));
      } else {
        const float4 *f = (const float4 *)((const float *)x + (long)t * H + i);
        const float4 f0 = f[0], f1 = f[1];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f0.z), fabsf(f0.w))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f1.x), fabsf(f1.y)), fmaxf(fabsf(f1.z), fabsf(f1.w))));
      }
    }
    m = warp_max(m);
    if (lane == 0) tscale[t] = token_scale(m);
  }
  MOE_RT_TRACE(6);
  float sel[kMaxV], wsrc[kMaxV];
  float mx = -INFINITY;
  // the H-split partial logits, all loaded before they are added (in split order)
  float part[kMaxV][kRouterHS], bv[kMaxV];  // ... and the selection biases, loaded with them
#pragma unroll
  for (int v = 0; v < kMaxV; v++) {
    const int e = lane + 32 * v;
    bv[v] = (grouped && e < E) ? bias[e] : 0.f;
#pragma unroll
    for (int hs = 0; hs < kRouterHS; hs++)
      part[v][hs] = (e < E && hs < hsplits) ? partials[((long)hs * T + t) * E + e] : 0.f;
  }
  bool nonfinite = false;
#pragma unroll
  for (int v = 0; v < kMaxV; v++) {
    int e = lane + 32 * v;
    float l = -INFINITY;
    if (e < E) {
      l = 0.f;
#pragma unroll
      for (int hs = 0; hs < kRouterHS; hs++)
        if (hs < hsplits) l += part[v][hs];
      if (!isfinite(l)) {  // keep the selection total and in range; reported below
        nonfinite = true;
        l = -INFINITY;
      }
    }
    sel[v] = l;
    mx = fmaxf(mx, l);
  }
  if (nonfinite) record_status(ctrl, MOE_ERR_NUMERIC, kKTopk);  // after all loads were issued
  MOE_RT_TRACE(1);
  float sum_all = 1.f;
  if (!grouped) {
    mx = warp_max(mx);
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < kMaxV; v++) {
      int e = lane + 32 * v;
      wsrc[v] = e < E ? expf(sel[v] - mx) : 0.f;
      s += wsrc[v];
    }
    sum_all = warp_sum(s);
  } else {
#pragma unroll
    for (int v = 0; v < kMaxV; v++) {
      int e = lane + 32 * v;
      if (e < E) {
        float sg = 1.0f / (1.0f + expf(-sel[v]));
        wsrc[v] = sg;
        sel[v] = sg + bv[v];
        if (isnan(sel[v])) sel[v] = -INFINITY;
        csm[warp][e] = sel[v];
      } else {
        wsrc[v] = 0.f;
      }
    }
  }
  MOE_RT_TRACE(2);
  unsigned allowed_groups = 0xffffffffu;
  int gs = E;
  if (grouped) {
    __syncwarp();
    const int G = c.n_group;
    gs = E / G;
    Cand gc{-INFINITY, 1 << 30, 0.f};
    if (lane < G) {
      float b1 = -INFINITY, b2 = -INFINITY;
      for (int i = 0; i < gs; i++) {
        float v = csm[warp][lane * gs + i];
        if (v > b1) { b2 = b1; b1 = v; }
        else if (v > b2) { b2 = v; }
      }
      gc.s = gs > 1 ? b1 + b2 : b1;
      gc.e = lane;
    }
    allowed_groups = 0;
    uint32_t gkey = lane < G ? order_key(gc.s) : 0u;
    for (int j = 0; j < c.topk_group; j++) {
      const int b = warp_argmax(gkey, lane);
      allowed_groups |= 1u << b;
      if (lane == b) gkey = 0u;
    }
  }
  MOE_RT_TRACE(3);
  // this lane's candidates (bit v: expert lane + 32 v) in the kept groups
  unsigned avail = 0;
#pragma unroll
  for (int v = 0; v < kMaxV; v++) {
    const int e = lane + 32 * v;
    if (e < E && ((allowed_groups >> (e / gs)) & 1)) avail |= 1u << v;
  }
  float my_w = 0.f, wsum = 0.f;
  int my_id = 0;
  uint32_t skey[kMaxV];  // selection keys (0: not a candidate)
#pragma unroll
  for (int v = 0; v < kMaxV; v++) skey[v] = order_key(sel[v]);
  for (int j = 0; j < k; j++) {
    // this lane's best remaining candidate: largest key, then lowest v (= lowest expert)
    uint32_t bk = 0u;
    int bvx = 0;
#pragma unroll
    for (int v = kMaxV - 1; v >= 0; v--)
      if (((avail >> v) & 1) && skey[v] >= bk) { bk = skey[v]; bvx = v; }
    const int e_best = warp_argmax(bk, lane + 32 * bvx);
    const int owner = e_best & 31, vb = e_best >> 5;
    float wsel = 0.f;
#pragma unroll
    for (int v = 0; v < kMaxV; v++)
      if (v == vb) wsel = wsrc[v];
    const float wb = __shfl_sync(0xffffffffu, wsel, owner);
    if (lane == owner) avail &= ~(1u << vb);
    wsum += wb;
    if (lane == j) { my_id = e_best; my_w = wb; }
  }
  MOE_RT_TRACE(4);
  if (lane < k) {
    float v;
    if (c.norm_topk) v = my_w / wsum;
    else v = grouped ? my_w : my_w / sum_all;
    ids[(long)t * k + lane] = my_id;
    w[(long)t * k + lane] = v * c.routed_scaling_factor;
  }
  MOE_RT_TRACE(5);
}

int launch_router(const moe_layer_config &c, const uint8_t *packed, const void *x, moe_dtype dt,
                  int T, int32_t *ids, float *w, uint8_t *ws, const WsLayout &W,
                  cudaStream_t st) {
  const PackLayout P = pack_layout(c);
  const float *wr = (const float *)(packed + P.router_w_off);
  float *partials = (float *)(ws + W.partials);
  Ctrl *ctrl = (Ctrl *)(ws + W.ctrl);
  int is_bf16 = dt == MOE_DT_BF16;
  int hsplits;
  // per-slice max |x| of the GEMV path (after the partial logits in the same region)
  float *xmax = W.tc ? partials + (size_t)kRouterHS * T * c.n_experts : nullptr;
  const bool gemv = T <= 16 && (size_t)T * (c.hidden / kRouterHS) * 4 <= 96 * 1024;
  if (gemv) {
    hsplits = 1;  // the GEMV adds its H slices into slice 0 itself
    dim3 grid((c.n_experts + 7) / 8, kRouterHS);
    size_t smem = (size_t)T * (c.hidden / kRouterHS) * 4;
    // the dynamic x slice plus the block's static flag may pass the 48 KB default
    auto launch = [&](auto k) {
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      k<<<grid, 256, smem, st>>>(c, packed, wr, x, is_bf16, T, partials, ctrl, xmax);
    };
    if (T <= 1) launch(router_gemv_kernel<1>);
    else if (T <= 2) launch(router_gemv_kernel<2>);
    else if (T <= 4) launch(router_gemv_kernel<4>);
    else if (T <= 8) launch(router_gemv_kernel<8>);
    else launch(router_gemv_kernel<16>);
  } else {
    // 128 x 128 tiles for large T, 64 x 64 below; H split (partial sums added in order by
    // the selection kernel) until the grid covers the SMs twice
    const bool big = T >= 256;
    const int BM = big ? 128 : 64, BN = big ? 128 : 64;
    const int tiles = ((T + BM - 1) / BM) * ((c.n_experts + BN - 1) / BN);
    const int sms = dev_info().sms;
    hsplits = 1;
    while (hsplits < kRouterHS && tiles * hsplits < 2 * sms) hsplits *= 2;
    const int hslice = c.hidden / hsplits;  // a multiple of 16: hidden % 128 == 0
    dim3 grid((c.n_experts + BN - 1) / BN, (T + BM - 1) / BM, hsplits);
    if (big)
      router_gemm_kernel<128, 128, 8, 8><<<grid, 256, 0, st>>>(c, packed, wr, x, is_bf16, T, hslice,
                                                               partials, ctrl);
    else
      router_gemm_kernel<64, 64, 4, 4><<<grid, 256, 0, st>>>(c, packed, wr, x, is_bf16, T, hslice,
                                                             partials, ctrl);
  }
  const float *bias = (const float *)(packed + P.router_b_off);
  float *tscale = W.tc ? (float *)(ws + W.tscale) : nullptr;
  router_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(c, bias, partials, hsplits, T, ids, w, ctrl, x,
                                                  is_bf16, tscale, gemv ? xmax : nullptr,
#ifdef MOE_TRACE
                                                  g_router_trace
#else
                                                  nullptr
#endif
  );
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

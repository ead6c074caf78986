// router.cu -- router logits and top-k selection.
//
// Logits: logits[t][e] = sum_h x[t][h] * Wr[e][h] in fp32 ("Colibri——面向前沿大模型推理的轻量级
// MoE引擎", §3.2 Step 1 gate projection; "colibrì 深度拆解", §4.3 router_forward).
//  - T <= 16: a GEMV split over (16 experts) x (H/8 slices) per CTA so that all SMs stream the
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
#include <cuda_fp16.h>

#include "dev.cuh"
#include "moe_internal.cuh"
#include "rows.cuh"

namespace moe {

#ifdef MOE_TRACE
extern long long *g_router_trace;
#define MOE_RT_TRACE(i)                                                     \
  do {                                                                      \
    if ((t == 0 || t == T - 1) && lane == 0 && rtrace)                      \
      rtrace[(t == 0 ? 0 : 16) + (i)] = clock64();                          \
  } while (0)
// fused front: the global timer (ns) at its phases, slots 8.. of the same row
#define MOE_FRONT_TRACE(i)                                                     \
  do {                                                                         \
    if (f.trace && threadIdx.x == 0) {                                         \
      unsigned long long ns_;                                                  \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns_));                  \
      f.trace[i] = (long long)ns_;                                             \
    }                                                                          \
  } while (0)
#else
#define MOE_RT_TRACE(i) \
  do {                  \
  } while (0)
#define MOE_FRONT_TRACE(i) \
  do {                     \
  } while (0)
#endif


// Router GEMV CTAs: a warp per expert row slice; the fused front's tail selects a token
// per warp, so 16 warps take a batch of up to 16 tokens in one round.
constexpr int kGemvWarps = 16, kGemvThreads = 32 * kGemvWarps;

// What the fused decode front writes besides the logits: the selection (ids, w, tscale),
// the permutation (offsets, perm, slot_pos, groups) and the token rows (xt, rscale).
struct FrontArgs {
  const float *bias;
  int32_t *ids;
  float *w;
  float *tscale;
  int32_t *offsets, *perm, *slot_pos;
  Group *groups;
  uint8_t *xt;
  float *rscale;
  int P, GN;
  int e0, e1, shared;  // the call's share: routed experts [e0, e1), the shared expert
  long long *trace;  // development builds: phase times of the fused front
};

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
  pdl_trigger();  // the selection kernel only prepares until this grid has completed
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

constexpr int kMaxV = 8;  // experts per lane (E <= 256)

// Order-preserving map of a float (not NaN) to an unsigned key: a > b iff key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The float whose order_key is `k`.
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The warp's best (key, index) pair: the largest key, ties to the lowest index, by a
// butterfly of shuffles (every lane ends with the result; lanes without a candidate pass
// key 0).  Shuffles rather than warp-reduction instructions: with a warp per token, many
// selections run side by side on one SM, and shuffles sustain the higher rate there.
__device__ __forceinline__ int warp_argmax(uint32_t key, int idx) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint32_t k2 = __shfl_xor_sync(0xffffffffu, key, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (k2 > key || (k2 == key && i2 < idx)) {
      key = k2;
      idx = i2;
    }
  }
  return idx;
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

// Selection for token t by one full warp; csm: 256 floats of this warp's shared memory.
// Partial logits and the per-slice max |x| are read through L2 (they may come from other
// CTAs of the same grid in the fused decode front); every load is issued before any of
// them is used.  sids / stscale (may be null): copies of the token's expert ids and
// activation scale in the caller's shared memory.
__device__ __forceinline__ void topk_token(const moe_layer_config &c, const float *bias,
                                           const float *partials, int hsplits, int T, int t,
                                           int32_t *ids, float *w, Ctrl *ctrl, const void *x,
                                           int is_bf16, float *tscale, const float *xmax,
                                           long long *rtrace, float *csm, int *sids,
                                           float *stscale) {
  const int lane = threadIdx.x & 31;
  MOE_RT_TRACE(0);
  const int E = c.n_experts, k = c.top_k;
  const bool grouped = c.router == MOE_ROUTER_SIGMOID_GROUPED;
  // the slice maxima of |x_t|, the H-split partial logits and the selection biases
  const float xm = (tscale && xmax && lane < kRouterHS) ? __ldcg(xmax + lane * T + t) : 0.f;
  float part[kMaxV][kRouterHS], bv[kMaxV];
#pragma unroll
  for (int v = 0; v < kMaxV; v++) {
    const int e = lane + 32 * v;
    bv[v] = (grouped && e < E) ? bias[e] : 0.f;
#pragma unroll
    for (int hs = 0; hs < kRouterHS; hs++)
      part[v][hs] = (e < E && hs < hsplits) ? __ldcg(partials + ((long)hs * T + t) * E + e) : 0.f;
  }
  if (tscale) {
    float m = 0.f;
    if (xmax) {
      m = warp_max(xm);
    } else {
      const int H = c.hidden;
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
    }
    const float ts = token_scale(m);
    if (lane == 0) {
      tscale[t] = ts;
      if (stscale) stscale[t] = ts;
    }
  }
  MOE_RT_TRACE(6);
  float sel[kMaxV], wsrc[kMaxV];
  float mx = -INFINITY;
  bool nonfinite = false;
#pragma unroll
  for (int v = 0; v < kMaxV; v++) {
    int e = lane + 32 * v;
    float l = -INFINITY;
    if (e < E) {
      l = 0.f;
#pragma unroll
      for (int hs = 0; hs < kRouterHS; hs++)
        if (hs < hsplits) l += part[v][hs];  // in slice order
      if (!isfinite(l)) {  // keep the selection total and in range; reported below
        nonfinite = true;
        l = -INFINITY;
      }
    }
    sel[v] = l;
    mx = fmaxf(mx, l);
  }
  if (nonfinite) record_status(ctrl, MOE_ERR_NUMERIC, kKTopk);
  MOE_RT_TRACE(1);
  float sum_all = 1.f;
  const bool g32 = grouped && E == 32 * c.n_group;  // groups of 32: group v = the v-th value
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
        csm[e] = sel[v];
      } else {
        wsrc[v] = 0.f;
      }
    }
  }
  MOE_RT_TRACE(2);
  unsigned allowed_groups = 0xffffffffu;
  if (grouped) {
    __syncwarp();
    const int G = c.n_group, gs = E / G;
    float gsc = -INFINITY;  // lane g < G: group g's score (the sum of its two best)
    if (g32 && G <= 8) {
      // four lanes per group: lane 4g + q takes the top two of scores 8q..8q+7 of group g,
      // then two shuffle rounds merge the four pairs (b1 >= b2)
      const int g = lane >> 2, q = lane & 3;
      float b1 = -INFINITY, b2 = -INFINITY;
      if (g < G) {
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const float v = csm[g * 32 + q * 8 + i];
          if (v > b1) { b2 = b1; b1 = v; }
          else if (v > b2) { b2 = v; }
        }
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        const float c1 = __shfl_xor_sync(0xffffffffu, b1, o);
        const float c2 = __shfl_xor_sync(0xffffffffu, b2, o);
        const float n2 = fmaxf(fminf(b1, c1), b1 >= c1 ? b2 : c2);
        b1 = fmaxf(b1, c1);
        b2 = n2;
      }
      const float s = b1 + b2;  // the same two values as a serial scan finds
      gsc = __shfl_sync(0xffffffffu, s, 4 * (lane & 7));  // lane g < G: group g
    } else if (lane < G) {
      float b1 = -INFINITY, b2 = -INFINITY;
      for (int i = 0; i < gs; i++) {
        float v = csm[lane * gs + i];
        if (v > b1) { b2 = b1; b1 = v; }
        else if (v > b2) { b2 = v; }
      }
      gsc = gs > 1 ? b1 + b2 : b1;
    }
    // keep the topk_group groups of best rank: higher score first, ties to the lower index
    const uint32_t gkey = lane < G ? order_key(gsc) : 0u;
    int rank = 0;
    for (int q = 0; q < G; q++) {
      const uint32_t kq = __shfl_sync(0xffffffffu, gkey, q);
      rank += (kq > gkey) || (kq == gkey && q < lane);
    }
    allowed_groups = __ballot_sync(0xffffffffu, lane < G && rank < c.topk_group);
  }
  MOE_RT_TRACE(3);
  // this lane's candidates (expert lane + 32 v in a kept group), sorted best first: key
  // descending, ties to the lower v (= lower expert); key 0 marks no candidate
  uint32_t ck[kMaxV];
  int cv[kMaxV];
  float cw[kMaxV];
#pragma unroll
  for (int v = 0; v < kMaxV; v++) {
    const int e = lane + 32 * v;
    const int grp = grouped ? (E == 32 * c.n_group ? v : e / (E / c.n_group)) : 0;
    const bool cand = e < E && ((allowed_groups >> grp) & 1);
    ck[v] = cand ? order_key(sel[v]) : 0u;
    cv[v] = v;
    cw[v] = wsrc[v];
  }
  {
    // a 19-comparator sorting network for 8 entries
    constexpr int net[19][2] = {{0, 2}, {1, 3}, {4, 6}, {5, 7}, {0, 4}, {1, 5}, {2, 6},
                                {3, 7}, {0, 1}, {2, 3}, {4, 5}, {6, 7}, {2, 4}, {3, 5},
                                {1, 4}, {3, 6}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
    for (int q = 0; q < 19; q++) {
      const int i = net[q][0], j = net[q][1];
      const bool sw = ck[j] > ck[i] || (ck[j] == ck[i] && cv[j] < cv[i]);
      const uint32_t tk = ck[i];
      const int tv = cv[i];
      const float tw = cw[i];
      ck[i] = sw ? ck[j] : ck[i];
      cv[i] = sw ? cv[j] : cv[i];
      cw[i] = sw ? cw[j] : cw[i];
      ck[j] = sw ? tk : ck[j];
      cv[j] = sw ? tv : cv[j];
      cw[j] = sw ? tw : cw[j];
    }
  }
  float my_w = 0.f, wsum = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; j++) {
    // the warp's best head: largest key, then lowest expert; its lane drops it
    const int e_best = warp_argmax(ck[0], lane + 32 * cv[0]);
    const int owner = e_best & 31;
    const float wb = __shfl_sync(0xffffffffu, cw[0], owner);
    const bool pop = lane == owner;  // branch-free: every lane selects
#pragma unroll
    for (int q = 0; q < kMaxV - 1; q++) {
      ck[q] = pop ? ck[q + 1] : ck[q];
      cv[q] = pop ? cv[q + 1] : cv[q];
      cw[q] = pop ? cw[q + 1] : cw[q];
    }
    ck[kMaxV - 1] = pop ? 0u : ck[kMaxV - 1];
    wsum += wb;
    if (lane == j) { my_id = e_best; my_w = wb; }
  }
  MOE_RT_TRACE(4);
  // adaptive expert top-p (opt-in): slot j stays while the share of slots 0..j-1 in the
  // selection's weight sources is below p (slot 0 always); the kept weights are then
  // normalised over the kept slots
  bool keep = lane < k;
  if (c.expert_top_p > 0.f && c.expert_top_p < 1.f) {
    const float share = lane < k ? my_w / wsum : 0.f;
    float incl = share;  // inclusive scan of the shares over the slot lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    float before = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) before = 0.f;
    keep = lane < k && (lane == 0 || before < c.expert_top_p);
    wsum = warp_sum(keep ? my_w : 0.f);
  }
  if (lane < k) {
    float v;
    if (c.norm_topk) v = my_w / wsum;
    else v = grouped ? my_w : my_w / sum_all;
    ids[(long)t * k + lane] = keep ? my_id : -1;
    w[(long)t * k + lane] = keep ? v * c.routed_scaling_factor : 0.f;
    if (sids) sids[t * k + lane] = keep ? my_id : -1;
  }
  MOE_RT_TRACE(5);
}

__global__ void __launch_bounds__(256) router_topk_kernel(moe_layer_config c, const float *bias,
                                                          const float *partials, int hsplits,
                                                          int T, int32_t *ids, float *w,
                                                          Ctrl *ctrl, const void *x, int is_bf16,
                                                          float *tscale, const float *xmax,
                                                          long long *rtrace) {
  __shared__ float csm[8][256];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  topk_token(c, bias, partials, hsplits, T, t, ids, w, ctrl, x, is_bf16, tscale, xmax, rtrace,
             csm[warp], nullptr, nullptr);
}

// ---------------------------------------------------------------- fused decode front
// For decode-sized batches the router GEMV's last CTA also does what the selection, permute
// and token-row kernels do, so the expert GEMMs follow a single launch.

// Shared memory of the fused front's last CTA.
struct FrontSmem {
  float csm[kGemvWarps][256];  // per warp: selection scores (groups not of 32)
  uint32_t emask[256];         // per expert: bit t = token t chose it
  int ids[256];                // slot -> expert
  int offs[257];               // per expert: first position
  int xrow0[256];              // per expert: first B row of its group
  int wsum[kGemvWarps], wused[kGemvWarps];
  float tscale[16];
};

// Selection (a warp per token), then by the whole CTA: the permutation (the same offsets,
// perm, slot_pos and groups as permute_kernel; every expert's count is at most T <= GN,
// so each expert in use has one group) and every group row's 1 / scale.  Runs after every
// partial logit, token row and token scale of the batch has been written.
__device__ void front_tail(const moe_layer_config &c, const FrontArgs &f, const float *partials,
                           int T, Ctrl *ctrl, const void *x, int is_bf16, const float *xmax,
                           FrontSmem &sm) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = c.n_experts, k = c.top_k, n = T * k, P = f.P, GN = f.GN;
  MOE_FRONT_TRACE(9);
  for (int t = warp; t < T; t += kGemvWarps)
    topk_token(c, f.bias, partials, kRouterHS, T, t, f.ids, f.w, ctrl, x, is_bf16, nullptr,
               nullptr, f.trace, sm.csm[warp], sm.ids, nullptr);
  for (int e = tid; e < E; e += blockDim.x) sm.emask[e] = 0u;
  if (tid < T) sm.tscale[tid] = __ldcg(f.tscale + tid);  // written by the GEMV CTAs
  __syncthreads();
  MOE_FRONT_TRACE(10);
  if (tid < n && sm.ids[tid] >= 0) atomicOr(&sm.emask[sm.ids[tid]], 1u << (tid / k));
  __syncthreads();
  // exclusive scans over the experts (thread e): slot offsets and group numbers
  const uint32_t m = tid < E ? sm.emask[tid] : 0u;
  const int cnt = __popc(m);
  const bool mine = tid >= f.e0 && tid < f.e1;  // the expert is in the call's share
  int inc = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  const unsigned used = __ballot_sync(0xffffffffu, cnt > 0 && mine);
  if (lane == 31) sm.wsum[warp] = inc;
  if (lane == 0) sm.wused[warp] = __popc(used);
  __syncthreads();
  int base = 0, gbase = 0, gtotal = 0, total = 0;
  for (int q = 0; q < kGemvWarps; q++) {
    if (q < warp) {
      base += sm.wsum[q];
      gbase += sm.wused[q];
    }
    gtotal += sm.wused[q];
    total += sm.wsum[q];
  }
  const int ns = c.n_shared && f.shared ? (T + GN - 1) / GN : 0;
  const int rbase = c.n_shared ? T : 0;  // routed rows follow the shared expert's T rows
  const int ng = ns + gtotal;
  if (tid < E) {
    const int off = base + inc - cnt;
    sm.offs[tid] = off;
    f.offsets[tid] = off;
    const int g0 = ns + gbase + __popc(used & ((1u << lane) - 1u));
    sm.xrow0[tid] = P * (rbase + off) + 7 * g0;
    if (cnt && mine)
      f.groups[g0] = Group{tid, off, cnt, P * (rbase + off) + 7 * g0, rbase + off + 7 * g0,
                           0, 0, 0};
  }
  if (tid == 0) {
    f.offsets[E] = total;  // slots kept (all T k unless top-p dropped some)
    ctrl->n_groups = ng;
  }
  for (int i = total + tid; i < n; i += blockDim.x) f.perm[i] = -1;
  for (int i = tid; i < ns; i += blockDim.x)
    f.groups[i] = Group{E, i * GN, min(GN, T - i * GN), P * i * GN + 7 * i, i * GN + 7 * i,
                        0, 0, 0};
  __syncthreads();
  // stable scatter: slot (t, j) goes after the earlier tokens of its expert; its B rows'
  // 1 / scale go to the rows of its group
  if (tid < n && sm.ids[tid] < 0) f.slot_pos[tid] = -1;  // dropped by top-p
  if (tid < n && sm.ids[tid] >= 0) {
    const int e = sm.ids[tid], t = tid / k;
    const int r = __popc(sm.emask[e] & ((1u << t) - 1u)), pos = sm.offs[e] + r;
    f.perm[pos] = tid;
    // a slot of an expert outside the call's share has no group and no output row
    const bool mine_e = e >= f.e0 && e < f.e1;
    f.slot_pos[tid] = mine_e ? pos : -1;
    const float inv = 1.0f / sm.tscale[t];
    if (mine_e)
      for (int p = 0; p < P; p++) f.rscale[sm.xrow0[e] + P * r + p] = inv;
  }
  // the shared expert's rows: token t is row t of group t / GN
  for (int i = tid; i < (ns ? T : 0); i += blockDim.x) {
    const int g = i / GN, r = i - g * GN;
    const float inv = 1.0f / sm.tscale[i];
    for (int p = 0; p < P; p++) f.rscale[P * g * GN + 7 * g + P * r + p] = inv;
  }
  MOE_FRONT_TRACE(11);
  MOE_FRONT_TRACE(12);
}

template <int TM>
__global__ void __launch_bounds__(kGemvThreads) router_gemv_kernel(moe_layer_config c, const uint8_t *packed,
                                                          const float *wr, const void *x,
                                                          int is_bf16, int T, float *partials,
                                                          Ctrl *ctrl, float *xmax, int fused,
                                                          FrontArgs f) {
  extern __shared__ float xs[];  // [T][HL]
  const int H = c.hidden, E = c.n_experts;
  const int HL = H / kRouterHS;
  const int hs = blockIdx.y;
  pdl_trigger();  // the next launch only prepares until this grid has completed
  if (blockIdx.x == 0 && blockIdx.y == 0) MOE_FRONT_TRACE(8);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) check_header(packed, c, ctrl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kGemvWarps + warp;
  const bool live = e < E;  // no early return: the block synchronises below
  const float4 *wrow = (const float4 *)(wr + (long)(live ? e : 0) * H + (long)hs * HL);
  // the first kPre float4 of this lane's share of the row slice are loaded before the
  // activations, so that the two memory round trips overlap
  constexpr int kPre = 6;
  float4 wpre[kPre];
#pragma unroll
  for (int j = 0; j < kPre; j++) {
    const int q = lane + 32 * j;
    wpre[j] = (live && q < HL / 4) ? __ldg(wrow + q) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // fused front: this CTA converts slice hs of the rows of tokens blockIdx.x,
  // blockIdx.x + gridDim.x, ..., each with its scale from max |x_t| over the whole row;
  // the first token's row is read together with the slice
  auto row_absmax = [&](int t) {
    float m = 0.f;
#pragma unroll 2
    for (int i = 8 * threadIdx.x; i < H; i += 8 * blockDim.x) {
      if (is_bf16) {
        const uint4 u = *(const uint4 *)((const uint16_t *)x + (long)t * H + i);
        const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; j++)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(q[j] << 16)),
                             fabsf(__uint_as_float(q[j] & 0xFFFF0000u))));
      } else {
        const float4 *p = (const float4 *)((const float *)x + (long)t * H + i);
        const float4 f0 = p[0], f1 = p[1];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f0.z), fabsf(f0.w))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(f1.x), fabsf(f1.y)), fmaxf(fabsf(f1.z), fabsf(f1.w))));
      }
    }
    return m;
  };
  const float first_max = (fused && (int)blockIdx.x < T) ? row_absmax(blockIdx.x) : 0.f;
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
  if (fused) {
    __shared__ float red[kGemvWarps];
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      float m = warp_max(t == (int)blockIdx.x ? first_max : row_absmax(t));
      if (lane == 0) red[warp] = m;
      __syncthreads();
      m = red[0];
      for (int q = 1; q < kGemvWarps; q++) m = fmaxf(m, red[q]);
      __syncthreads();  // red is reused by the next token
      const float sc = token_scale(m);
      if (hs == 0 && threadIdx.x == 0) f.tscale[t] = sc;
      for (int i = 8 * threadIdx.x; i < HL; i += 8 * blockDim.x) {
        const float4 f0 = *(const float4 *)(xs + t * HL + i);
        const float4 f1 = *(const float4 *)(xs + t * HL + i + 4);
        const float e[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const float v0 = e[2 * j] * sc, v1 = e[2 * j + 1] * sc;  // exact: 2^e scale
          const __half2 h = __floats2half2_rn(v0, v1);
          const __half2 l = __floats2half2_rn(v0 - __low2float(h), v1 - __high2float(h));
          hi[j] = *(const uint32_t *)&h;
          lo[j] = *(const uint32_t *)&l;
        }
        uint8_t *row = f.xt + ((size_t)t * f.P * H + (size_t)hs * HL + i) * 2;
        *(uint4 *)row = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (f.P == 2) *(uint4 *)(row + (size_t)H * 2) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
  }
  // the first expert block also reduces max |x| over its H slice, per token: the
  // selection kernel combines the slices into the token's activation scale
  if (xmax && !fused && blockIdx.x == 0)
    for (int t = warp; t < T; t += kGemvWarps) {
      float m = 0.f;
      for (int i = lane; i < HL; i += 32) m = fmaxf(m, fabsf(xs[t * HL + i]));
      m = warp_max(m);
      if (lane == 0) xmax[hs * T + t] = m;
    }
  float acc[TM];
#pragma unroll
  for (int t = 0; t < TM; t++) acc[t] = 0.f;
  auto dot = [&](const float4 &wv, int q) {
#pragma unroll
    for (int t = 0; t < TM; t++) {
      if (t < T) {
        const float4 xv = *(const float4 *)(xs + t * HL + 4 * q);
        acc[t] = fmaf(wv.x, xv.x, acc[t]);
        acc[t] = fmaf(wv.y, xv.y, acc[t]);
        acc[t] = fmaf(wv.z, xv.z, acc[t]);
        acc[t] = fmaf(wv.w, xv.w, acc[t]);
      }
    }
  };
#pragma unroll
  for (int j = 0; j < kPre; j++) {
    const int q = lane + 32 * j;
    if (live && q < HL / 4) dot(wpre[j], q);
  }
#pragma unroll 8
  for (int q = lane + 32 * kPre; live && q < HL / 4; q += 32) dot(__ldg(wrow + q), q);
  // the slice's partial logits; the selection adds the kRouterHS slices in slice order
#pragma unroll
  for (int t = 0; t < TM; t++) {
    if (t < T) {
      float s = warp_sum(acc[t]);
      if (lane == 0 && live) partials[((long)hs * T + t) * E + e] = s;
    }
  }
#ifdef MOE_TRACE
  if (f.trace && threadIdx.x == 0) {  // the latest end of a block's dot products
    unsigned long long ns_;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(ns_));
    atomicMax((unsigned long long *)&f.trace[13], ns_);
  }
#endif
  if (!fused) return;
  // The last CTA to finish runs the rest of the decode front.
  __shared__ int tail;
  __threadfence();  // this thread's partials are visible before the CTA is counted
  __syncthreads();
  if (threadIdx.x == 0)
    tail = atomicAdd(&ctrl->front_done, 1) == (int)(gridDim.x * gridDim.y) - 1;
  __syncthreads();
  if (!tail) return;
  __threadfence();
  __shared__ FrontSmem sm;
  front_tail(c, f, partials, T, ctrl, x, is_bf16, xmax, sm);
}

int launch_router(const moe_layer_config &c, const uint8_t *packed, const void *x, moe_dtype dt,
                  int T, int32_t *ids, float *w, uint8_t *ws, const WsLayout &W,
                  cudaStream_t st, bool fused) {
  const PackLayout P = pack_layout(c);
  const float *wr = (const float *)(packed + P.router_w_off);
  const float *bias = (const float *)(packed + P.router_b_off);
  float *partials = (float *)(ws + W.partials);
  Ctrl *ctrl = (Ctrl *)(ws + W.ctrl);
  float *tscale = W.tc ? (float *)(ws + W.tscale) : nullptr;
  int is_bf16 = dt == MOE_DT_BF16;
  int hsplits;
  // per-slice max |x| of the GEMV path (after the partial logits in the same region)
  float *xmax = W.tc ? partials + (size_t)kRouterHS * T * c.n_experts : nullptr;
  const bool gemv = router_gemv(c, T);
  if (fused && !(gemv && W.tc)) return MOE_ERR_UNSUPPORTED;
  if (gemv) {
    hsplits = kRouterHS;  // the selection adds the GEMV's H slices
    dim3 grid((c.n_experts + kGemvWarps - 1) / kGemvWarps, kRouterHS);
    size_t smem = (size_t)T * (c.hidden / kRouterHS) * 4;
    FrontArgs f{};
    if (fused) {
      f.bias = bias;
      f.ids = ids;
      f.w = w;
      f.tscale = tscale;
      f.offsets = (int32_t *)(ws + W.offsets);
      f.perm = (int32_t *)(ws + W.perm);
      f.slot_pos = (int32_t *)(ws + W.slot_pos);
      f.groups = (Group *)(ws + W.groups);
      f.xt = ws + W.xg;
      f.rscale = (float *)(ws + W.rscale);
      f.P = W.pieces;
      f.GN = W.group_n;
      f.e0 = W.e0;
      f.e1 = W.e1;
      f.shared = W.shared ? 1 : 0;
#ifdef MOE_TRACE
      f.trace = g_router_trace;
#endif
    }
    // the dynamic x slice plus the block's static arrays may pass the 48 KB default
    auto launch = [&](auto k) {
      set_dyn_smem((const void *)k, (int)smem);
      k<<<grid, kGemvThreads, smem, st>>>(c, packed, wr, x, is_bf16, T, partials, ctrl, xmax,
                                          fused ? 1 : 0, f);
    };
    if (T <= 1) launch(router_gemv_kernel<1>);
    else if (T <= 2) launch(router_gemv_kernel<2>);
    else if (T <= 4) launch(router_gemv_kernel<4>);
    else if (T <= 8) launch(router_gemv_kernel<8>);
    else launch(router_gemv_kernel<16>);
    if (fused) return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  } else if (router_tc_applies(c, dt, T)) {
    // tensor cores: 128 experts x 256 tokens a CTA, H split until the grid covers the SMs
    const int tiles = router_mtiles(c) * ((T + 255) / 256), KC = c.hidden / 64;
    const int sms = dev_info().sms;
    hsplits = 1;
    while (hsplits < kRouterHS && tiles * hsplits < sms && KC % (2 * hsplits) == 0) hsplits *= 2;
    const int r = launch_router_tc(c, packed, x, T, partials, hsplits, ctrl, st);
    if (r) return r;
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
  long long *rtrace = nullptr;
#ifdef MOE_TRACE
  rtrace = g_router_trace;
#endif
  if (launch_pdl(router_topk_kernel, dim3((T + 7) / 8), dim3(256), 0, st, c, bias,
                 (const float *)partials, hsplits, T, ids, w, ctrl, x, is_bf16, tscale,
                 (const float *)(gemv ? xmax : nullptr), rtrace) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

/*
 * moe_oracle.c -- plain single-threaded fp64 CPU oracle of one MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h).  Written for a reader to check
 * against the pages by eye: no blocking, no fusion, no reordering beyond what
 * each step's definition states.  Build: cc -std=c99 -O2 -ffp-contract=off.
 *
 * Pages cited: [README], [DEEP], [ENGINE], [SITE] as named in moe_oracle.h.
 *
 * Readings taken where the pages are silent or ambiguous:
 *  - Softmax router: softmax over all E logits with the maximum subtracted
 *    ([ENGINE] §3.2 Step 2), the k largest probabilities selected ([ENGINE]
 *    §3.2 Step 3), then renormalised over the selected k (norm_topk = 1).
 *    [SITE] §3.2 selects on raw logits; softmax is monotone, so the ids are the
 *    same.  Ties go to the lower expert index; slot order is descending score.
 *  - Sigmoid grouped router: [README] 已实现的功能 names only a "DeepSeek-V3
 *    style sigmoid router (noaux_tc, routed_scaling_factor)".  Reading (the
 *    DeepSeek-V3 method): s = sigmoid(logit), c = s + bias; groups are E/n_group
 *    consecutive experts; a group's score is the sum of its two largest c; the
 *    topk_group best groups are kept; the k largest c among the kept groups'
 *    experts are selected; weights are s (not c) renormalised over the
 *    selection and multiplied by routed_scaling_factor.
 *  - Shared expert: added with weight 1 ([DEEP] §4.3 merges shared_output
 *    with the accumulated routed outputs).
 *  - SwiGLU expert: y = W_down (silu(W_gate x) * (W_up x)), silu(z) = z/(1+e^-z)
 *    ([SITE] §3.1 names the SwiGLU gate_proj output; [README] routed-expert
 *    SwiGLU); weights are per-row scaled codes, W[r][c] = s[r] * q[r][c]
 *    ([DEEP] §5.1 逐行缩放; [README] 量化内核: 逐行缩放, 使用时反量化).
 *  - Combine: out[t] = shared(x_t) + sum_j w[t][j] * y_{ids[t][j]}(x_t), summed
 *    in slot order ([DEEP] §4.3: accumulator += expert_output * routing_weights).
 *  - Batched union ([README] 批处理并集 MoE): each selected expert is evaluated
 *    once on all the tokens routed to it; the result equals the per-token loop.
 *  - Q8_0 ([README] 整数点积内核): blocks of 32 along the contraction, one fp32
 *    scale d = amax/127 per block, q = round-half-away-from-zero(v/d) in fp32,
 *    d = 0 gives q = 0; every expert matmul's activation is Q8_0 in that mode
 *    (x before gate/up, h before down); h is rounded to fp32 before encoding.
 *  - int4 packing ([DEEP] §5.1): two's complement nibbles, first element in the
 *    high nibble.  The printed dequantiser ORs 0xF0 into an int, which would
 *    give 240..255; the reading is ordinary 4-bit sign extension.  int2 (pages
 *    silent): values [-2,1], four per byte, first element in bits 7..6.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* [ENGINE] §3.2 Step 1 gate projection; [SITE] §3.2 linear router. */
void orc_router_logits(const orc_config *c, const double *x, int T, const float *wr,
                       double *logits) {
  const int H = c->hidden, E = c->n_experts;
  for (int t = 0; t < T; t++)
    for (int e = 0; e < E; e++) {
      double acc = 0.0;
      for (int h = 0; h < H; h++) acc += x[(size_t)t * H + h] * (double)wr[(size_t)e * H + h];
      logits[(size_t)t * E + e] = acc;
    }
}

/* Order n candidate indices by (score descending, index ascending): selection sort,
 * strict '>' so that equal scores keep the lower index first. */
static void order_desc(const double *score, const int *cand, int n, int *sorted) {
  char *used = (char *)calloc((size_t)n, 1);
  for (int j = 0; j < n; j++) {
    int best = -1;
    for (int i = 0; i < n; i++) {
      if (used[i]) continue;
      if (best < 0 || score[cand[i]] > score[cand[best]]) best = i;
    }
    used[best] = 1;
    sorted[j] = cand[best];
  }
  free(used);
}

/* smallest gap score[s[j]] - score[s[j+1]] over j < upto (s sorted descending) */
static double min_gap(const double *score, const int *s, int n, int upto) {
  double m = INFINITY;
  for (int j = 0; j < upto && j + 1 < n; j++) {
    double g = score[s[j]] - score[s[j + 1]];
    if (g < m) m = g;
  }
  return m;
}

/* Routing of one token.  The decision boundaries whose gaps make up the margin:
 * every consecutive pair among the k selected (slot order), the k-th selected vs
 * the best unselected candidate, and (grouped router) the topk_group-th kept
 * group vs the best dropped group. */
static int route_one(const orc_config *c, const double *l, const float *bias, int32_t *ids,
                     double *w, double *margin) {
  const int E = c->n_experts, k = c->top_k;
  double *p = (double *)malloc(sizeof(double) * (size_t)E);
  double *sel_score = (double *)malloc(sizeof(double) * (size_t)E); /* score used to select */
  double *wsrc = (double *)malloc(sizeof(double) * (size_t)E);      /* score used as weight */
  int *cand = (int *)malloc(sizeof(int) * (size_t)E);
  int *sorted = (int *)malloc(sizeof(int) * (size_t)E);
  int ncand = 0;
  double mg = INFINITY;

  if (c->router == ORC_ROUTER_SOFTMAX) {
    /* [ENGINE] §3.2 Step 2: softmax with the maximum subtracted */
    double mx = -INFINITY, sum = 0.0;
    for (int e = 0; e < E; e++) if (l[e] > mx) mx = l[e];
    for (int e = 0; e < E; e++) { p[e] = exp(l[e] - mx); sum += p[e]; }
    for (int e = 0; e < E; e++) { p[e] = p[e] / sum; sel_score[e] = p[e]; wsrc[e] = p[e]; }
    for (int e = 0; e < E; e++) cand[ncand++] = e;
  } else if (c->router == ORC_ROUTER_SIGMOID_GROUPED) {
    const int G = c->n_group, gs = E / G;
    for (int e = 0; e < E; e++) {
      double s = 1.0 / (1.0 + exp(-l[e]));
      wsrc[e] = s;
      sel_score[e] = s + (bias ? (double)bias[e] : 0.0);
    }
    /* group score = sum of the (up to) two largest corrected scores in the group */
    double *gscore = (double *)malloc(sizeof(double) * (size_t)G);
    int *gidx = (int *)malloc(sizeof(int) * (size_t)G);
    int *gsorted = (int *)malloc(sizeof(int) * (size_t)G);
    int *members = (int *)malloc(sizeof(int) * (size_t)gs);
    int *msorted = (int *)malloc(sizeof(int) * (size_t)gs);
    for (int g = 0; g < G; g++) {
      for (int i = 0; i < gs; i++) members[i] = g * gs + i;
      order_desc(sel_score, members, gs, msorted);
      gscore[g] = sel_score[msorted[0]] + (gs > 1 ? sel_score[msorted[1]] : 0.0);
      gidx[g] = g;
    }
    order_desc(gscore, gidx, G, gsorted);
    if (c->topk_group < G) {
      double gg = gscore[gsorted[c->topk_group - 1]] - gscore[gsorted[c->topk_group]];
      if (gg < mg) mg = gg;
    }
    /* candidates: experts of the kept groups, in expert order */
    for (int e = 0; e < E; e++) {
      int g = e / gs, kept = 0;
      for (int j = 0; j < c->topk_group; j++) if (gsorted[j] == g) kept = 1;
      if (kept) cand[ncand++] = e;
    }
    free(gscore); free(gidx); free(gsorted); free(members); free(msorted);
  } else {
    free(p); free(sel_score); free(wsrc); free(cand); free(sorted);
    return -1;
  }

  /* [ENGINE] §3.2 Step 3: the k largest */
  order_desc(sel_score, cand, ncand, sorted);
  double eg = min_gap(sel_score, sorted, ncand, k);
  if (eg < mg) mg = eg;
  double wsum = 0.0;
  for (int j = 0; j < k; j++) { ids[j] = sorted[j]; wsum += wsrc[sorted[j]]; }
  /* Adaptive expert top-p ("Show HN" 实用调节项 --topp, an explicit lossy override; the
   * pages give no formula, reading): in slot order keep the shortest prefix of the
   * selected experts whose share of the selection's weight sources reaches top_p (at
   * least the first); the rest are dropped and the kept weights normalised over the kept
   * experts.  Its decisions are "share before slot j < top_p"; the gaps at the crossing
   * enter the margin. */
  int m = k;
  if (c->top_p > 0.0 && c->top_p < 1.0) {
    double before = 0.0, before_last = 0.0;
    m = 0;
    for (int j = 0; j < k; j++) {
      if (before >= c->top_p) break;
      before_last = before;
      before += wsrc[sorted[j]] / wsum;
      m = j + 1;
    }
    double g1 = c->top_p - before_last;  /* the last kept slot */
    if (g1 < mg) mg = g1;
    if (m < k) {
      double g2 = before - c->top_p;     /* the first dropped slot */
      if (g2 < mg) mg = g2;
    }
    wsum = 0.0;
    for (int j = 0; j < m; j++) wsum += wsrc[sorted[j]];
  }
  for (int j = 0; j < k; j++) {
    if (j >= m) { ids[j] = -1; w[j] = 0.0; continue; }
    double v = wsrc[sorted[j]];
    if (c->norm_topk) v = v / wsum;
    w[j] = v * c->rsf;
  }
  if (margin) *margin = mg;
  free(p); free(sel_score); free(wsrc); free(cand); free(sorted);
  return 0;
}

int orc_route(const orc_config *c, const double *logits, const float *bias, int T,
              int32_t *ids, double *w, double *margin) {
  const int E = c->n_experts, k = c->top_k;
  if (k < 1 || k > E) return -1;
  if (c->router == ORC_ROUTER_SIGMOID_GROUPED) {
    if (c->n_group < 1 || E % c->n_group != 0) return -1;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return -1;
    if (c->topk_group * (E / c->n_group) < k) return -1;
  }
  for (int t = 0; t < T; t++) {
    int r = route_one(c, logits + (size_t)t * E, bias, ids + (size_t)t * k, w + (size_t)t * k,
                      margin ? margin + t : NULL);
    if (r) return r;
  }
  return 0;
}

/* [README] 批处理并集 MoE: group the (token, slot) pairs by expert. */
void orc_permutation(int T, int k, int E, const int32_t *ids, int32_t *offsets, int32_t *perm) {
  for (int e = 0; e <= E; e++) offsets[e] = 0;
  for (int i = 0; i < T * k; i++)
    if (ids[i] >= 0) offsets[ids[i] + 1]++;
  for (int e = 0; e < E; e++) offsets[e + 1] += offsets[e];
  int pos = 0;
  for (int e = 0; e < E; e++)
    for (int t = 0; t < T; t++)
      for (int j = 0; j < k; j++)
        if (ids[t * k + j] == e) perm[pos++] = t * k + j;
  while (pos < T * k) perm[pos++] = -1;
}

/* y[n][rows] = W x with W[r][c] = s[r] * q[r][c] (plain fp64) */
static void dequant_matvec(const int8_t *q, const float *s, int rows, int cols, const double *x,
                           int n, double *y) {
  double *wrow = (double *)malloc(sizeof(double) * (size_t)cols);
  for (int r = 0; r < rows; r++) {
    for (int cc = 0; cc < cols; cc++) wrow[cc] = (double)s[r] * (double)q[(size_t)r * cols + cc];
    for (int i = 0; i < n; i++) {
      double acc = 0.0;
      for (int cc = 0; cc < cols; cc++) acc += wrow[cc] * x[(size_t)i * cols + cc];
      y[(size_t)i * rows + r] = acc;
    }
  }
  free(wrow);
}

/* ---- Q8_0 ---- */
void orc_q8_0_encode(const float *v, int n, int8_t *q, float *d) {
  for (int b = 0; b < n / 32; b++) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
      float a = fabsf(v[b * 32 + i]);
      if (a > amax) amax = a;
    }
    volatile float db = amax / 127.0f; /* fp32 IEEE division */
    d[b] = db;
    for (int i = 0; i < 32; i++) {
      int qi = 0;
      if (db != 0.0f) {
        volatile float r = v[b * 32 + i] / db;
        float rr = roundf(r); /* half away from zero */
        if (rr > 127.0f) rr = 127.0f;
        if (rr < -127.0f) rr = -127.0f;
        qi = (int)rr;
      }
      q[b * 32 + i] = (int8_t)qi;
    }
  }
}

int32_t orc_block_dot(const int8_t *a, const int8_t *b) {
  int32_t acc = 0;
  for (int i = 0; i < 32; i++) acc += (int32_t)a[i] * (int32_t)b[i];
  return acc;
}

/* y[n][rows] = s[r] * sum_b d_x[i][b] * D(q[r] block b, q_x[i] block b) */
static void q8_matvec(const int8_t *q, const float *s, int rows, int cols, const int8_t *qx,
                      const float *dx, int n, double *y) {
  const int nb = cols / 32;
  for (int r = 0; r < rows; r++)
    for (int i = 0; i < n; i++) {
      double acc = 0.0;
      for (int b = 0; b < nb; b++)
        acc += (double)dx[(size_t)i * nb + b] *
               (double)orc_block_dot(q + (size_t)r * cols + b * 32, qx + (size_t)i * cols + b * 32);
      y[(size_t)i * rows + r] = (double)s[r] * acc;
    }
}

/* One SwiGLU expert ([SITE] §3.1, [README]): h = silu(W_g x) * (W_u x), y = W_d h. */
void orc_expert_forward(const orc_config *c, const orc_expert *ex, const double *x, int n,
                        double *y) {
  const int H = c->hidden, I = ex->inter;
  double *g = (double *)malloc(sizeof(double) * (size_t)n * I);
  double *u = (double *)malloc(sizeof(double) * (size_t)n * I);
  double *h = (double *)malloc(sizeof(double) * (size_t)n * I);
  if (!c->act_q8_0) {
    dequant_matvec(ex->gate, ex->s_gate, I, H, x, n, g);
    dequant_matvec(ex->up, ex->s_up, I, H, x, n, u);
    for (size_t i = 0; i < (size_t)n * I; i++) h[i] = orc_silu(g[i]) * u[i];
    dequant_matvec(ex->down, ex->s_down, H, I, h, n, y);
  } else {
    float *xf = (float *)malloc(sizeof(float) * (size_t)n * H);
    int8_t *qx = (int8_t *)malloc((size_t)n * H);
    float *dx = (float *)malloc(sizeof(float) * (size_t)n * (H / 32));
    for (size_t i = 0; i < (size_t)n * H; i++) xf[i] = (float)x[i];
    for (int i = 0; i < n; i++)
      orc_q8_0_encode(xf + (size_t)i * H, H, qx + (size_t)i * H, dx + (size_t)i * (H / 32));
    q8_matvec(ex->gate, ex->s_gate, I, H, qx, dx, n, g);
    q8_matvec(ex->up, ex->s_up, I, H, qx, dx, n, u);
    float *hf = (float *)malloc(sizeof(float) * (size_t)n * I);
    int8_t *qh = (int8_t *)malloc((size_t)n * I);
    float *dh = (float *)malloc(sizeof(float) * (size_t)n * (I / 32));
    for (size_t i = 0; i < (size_t)n * I; i++) hf[i] = (float)(orc_silu(g[i]) * u[i]);
    for (int i = 0; i < n; i++)
      orc_q8_0_encode(hf + (size_t)i * I, I, qh + (size_t)i * I, dh + (size_t)i * (I / 32));
    q8_matvec(ex->down, ex->s_down, H, I, qh, dh, n, y);
    free(xf); free(qx); free(dx); free(hf); free(qh); free(dh);
  }
  free(g); free(u); free(h);
}

int orc_layer_experts(const orc_config *c, const double *x, int T, const int32_t *ids,
                      const double *w, const orc_expert *experts, const orc_expert *shared,
                      int mode, double *out) {
  const int H = c->hidden, k = c->top_k, E = c->n_experts;
  if (c->n_shared && !shared) return -1;
  if (mode == 0) {
    /* per-token: out[t] = shared(x_t) + sum_j w[t][j] * y_{e_j}(x_t) */
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    for (int t = 0; t < T; t++) {
      double *o = out + (size_t)t * H;
      if (c->n_shared) orc_expert_forward(c, shared, x + (size_t)t * H, 1, o);
      else for (int h = 0; h < H; h++) o[h] = 0.0;
      for (int j = 0; j < k; j++) {
        if (ids[t * k + j] < 0) continue;  /* dropped by top-p */
        const orc_expert *ex = &experts[ids[t * k + j]];
        if (!ex->gate) { free(y); return -2; }
        orc_expert_forward(c, ex, x + (size_t)t * H, 1, y);
        for (int h = 0; h < H; h++) o[h] += w[t * k + j] * y[h];
      }
    }
    free(y);
    return 0;
  }
  /* batched union: each selected expert once, on all of its tokens */
  int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
  double *yslot = (double *)malloc(sizeof(double) * (size_t)T * k * H);
  orc_permutation(T, k, E, ids, offsets, perm);
  for (int e = 0; e < E; e++) {
    int n = offsets[e + 1] - offsets[e];
    if (n == 0) continue;
    if (!experts[e].gate) { free(offsets); free(perm); free(yslot); return -2; }
    double *xe = (double *)malloc(sizeof(double) * (size_t)n * H);
    double *ye = (double *)malloc(sizeof(double) * (size_t)n * H);
    for (int i = 0; i < n; i++) {
      int t = perm[offsets[e] + i] / k;
      memcpy(xe + (size_t)i * H, x + (size_t)t * H, sizeof(double) * (size_t)H);
    }
    orc_expert_forward(c, &experts[e], xe, n, ye);
    for (int i = 0; i < n; i++)
      memcpy(yslot + (size_t)perm[offsets[e] + i] * H, ye + (size_t)i * H,
             sizeof(double) * (size_t)H);
    free(xe); free(ye);
  }
  if (c->n_shared) orc_expert_forward(c, shared, x, T, out);
  else for (size_t i = 0; i < (size_t)T * H; i++) out[i] = 0.0;
  for (int t = 0; t < T; t++)
    for (int j = 0; j < k; j++) {
      if (ids[t * k + j] < 0) continue;  /* dropped by top-p */
      for (int h = 0; h < H; h++)
        out[(size_t)t * H + h] += w[t * k + j] * yslot[((size_t)t * k + j) * H + h];
    }
  free(offsets); free(perm); free(yslot);
  return 0;
}

int orc_layer_forward(const orc_config *c, const double *x, int T, const float *wr,
                      const float *bias, const orc_expert *experts, const orc_expert *shared,
                      int mode, int32_t *ids, double *w, double *out) {
  double *logits = (double *)malloc(sizeof(double) * (size_t)T * c->n_experts);
  orc_router_logits(c, x, T, wr, logits);
  int r = orc_route(c, logits, bias, T, ids, w, NULL);
  free(logits);
  if (r) return r;
  return orc_layer_experts(c, x, T, ids, w, experts, shared, mode, out);
}

/* ---- packing ([DEEP] §5.1; [README] 量化内核: 打包与 int8 容器逐位一致) ---- */
void orc_pack_int4(const int8_t *q, size_t n, uint8_t *out) {
  for (size_t i = 0; i < n; i += 2)
    out[i / 2] = (uint8_t)(((q[i] & 0xF) << 4) | (q[i + 1] & 0xF));
}

static int8_t sext(int v, int bits) {
  int m = 1 << (bits - 1);
  return (int8_t)(v >= m ? v - (1 << bits) : v);
}

void orc_unpack_int4(const uint8_t *p, size_t n, int8_t *q) {
  for (size_t i = 0; i < n; i += 2) {
    q[i] = sext(p[i / 2] >> 4, 4);
    q[i + 1] = sext(p[i / 2] & 0xF, 4);
  }
}

void orc_pack_int2(const int8_t *q, size_t n, uint8_t *out) {
  for (size_t i = 0; i < n; i += 4)
    out[i / 4] = (uint8_t)(((q[i] & 3) << 6) | ((q[i + 1] & 3) << 4) | ((q[i + 2] & 3) << 2) |
                           (q[i + 3] & 3));
}

void orc_unpack_int2(const uint8_t *p, size_t n, int8_t *q) {
  for (size_t i = 0; i < n; i++) q[i] = sext((p[i / 4] >> (6 - 2 * (int)(i % 4))) & 3, 2);
}

/* Round an fp64 value to bf16 (8 significant bits), to nearest, ties to even; returns the
 * bf16 value exactly as a double.  Values beyond the bf16 range become +-inf. */
static double round_bf16(double v) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  int e;
  double m = frexp(v, &e);              /* v = m * 2^e, 0.5 <= |m| < 1 */
  if (e < -125) {                       /* bf16 subnormals: fixed step 2^-133 */
    double q = nearbyint(ldexp(v, 133)); /* current rounding mode: to nearest even */
    return ldexp(q, -133);
  }
  double q = nearbyint(ldexp(m, 8));    /* 8 significant bits */
  double r = ldexp(q, e - 8);
  if (fabs(r) >= 0x1.ffp127 * (1.0 + 0x1p-9)) return v > 0 ? INFINITY : -INFINITY;
  return r;
}

void orc_residual_rmsnorm(int T, int H, double *r, const double *add, double eps,
                          double *xn) {
  for (int t = 0; t < T; t++) {
    double *rt = r + (size_t)t * H;
    if (add)
      for (int h = 0; h < H; h++) rt[h] += add[(size_t)t * H + h];
    double ss = 0.0;
    for (int h = 0; h < H; h++) ss += rt[h] * rt[h];
    const double inv = 1.0 / sqrt(ss / H + eps);
    for (int h = 0; h < H; h++) xn[(size_t)t * H + h] = round_bf16(rt[h] * inv);
  }
}

int orc_quantize_rows(const float *w, int rows, int cols, int bits, int8_t *q, float *s) {
  if (bits != 8 && bits != 4 && bits != 2) return -1;
  const int qmax = (1 << (bits - 1)) - 1, qmin = -(1 << (bits - 1));
  for (int r = 0; r < rows; r++) {
    const float *row = w + (size_t)r * cols;
    float amax = 0.0f;
    for (int c = 0; c < cols; c++) {
      const float a = fabsf(row[c]);
      if (a > amax) amax = a;
    }
    volatile float sc = amax / (float)qmax; /* fp32, as the quantiser does it */
    s[r] = sc;
    for (int c = 0; c < cols; c++) {
      int v = 0;
      if (sc != 0.0f) {
        volatile float ratio = row[c] / sc;
        if (ratio == ratio) { /* a NaN ratio (inf / inf, NaN weights) gives code 0 */
          const float rr = roundf(ratio);
          v = rr < (float)qmin ? qmin : (rr > (float)qmax ? qmax : (int)rr);
        }
      }
      q[(size_t)r * cols + c] = (int8_t)v;
    }
  }
  return 0;
}

/*
 * moe_oracle.h -- plain, slow, single-threaded CPU oracle of one MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this code: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library; the two meet only through the seeded input generator.
 *
 * Arithmetic: fp64 everywhere (compiled with -ffp-contract=off), except the
 * Q8_0 activation encoding, which is an fp32 encoding by definition.
 *
 * Pages cited (by title and section):
 *   [README]  "Show HN: 如何在我的低配置电脑上运行 GLM-5.2" (the colibrì README),
 *             section 已实现的功能 (implemented features).
 *   [DEEP]    "colibrì 深度拆解：当1300行纯C在25GB笔记本上跑起744B大模型",
 *             §4.3 路由机制详解, §5.1 量化, §5.2 AVX2 SIMD手写矩阵乘法.
 *   [ENGINE]  "Colibri——面向前沿大模型推理的轻量级MoE引擎",
 *             §3.2 路由算法的工程实现 (Step 1 gate projection, Step 2 softmax, Step 3 top-k).
 *   [SITE]    "企业官网建设流程全解析" (a Colibri article), §3.1 激活内存池化 (SwiGLU
 *             gate_proj output), §3.2 路由器实现.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_ROUTER_SOFTMAX 0
#define ORC_ROUTER_SIGMOID_GROUPED 1

typedef struct {
  int hidden;        /* H */
  int inter;         /* I of the routed experts */
  int n_experts;     /* E */
  int top_k;         /* k */
  int n_shared;      /* 0 or 1 */
  int inter_shared;  /* I of the shared expert */
  int router;        /* ORC_ROUTER_* */
  int n_group;       /* grouped router: groups of E/n_group consecutive experts */
  int topk_group;    /* grouped router: groups kept */
  int norm_topk;     /* 1: renormalise the selected weights */
  double rsf;        /* routed_scaling_factor */
  int act_q8_0;      /* 1: Q8_0 int8 activations for every expert matmul */
  double top_p;      /* 0 < top_p < 1: adaptive expert top-p (lossy, opt-in); else off */
} orc_config;

/* One expert: int8 containers (code per weight) and fp32 per-row scales. */
typedef struct {
  const int8_t *gate;   /* [inter][H] */
  const int8_t *up;     /* [inter][H] */
  const int8_t *down;   /* [H][inter] */
  const float *s_gate;  /* [inter] */
  const float *s_up;    /* [inter] */
  const float *s_down;  /* [H] */
  int inter;
} orc_expert;

/* silu(z) = z / (1 + exp(-z)) */
double orc_silu(double z);

/* logits[t][e] = sum_h x[t][h] * wr[e][h] */
void orc_router_logits(const orc_config *c, const double *x, int T, const float *wr,
                       double *logits);

/* Routing of T tokens from their logits.  Writes ids[T][k] (slot order = descending
 * selection score, ties to the lower expert index), w[T][k], and, if margin != NULL,
 * margin[t] = the smallest gap at any decision boundary of token t (see the .c file).
 * With top_p on, slots past the kept prefix have id -1 and weight 0.
 * bias may be NULL (= zeros).  Returns 0, or -1 on an unsupported config. */
int orc_route(const orc_config *c, const double *logits, const float *bias, int T,
              int32_t *ids, double *w, double *margin);

/* Canonical permutation: offsets[E+1] (exclusive scan of per-expert counts) and
 * perm[T*k] = slot indices t*k+j ordered by (expert ascending, token ascending); slots with
 * id -1 (dropped by top-p) are left out and the tail of perm is -1. */
void orc_permutation(int T, int k, int E, const int32_t *ids, int32_t *offsets, int32_t *perm);

/* One SwiGLU expert on n rows of x (fp64 [n][H]) -> y [n][H]. */
void orc_expert_forward(const orc_config *c, const orc_expert *ex, const double *x, int n,
                        double *y);

/* Whole layer.  mode 0 = per-token loop, mode 1 = batched union (each expert once).
 * experts[E] may hold NULL weight pointers for experts no token selects.
 * shared may be NULL when c->n_shared == 0.  out[T][H]. */
int orc_layer_forward(const orc_config *c, const double *x, int T, const float *wr,
                      const float *bias, const orc_expert *experts, const orc_expert *shared,
                      int mode, int32_t *ids, double *w, double *out);

/* Same layer, given the routing (ids, w) already: only the expert part and the combine. */
int orc_layer_experts(const orc_config *c, const double *x, int T, const int32_t *ids,
                      const double *w, const orc_expert *experts, const orc_expert *shared,
                      int mode, double *out);

/* ---- Q8_0 activations ([README] 已实现的功能: 整数点积内核, Q8_0 风格 int8 激活) ---- */
/* n a multiple of 32.  Per block b: d[b] = amax/127 (fp32), q = round-half-away(v/d)
 * clamped to [-127,127] (fp32 division), d == 0 => q = 0. */
void orc_q8_0_encode(const float *v, int n, int8_t *q, float *d);
/* int32 dot of two 32-element int8 blocks */
int32_t orc_block_dot(const int8_t *a, const int8_t *b);

/* ---- packing ([DEEP] §5.1: two int4 per byte, first element in the high nibble) ---- */
void orc_pack_int4(const int8_t *q, size_t n, uint8_t *out);     /* n even */
void orc_unpack_int4(const uint8_t *p, size_t n, int8_t *q);
void orc_pack_int2(const int8_t *q, size_t n, uint8_t *out);     /* n multiple of 4 */
void orc_unpack_int2(const uint8_t *p, size_t n, int8_t *q);

/* ---- quantiser ([DEEP] §5.1 quantize_row, per-row scaling) ----
 * For each row r of w [rows][cols] (fp32): amax = max |w|, s = amax / qmax (fp32 IEEE
 * division), q = roundf(w / s) (fp32 division, half away from zero) clamped to
 * [-2^(bits-1), qmax], qmax = 2^(bits-1) - 1 (7 for int4 as printed; 127 and 1 for int8 and
 * int2 by the same pattern); a row with amax == 0 gets s = 0 and q = 0, a NaN ratio gives
 * q = 0 (non-finite weights are outside the pages' scheme).  Codes go to an
 * int8 container [rows][cols], scales to s [rows].  bits: 8, 4 or 2. */
int orc_quantize_rows(const float *w, int rows, int cols, int bits, int8_t *q, float *s);

/* ---- a stack of layers ([DEEP] §4.3: a layer's merged output feeds the next layer) ----
 * The pages leave the stacking arithmetic open.  Reading: the stack keeps a residual
 * stream r [T][H]; after a layer, r <- r + out (out = the layer's MoE output), and the next
 * layer's input is the unweighted RMSNorm of r, x = r / sqrt(mean_h(r^2) + eps), rounded to
 * bf16 (the layers' activation type).  `add` may be NULL (the first layer: r = x_0).
 * Writes r in place, xn [T][H] in fp64 (the rounded bf16 values, exactly). */
void orc_residual_rmsnorm(int T, int H, double *r, const double *add, double eps,
                          double *xn);

#ifdef __cplusplus
}
#endif
#endif

/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE-layer library.
 *
 * One Mixture-of-Experts layer forward on one GPU:
 *   router (softmax top-k, or DeepSeek-V3-style sigmoid router with bias-corrected
 *   grouped top-k) -> token-by-expert permutation ("batched union": every selected
 *   expert's weights are read once for all tokens routed to it) -> SwiGLU experts on
 *   per-row-scaled int4 / int8 / int2 weights dequantised on use -> gate-weighted
 *   combine plus the shared expert.
 *
 * Pages that define the operations (cited by title and section):
 *   [README] "Show HN: 如何在我的低配置电脑上运行 GLM-5.2" (the colibrì README), section
 *            已实现的功能: DeepSeek-V3 sigmoid router (noaux_tc, routed_scaling_factor) and
 *            shared expert; integer dot kernels with Q8_0-style int8 activations;
 *            int8 / packed int4 / packed int2 kernels with per-row scales, dequantised on
 *            use, packing bit-identical to the int8 container; batched union MoE.
 *   [DEEP]   "colibrì 深度拆解：当1300行纯C在25GB笔记本上跑起744B大模型", §4.3 路由机制详解
 *            (router, per-expert forward, weighted accumulate, merge with the shared
 *            expert), §5.1 量化 (per-row scaled int4, two codes per byte).
 *   [ENGINE] "Colibri——面向前沿大模型推理的轻量级MoE引擎", §3.2 路由算法的工程实现
 *            (gate projection, softmax with the maximum subtracted, top-k).
 *   [SITE]   "企业官网建设流程全解析" (a Colibri article), §3.1 激活内存池化 (SwiGLU).
 *
 * Conventions (all entry points):
 *  - Pointers are DEVICE pointers owned by the caller unless stated otherwise; the
 *    library allocates no device memory and keeps no per-call global state.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Work is stream-ordered and asynchronous; nothing synchronises the host except
 *    moe_read_status and the debug entry points that say so.
 *  - Argument and shape errors are returned synchronously, before any launch.
 *    Conditions found on the device (a packed blob whose header does not match the
 *    config, a bounded wait that gave up) are written to a status word inside the
 *    workspace and returned by moe_read_status.
 *  - Supported shapes: hidden H and inter I (and inter_shared) multiples of 128;
 *    1 <= top_k <= 16, top_k <= n_experts <= 256; grouped router: n_experts divisible
 *    by n_group, 1 <= topk_group <= n_group <= 32.  weight_bits 4, 8 or 2; act_q8_0
 *    requires weight_bits == 8.  Anything else returns MOE_ERR_UNSUPPORTED.
 *  - The output of the layer is fp32 [T][H].
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* NULL pointer, negative size, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2,  /* shape or option outside the supported set */
  MOE_ERR_WORKSPACE = -3,    /* workspace or packed buffer too small */
  MOE_ERR_CUDA = -4,         /* a CUDA launch or copy failed */
  MOE_ERR_TIMEOUT = -5,      /* device: a bounded wait gave up */
  MOE_ERR_NUMERIC = -6,      /* device: non-finite value in an intermediate */
  MOE_ERR_PACKED = -7        /* device: packed blob header does not match the config */
} moe_status;

typedef enum { MOE_ROUTER_SOFTMAX = 0, MOE_ROUTER_SIGMOID_GROUPED = 1 } moe_router_kind;
typedef enum { MOE_DT_F32 = 0, MOE_DT_BF16 = 1 } moe_dtype;

/* Layer shape and routing options. */
typedef struct {
  int hidden;          /* H */
  int inter;           /* I, intermediate size of a routed expert */
  int n_experts;       /* E routed experts */
  int top_k;           /* k experts per token */
  int n_shared;        /* 0 or 1 shared expert (always applied, weight 1) */
  int inter_shared;    /* intermediate size of the shared expert (0 = inter) */
  int router;          /* moe_router_kind */
  int n_group;         /* grouped router: number of expert groups */
  int topk_group;      /* grouped router: groups kept per token */
  int norm_topk;       /* 1 = renormalise the k selected weights to sum to 1 */
  float routed_scaling_factor; /* multiplies the routed weights (1 for softmax layers) */
  int weight_bits;     /* 4, 8 or 2 */
  int act_q8_0;        /* 1 = Q8_0 int8 activations (blocks of 32, fp32 scale) */
  float expert_top_p;  /* adaptive expert top-p, lossy and opt-in ("Show HN: 如何在我的低配置
                        * 电脑上运行 GLM-5.2", 实用调节项 --topp): 0 < p < 1 keeps, in slot
                        * order, the shortest prefix of a token's k selected experts whose
                        * share of their weight sources reaches p (at least one); dropped
                        * slots get id -1 and weight 0 and are not computed, and the kept
                        * weights are normalised over the kept experts.  0 (or >= 1) = off. */
} moe_layer_config;

/* Source weights for packing: int8 containers (one code per byte, row-major, codes in
 * the weight_bits range) and fp32 per-row scales.  Device pointers. */
typedef struct {
  const int8_t *gate, *up, *down;       /* [E][I][H], [E][I][H], [E][H][I] */
  const float *s_gate, *s_up, *s_down;  /* [E][I], [E][I], [E][H] */
  const int8_t *sh_gate, *sh_up, *sh_down;     /* shared: [Is][H], [Is][H], [H][Is] */
  const float *sh_s_gate, *sh_s_up, *sh_s_down;/* [Is], [Is], [H] */
  const float *router_w;                /* [E][H] fp32 */
  const float *router_bias;             /* [E] fp32, or NULL (= zeros) */
} moe_weight_src;

/* Library version (major*10000 + minor*100 + patch). */
int moe_version(void);

/* Human-readable name of a moe_status code (static string). */
const char *moe_status_str(int status);

/* Validate a config: MOE_OK, MOE_ERR_INVALID_ARG (NULL) or MOE_ERR_UNSUPPORTED. */
int moe_check_config(const moe_layer_config *cfg);

/* Bytes of the packed weight blob for `cfg` (0 if the config is unsupported).
 * The blob holds a header, the router weights and bias, and every expert's packed
 * codes and row scales in a private GPU layout ([README] 量化内核; [DEEP] §5.1). */
size_t moe_packed_bytes(const moe_layer_config *cfg);

/* Workspace bytes for calls with up to `max_tokens` tokens (0 if unsupported).
 * Workspace: caller-owned device memory, 256-byte aligned; one workspace per
 * concurrently running call (calls sharing a workspace must be stream-ordered). */
size_t moe_workspace_bytes(const moe_layer_config *cfg, int max_tokens);

/* Pack every expert, the shared expert and the router into `packed` (device,
 * 256-byte aligned, packed_bytes >= moe_packed_bytes).  Codes outside the
 * weight_bits range are masked to their low bits.  Returns MOE_ERR_WORKSPACE if
 * packed_bytes is too small. */
int moe_pack_weights(const moe_layer_config *cfg, const moe_weight_src *src, void *packed,
                     size_t packed_bytes, void *stream);

/* Incremental packing: write the header + router (router_bias may be NULL) ... */
int moe_pack_router(const moe_layer_config *cfg, const float *router_w, const float *router_bias,
                    void *packed, size_t packed_bytes, void *stream);
/* ... then one expert at a time: expert in [0, E) is a routed expert, expert == E the
 * shared expert.  gate/up [I][H], down [H][I] int8 containers; scales [I],[I],[H]. */
int moe_pack_expert(const moe_layer_config *cfg, int expert, const int8_t *gate,
                    const int8_t *up, const int8_t *down, const float *s_gate,
                    const float *s_up, const float *s_down, void *packed, size_t packed_bytes,
                    void *stream);

/* Inverse of packing for one expert (expert == E: the shared expert): writes the int8
 * containers and scales back.  unpack(pack(q)) == q bit for bit ([README] 打包与 int8
 * 容器逐位一致).  Any output pointer may be NULL to skip it. */
int moe_unpack_weights(const moe_layer_config *cfg, const void *packed, int expert,
                       int8_t *gate, int8_t *up, int8_t *down, float *s_gate, float *s_up,
                       float *s_down, void *stream);

/* Router only ([ENGINE] §3.2; [README] sigmoid router; [DEEP] §4.3 router_forward):
 * x [T][H] (fp32 or bf16, per `dtype`) -> ids [T][k] int32 in slot order (descending
 * selection score, ties to the lower expert index) and w [T][k] fp32 routed weights
 * (softmax: p / sum of selected p; grouped: sigmoid / sum of selected sigmoids, times
 * routed_scaling_factor).  With expert_top_p on, the slots it drops have id -1 and
 * weight 0 and the sums run over the kept slots.  T == 0 is a no-op.  T <= the
 * workspace's max_tokens. */
int moe_route_topk(const moe_layer_config *cfg, const void *packed, const void *x,
                   moe_dtype dtype, int T, int32_t *ids, float *w, void *ws, size_t ws_bytes,
                   void *stream);

/* Whole layer ([DEEP] §4.3; [README] 批处理并集 MoE, 量化内核, 整数点积内核):
 * out[t] = shared(x_t) + sum_j w[t][j] * expert_{ids[t][j]}(x_t), fp32 [T][H], with
 * expert(x) = W_down (silu(W_gate x) * (W_up x)).  Also returns ids and w as
 * moe_route_topk does.  x, out, ids and w must not alias. */
int moe_layer_forward(const moe_layer_config *cfg, const void *packed, const void *x,
                      moe_dtype dtype, int T, float *out, int32_t *ids, float *w, void *ws,
                      size_t ws_bytes, void *stream);

/* Expert-parallel share of the layer ("Show HN: 如何在我的低配置电脑上运行 GLM-5.2",
 * 实验性常驻 CUDA 后端: whole experts are placed on devices, an expert is never split; the
 * per-device partial results are added): the router and the permutation run over every
 * expert as in moe_layer_forward, and ids / w receive the full routing, but only routed
 * experts e with expert_begin <= e < expert_end (and the shared expert when with_shared is
 * 1) are computed:
 *   out[t] = [with_shared] shared(x_t) + sum over j with ids[t][j] in [begin, end) of
 *            w[t][j] * expert_{ids[t][j]}(x_t),   fp32 [T][H].
 * Devices that own disjoint expert ranges covering [0, E), exactly one of them with the
 * shared expert, produce partial outputs whose sum is moe_layer_forward's output (up to
 * the order of the fp32 additions).  Only the owned experts' regions of `packed` are read
 * (the router weights and the header always are), so a device may pack just its own
 * experts.  0 <= expert_begin <= expert_end <= n_experts and with_shared in {0, 1}, else
 * MOE_ERR_INVALID_ARG; everything else as moe_layer_forward (same workspace size). */
int moe_layer_forward_experts(const moe_layer_config *cfg, const void *packed, const void *x,
                              moe_dtype dtype, int T, int expert_begin, int expert_end,
                              int with_shared, float *out, int32_t *ids, float *w, void *ws,
                              size_t ws_bytes, void *stream);

/* moe_layer_forward for one layer of a stack of layers ("colibrì 深度拆解" §4.3: a layer's
 * merged output feeds the next layer; "Show HN: 如何在我的低配置电脑上运行 GLM-5.2", 已实现的功能:
 * 异步专家预读, the next weights are read ahead while the current ones are in use): the same
 * forward, whose last kernel (the combine) also starts loading the NEXT layer's router
 * weights and bias (next_cfg, next_packed: that layer's config and packed blob, device,
 * 256-byte aligned) into L2, so that the next layer's router finds them there.  A hint: the
 * results are those of moe_layer_forward, bit for bit.  next_cfg / next_packed NULL or an
 * unsupported next_cfg: MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED before any launch. */
int moe_layer_forward_next(const moe_layer_config *cfg, const void *packed, const void *x,
                           moe_dtype dtype, int T, float *out, int32_t *ids, float *w, void *ws,
                           size_t ws_bytes, const moe_layer_config *next_cfg,
                           const void *next_packed, void *stream);

/* moe_layer_forward with stage timing: records the caller's CUDA events (cudaEvent_t
 * passed as void*) on `stream` around the stages, events[0] before the first kernel and
 * events[i+1] after stage i, for the stages 0 router (logits + top-k), 1 permutation,
 * 2 activation encoding (Q8_0 codes with act_q8_0, else the fp16 tensor-core tiles),
 * 3 gate/up + SwiGLU, 4 down projection, 5 combine.  Decode-sized batches (every gate/up
 * group at most 16 activation rows, router on the GEMV) run selection, permutation and
 * the fp16 token rows inside the router's launch, so stage 0 covers them and stages 1-2
 * are empty.  n_events must be >= 7.  Same results as moe_layer_forward.  The call may be captured into a CUDA graph: while the stream is
 * capturing, the events are recorded as graph nodes (cudaEventRecordExternal), so each
 * replay records them. */
int moe_layer_forward_timed(const moe_layer_config *cfg, const void *packed, const void *x,
                            moe_dtype dtype, int T, float *out, int32_t *ids, float *w, void *ws,
                            size_t ws_bytes, void *const *events, int n_events, void *stream);

/* Allocation-free moe_layer_forward, for callers that cannot provide device scratch
 * (plugin hosts that pass an op only its input and output tensors, serving loops whose
 * device memory is fixed at start-up, code that must not call cudaMalloc because it may
 * synchronise the device).  The pages have no counterpart: it is a property of this
 * library's interface, not of the method.
 * Same kernels and results as moe_layer_forward; the scratch is a file-scope device array
 * of 32 MiB inside the library, held by every GPU that loads the library until the
 * process exits.  Calls are accepted while their workspace (moe_workspace_bytes(cfg, T)) fits
 * in 32 MiB, larger ones are rejected with MOE_ERR_WORKSPACE before any launch (for the
 * DeepSeek-V3-style layer, H = 6144, I = 2048, 256 experts, top-8: T <= 23).  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current and keeps it for later calls on that device; make that first call before
 * any stream capture.  The kept address does not survive cudaDeviceReset (the library's
 * module may load at another address in the new context): do not call this entry point
 * after resetting a device it was used on.  No cudaMalloc,
 * cudaFree or allocating routine is called.  All calls on a device share the one array,
 * which keeps the last call's contents (each call clears the status word it uses first):
 * calls that overlap on the GPU (issued on different streams, or from several host
 * threads without ordering) race on it, so serialise them.  status: optional device int32 that receives the
 * device status word (MOE_OK, MOE_ERR_NUMERIC, MOE_ERR_PACKED ...) at the end of the call,
 * stream-ordered; may be NULL.  It is written only when the call returns MOE_OK: after an
 * error return it keeps whatever it held. */
int moe_layer_forward_static(const moe_layer_config *cfg, const void *packed, const void *x,
                             moe_dtype dtype, int T, float *out, int32_t *ids, float *w,
                             int32_t *status, void *stream);

/* Number of kernel launches one moe_layer_forward makes for `cfg`, hidden states of
 * `dtype` and T tokens (0 for T == 0; negative moe_status for an unsupported config or
 * dtype). */
int moe_forward_launches(const moe_layer_config *cfg, moe_dtype dtype, int T);

/* Synchronise `stream`, then return and clear the device status word of `ws`
 * (MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_NUMERIC, MOE_ERR_PACKED). */
int moe_read_status(void *ws, void *stream);

/* Debug: copy the permutation of the last call that used `ws` (T tokens):
 * offsets [E+1] (exclusive scan of per-expert token counts) and perm [T*k] (slot
 * indices t*k+j ordered by expert, then token; with expert_top_p the slots it dropped are
 * left out and the tail of perm is -1).  Device pointers; stream-ordered. */
int moe_debug_permutation(const moe_layer_config *cfg, const void *ws, int T, int32_t *offsets,
                          int32_t *perm, void *stream);

/* Q8_0 encoding of activations ([README] 整数点积内核), exactly as the layer does it:
 * x [T][n] (fp32 or bf16), n a multiple of 32 -> q [T][n] int8 and d [T][n/32] fp32,
 * d = amax/127 (IEEE fp32 division), q = round-half-away-from-zero(x/d) clamped to
 * [-127,127], d == 0 -> q = 0. */
int moe_q8_0_quantize(const void *x, moe_dtype dtype, int T, int n, int8_t *q, float *d,
                      void *stream);

/* Debug: int32 block dot products of packed int8 weight rows with Q8_0 codes, computed
 * by the same device routine the layer uses.  which: 0 gate, 1 up, 2 down.
 * rows [n_rows] (row indices of that matrix), qa [n_tok][K] int8 (K = the matrix's
 * contraction length) -> dots [n_rows][n_tok][K/32] int32.  Needs weight_bits == 8. */
int moe_debug_block_dots(const moe_layer_config *cfg, const void *packed, int expert, int which,
                         const int32_t *rows, int n_rows, const int8_t *qa, int n_tok,
                         int32_t *dots, void *stream);

/* Per-row weight quantiser ("colibrì 深度拆解" §5.1 quantize_row, per-row scaling): for each
 * row r of w [rows][cols] (fp32 or bf16, device): amax = max |w|, scale[r] = amax / qmax
 * (IEEE fp32 division), q = roundf(w / scale) (IEEE fp32 division, half away from zero)
 * clamped to [-2^(bits-1), qmax], qmax = 2^(bits-1) - 1 (int4 as printed on the page; int8
 * and int2 by the same pattern).  A zero row gives scale 0 and codes 0; a NaN ratio gives
 * code 0.  q [rows][cols] int8 container and scale [rows] fp32 (device) are what
 * moe_pack_weights / moe_pack_expert take.  bits: 8, 4 or 2. */
int moe_quantize_rows(const void *w, moe_dtype dtype, int rows, int cols, int bits, int8_t *q,
                      float *scale, void *stream);

/* Debug: launch a one-block kernel whose bounded wait on a flag that nothing sets gives
 * up after `iterations` polls; it records MOE_ERR_TIMEOUT in the status word of `ws`
 * (read it with moe_read_status).  Exercises the timeout path without a fault. */
int moe_debug_wait_timeout(void *ws, size_t ws_bytes, int iterations, void *stream);

/* The step between two stacked layers ("colibrì 深度拆解" §4.3: a layer's merged output
 * feeds the next layer; the stacking arithmetic is this library's reading): for every
 * token t, resid[t] = x0[t] when x0 is given (the stack's input, bf16; add is then
 * ignored), else resid[t] += add[t] (fp32, in place; add may be NULL), then
 * x_next[t] = bf16(resid[t] / sqrt(mean(resid[t]^2) + eps)), unweighted RMSNorm rounded to
 * nearest: the next layer's input.  resid, add [T][H] fp32, x0 and x_next [T][H] bf16
 * (uint16 bit patterns) are device pointers, 16-byte aligned; H a multiple of 8; eps >= 0.
 * Returns MOE_ERR_INVALID_ARG before any launch when an argument is out of range. */
int moe_residual_rmsnorm(int T, int H, float *resid, const float *add, const uint16_t *x0,
                         float eps, uint16_t *x_next, void *stream);

#ifdef __cplusplus
}
#endif
#endif

// moe_api.cu -- the C ABI entry points: validation, layouts, and the launch sequence of
// one MoE layer forward on one stream (router -> permute -> experts -> combine).
#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "moe_internal.cuh"

namespace moe {

// Host-side per-launch work cached per (kernel, device): the dynamic shared-memory limit
// (the attribute persists once set) and occupancy queries (fixed for a kernel and launch
// shape), so an eager forward costs little more host time than its launches.
static uint64_t func_key(const void *func, int extra) {
  int dev = 0;
  cudaGetDevice(&dev);
  return ((uint64_t)(uintptr_t)func * 1000003ull) ^ ((uint64_t)dev << 56) ^ (uint64_t)extra;
}

void set_dyn_smem(const void *func, int bytes) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> done;
  const uint64_t key = func_key(func, 0);
  std::lock_guard<std::mutex> g(mu);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return;
  cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  done[key] = bytes;
}

template <typename Q>
static int cached(const void *func, int shape, Q query) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> memo;
  const uint64_t key = func_key(func, shape);
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  const int v = query();
  std::lock_guard<std::mutex> g(mu);
  memo[key] = v;
  return v;
}

int cached_blocks_per_sm(const void *func, int threads, size_t smem) {
  return cached(func, (int)smem ^ (threads << 20), [&]() {
    int v = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, func, threads, smem) == cudaSuccess
               ? v
               : 0;
  });
}

DevInfo dev_info() {
  static std::mutex mu;
  static DevInfo cache[64];
  static bool have[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> g(mu);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!have[dev]) {
    DevInfo d{};
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cache[dev] = d;
    have[dev] = true;
  }
  return cache[dev];
}

// tokens per expert group of the CUDA-core expert kernels: the largest power of two
// <= 8 whose fp32 activation rows fit the shared-memory budget, capped near T.
int choose_group_n(const moe_layer_config &c, int T) {
  int Is = c.inter_shared ? c.inter_shared : c.inter;
  long kmax = c.hidden;
  if (c.inter > kmax) kmax = c.inter;
  if (Is > kmax) kmax = Is;
  int g = 8;
  while (g > 1 && (long)g * 4 * kmax > 200 * 1024) g >>= 1;
  int cap = 1;
  while (cap < T && cap < 8) cap <<= 1;
  return g < cap ? g : cap;
}

static int check(const moe_layer_config *c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  int Is = c->inter_shared ? c->inter_shared : c->inter;
  if (c->hidden <= 0 || c->hidden % 128 || c->inter <= 0 || c->inter % 128) return MOE_ERR_UNSUPPORTED;
  if (Is <= 0 || Is % 128) return MOE_ERR_UNSUPPORTED;
  if (c->hidden > 32768 || c->inter > 32768 || Is > 32768) return MOE_ERR_UNSUPPORTED;
  if (c->top_k < 1 || c->top_k > 16 || c->n_experts < c->top_k || c->n_experts > 256)
    return MOE_ERR_UNSUPPORTED;
  if (c->n_shared != 0 && c->n_shared != 1) return MOE_ERR_UNSUPPORTED;
  if (c->norm_topk != 0 && c->norm_topk != 1) return MOE_ERR_UNSUPPORTED;
  if (!std::isfinite(c->routed_scaling_factor)) return MOE_ERR_UNSUPPORTED;
  if (c->router == MOE_ROUTER_SIGMOID_GROUPED) {
    if (c->n_group < 1 || c->n_group > 32 || c->n_experts % c->n_group) return MOE_ERR_UNSUPPORTED;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_UNSUPPORTED;
    if (c->topk_group * (c->n_experts / c->n_group) < c->top_k) return MOE_ERR_UNSUPPORTED;
  } else if (c->router != MOE_ROUTER_SOFTMAX) {
    return MOE_ERR_UNSUPPORTED;
  }
  if (c->weight_bits != 4 && c->weight_bits != 8 && c->weight_bits != 2) return MOE_ERR_UNSUPPORTED;
  if (c->act_q8_0 != 0 && c->act_q8_0 != 1) return MOE_ERR_UNSUPPORTED;
  if (c->act_q8_0 && c->weight_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (!(c->expert_top_p >= 0.f) || !std::isfinite(c->expert_top_p)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// largest T one call supports (slot positions and token indices stay well inside int)
static bool tokens_supported(const moe_layer_config &c, int T) {
  if (T > 65535) return false;
  return (long)permute_smem(T, c.n_experts) <= (long)dev_info().smem_optin;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char *moe_status_str(int s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_NUMERIC: return "MOE_ERR_NUMERIC";
    case MOE_ERR_PACKED: return "MOE_ERR_PACKED";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_check_config(const moe_layer_config *cfg) { return check(cfg); }

size_t moe_packed_bytes(const moe_layer_config *cfg) {
  if (check(cfg) != MOE_OK) return 0;
  return (size_t)pack_layout(*cfg).total;
}

size_t moe_workspace_bytes(const moe_layer_config *cfg, int max_tokens) {
  if (check(cfg) != MOE_OK || max_tokens < 0 || max_tokens > (1 << 20)) return 0;
  return (size_t)ws_layout(*cfg, max_tokens < 1 ? 1 : max_tokens).total;
}

int moe_pack_router(const moe_layer_config *cfg, const float *router_w, const float *router_bias,
                    void *packed, size_t packed_bytes, void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (!router_w || !packed || !aligned(packed, 256)) return MOE_ERR_INVALID_ARG;
  PackLayout P = pack_layout(*cfg);
  if (packed_bytes < P.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *base = (uint8_t *)packed;
  if ((r = launch_write_header(*cfg, base, st))) return r;
  size_t wbytes = (size_t)cfg->n_experts * cfg->hidden * 4;
  if (cudaMemcpyAsync(base + P.router_w_off, router_w, wbytes, cudaMemcpyDeviceToDevice, st))
    return MOE_ERR_CUDA;
  size_t bbytes = (size_t)cfg->n_experts * 4;
  cudaError_t e = router_bias
      ? cudaMemcpyAsync(base + P.router_b_off, router_bias, bbytes, cudaMemcpyDeviceToDevice, st)
      : cudaMemsetAsync(base + P.router_b_off, 0, bbytes, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return launch_router_tiles(*cfg, (const float *)(base + P.router_w_off),
                             base + P.router_t_off, st);
}

int moe_pack_expert(const moe_layer_config *cfg, int expert, const int8_t *gate, const int8_t *up,
                    const int8_t *down, const float *s_gate, const float *s_up, const float *s_down,
                    void *packed, size_t packed_bytes, void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (!packed || !gate || !up || !down || !s_gate || !s_up || !s_down || !aligned(packed, 256))
    return MOE_ERR_INVALID_ARG;
  if (expert < 0 || expert > cfg->n_experts || (expert == cfg->n_experts && !cfg->n_shared))
    return MOE_ERR_INVALID_ARG;
  PackLayout P = pack_layout(*cfg);
  if (packed_bytes < P.total) return MOE_ERR_WORKSPACE;
  bool sh = expert == cfg->n_experts;
  uint8_t *base = (uint8_t *)packed + (sh ? P.shared_off : P.experts_off + P.routed.bytes * expert);
  return launch_pack_expert(*cfg, sh ? P.shared : P.routed, gate, up, down, s_gate, s_up, s_down,
                            base, (cudaStream_t)stream);
}

int moe_pack_weights(const moe_layer_config *cfg, const moe_weight_src *src, void *packed,
                     size_t packed_bytes, void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (!src) return MOE_ERR_INVALID_ARG;
  if ((r = moe_pack_router(cfg, src->router_w, src->router_bias, packed, packed_bytes, stream)))
    return r;
  const size_t H = cfg->hidden, I = cfg->inter;
  for (int e = 0; e < cfg->n_experts; e++) {
    if (!src->gate || !src->up || !src->down || !src->s_gate || !src->s_up || !src->s_down)
      return MOE_ERR_INVALID_ARG;
    r = moe_pack_expert(cfg, e, src->gate + e * I * H, src->up + e * I * H, src->down + e * H * I,
                        src->s_gate + e * I, src->s_up + e * I, src->s_down + e * H, packed,
                        packed_bytes, stream);
    if (r) return r;
  }
  if (cfg->n_shared)
    return moe_pack_expert(cfg, cfg->n_experts, src->sh_gate, src->sh_up, src->sh_down,
                           src->sh_s_gate, src->sh_s_up, src->sh_s_down, packed, packed_bytes,
                           stream);
  return MOE_OK;
}

int moe_unpack_weights(const moe_layer_config *cfg, const void *packed, int expert, int8_t *gate,
                       int8_t *up, int8_t *down, float *s_gate, float *s_up, float *s_down,
                       void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (!packed || !aligned(packed, 256)) return MOE_ERR_INVALID_ARG;
  if (expert < 0 || expert > cfg->n_experts || (expert == cfg->n_experts && !cfg->n_shared))
    return MOE_ERR_INVALID_ARG;
  PackLayout P = pack_layout(*cfg);
  bool sh = expert == cfg->n_experts;
  const uint8_t *base =
      (const uint8_t *)packed + (sh ? P.shared_off : P.experts_off + P.routed.bytes * expert);
  return launch_unpack_expert(*cfg, sh ? P.shared : P.routed, base, gate, up, down, s_gate, s_up,
                              s_down, (cudaStream_t)stream);
}

static int common_args(const moe_layer_config *cfg, const void *packed, const void *x,
                       moe_dtype dt, int T, int32_t *ids, float *w, void *ws, size_t ws_bytes,
                       WsLayout *W) {
  int r = check(cfg);
  if (r) return r;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (dt != MOE_DT_F32 && dt != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!packed || !x || !ids || !w || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(ids, 4) ||
      !aligned(w, 4))
    return MOE_ERR_INVALID_ARG;
  *W = ws_layout(*cfg, T, dt == MOE_DT_F32 ? 2 : 1);
  if (ws_bytes < W->total) return MOE_ERR_WORKSPACE;
  if (!tokens_supported(*cfg, T)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int moe_route_topk(const moe_layer_config *cfg, const void *packed, const void *x, moe_dtype dtype,
                   int T, int32_t *ids, float *w, void *ws, size_t ws_bytes, void *stream) {
  WsLayout W;
  int r = common_args(cfg, packed, x, dtype, T, ids, w, ws, ws_bytes, &W);
  if (r || T == 0) return r;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, sizeof(Ctrl), st) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_router(*cfg, (const uint8_t *)packed, x, dtype, T, ids, w, (uint8_t *)ws, W, st);
}

// One forward; share (optional): {e0, e1, shared} restricts the computed experts to an
// expert-parallel share of the layer.
static int forward_impl(const moe_layer_config *cfg, const void *packed, const void *x,
                        moe_dtype dtype, int T, float *out, int32_t *ids, float *w, void *ws,
                        size_t ws_bytes, void *const *ev, void *stream,
                        const int *share = nullptr, const uint8_t *pf = nullptr,
                        uint64_t pf_bytes = 0) {
  WsLayout W;
  int r = common_args(cfg, packed, x, dtype, T, ids, w, ws, ws_bytes, &W);
  if (r || T == 0) return r;
  if (share) {
    W.e0 = share[0];
    W.e1 = share[1];
    W.shared = share[2] != 0 && cfg->n_shared != 0;
  }
  if (!out || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *wsb = (uint8_t *)ws;
  const uint8_t *pk = (const uint8_t *)packed;
  auto mark = [&](int i) {
    return ev ? record_stage_event(ev[i], st) == cudaSuccess : true;
  };
  // decode-sized batches: selection, permutation and token rows in the router's launch
  const bool fused = fused_front(*cfg, T, W.pieces);
  if (cudaMemsetAsync(ws, 0, sizeof(Ctrl), st) != cudaSuccess || !mark(0)) return MOE_ERR_CUDA;
  if ((r = launch_router(*cfg, pk, x, dtype, T, ids, w, wsb, W, st, fused))) return r;
  if (!mark(1)) return MOE_ERR_CUDA;
  if (!fused && (r = launch_permute(*cfg, T, ids, wsb, W, st))) return r;
  if (!mark(2)) return MOE_ERR_CUDA;
  if (cfg->act_q8_0 && (r = launch_quant_x(*cfg, x, dtype, T, wsb, W, st))) return r;
  // stage 2 ends when the activations are encoded: Q8_0 codes, or the tensor-core path's
  // fp16 tiles or token rows (written inside launch_experts unless the front wrote them)
  if ((r = launch_experts(*cfg, pk, x, dtype, T, wsb, W, st, ev ? ev[3] : nullptr,
                          ev ? ev[4] : nullptr, fused)))
    return r;
  if (!mark(5)) return MOE_ERR_CUDA;
  if ((r = launch_combine(*cfg, T, w, out, wsb, W, st, pf, pf_bytes))) return r;
  return mark(6) ? MOE_OK : MOE_ERR_CUDA;
}

int moe_layer_forward(const moe_layer_config *cfg, const void *packed, const void *x,
                      moe_dtype dtype, int T, float *out, int32_t *ids, float *w, void *ws,
                      size_t ws_bytes, void *stream) {
  return forward_impl(cfg, packed, x, dtype, T, out, ids, w, ws, ws_bytes, nullptr, stream);
}

int moe_layer_forward_experts(const moe_layer_config *cfg, const void *packed, const void *x,
                              moe_dtype dtype, int T, int expert_begin, int expert_end,
                              int with_shared, float *out, int32_t *ids, float *w, void *ws,
                              size_t ws_bytes, void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (expert_begin < 0 || expert_end < expert_begin || expert_end > cfg->n_experts ||
      (with_shared != 0 && with_shared != 1))
    return MOE_ERR_INVALID_ARG;
  const int share[3] = {expert_begin, expert_end, with_shared};
  return forward_impl(cfg, packed, x, dtype, T, out, ids, w, ws, ws_bytes, nullptr, stream,
                      share);
}

int moe_layer_forward_next(const moe_layer_config *cfg, const void *packed, const void *x,
                           moe_dtype dtype, int T, float *out, int32_t *ids, float *w, void *ws,
                           size_t ws_bytes, const moe_layer_config *next_cfg,
                           const void *next_packed, void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (!next_cfg || !next_packed) return MOE_ERR_INVALID_ARG;
  if ((r = check(next_cfg))) return r;
  if (!aligned(next_packed, 256)) return MOE_ERR_INVALID_ARG;
  // the next layer's router weights and bias (contiguous in its blob)
  const PackLayout P = pack_layout(*next_cfg);
  const uint64_t bytes = align_up((uint64_t)next_cfg->n_experts * 4, 16) +
                         (P.router_b_off - P.router_w_off);
  return forward_impl(cfg, packed, x, dtype, T, out, ids, w, ws, ws_bytes, nullptr, stream, nullptr,
                      (const uint8_t *)next_packed + P.router_w_off, bytes);
}

int moe_layer_forward_timed(const moe_layer_config *cfg, const void *packed, const void *x,
                            moe_dtype dtype, int T, float *out, int32_t *ids, float *w, void *ws,
                            size_t ws_bytes, void *const *events, int n_events, void *stream) {
  if (!events || n_events < 7) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 7; i++)
    if (!events[i]) return MOE_ERR_INVALID_ARG;
  return forward_impl(cfg, packed, x, dtype, T, out, ids, w, ws, ws_bytes, events, stream);
}

int moe_forward_launches(const moe_layer_config *cfg, moe_dtype dtype, int T) {
  int r = check(cfg);
  if (r) return r;
  if (dtype != MOE_DT_F32 && dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (T <= 0) return 0;
  const int pieces = dtype == MOE_DT_F32 ? 2 : 1;
  // decode front (router, selection, permutation, token rows), gate/up, down, combine
  if (fused_front(*cfg, T, pieces)) return 4;
  // router logits + selection, permute, [Q8_0 encode], [activation tiles or token rows],
  // gate/up, down, combine
  return 2 + 1 + (cfg->act_q8_0 ? 1 : 0) + (use_tc(*cfg) ? 1 : 0) + 2 + 1;
}

int moe_read_status(void *ws, void *stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int s = 0;
  if (cudaMemcpy(&s, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemset(ws, 0, 2 * sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  return s;
}

int moe_debug_permutation(const moe_layer_config *cfg, const void *ws, int T, int32_t *offsets,
                          int32_t *perm, void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (!ws || !offsets || !perm || T <= 0) return MOE_ERR_INVALID_ARG;
  WsLayout W = ws_layout(*cfg, T);
  cudaStream_t st = (cudaStream_t)stream;
  const uint8_t *b = (const uint8_t *)ws;
  if (cudaMemcpyAsync(offsets, b + W.offsets, (cfg->n_experts + 1) * 4, cudaMemcpyDeviceToDevice, st))
    return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(perm, b + W.perm, (size_t)T * cfg->top_k * 4, cudaMemcpyDeviceToDevice, st))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_q8_0_quantize(const void *x, moe_dtype dtype, int T, int n, int8_t *q, float *d,
                      void *stream) {
  if (T < 0 || n <= 0 || n % 32) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_DT_F32 && dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !q || !d) return MOE_ERR_INVALID_ARG;
  return launch_q8_quantize(x, dtype, T, n, q, d, (cudaStream_t)stream);
}

int moe_quantize_rows(const void *w, moe_dtype dtype, int rows, int cols, int bits, int8_t *q,
                      float *scale, void *stream) {
  if (rows < 0 || cols <= 0 || (bits != 8 && bits != 4 && bits != 2)) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_DT_F32 && dtype != MOE_DT_BF16) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!w || !q || !scale) return MOE_ERR_INVALID_ARG;
  return launch_quantize_rows(w, dtype, rows, cols, bits, q, scale, (cudaStream_t)stream);
}

int moe_debug_block_dots(const moe_layer_config *cfg, const void *packed, int expert, int which,
                         const int32_t *rows, int n_rows, const int8_t *qa, int n_tok,
                         int32_t *dots, void *stream) {
  int r = check(cfg);
  if (r) return r;
  if (cfg->weight_bits != 8) return MOE_ERR_UNSUPPORTED;
  if (!packed || !rows || !qa || !dots || n_rows <= 0 || n_tok <= 0) return MOE_ERR_INVALID_ARG;
  if (which < 0 || which > 2) return MOE_ERR_INVALID_ARG;
  if (expert < 0 || expert > cfg->n_experts || (expert == cfg->n_experts && !cfg->n_shared))
    return MOE_ERR_INVALID_ARG;
  PackLayout P = pack_layout(*cfg);
  bool sh = expert == cfg->n_experts;
  const ExpertLayout &L = sh ? P.shared : P.routed;
  const uint8_t *base =
      (const uint8_t *)packed + (sh ? P.shared_off : P.experts_off + P.routed.bytes * expert);
  const uint8_t *mat = base + (which == 2 ? L.down_off : L.gu_off);
  int K = which == 2 ? L.inter : cfg->hidden;
  int nrows = which == 2 ? cfg->hidden : L.inter;
  return launch_block_dots(*cfg, mat, K, nrows, which, rows, n_rows, qa, n_tok, dots,
                           (cudaStream_t)stream);
}

int moe_debug_wait_timeout(void *ws, size_t ws_bytes, int iterations, void *stream) {
  if (!ws || ws_bytes < sizeof(Ctrl) || iterations < 1) return MOE_ERR_INVALID_ARG;
  return launch_debug_wait((uint8_t *)ws, iterations, (cudaStream_t)stream);
}

}  // extern "C"

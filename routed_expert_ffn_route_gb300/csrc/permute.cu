// permute.cu -- the token-by-expert permutation of the batched union forward
// ("Show HN: 如何在我的低配置电脑上运行 GLM-5.2", 已实现的功能: 批处理并集 MoE -- each unique
// expert of the batch is read once and applied to every position routed to it).
//
// One CTA of 1024 threads:
//  1. per 32-token chunk, a bitmask per expert of the chunk's tokens that chose it
//     (shared-memory atomicOr), giving per-chunk per-expert counts;
//  2. exclusive scans: per-expert offsets (expert_offsets), per-expert chunk bases, and
//     the work-list positions (first group of each expert);
//  3. stable scatter: the rank of slot (t, j) inside expert e is its chunk base plus
//     popc(mask & lanes-below), so perm lists t*k+j ordered by (expert, token) exactly,
//     without any order decided by atomics;
//  4. the work list of the expert kernels: groups of at most GN rows of one expert
//     (shared-expert groups first, over the tokens in order; only the experts of the
//     call's share, see WsLayout), each with its first row in
//     the tensor-core activation tiles (row index + 7 x group index: room to pad each
//     group's rows to a multiple of 8).
#include "dev.cuh"
#include "moe_internal.cuh"

namespace moe {

// shared memory: masks [32][E] u32 | chunk bases [n_chunks][E] u16 | 2 x [E+1] int
__global__ void __launch_bounds__(1024) permute_kernel(int T, int k, int E, int n_shared, int GN,
                                                       int P, int e0, int e1, int sh_on,
                                                       const int32_t *ids,
                                                       int32_t *offsets_out, int32_t *perm,
                                                       int32_t *slot_pos, Group *groups,
                                                       Ctrl *ctrl) {
  extern __shared__ uint32_t sm[];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_chunks = (T + 31) / 32;
  uint32_t *masks = sm;                                    // [32][E]
  uint16_t *cbase = (uint16_t *)(sm + 32 * E);             // [n_chunks][E]
  int *offs = (int *)(cbase + ((n_chunks * E + 1) & ~1));  // [E+1] token offsets
  int *gstart = offs + (E + 1);                            // [E+1] first group
  uint32_t *my = masks + warp * E;

  // 1. per-chunk per-expert counts
  for (int c = warp; c < n_chunks; c += 32) {
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    int t = c * 32 + lane;
    if (t < T)
      for (int j = 0; j < k; j++)
        if (ids[t * k + j] >= 0) atomicOr(&my[ids[t * k + j]], 1u << lane);
    __syncwarp();
    for (int e = lane; e < E; e += 32) cbase[c * E + e] = (uint16_t)__popc(my[e]);
    __syncwarp();
  }
  __syncthreads();
  // 2a. per-expert totals and chunk bases (relative to the expert's start)
  if (threadIdx.x < E) {
    int e = threadIdx.x, run = 0;
    for (int c = 0; c < n_chunks; c++) {
      int v = cbase[c * E + e];
      cbase[c * E + e] = (uint16_t)run;
      run += v;
    }
    offs[e] = run;  // counts for now
    // groups of this expert (none for an expert outside the call's share)
    gstart[e] = e >= e0 && e < e1 ? (run + GN - 1) / GN : 0;
  }
  __syncthreads();
  // 2b. exclusive scans of the per-expert counts and group counts (one warp, E <= 256)
  if (warp == 0) {
    int *arr[2] = {offs, gstart};
    int per = (E + 31) / 32;
    int s[2] = {0, 0};
    for (int i = 0; i < per; i++) {
      int e = lane * per + i;
      if (e < E)
        for (int q = 0; q < 2; q++) s[q] += arr[q][e];
    }
    int inc[2];
    for (int q = 0; q < 2; q++) {
      inc[q] = s[q];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, inc[q], o);
        if (lane >= o) inc[q] += v;
      }
    }
    int r[2];
    for (int q = 0; q < 2; q++) r[q] = inc[q] - s[q];
    for (int i = 0; i < per; i++) {
      int e = lane * per + i;
      if (e < E)
        for (int q = 0; q < 2; q++) {
          int v = arr[q][e];
          arr[q][e] = r[q];
          r[q] += v;
        }
    }
    if (lane == 31)
      for (int q = 0; q < 2; q++) arr[q][E] = inc[q];
  }
  __syncthreads();
  const int ns = n_shared && sh_on ? (T + GN - 1) / GN : 0;
  const int rbase = n_shared ? T : 0;  // routed rows follow the shared expert's T rows
  if (threadIdx.x == 0) ctrl->n_groups = ns + gstart[E];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets_out[e] = offs[e];
  // slots dropped by top-p (id -1) are not permuted: the tail of perm is -1
  for (int i = offs[E] + threadIdx.x; i < T * k; i += blockDim.x) perm[i] = -1;
  // 3. stable scatter
  for (int c = warp; c < n_chunks; c += 32) {
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    int t = c * 32 + lane;
    if (t < T)
      for (int j = 0; j < k; j++)
        if (ids[t * k + j] >= 0) atomicOr(&my[ids[t * k + j]], 1u << lane);
    __syncwarp();
    if (t < T) {
      unsigned below = (1u << lane) - 1u;
      for (int j = 0; j < k; j++) {
        int e = ids[t * k + j];
        if (e < 0) {  // dropped by top-p
          slot_pos[t * k + j] = -1;
          continue;
        }
        int pos = offs[e] + cbase[c * E + e] + __popc(my[e] & below);
        perm[pos] = t * k + j;
        // a slot of an expert outside the call's share has no output row to combine
        slot_pos[t * k + j] = e >= e0 && e < e1 ? pos : -1;
      }
    }
    __syncwarp();
  }
  // 4. groups
  for (int i = threadIdx.x; i < ns; i += blockDim.x)
    groups[i] = Group{E, i * GN, min(GN, T - i * GN), P * i * GN + 7 * i, i * GN + 7 * i, 0, 0, 0};
  for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
    int n = offs[e + 1] - offs[e];
    int g0 = ns + gstart[e];
    for (int g = 0; g * GN < n; g++)
      groups[g0 + g] = Group{e, offs[e] + g * GN, min(GN, n - g * GN),
                             P * (rbase + offs[e] + g * GN) + 7 * (g0 + g),
                             rbase + offs[e] + g * GN + 7 * (g0 + g), 0, 0, 0};
  }
}

size_t permute_smem(int T, int E) {
  int n_chunks = (T + 31) / 32;
  return (size_t)32 * E * 4 + (size_t)((n_chunks * E + 1) & ~1) * 2 + (size_t)2 * (E + 1) * 4;
}

int launch_permute(const moe_layer_config &c, int T, const int32_t *ids, uint8_t *ws,
                   const WsLayout &W, cudaStream_t st) {
  size_t smem = permute_smem(T, c.n_experts);
  DevInfo d = dev_info();
  if ((long)smem > d.smem_optin) return MOE_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    set_dyn_smem((const void *)permute_kernel, (int)smem);
  if (launch_pdl(permute_kernel, dim3(1), dim3(1024), smem, st, T, c.top_k, c.n_experts,
                 c.n_shared, W.group_n, W.pieces, W.e0, W.e1, W.shared ? 1 : 0, ids,
                 (int32_t *)(ws + W.offsets),
                 (int32_t *)(ws + W.perm), (int32_t *)(ws + W.slot_pos), (Group *)(ws + W.groups),
                 (Ctrl *)(ws + W.ctrl)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// permute.cu -- the token-by-expert permutation of the batched union forward
// ("Show HN: 如何在我的低配置电脑上运行 GLM-5.2", 已实现的功能: 批处理并集 MoE -- each unique
// expert of the batch is read once and applied to every position routed to it).
//
// One CTA of 1024 threads:
//  1. per 32-token chunk, a bitmask per expert of the chunk's tokens that chose it
//     (shared-memory atomicOr), giving per-chunk per-expert counts;
//  2. exclusive scans: per-expert offsets (expert_offsets), per-expert chunk bases;
//  3. stable scatter: the rank of slot (t, j) inside expert e is its chunk base plus
//     popc(mask & lanes-below), so perm lists t*k+j ordered by (expert, token) exactly,
//     without any order decided by atomics;
//  4. the work list of the expert kernels: groups of at most GN rows of one expert
//     (shared-expert groups first, over the tokens in order).
#include "dev.cuh"
#include "moe_internal.cuh"

namespace moe {

// shared memory: masks [32][E] u32 | chunk bases [n_chunks][E] u16 | offs [E+1] | gstart [E+1]
__global__ void __launch_bounds__(1024) permute_kernel(int T, int k, int E, int n_shared, int GN,
                                                       const int32_t *ids, int32_t *offsets_out,
                                                       int32_t *perm, int32_t *slot_pos,
                                                       Group *groups, Ctrl *ctrl) {
  extern __shared__ uint32_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_chunks = (T + 31) / 32;
  uint32_t *masks = sm;                                    // [32][E]
  uint16_t *cbase = (uint16_t *)(sm + 32 * E);             // [n_chunks][E]
  int *offs = (int *)(cbase + ((n_chunks * E + 1) & ~1));  // [E+1]
  int *gstart = offs + (E + 1);                            // [E+1]
  uint32_t *my = masks + warp * E;

  // 1. per-chunk per-expert counts
  for (int c = warp; c < n_chunks; c += 32) {
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    int t = c * 32 + lane;
    if (t < T)
      for (int j = 0; j < k; j++) atomicOr(&my[ids[t * k + j]], 1u << lane);
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
    offs[e] = run;                          // count for now
    gstart[e] = (run + GN - 1) / GN;        // groups of this expert
  }
  __syncthreads();
  // 2b. exclusive scans of counts and group counts (one warp, E <= 256)
  if (warp == 0) {
    int per = (E + 31) / 32;
    int s0 = 0, s1 = 0;
    for (int i = 0; i < per; i++) {
      int e = lane * per + i;
      if (e < E) { s0 += offs[e]; s1 += gstart[e]; }
    }
    int i0 = s0, i1 = s1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int a = __shfl_up_sync(0xffffffffu, i0, o), b = __shfl_up_sync(0xffffffffu, i1, o);
      if (lane >= o) { i0 += a; i1 += b; }
    }
    int r0 = i0 - s0, r1 = i1 - s1;  // exclusive
    for (int i = 0; i < per; i++) {
      int e = lane * per + i;
      if (e < E) {
        int c0 = offs[e], c1 = gstart[e];
        offs[e] = r0;
        gstart[e] = r1;
        r0 += c0;
        r1 += c1;
      }
    }
    if (lane == 31) {
      offs[E] = i0;
      gstart[E] = i1;
    }
  }
  __syncthreads();
  const int ns = n_shared ? (T + GN - 1) / GN : 0;
  if (threadIdx.x == 0) ctrl->n_groups = ns + gstart[E];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) offsets_out[e] = offs[e];
  // 3. stable scatter
  for (int c = warp; c < n_chunks; c += 32) {
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    int t = c * 32 + lane;
    if (t < T)
      for (int j = 0; j < k; j++) atomicOr(&my[ids[t * k + j]], 1u << lane);
    __syncwarp();
    if (t < T) {
      unsigned below = (1u << lane) - 1u;
      for (int j = 0; j < k; j++) {
        int e = ids[t * k + j];
        int pos = offs[e] + cbase[c * E + e] + __popc(my[e] & below);
        perm[pos] = t * k + j;
        slot_pos[t * k + j] = pos;
      }
    }
    __syncwarp();
  }
  // 4. groups
  for (int i = threadIdx.x; i < ns; i += blockDim.x)
    groups[i] = Group{E, i * GN, min(GN, T - i * GN), 0};
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int n = offs[e + 1] - offs[e];
    int g0 = ns + gstart[e];
    for (int g = 0; g * GN < n; g++)
      groups[g0 + g] = Group{e, offs[e] + g * GN, min(GN, n - g * GN), 0};
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
    cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  permute_kernel<<<1, 1024, smem, st>>>(
      T, c.top_k, c.n_experts, c.n_shared, W.group_n, ids, (int32_t *)(ws + W.offsets),
      (int32_t *)(ws + W.perm), (int32_t *)(ws + W.slot_pos), (Group *)(ws + W.groups),
      (Ctrl *)(ws + W.ctrl));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

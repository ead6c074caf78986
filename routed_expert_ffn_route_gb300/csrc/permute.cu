// permute.cu -- the token-by-expert permutation of the batched union forward
// ("Show HN: 如何在我的低配置电脑上运行 GLM-5.2", 已实现的功能: 批处理并集 MoE -- each unique
// expert of the batch is read once and applied to every position routed to it).
//
// One CTA per run of 32-token chunks; no CTA waits on another:
//  1. every CTA counts the slots of each expert over the whole batch and over the tokens
//     before its first chunk (the id array is small and L2-resident);
//  2. exclusive scans over the experts: per-expert offsets (expert_offsets) and the
//     work-list positions (first group of each expert);
//  3. stable scatter, chunk by chunk: slot (t, j) of expert e goes to offset[e] + the
//     expert's slots in earlier chunks + popc(the chunk's mask of e & lanes below t), so
//     perm lists t*k+j ordered by (expert, token) exactly, without any order decided by
//     atomics;
//  4. CTA 0 writes the offsets, the group count, the -1 tail of perm and the work list of
//     the expert kernels: groups of at most GN rows of one expert (shared-expert groups
//     first, over the tokens in order; only the experts of the call's share, see
//     WsLayout), each with its first row in the tensor-core activation tiles (row index +
//     7 x group index: room to pad each group's rows to a multiple of 8).
#include <algorithm>

#include "dev.cuh"
#include "moe_internal.cuh"

namespace moe {

constexpr int kPermThreads = 1024;
constexpr int kPermChunk = 32;  // tokens per chunk (one per lane of the scattering warp)

// shared memory: 5 arrays of E (+1) ints and the ids of one chunk
__global__ void __launch_bounds__(kPermThreads) permute_kernel(int T, int k, int E, int n_shared, int GN,
                                                               int P, int e0, int e1, int sh_on,
                                                               int chunks_per_cta,
                                                               const int32_t *ids,
                                                               int32_t *offsets_out, int32_t *perm,
                                                               int32_t *slot_pos, Group *groups,
                                                               Ctrl *ctrl) {
  extern __shared__ int psm[];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int *tot = psm;                                 // [E] slots per expert, whole batch
  int *before = tot + E;                          // [E] slots per expert before the chunk
  int *offs = before + E;                         // [E+1] first position per expert
  int *gstart = offs + (E + 1);                   // [E+1] first group per expert
  uint32_t *mask = (uint32_t *)(gstart + E + 1);  // [E] the chunk's tokens per expert
  int *cid = (int *)(mask + E);                   // [32 k] the chunk's expert ids
  const int n = T * k;
  const int c0 = blockIdx.x * chunks_per_cta;
  const int c1 = min(c0 + chunks_per_cta, (T + kPermChunk - 1) / kPermChunk);
  const int lo = c0 * kPermChunk * k;  // slots of the tokens before the first chunk

  // 1. counts (eight independent loads per thread in flight before their atomics)
  for (int e = tid; e < E; e += blockDim.x) tot[e] = before[e] = 0, mask[e] = 0u;
  __syncthreads();
  constexpr int kU = 8;
  for (int i0 = 0; i0 < n; i0 += kU * kPermThreads) {
    int ev[kU];
#pragma unroll
    for (int u = 0; u < kU; u++) {
      const int i = i0 + u * kPermThreads + tid;
      ev[u] = i < n ? ids[i] : -1;
    }
#pragma unroll
    for (int u = 0; u < kU; u++) {
      const int i = i0 + u * kPermThreads + tid;
      if (ev[u] >= 0) {
        atomicAdd(&tot[ev[u]], 1);
        if (i < lo) atomicAdd(&before[ev[u]], 1);
      }
    }
  }
  __syncthreads();
  // 2. exclusive scans of the slot counts and group counts (one warp, E <= 256)
  if (warp == 0) {
    const int per = (E + 31) / 32;
    int s0 = 0, s1 = 0;
    for (int i = 0; i < per; i++) {
      const int e = lane * per + i;
      if (e < E) {
        s0 += tot[e];
        // groups of this expert (none for an expert outside the call's share)
        s1 += e >= e0 && e < e1 ? (tot[e] + GN - 1) / GN : 0;
      }
    }
    int i0 = s0, i1 = s1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v0 = __shfl_up_sync(0xffffffffu, i0, o), v1 = __shfl_up_sync(0xffffffffu, i1, o);
      if (lane >= o) i0 += v0, i1 += v1;
    }
    int r0 = i0 - s0, r1 = i1 - s1;
    for (int i = 0; i < per; i++) {
      const int e = lane * per + i;
      if (e < E) {
        offs[e] = r0;
        gstart[e] = r1;
        r0 += tot[e];
        r1 += e >= e0 && e < e1 ? (tot[e] + GN - 1) / GN : 0;
      }
    }
    if (lane == 31) offs[E] = i0, gstart[E] = i1;
  }
  __syncthreads();
  // 3. stable scatter of this CTA's chunks (one warp, a token per lane; the chunk's ids are
  //    staged in shared memory by coalesced loads)
  if (warp == 0) {
    const unsigned below = (1u << lane) - 1u;
    for (int c = c0; c < c1; c++) {
      const int t = c * kPermChunk + lane;
      const int s0 = c * kPermChunk * k, cn = min(kPermChunk * k, n - s0);
      for (int i = lane; i < cn; i += 32) cid[i] = ids[s0 + i];
      __syncwarp();
      const int *my_ids = cid + lane * k;  // this lane's token's slots
      if (t < T)
        for (int j = 0; j < k; j++) {
          const int e = my_ids[j];
          if (e >= 0) atomicOr(&mask[e], 1u << lane);
        }
      __syncwarp();
      if (t < T)
        for (int j = 0; j < k; j++) {
          const int e = my_ids[j];
          if (e < 0) {  // dropped by top-p
            slot_pos[t * k + j] = -1;
            continue;
          }
          const int pos = offs[e] + before[e] + __popc(mask[e] & below);
          perm[pos] = t * k + j;
          // a slot of an expert outside the call's share has no output row to combine
          slot_pos[t * k + j] = e >= e0 && e < e1 ? pos : -1;
        }
      __syncwarp();
      // the chunk's slots now come before the next chunk's; its masks are cleared
      if (t < T)
        for (int j = 0; j < k; j++) {
          const int e = my_ids[j];
          if (e >= 0) {
            const uint32_t m = mask[e];
            if (m) {
              // the lowest lane of the expert's mask moves its count forward
              if ((m & below) == 0) before[e] += __popc(m), mask[e] = 0u;
            }
          }
        }
      __syncwarp();
    }
  }
  if (blockIdx.x != 0) return;
  // 4. CTA 0: offsets, group count, perm tail, work list
  const int ns = n_shared && sh_on ? (T + GN - 1) / GN : 0;
  const int rbase = n_shared ? T : 0;  // routed rows follow the shared expert's T rows
  if (tid == 0) ctrl->n_groups = ns + gstart[E];
  for (int e = tid; e <= E; e += blockDim.x) offsets_out[e] = offs[e];
  // slots dropped by top-p (id -1) are not permuted: the tail of perm is -1
  for (int i = offs[E] + tid; i < n; i += blockDim.x) perm[i] = -1;
  for (int i = tid; i < ns; i += blockDim.x)
    groups[i] = Group{E, i * GN, min(GN, T - i * GN), P * i * GN + 7 * i, i * GN + 7 * i, 0, 0, 0};
  for (int e = e0 + tid; e < e1; e += blockDim.x) {
    const int cnt = offs[e + 1] - offs[e];
    const int g0 = ns + gstart[e];
    for (int g = 0; g * GN < cnt; g++)
      groups[g0 + g] = Group{e, offs[e] + g * GN, min(GN, cnt - g * GN),
                             P * (rbase + offs[e] + g * GN) + 7 * (g0 + g),
                             rbase + offs[e] + g * GN + 7 * (g0 + g), 0, 0, 0};
  }
}

size_t permute_smem(int T, int E) {
  (void)T;  // the tables are per expert; the token count only sets the grid
  return (size_t)(5 * E + 2 + kPermChunk * 16) * 4;  // top_k <= 16
}

int launch_permute(const moe_layer_config &c, int T, const int32_t *ids, uint8_t *ws,
                   const WsLayout &W, cudaStream_t st) {
  const size_t smem = permute_smem(T, c.n_experts);
  DevInfo d = dev_info();
  if ((long)smem > d.smem_optin) return MOE_ERR_UNSUPPORTED;
  // a CTA per chunk up to two per SM; past that each CTA scatters a run of chunks (every
  // CTA reads the whole id array once)
  const int n_chunks = (T + kPermChunk - 1) / kPermChunk;
  const int per = std::max(1, (n_chunks + 2 * d.sms - 1) / (2 * d.sms));
  const int ctas = std::max(1, (n_chunks + per - 1) / per);
  if (launch_pdl(permute_kernel, dim3(ctas), dim3(kPermThreads), smem, st, T, c.top_k,
                 c.n_experts, c.n_shared, W.group_n, W.pieces, W.e0, W.e1, W.shared ? 1 : 0,
                 per, ids, (int32_t *)(ws + W.offsets), (int32_t *)(ws + W.perm),
                 (int32_t *)(ws + W.slot_pos), (Group *)(ws + W.groups),
                 (Ctrl *)(ws + W.ctrl)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe

// bucket.cuh -- per-expert bucketing of the routed (token, slot) pairs, done
// by one thread block: counts, offsets, the (token, slot) list of every
// expert, and the active-expert list (shared expert first, then the routed
// experts with at least one token in ascending id). The order of pairs
// within an expert's list does not affect any result: every (token, slot) is
// computed on its own.
#pragma once
#include "common.cuh"

namespace ds4 {

// Block-wide exclusive scan of v (one value per thread, blockDim.x <= 1024).
// Returns the exclusive prefix; *total receives the sum. Uses sh[32].
__device__ __forceinline__ int block_exscan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;  // inclusive prefix over warps
  }
  __syncthreads();
  const int before = (warp ? sh[warp - 1] : 0) + x - v;
  *total = sh[nw - 1];
  __syncthreads();
  return before;
}

// Shared-memory need of bucket_block, in ints.
__host__ __device__ constexpr int bucket_smem_ints(int E) { return 2 * (E + 2) + 32; }

// ids: [T][k] routed expert ids (-1 = none), written before the call (shared
// or global memory). Writes cnt[0..E] (cnt[E] = T if
// a shared expert exists), off[0..E+1], active[], *n_active and list[].
// Must be called by every thread of the block.
__device__ void bucket_block(const int32_t *ids, int T, int E, int k, int NS, int n_shared, int32_t *sm,
                             int32_t *cnt_g, int32_t *off_g, int32_t *act_g, int32_t *nact_g, int32_t *list,
                             uint32_t *err) {
  int32_t *cnt = sm, *cur = sm + (E + 2), *scan = sm + 2 * (E + 2);
  const int tid = threadIdx.x, nth = blockDim.x;
  for (int e = tid; e < E + 2; e += nth) cnt[e] = 0, cur[e] = 0;
  __syncthreads();
  const int n = T * k;
  for (int i = tid; i < n; i += nth) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else if (e >= E) raise_flag(err, DS4MOE_DEVERR_INTERNAL);
  }
  if (tid == 0) cnt[E] = n_shared ? T : 0;
  __syncthreads();
  // Each thread owns a contiguous run of experts [e0, e1) of E+1 entries.
  const int per = (E + 1 + nth - 1) / nth;
  const int e0 = min(tid * per, E + 1), e1 = min(e0 + per, E + 1);
  int c_sum = 0, a_sum = 0;
  for (int e = e0; e < e1; e++) {
    c_sum += cnt[e];
    if (e < E && cnt[e] > 0) a_sum++;
  }
  int c_tot, a_tot;
  int c_pre = block_exscan(c_sum, scan, &c_tot);
  int a_pre = block_exscan(a_sum, scan, &a_tot);
  for (int e = e0; e < e1; e++) {
    cur[e] = c_pre;  // temporarily: offset of e
    off_g[e] = c_pre;
    cnt_g[e] = cnt[e];
    if (e < E && cnt[e] > 0) act_g[n_shared + a_pre++] = e;
    c_pre += cnt[e];
  }
  if (tid == 0) {
    off_g[E + 1] = c_tot;
    if (n_shared) act_g[0] = E;
    *nact_g = a_tot + n_shared;
  }
  __syncthreads();
  for (int i = tid; i < n; i += nth) {
    const int e = ids[i];
    if (e >= 0 && e < E) {
      const int p = atomicAdd(&cur[e], 1);
      list[p] = (i / k) * NS + (i % k);
    }
  }
  if (n_shared)
    for (int t = tid; t < T; t += nth) list[cur[E] + t] = t * NS + k;
}

}  // namespace ds4

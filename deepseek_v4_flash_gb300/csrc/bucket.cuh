// bucket.cuh -- per-expert bucketing of the routed (token, slot) pairs of one
// call, done by one thread block, into a compact table:
//
//   int32 header[4]    n_active, n_pairs (routed pairs with a valid id), 0, 0
//   int4  act[A_cap]   {expert, pair count, offset into list, 0}: the shared
//                      expert first (expert = E, all tokens), then the routed
//                      experts with at least one pair in ascending id
//   int32 list[T*NS]   (token t << 5) | slot j, grouped by expert in act
//                      order; within an expert in (token, slot) order
//
// Every position is a rank count (how many pairs sort before this one), so
// the table is the same on every run. The order of pairs within an expert
// does not affect any result: every (token, slot) is computed on its own.
#pragma once
#include "common.cuh"

namespace ds4 {

constexpr int BKT_HDR = 4;  // header ints before the act table

__host__ __device__ constexpr int bucket_table_ints(int A_cap, int T, int NS) { return BKT_HDR + 4 * A_cap + T * NS; }

// Shared-memory ints bucket_rank needs for n = T*k pairs.
__host__ __device__ constexpr int bucket_rank_smem_ints(int n) { return 3 * n + 4; }

// ids: [T][k] routed expert ids in shared memory (-1 = none; >= E raises
// DS4MOE_DEVERR_INTERNAL and is dropped). sm: bucket_rank_smem_ints(T*k)
// ints. out: the table above in global memory, A_cap >= its rows. All
// threads of the block call it.
__device__ inline void bucket_rank(const int32_t *ids, int T, int E, int k, int NS, int n_shared, int32_t *sm,
                                   int32_t *out, int A_cap, uint32_t *err) {
  const int n = T * k, tid = threadIdx.x, nth = blockDim.x;
  int32_t *rank = sm, *first = sm + n, *count = sm + 2 * n, *tot = sm + 3 * n;  // tot: pairs, experts
  if (tid < 2) tot[tid] = 0;
  __syncthreads();
  int4 *act = (int4 *)(out + BKT_HDR);
  int32_t *list = out + BKT_HDR + 4 * A_cap;
  for (int i = tid; i < n; i += nth) {
    const int e = ids[i];
    const bool ok = e >= 0 && e < E;
    if (e >= E) raise_flag(err, DS4MOE_DEVERR_INTERNAL);
    int r = 0, c = 0, f = 1;
    if (ok) {
      for (int j = 0; j < n; j++) {
        const int ej = ids[j];
        if (ej < 0 || ej >= E) continue;
        r += (ej < e || (ej == e && j < i)) ? 1 : 0;
        c += ej == e ? 1 : 0;
        f &= (ej == e && j < i) ? 0 : 1;
      }
      list[r] = ((i / k) << 5) | (i % k);
      atomicAdd(&tot[0], 1);
      if (f) atomicAdd(&tot[1], 1);
    }
    rank[i] = r;
    first[i] = ok && f;
    count[i] = c;
  }
  __syncthreads();
  const int n_pairs = tot[0], n_exp = tot[1];
  for (int i = tid; i < n; i += nth) {
    if (!first[i]) continue;
    const int e = ids[i];
    int d = 0;  // distinct experts below e
    for (int j = 0; j < n; j++) d += (first[j] && ids[j] < e) ? 1 : 0;
    act[n_shared + d] = make_int4(e, count[i], rank[i], 0);
  }
  if (n_shared) {
    for (int t = tid; t < T; t += nth) list[n_pairs + t] = (t << 5) | k;
    if (tid == 0) act[0] = make_int4(E, T, n_pairs, 0);
  }
  if (tid == 0) {
    out[0] = n_exp + n_shared;
    out[1] = n_pairs;
    out[2] = 0;
    out[3] = 0;
  }
  __syncthreads();
}

// The same table for a single token, by one warp (lane j < k: slot j); every
// lane of the warp calls it. ids: the token's k routed ids (-1 = none; >= E
// raises DS4MOE_DEVERR_INTERNAL and is dropped).
__device__ inline void bucket_one_token_ids(int e, int E, int k, int n_shared, int32_t *out, int A_cap,
                                            uint32_t *err, int lane);
__device__ inline void bucket_one_token(const int32_t *ids, int E, int k, int n_shared, int32_t *out, int A_cap,
                                        uint32_t *err, int lane) {
  bucket_one_token_ids(lane < k ? ids[lane] : -1, E, k, n_shared, out, A_cap, err, lane);
}
// The same with lane j < k holding slot j's id e (others: -1); `out` may be
// shared memory.
__device__ inline void bucket_one_token_ids(int e, int E, int k, int n_shared, int32_t *out, int A_cap,
                                            uint32_t *err, int lane) {
  const bool ok = e >= 0 && e < E;
  if (lane < k && e >= E) raise_flag(err, DS4MOE_DEVERR_INTERNAL);
  const unsigned valid = __ballot_sync(0xffffffffu, ok);
  const unsigned same = __match_any_sync(0xffffffffu, ok ? e : -1) & valid;  // this lane's expert
  const bool f = ok && (same & ((1u << lane) - 1u)) == 0;                    // first slot of it
  const unsigned first = __ballot_sync(0xffffffffu, f);
  int below = 0, dbelow = 0;  // valid slots / distinct experts with a lower id
#pragma unroll
  for (int i = 0; i < 32; i++) {
    if (i >= k) break;
    const int ei = __shfl_sync(0xffffffffu, e, i);
    below += ((valid >> i) & 1u) && ei < e;
    dbelow += ((first >> i) & 1u) && ei < e;
  }
  const int r = below + __popc(same & ((1u << lane) - 1u)), c = __popc(same);
  const int n_pairs = __popc(valid), n_exp = __popc(first);
  int4 *act = (int4 *)(out + BKT_HDR);
  int32_t *list = out + BKT_HDR + 4 * A_cap;
  if (ok) {
    list[r] = lane;  // token 0, slot lane
    if (f) act[n_shared + dbelow] = make_int4(e, c, r, 0);
  }
  if (lane == 0) {
    if (n_shared) {
      list[n_pairs] = k;
      act[0] = make_int4(E, 1, n_pairs, 0);
    }
    out[0] = n_exp + n_shared;
    out[1] = n_pairs;
    out[2] = 0;
    out[3] = 0;
  }
}

}  // namespace ds4

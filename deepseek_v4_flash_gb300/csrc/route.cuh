// route.cuh -- block-parallel routing of one token from its router logits:
// sigmoid scores, selection keys (score + bias), the top-k of the keys and
// the renormalised weights (CAS steps 5-7).
//
// The top-k is a two-level rank count instead of k rounds of arg-max: every
// key is made unique by appending its expert index, so "the j-th pick of
// repeated arg-max with ties to the lower index" is exactly "the key with
// j larger keys". Level 1 ranks each key within its chunk of 32; the at most
// k keys of each chunk that rank below k are the only candidates; level 2
// ranks the candidates among themselves.
#pragma once
#include "common.cuh"

namespace ds4 {

// 64-bit selection key, larger = picked earlier. High word: the float key
// mapped so that unsigned order is float order (-0 ranks as +0, NaN lowest);
// low word: ~e, so that of two equal keys the lower index ranks first.
__device__ __forceinline__ uint64_t sel_key(float key, int e) {
  uint32_t u = __float_as_uint(key);
  if (key == 0.0f) u = 0u;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  if (key != key) u = 0u;
  return ((uint64_t)u << 32) | (uint64_t)(~(uint32_t)e);
}

// Shared-memory bytes of the routing scratch for E experts (E_pad = E
// rounded up to 32) and top-k: K [E_pad] u64 | cand [(E_pad/32)*k] u64 |
// s [E_pad] f32 | sel [16] i32.
__host__ __device__ constexpr int route_block_smem(int E_pad, int k) {
  return E_pad * 8 + (E_pad / 32) * k * 8 + E_pad * 4 + 16 * 4;
}

struct RouteScratch {
  uint64_t *K, *cand;
  float *s;
  int *sel;
};

// sm: route_block_smem bytes, 8-byte aligned.
__device__ __forceinline__ RouteScratch route_scratch(uint8_t *sm, int E_pad, int k) {
  RouteScratch r;
  r.K = (uint64_t *)sm;
  r.cand = r.K + E_pad;
  r.s = (float *)(r.cand + (E_pad >> 5) * k);
  r.sel = (int *)(r.s + E_pad);
  return r;
}

// Score and selection key of expert e from its logit (CAS step 5); padding
// entries (E <= e < E_pad) get a key below every expert's.
__device__ __forceinline__ void route_score(const RouteScratch &r, int e, int E, float lg, float bias) {
  if (e < E) {
    const float sv = cas_sigmoid(lg);
    r.s[e] = sv;
    r.K[e] = sel_key(__fadd_rn(sv, bias), e);
  } else {
    r.K[e] = (uint64_t)(~(uint32_t)e);
  }
}

// Top-k of the keys and the renormalised weights (CAS steps 6-7), once every
// K[e] and s[e] has been written by the block. Writes ids[0..k) (descending
// key order) and w[0..k). All threads of the block call it (blockDim.x a
// multiple of 32); it starts and ends with a barrier.
__device__ inline void route_select(const RouteScratch &r, int E_pad, int k, float scale, int32_t *ids, float *w) {
  const int tid = threadIdx.x, nth = blockDim.x;
  __syncthreads();
  for (int e = tid; e < E_pad; e += nth) {
    const uint64_t me = r.K[e];
    const uint64_t *c = r.K + (e & ~31);
    int n = 0;
#pragma unroll 8
    for (int j = 0; j < 32; j++) n += c[j] > me ? 1 : 0;
    if (n < k) r.cand[(e >> 5) * k + n] = me;
  }
  __syncthreads();
  const int nc = (E_pad >> 5) * k;
  for (int i = tid; i < nc; i += nth) {
    const uint64_t me = r.cand[i];
    int n = 0;
#pragma unroll 8
    for (int j = 0; j < nc; j++) n += r.cand[j] > me ? 1 : 0;
    if (n < k) r.sel[n] = (int)(~(uint32_t)me);
  }
  __syncthreads();
  if (tid < k) {
    float sum = 0.0f;  // in selection order
    for (int j = 0; j < k; j++) sum = __fadd_rn(sum, r.s[r.sel[j]]);
    const int e = r.sel[tid];
    ids[tid] = e;
    w[tid] = __fmul_rn(__fdiv_rn(r.s[e], sum), scale);
  }
  __syncthreads();
}

// Routes one token from its router segment sums part [ROUTER_SEGS][E_pad]
// (global memory, read through L2: other blocks may have written them);
// logit = the segment sums added in segment order. bias [E]. sm:
// route_block_smem bytes. All threads of the block call it.
__device__ inline void route_token_block(const float *part, int E, int E_pad, int k, const float *bias, float scale,
                                         uint8_t *sm, int32_t *ids, float *w) {
  const RouteScratch r = route_scratch(sm, E_pad, k);
  for (int e = threadIdx.x; e < E_pad; e += blockDim.x) {
    float lg = 0.0f;
    if (e < E) {
#pragma unroll
      for (int g = 0; g < ROUTER_SEGS; g++) lg = __fadd_rn(lg, __ldcg(part + (size_t)g * E_pad + e));
    }
    route_score(r, e, E, lg, e < E ? __ldg(bias + e) : 0.0f);
  }
  route_select(r, E_pad, k, scale, ids, w);
}

}  // namespace ds4

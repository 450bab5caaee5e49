// route.cuh -- block-parallel routing of one token from its router segment
// sums: logits, sigmoid scores, selection keys (score + bias), the top-k of
// the keys and the renormalised weights (CAS steps 5-7).
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

// Shared-memory bytes of route_token_block for E experts (E_pad = E rounded
// up to 32) and top-k.
__host__ __device__ constexpr int route_block_smem(int E_pad, int k) {
  return E_pad * 8 + (E_pad / 32) * k * 8 + E_pad * 4 + 16 * 4;
}

// Routes one token with every thread of the block (blockDim.x a multiple of
// 32). part: the token's segment sums [ROUTER_SEGS][E_pad]; bias [E].
// Writes ids[0..k) (descending key order) and w[0..k). sm: route_block_smem
// bytes, 8-byte aligned. Must be called by all threads; ends with a barrier.
__device__ void route_token_block(const float *part, int E, int E_pad, int k, const float *bias, float scale,
                                  uint8_t *sm, int32_t *ids, float *w) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int nch = E_pad >> 5;
  uint64_t *K = (uint64_t *)sm;
  uint64_t *cand = K + E_pad;                 // [nch][k]
  float *s = (float *)(cand + nch * k);       // [E_pad]
  int *sel = (int *)(s + E_pad);              // [k]
  for (int e = tid; e < E_pad; e += nth) {
    if (e < E) {
      float lg = 0.0f;
#pragma unroll
      for (int g = 0; g < ROUTER_SEGS; g++) lg = __fadd_rn(lg, part[(size_t)g * E_pad + e]);
      const float sv = cas_sigmoid(lg);
      s[e] = sv;
      K[e] = sel_key(__fadd_rn(sv, __ldg(bias + e)), e);
    } else {
      K[e] = (uint64_t)(~(uint32_t)e);  // padding: below every expert, still unique
    }
  }
  __syncthreads();
  for (int e = tid; e < E_pad; e += nth) {
    const uint64_t me = K[e];
    const uint64_t *c = K + (e & ~31);
    int r = 0;
#pragma unroll 8
    for (int j = 0; j < 32; j++) r += c[j] > me ? 1 : 0;
    if (r < k) cand[(e >> 5) * k + r] = me;
  }
  __syncthreads();
  const int nc = nch * k;
  for (int i = tid; i < nc; i += nth) {
    const uint64_t me = cand[i];
    int r = 0;
    for (int j = 0; j < nc; j++) r += cand[j] > me ? 1 : 0;
    if (r < k) sel[r] = (int)(~(uint32_t)me);
  }
  __syncthreads();
  if (tid < k) {
    float sum = 0.0f;  // in selection order
    for (int j = 0; j < k; j++) sum = __fadd_rn(sum, s[sel[j]]);
    const int e = sel[tid];
    ids[tid] = e;
    w[tid] = __fmul_rn(__fdiv_rn(s[e], sum), scale);
  }
  __syncthreads();
}

}  // namespace ds4

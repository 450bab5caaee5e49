// tiles.cuh -- per-K-step dot products of one RG16 weight tile (16 rows, two
// lanes per row) against up to TT activation rows, accumulated in CAS order.
#pragma once
#include "common.cuh"

namespace ds4 {

constexpr uint32_t M2 = 0x03030303u;

// Activation reads: through the read-only data path from global memory, or
// plain loads when the activations were staged in shared memory (ACT_SMEM).
template <bool ACT_SMEM, typename T>
__device__ __forceinline__ T act_load(const T *p) {
  if constexpr (ACT_SMEM) return *p;
  else return __ldg(p);
}

// Sum over one 16-weight group of q * x: 4 dp4a on the transposed word W.
__device__ __forceinline__ int grp_dot(uint32_t W, uint4 x) {
  int a = __dp4a((int)(W & M2), (int)x.x, 0);
  a = __dp4a((int)((W >> 2) & M2), (int)x.y, a);
  a = __dp4a((int)((W >> 4) & M2), (int)x.z, a);
  a = __dp4a((int)((W >> 6) & M2), (int)x.w, a);
  return a;
}

// One Q2S tile (16 rows x 256 K, superblock s) against TT activation rows.
// Lane 2r+h computes, for each block b, sc*dot and mn*gs of group 2b+h; the
// partner lane's halves complete A_b and B_b exactly (CAS step 2); both lanes
// then add the block term to the row sum in block order (CAS steps 3-4).
template <int TT, bool ACT_SMEM = false>
__device__ __forceinline__ void q2s_tile(uint32_t tile, int lane, int s, int K, const int *tok,
                                         const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                         const int16_t *__restrict__ ag, float *acc) {
  const int h = lane & 1, r = lane >> 1;
  const uint2 sm = ld_shared_v2(tile + Q2S_SM + 8 * lane);
  const uint32_t dd = ld_shared_u32(tile + Q2S_DD + 4 * r);
  const float d = half_bits_to_float(dd), dmin = half_bits_to_float(dd >> 16);
  const int nb = K >> 5;
  constexpr int UNROLL_C = TT >= 4 ? 1 : 2;  // bound register use for wide token tiles
#pragma unroll UNROLL_C
  for (int c = 0; c < 2; c++) {
    const uint4 q = ld_shared_v4(tile + Q2S_QS + 512 * c + 16 * lane);
    const uint32_t smw = c ? sm.y : sm.x;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int j = 4 * c + i;  // block within the superblock
      const uint32_t W = i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
      const int byte = (int)((smw >> (8 * i)) & 0xFFu);
      const int sc = byte & 15, mn = byte >> 4;
      const int blk = 8 * s + j;
#pragma unroll
      for (int t = 0; t < TT; t++) {
        const uint4 x = act_load<ACT_SMEM>((const uint4 *)(aq + (size_t)tok[t] * K + 32 * blk + 16 * h));
        const int gsv = (int)act_load<ACT_SMEM>(ag + (size_t)tok[t] * (K >> 4) + 2 * blk + h);
        const int pa = sc * grp_dot(W, x), pb = mn * gsv;
        const int A = pa + __shfl_xor_sync(0xffffffffu, pa, 1);
        const int B = pb + __shfl_xor_sync(0xffffffffu, pb, 1);
        acc[t] = __fadd_rn(acc[t], q2s_term(act_load<ACT_SMEM>(ad + (size_t)tok[t] * nb + blk), d, dmin, A, B));
      }
    }
  }
}

// One Q8 tile (16 rows x one 32-block: K-step s = block s) against TT rows.
// Lane 2r+h takes elements 16h..16h+15; the partner lane completes I exactly.
template <int TT, bool ACT_SMEM = false>
__device__ __forceinline__ void q8_tile(uint32_t tile, int lane, int s, int K, const int *tok,
                                        const int8_t *__restrict__ aq, const float *__restrict__ ad, float *acc) {
  const int h = lane & 1, r = lane >> 1;
  const uint32_t dw = ld_shared_u32(tile + 4 * (r >> 1));
  const float d = half_bits_to_float((r & 1) ? dw >> 16 : dw);
  const uint4 q = ld_shared_v4(tile + Q8_Q + 16 * lane);
  const int nb = K >> 5;
#pragma unroll
  for (int t = 0; t < TT; t++) {
    const uint4 x = act_load<ACT_SMEM>((const uint4 *)(aq + (size_t)tok[t] * K + 32 * s + 16 * h));
    int I = dot16(q, x, 0);
    I += __shfl_xor_sync(0xffffffffu, I, 1);
    acc[t] = __fadd_rn(acc[t], q8_term(d, act_load<ACT_SMEM>(ad + (size_t)tok[t] * nb + s), I));
  }
}

}  // namespace ds4

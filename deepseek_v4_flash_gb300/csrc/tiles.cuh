// tiles.cuh -- per-K-step dot products of one RG32 weight tile (one row per
// lane) against up to TT activation rows, accumulated in CAS order.
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

__device__ __forceinline__ int byte_of(uint4 v, int i) {
  const uint32_t w = i < 4 ? v.x : i < 8 ? v.y : i < 12 ? v.z : v.w;
  return (int)((w >> (8 * (i & 3))) & 0xFFu);
}

// Sum over one 16-weight group of q * x: 4 dp4a on the transposed word W.
__device__ __forceinline__ int grp_dot(uint32_t W, uint4 x) {
  int a = __dp4a((int)(W & M2), (int)x.x, 0);
  a = __dp4a((int)((W >> 2) & M2), (int)x.y, a);
  a = __dp4a((int)((W >> 4) & M2), (int)x.z, a);
  a = __dp4a((int)((W >> 6) & M2), (int)x.w, a);
  return a;
}

// One Q2S tile (32 rows x 256 K) against TT activation rows: blocks 8s..8s+7
// of each row, accumulated in order into acc[] (CAS steps 2-4).
template <int TT, bool ACT_SMEM = false>
__device__ __forceinline__ void q2s_tile(uint32_t tile, int lane, int s, int K, const int *tok,
                                         const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                         const int16_t *__restrict__ ag, float *acc) {
  const uint4 sm = ld_shared_v4(tile + 16 * lane);
  const uint32_t dd = ld_shared_u32(tile + Q2S_DD + 4 * lane);
  const float d = half_bits_to_float(dd), dmin = half_bits_to_float(dd >> 16);
  const int nb = K >> 5;
  constexpr int UNROLL_C = TT >= 4 ? 1 : 4;  // bound register use for wide token tiles
#pragma unroll UNROLL_C
  for (int c = 0; c < 4; c++) {
    const uint4 q = ld_shared_v4(tile + Q2S_QS + 512 * c + 16 * lane);
#pragma unroll
    for (int hb = 0; hb < 2; hb++) {
      const int j = 2 * c + hb;  // block within the superblock
      const uint32_t w0 = hb ? q.z : q.x, w1 = hb ? q.w : q.y;
      const int b0 = byte_of(sm, 2 * j), b1 = byte_of(sm, 2 * j + 1);
      const int sc0 = b0 & 15, mn0 = b0 >> 4, sc1 = b1 & 15, mn1 = b1 >> 4;
      const int blk = 8 * s + j;
#pragma unroll
      for (int i = 0; i < TT; i++) {
        const uint4 *xv = (const uint4 *)(aq + (size_t)tok[i] * K + 32 * blk);
        const uint4 x0 = act_load<ACT_SMEM>(xv), x1 = act_load<ACT_SMEM>(xv + 1);
        const uint32_t g2 = act_load<ACT_SMEM>((const uint32_t *)(ag + (size_t)tok[i] * (K >> 4) + 2 * blk));
        const int gs0 = (int)(int16_t)(g2 & 0xFFFFu), gs1 = (int)(int16_t)(g2 >> 16);
        const int A = sc0 * grp_dot(w0, x0) + sc1 * grp_dot(w1, x1);
        const int B = mn0 * gs0 + mn1 * gs1;
        acc[i] = __fadd_rn(acc[i], q2s_term(act_load<ACT_SMEM>(ad + (size_t)tok[i] * nb + blk), d, dmin, A, B));
      }
    }
  }
}

// One Q8 tile (32 rows x one 32-block: K-step s = block s) against TT rows.
template <int TT, bool ACT_SMEM = false>
__device__ __forceinline__ void q8_tile(uint32_t tile, int lane, int s, int K, const int *tok,
                                        const int8_t *__restrict__ aq, const float *__restrict__ ad, float *acc) {
  const uint32_t dw = ld_shared_u32(tile + 4 * (lane >> 1));
  const float d = half_bits_to_float((lane & 1) ? dw >> 16 : dw);
  const uint4 q0 = ld_shared_v4(tile + Q8_Q + 16 * lane);
  const uint4 q1 = ld_shared_v4(tile + Q8_Q + 512 + 16 * lane);
  const int nb = K >> 5;
#pragma unroll
  for (int i = 0; i < TT; i++) {
    const uint4 *xv = (const uint4 *)(aq + (size_t)tok[i] * K + 32 * s);
    const int I = dot16(q1, act_load<ACT_SMEM>(xv + 1), dot16(q0, act_load<ACT_SMEM>(xv), 0));
    acc[i] = __fadd_rn(acc[i], q8_term(d, act_load<ACT_SMEM>(ad + (size_t)tok[i] * nb + s), I));
  }
}

}  // namespace ds4

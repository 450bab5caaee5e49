// tiles.cuh -- dot products of one K-step of RG16 weight tiles (16 rows)
// against up to TT activation rows, accumulated in CAS order. MATS tiles of
// the same K-step (gate and up: 2) share the activation loads.
#pragma once
#include "common.cuh"

namespace ds4 {

constexpr uint32_t M2 = 0x03030303u;

// Activation reads: plain loads from shared memory (staged) or through the
// read-only path from global memory.
template <bool ACT_SMEM, typename T>
__device__ __forceinline__ T act_load(const T *p) {
  if constexpr (ACT_SMEM) return *p;
  else return __ldg(p);
}

// Sum over one 16-weight group of q * x: 4 dp4a on the transposed word W.
// Two independent chains of two, for latency.
__device__ __forceinline__ int grp_dot(uint32_t W, uint4 x) {
  const int a = __dp4a((int)((W >> 2) & M2), (int)x.y, __dp4a((int)(W & M2), (int)x.x, 0));
  const int b = __dp4a((int)((W >> 6) & M2), (int)x.w, __dp4a((int)((W >> 4) & M2), (int)x.z, 0));
  return a + b;
}

// a.h0 * b.byte0 + a.h1 * b.byte1 (hi: bytes 2, 3) + c; a's halves signed,
// b's bytes unsigned.
template <bool HI>
__device__ __forceinline__ int dp2a_su(uint32_t a, uint32_t b, int c) {
  int d;
  if constexpr (HI) asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One Q2S K-step (superblock s) of MATS tiles at t0, t0 + Q2S_TILE, ...
// Lane 2r + h owns blocks h, h+2, h+4, h+6 of row r (both groups of each):
// A_b = sc0*dot0 + sc1*dot1 and B_b = mn0*gs0 + mn1*gs1 are complete in the
// lane (CAS step 2); the lane computes its blocks' terms (CAS step 3) and
// trades them with its partner, so lane h = 0 adds all eight terms to the
// row chain in block order (CAS step 4). acc of lanes with h = 1 is not used.
template <int TT, int MATS, bool ACT_SMEM>
__device__ __forceinline__ void q2s_step(uint32_t t0, int lane, int s, int K, const int *arow, int nt,
                                         const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                         const int16_t *__restrict__ ag, float (&acc)[MATS][TT]) {
  const int h = lane & 1, r = lane >> 1;
  uint32_t sc[MATS][2], mn[MATS][2];
  float d[MATS], dmin[MATS];
#pragma unroll
  for (int m = 0; m < MATS; m++) {
    const uint32_t tm = t0 + m * Q2S_TILE;
    const uint2 smw = ld_shared_v2(tm + Q2S_SM + 8 * lane);
    const uint32_t dd = ld_shared_u32(tm + Q2S_DD + 4 * r);
    sc[m][0] = smw.x & 0x0F0F0F0Fu, mn[m][0] = (smw.x >> 4) & 0x0F0F0F0Fu;
    sc[m][1] = smw.y & 0x0F0F0F0Fu, mn[m][1] = (smw.y >> 4) & 0x0F0F0F0Fu;
    d[m] = half_bits_to_float(dd), dmin[m] = half_bits_to_float(dd >> 16);
  }
  const int nb = K >> 5;
#pragma unroll
  for (int c = 0; c < 2; c++) {  // chunk c: blocks h + 4c, h + 4c + 2
    uint4 q[MATS];
#pragma unroll
    for (int m = 0; m < MATS; m++) q[m] = ld_shared_v4(t0 + m * Q2S_TILE + Q2S_QS + 512 * c + 16 * lane);
#pragma unroll
    for (int jj = 0; jj < 2; jj++) {
      const int blk = 8 * s + h + 4 * c + 2 * jj;
#pragma unroll
      for (int t = 0; t < TT; t++) {
        if (t >= nt) break;  // warp-uniform: only the unit's valid tokens
        const int8_t *xr = aq + (size_t)arow[t] * K + 32 * blk;
        const uint4 x0 = act_load<ACT_SMEM>((const uint4 *)xr);
        const uint4 x1 = act_load<ACT_SMEM>((const uint4 *)(xr + 16));
        const uint32_t gsw = act_load<ACT_SMEM>((const uint32_t *)(ag + (size_t)arow[t] * (K >> 4) + 2 * blk));
        const float dxv = act_load<ACT_SMEM>(ad + (size_t)arow[t] * nb + blk);
#pragma unroll
        for (int m = 0; m < MATS; m++) {
          const uint32_t W0 = jj ? q[m].z : q[m].x, W1 = jj ? q[m].w : q[m].y;
          const uint32_t P = __byte_perm((uint32_t)grp_dot(W0, x0), (uint32_t)grp_dot(W1, x1), 0x5410);
          int A, B;
          if (jj) {
            A = dp2a_su<true>(P, sc[m][c], 0);
            B = dp2a_su<true>(gsw, mn[m][c], 0);
          } else {
            A = dp2a_su<false>(P, sc[m][c], 0);
            B = dp2a_su<false>(gsw, mn[m][c], 0);
          }
          const float mine = q2s_term(dxv, d[m], dmin[m], A, B);
          const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
          acc[m][t] = __fadd_rn(__fadd_rn(acc[m][t], mine), other);
        }
      }
    }
  }
}

// One Q8_0 K-step (block s) of MATS tiles at t0, t0 + Q8_TILE, ...
// Lane 2r + h takes elements 16h .. 16h+15 of row r; the partner lane
// completes I exactly and both lanes add the same term.
template <int TT, int MATS, bool ACT_SMEM>
__device__ __forceinline__ void q8_step(uint32_t t0, int lane, int s, int K, const int *arow, int nt,
                                        const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                        float (&acc)[MATS][TT]) {
  const int h = lane & 1, r = lane >> 1;
  float d[MATS];
  uint4 q[MATS];
#pragma unroll
  for (int m = 0; m < MATS; m++) {
    const uint32_t tm = t0 + m * Q8_TILE;
    const uint32_t dw = ld_shared_u32(tm + 4 * (r >> 1));
    d[m] = half_bits_to_float((r & 1) ? dw >> 16 : dw);
    q[m] = ld_shared_v4(tm + Q8_Q + 16 * lane);
  }
  const int nb = K >> 5;
#pragma unroll
  for (int t = 0; t < TT; t++) {
    if (t >= nt) break;  // warp-uniform: only the unit's valid tokens
    const uint4 x = act_load<ACT_SMEM>((const uint4 *)(aq + (size_t)arow[t] * K + 32 * s + 16 * h));
    const float dxv = act_load<ACT_SMEM>(ad + (size_t)arow[t] * nb + s);
#pragma unroll
    for (int m = 0; m < MATS; m++) {
      int I = dot16(q[m], x, 0);
      I += __shfl_xor_sync(0xffffffffu, I, 1);
      acc[m][t] = __fadd_rn(acc[m][t], q8_term(d[m], dxv, I));
    }
  }
}

}  // namespace ds4

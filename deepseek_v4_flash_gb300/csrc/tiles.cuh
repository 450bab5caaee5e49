// tiles.cuh -- dot products of one K-step of RG16 weight tiles (16 rows)
// against up to TT activation rows, accumulated in CAS order. The two tiles
// of a K-step (gate and up, or the two 16-row halves of a down item) share
// the activation loads.
#pragma once
#include "common.cuh"

namespace ds4 {

// The two tiles' row chains of one token: a packed pair (two binary32 lanes
// per instruction, each rounded as the scalar operation) or two scalars.
// Packing saves instructions when several tokens share a K-step; for one
// token the scalar form schedules better under the register cap of two
// blocks per SM (measured).
template <bool PACK> struct Chains { float c[2]; };
template <> struct Chains<true> { unsigned long long v; };

template <bool PACK> __device__ __forceinline__ void chains_zero(Chains<PACK> &a) {
  if constexpr (PACK) a.v = 0ull;
  else a.c[0] = 0.0f, a.c[1] = 0.0f;
}
template <bool PACK> __device__ __forceinline__ void chains_get(const Chains<PACK> &a, float &c0, float &c1) {
  if constexpr (PACK) f2_unpack(a.v, c0, c1);
  else c0 = a.c[0], c1 = a.c[1];
}

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

// One Q2S K-step (superblock s) of the two tiles at t0, t0 + Q2S_TILE.
// Lane 2r + h owns blocks h, h+2, h+4, h+6 of row r (both groups of each):
// A_b = sc0*dot0 + sc1*dot1 and B_b = mn0*gs0 + mn1*gs1 are complete in the
// lane (CAS step 2); the lane computes its blocks' terms (CAS step 3) and
// trades them with its partner, so lane h = 0 adds all eight terms to the
// row chain in block order (CAS step 4). acc of lanes with h = 1 is not used.
template <int TT, bool ACT_SMEM, bool PACK>
__device__ __forceinline__ void q2s_step(uint32_t t0, int lane, int s, int K, const int *arow, int nt,
                                         const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                         const int16_t *__restrict__ ag, Chains<PACK> (&acc)[TT]) {
  const int h = lane & 1, r = lane >> 1;
  uint32_t sc[2][2], mn[2][2];
  float d[2], dmin[2];
#pragma unroll
  for (int m = 0; m < 2; m++) {
    const uint32_t tm = t0 + m * Q2S_TILE;
    const uint2 smw = ld_shared_v2(tm + Q2S_SM + 8 * lane);
    const uint32_t dd = ld_shared_u32(tm + Q2S_DD + 4 * r);
    sc[m][0] = smw.x & 0x0F0F0F0Fu, mn[m][0] = (smw.x >> 4) & 0x0F0F0F0Fu;
    sc[m][1] = smw.y & 0x0F0F0F0Fu, mn[m][1] = (smw.y >> 4) & 0x0F0F0F0Fu;
    d[m] = half_bits_to_float(dd), dmin[m] = half_bits_to_float(dd >> 16);
  }
  // packed: (-dmin) * B is exactly -(dmin * B), so the term
  // dx * fma(d, A, -(dmin * B)) takes one packed product for the min part
  unsigned long long d2 = 0ull, nm2 = 0ull;
  if constexpr (PACK) d2 = f2_pack(d[0], d[1]), nm2 = f2_pack(-dmin[0], -dmin[1]);
  const int nb = K >> 5;
#pragma unroll
  for (int c = 0; c < 2; c++) {  // chunk c: blocks h + 4c, h + 4c + 2
    uint4 q[2];
#pragma unroll
    for (int m = 0; m < 2; m++) q[m] = ld_shared_v4(t0 + m * Q2S_TILE + Q2S_QS + 512 * c + 16 * lane);
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
        int A[2], B[2];
#pragma unroll
        for (int m = 0; m < 2; m++) {
          const uint32_t W0 = jj ? q[m].z : q[m].x, W1 = jj ? q[m].w : q[m].y;
          const uint32_t P = __byte_perm((uint32_t)grp_dot(W0, x0), (uint32_t)grp_dot(W1, x1), 0x5410);
          if (jj) {
            A[m] = dp2a_su<true>(P, sc[m][c], 0);
            B[m] = dp2a_su<true>(gsw, mn[m][c], 0);
          } else {
            A[m] = dp2a_su<false>(P, sc[m][c], 0);
            B[m] = dp2a_su<false>(gsw, mn[m][c], 0);
          }
          if constexpr (!PACK) {
            const float mine = q2s_term(dxv, d[m], dmin[m], A[m], B[m]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
            acc[t].c[m] = __fadd_rn(__fadd_rn(acc[t].c[m], mine), other);
          }
        }
        if constexpr (PACK) {
          // both matrices' terms, this lane's and the partner's, in one
          // packed chain (the product `mine` also feeds the shuffle, so it
          // is rounded on its own before the add)
          const unsigned long long mine =
              f2_mul(f2_pack(dxv, dxv),
                     f2_fma(d2, f2_pack(__int2float_rn(A[0]), __int2float_rn(A[1])),
                            f2_mul(nm2, f2_pack(__int2float_rn(B[0]), __int2float_rn(B[1])))));
          float m0, m1;
          f2_unpack(mine, m0, m1);
          const unsigned long long other =
              f2_pack(__shfl_xor_sync(0xffffffffu, m0, 1), __shfl_xor_sync(0xffffffffu, m1, 1));
          acc[t].v = f2_add(f2_add(acc[t].v, mine), other);
        }
      }
    }
  }
}

// Sum over one 16-weight group of q * x for 4-bit codes: its two words (W0:
// elements 0-7, W1: 8-15; low nibbles the first four of each eight) against
// the group's 16 int8 activations.
__device__ __forceinline__ int grp_dot4(uint32_t W0, uint32_t W1, uint4 x) {
  constexpr uint32_t M4 = 0x0F0F0F0Fu;
  const int a = __dp4a((int)((W0 >> 4) & M4), (int)x.y, __dp4a((int)(W0 & M4), (int)x.x, 0));
  const int b = __dp4a((int)((W1 >> 4) & M4), (int)x.w, __dp4a((int)(W1 & M4), (int)x.z, 0));
  return a + b;
}

// One Q4S K-step (superblock s) of the two tiles at t0, t0 + Q4S_TILE: as
// q2s_step, with lane 2r + h owning blocks h + 2c (c = 0..3) of row r, each
// block's four group words in chunk c. A_b and B_b are complete in the lane
// (CAS step 2), the lane computes its blocks' terms (CAS step 3) and trades
// them with its partner, so that lane h = 0 adds all eight terms to the row
// chain in block order (CAS step 4). acc of lanes with h = 1 is not used.
template <int TT, bool ACT_SMEM, bool PACK>
__device__ __forceinline__ void q4s_step(uint32_t t0, int lane, int s, int K, const int *arow, int nt,
                                         const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                         const int16_t *__restrict__ ag, Chains<PACK> (&acc)[TT]) {
  const int h = lane & 1, r = lane >> 1;
  uint32_t sc[2][2], mn[2][2];
  float d[2], dmin[2];
#pragma unroll
  for (int m = 0; m < 2; m++) {
    const uint32_t tm = t0 + m * Q4S_TILE;
    const uint2 smw = ld_shared_v2(tm + Q4S_SM + 8 * lane);
    const uint32_t dd = ld_shared_u32(tm + Q4S_DD + 4 * r);
    sc[m][0] = smw.x & 0x0F0F0F0Fu, mn[m][0] = (smw.x >> 4) & 0x0F0F0F0Fu;
    sc[m][1] = smw.y & 0x0F0F0F0Fu, mn[m][1] = (smw.y >> 4) & 0x0F0F0F0Fu;
    d[m] = half_bits_to_float(dd), dmin[m] = half_bits_to_float(dd >> 16);
  }
  unsigned long long d2 = 0ull, nm2 = 0ull;
  if constexpr (PACK) d2 = f2_pack(d[0], d[1]), nm2 = f2_pack(-dmin[0], -dmin[1]);
  const int nb = K >> 5;
#pragma unroll
  for (int c = 0; c < 4; c++) {  // block h + 2c
    uint4 q[2];
#pragma unroll
    for (int m = 0; m < 2; m++) q[m] = ld_shared_v4(t0 + m * Q4S_TILE + Q4S_QS + 512 * c + 16 * lane);
    const int blk = 8 * s + h + 2 * c;
#pragma unroll
    for (int t = 0; t < TT; t++) {
      if (t >= nt) break;  // warp-uniform: only the unit's valid tokens
      const int8_t *xr = aq + (size_t)arow[t] * K + 32 * blk;
      const uint4 x0 = act_load<ACT_SMEM>((const uint4 *)xr);
      const uint4 x1 = act_load<ACT_SMEM>((const uint4 *)(xr + 16));
      const uint32_t gsw = act_load<ACT_SMEM>((const uint32_t *)(ag + (size_t)arow[t] * (K >> 4) + 2 * blk));
      const float dxv = act_load<ACT_SMEM>(ad + (size_t)arow[t] * nb + blk);
      int A[2], B[2];
#pragma unroll
      for (int m = 0; m < 2; m++) {
        const uint32_t P = __byte_perm((uint32_t)grp_dot4(q[m].x, q[m].y, x0), (uint32_t)grp_dot4(q[m].z, q[m].w, x1),
                                       0x5410);
        if (c & 1) {
          A[m] = dp2a_su<true>(P, sc[m][c >> 1], 0);
          B[m] = dp2a_su<true>(gsw, mn[m][c >> 1], 0);
        } else {
          A[m] = dp2a_su<false>(P, sc[m][c >> 1], 0);
          B[m] = dp2a_su<false>(gsw, mn[m][c >> 1], 0);
        }
        if constexpr (!PACK) {
          const float mine = q2s_term(dxv, d[m], dmin[m], A[m], B[m]);
          const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
          acc[t].c[m] = __fadd_rn(__fadd_rn(acc[t].c[m], mine), other);
        }
      }
      if constexpr (PACK) {
        const unsigned long long mine =
            f2_mul(f2_pack(dxv, dxv), f2_fma(d2, f2_pack(__int2float_rn(A[0]), __int2float_rn(A[1])),
                                             f2_mul(nm2, f2_pack(__int2float_rn(B[0]), __int2float_rn(B[1])))));
        float m0, m1;
        f2_unpack(mine, m0, m1);
        const unsigned long long other =
            f2_pack(__shfl_xor_sync(0xffffffffu, m0, 1), __shfl_xor_sync(0xffffffffu, m1, 1));
        acc[t].v = f2_add(f2_add(acc[t].v, mine), other);
      }
    }
  }
}

// One Q8_0 K-step (block s) of the two tiles at t0, t0 + Q8_TILE.
// Lane 2r + h takes elements 16h .. 16h+15 of row r; the partner lane
// completes I exactly and both lanes add the same term.
template <int TT, bool ACT_SMEM, bool PACK>
__device__ __forceinline__ void q8_step(uint32_t t0, int lane, int s, int K, const int *arow, int nt,
                                        const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                        Chains<PACK> (&acc)[TT]) {
  const int h = lane & 1, r = lane >> 1;
  float d[2];
  uint4 q[2];
#pragma unroll
  for (int m = 0; m < 2; m++) {
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
    int I[2];
#pragma unroll
    for (int m = 0; m < 2; m++) {
      I[m] = dot16(q[m], x, 0);
      I[m] += __shfl_xor_sync(0xffffffffu, I[m], 1);
      if constexpr (!PACK) acc[t].c[m] = __fadd_rn(acc[t].c[m], q8_term(d[m], dxv, I[m]));
    }
    if constexpr (PACK) {
      // (d * dx) * I for both matrices (CAS step 3); the second product is
      // scalar: ptxas merges a packed product whose only use is a packed
      // add into one single-rounding packed multiply-add, .rn notwithstanding
      float dd0, dd1;
      f2_unpack(f2_mul(f2_pack(d[0], d[1]), f2_pack(dxv, dxv)), dd0, dd1);
      acc[t].v = f2_add(acc[t].v, f2_pack(__fmul_rn(dd0, __int2float_rn(I[0])), __fmul_rn(dd1, __int2float_rn(I[1]))));
    }
  }
}

}  // namespace ds4

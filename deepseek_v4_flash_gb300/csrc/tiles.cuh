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


// ---------------------------------------------------------------------------
// Int8 tensor-core steps for units of eight tokens (mma.sync m16n8k32).
// Lane (g, t) = (lane / 4, lane % 4) holds A rows g and g + 8 of a 16-row
// tile at K 4t..4t+3 and 16+4t..16+4t+3, B column (token) g at the same K,
// and D rows g, g + 8 for tokens 2t, 2t + 1. A is the exact integer weight of
// CAS step 2 (sc*q for the superblock formats, q for Q8_0) and B the int8
// codes, so D holds the exact block dots A_b (I_b) of 16 rows and 8 tokens.
// The lane keeps the chains of rows g, g + 8 of both tiles for tokens 2t,
// 2t + 1 as packed pairs, adding the block terms in block order.
struct MChains {
  unsigned long long v[2][2];  // [tile][row g, g + 8]: tokens (2t, 2t + 1)
};

__device__ __forceinline__ void mchains_zero(MChains &c) {
#pragma unroll
  for (int i = 0; i < 4; i++) c.v[i >> 1][i & 1] = 0ull;
}

// Unsigned weights (sc*q <= 225) against signed codes.
__device__ __forceinline__ void mma_u8s8(const uint32_t (&a)[4], uint32_t b0, uint32_t b1, int (&d)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

__device__ __forceinline__ void mma_s8s8(const uint32_t (&a)[4], uint32_t b0, uint32_t b1, int (&d)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

// Four 8x8 b16 matrices: lane i gives the address of row i % 8 of matrix
// i / 8 and receives, from each, bytes 4*(i%4)..+3 of row i / 4.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// The lane's activation data of 32-block blk: B fragment (token g, rows
// ar_g), and scales and group sums of its D tokens (rows ar0, ar1).
struct MTok {
  uint32_t b0, b1, gs0, gs1;
  float dx0, dx1;
};

template <bool ACT_SMEM, bool GS>
__device__ __forceinline__ MTok m_tok(int blk, int t, int K, int ar_g, int ar0, int ar1, const int8_t *__restrict__ aq,
                                      const float *__restrict__ ad, const int16_t *__restrict__ ag) {
  MTok o;
  const int8_t *xr = aq + (size_t)ar_g * K + 32 * blk + 4 * t;
  o.b0 = act_load<ACT_SMEM>((const uint32_t *)xr);
  o.b1 = act_load<ACT_SMEM>((const uint32_t *)(xr + 16));
  const int nb = K >> 5;
  o.dx0 = act_load<ACT_SMEM>(ad + (size_t)ar0 * nb + blk);
  o.dx1 = act_load<ACT_SMEM>(ad + (size_t)ar1 * nb + blk);
  o.gs0 = o.gs1 = 0u;
  if constexpr (GS) {
    o.gs0 = act_load<ACT_SMEM>((const uint32_t *)(ag + (size_t)ar0 * (K >> 4) + 2 * blk));
    o.gs1 = act_load<ACT_SMEM>((const uint32_t *)(ag + (size_t)ar1 * (K >> 4) + 2 * blk));
  }
  return o;
}

// Superblock-format terms of one row for the lane's two tokens (CAS step 3:
// dx * fma(d, A, -(dmin * B))); the products by dx are scalar, so that no
// packed product is fused into the chain's add.
__device__ __forceinline__ void m_sb_terms(unsigned long long &acc, float d, float dmin, int A0, int A1, int B0,
                                           int B1, float dx0, float dx1) {
  const unsigned long long f =
      f2_fma(f2_pack(d, d), f2_pack(__int2float_rn(A0), __int2float_rn(A1)),
             f2_mul(f2_pack(-dmin, -dmin), f2_pack(__int2float_rn(B0), __int2float_rn(B1))));
  float f0, f1;
  f2_unpack(f, f0, f1);
  acc = f2_add(acc, f2_pack(__fmul_rn(dx0, f0), __fmul_rn(dx1, f1)));
}

// B_b = mn0 * gs0 + mn1 * gs1 of one row (scale/min byte pair smp) for a
// token's packed group sums.
__device__ __forceinline__ int m_minterm(uint32_t smp, uint32_t gsw) {
  return (int)((smp >> 4) & 15) * (int)(int16_t)(gsw & 0xFFFF) + (int)((smp >> 12) & 15) * (int)(int16_t)(gsw >> 16);
}

// One Q2S (4-bit: Q4S) K-step (superblock s) of the two tiles at t0.
// Row r's scale/min bytes: 16 at SM + 16r, block b = h + 2j, group gi at
// byte 8h + 2j + gi; its group words: lane L = 2r + h's chunk (see q2s_step,
// q4s_step).
template <bool ACT_SMEM, bool Q4>
__device__ __forceinline__ void sb_step_mma(uint32_t t0, int lane, int s, int K, int ar_g, int ar0, int ar1,
                                            const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                            const int16_t *__restrict__ ag, MChains &acc) {
  constexpr int TILE = Q4 ? Q4S_TILE : Q2S_TILE, SM = Q4 ? Q4S_SM : Q2S_SM, DD = Q4 ? Q4S_DD : Q2S_DD,
                QS = Q4 ? Q4S_QS : Q2S_QS;
  const int g = lane >> 2, t = lane & 3;
  uint4 smr[2][2];
  float d[2][2], dmin[2][2];
#pragma unroll
  for (int m = 0; m < 2; m++)
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
      const int r = g + 8 * hh;
      const uint32_t tm = t0 + m * TILE;
      smr[m][hh] = ld_shared_v4(tm + SM + 16 * r);
      const uint32_t dd = ld_shared_u32(tm + DD + 4 * r);
      d[m][hh] = half_bits_to_float(dd), dmin[m][hh] = half_bits_to_float(dd >> 16);
    }
#pragma unroll
  for (int b = 0; b < 8; b++) {
    const int h = b & 1, j = b >> 1, blk = 8 * s + b;
    const MTok tk = m_tok<ACT_SMEM, true>(blk, t, K, ar_g, ar0, ar1, aq, ad, ag);
    const int byte = 8 * h + 2 * j;  // scale/min bytes of groups 0, 1: byte, byte + 1
#pragma unroll
    for (int m = 0; m < 2; m++) {
      uint32_t af[4], smp[2];
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int r = g + 8 * hh;
        const uint32_t wsel = byte >> 2;
        const uint32_t sw = wsel == 0 ? smr[m][hh].x : wsel == 1 ? smr[m][hh].y : wsel == 2 ? smr[m][hh].z : smr[m][hh].w;
        smp[hh] = sw >> (8 * (byte & 3));  // byte pair (group 0, group 1) in the low 16 bits
        uint32_t w0, w1;                   // the lane's code words of groups 0, 1
        if constexpr (Q4) {
          const uint32_t base = t0 + m * TILE + QS + 512 * j + 16 * (2 * r + h) + 4 * (t >> 1);
          w0 = ld_shared_u32(base), w1 = ld_shared_u32(base + 8);
          w0 = (w0 >> (4 * (t & 1))) & 0x0F0F0F0Fu, w1 = (w1 >> (4 * (t & 1))) & 0x0F0F0F0Fu;
        } else {
          const uint2 w = ld_shared_v2(t0 + m * TILE + QS + 512 * (j >> 1) + 16 * (2 * r + h) + 8 * (j & 1));
          w0 = (w.x >> (2 * t)) & M2, w1 = (w.y >> (2 * t)) & M2;
        }
        af[hh] = w0 * (smp[hh] & 15u);              // rows g / g + 8, K 4t..: group 0
        af[2 + hh] = w1 * ((smp[hh] >> 8) & 15u);   // K 16+4t..: group 1
      }
      int D[4];
      mma_u8s8(af, tk.b0, tk.b1, D);
#pragma unroll
      for (int hh = 0; hh < 2; hh++)
        m_sb_terms(acc.v[m][hh], d[m][hh], dmin[m][hh], D[2 * hh], D[2 * hh + 1], m_minterm(smp[hh], tk.gs0),
                   m_minterm(smp[hh], tk.gs1), tk.dx0, tk.dx1);
    }
  }
}

// One Q8_0 K-step (block s) of the two tiles at t0: A straight from the
// tiles' int8 rows with ldmatrix; terms (d * dx) * I.
template <bool ACT_SMEM>
__device__ __forceinline__ void q8_step_mma(uint32_t t0, int lane, int s, int K, int ar_g, int ar0, int ar1,
                                            const int8_t *__restrict__ aq, const float *__restrict__ ad,
                                            MChains &acc) {
  const int g = lane >> 2, t = lane & 3;
  const MTok tk = m_tok<ACT_SMEM, false>(s, t, K, ar_g, ar0, ar1, aq, ad, nullptr);
  const unsigned long long dx2 = f2_pack(tk.dx0, tk.dx1);
  const uint32_t lm = Q8_Q + 32 * (((lane >> 3) & 1) * 8 + (lane & 7)) + 16 * (lane >> 4);
#pragma unroll
  for (int m = 0; m < 2; m++) {
    const uint32_t tm = t0 + m * Q8_TILE;
    uint32_t af[4];
    ldsm_x4(tm + lm, af);
    int D[4];
    mma_s8s8(af, tk.b0, tk.b1, D);
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
      const uint32_t dw = ld_shared_u32(tm + 4 * ((g + 8 * hh) >> 1));
      const float dr = half_bits_to_float((g & 1) ? dw >> 16 : dw);
      float dd0, dd1;
      f2_unpack(f2_mul(f2_pack(dr, dr), dx2), dd0, dd1);
      acc.v[m][hh] = f2_add(acc.v[m][hh], f2_pack(__fmul_rn(dd0, __int2float_rn(D[2 * hh])),
                                                  __fmul_rn(dd1, __int2float_rn(D[2 * hh + 1]))));
    }
  }
}

}  // namespace ds4

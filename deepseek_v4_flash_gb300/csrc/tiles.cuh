// tiles.cuh -- per-K-step dot products of one RG32 weight tile (one row per
// lane) against up to TT activation rows, accumulated in CAS order.
#pragma once
#include "common.cuh"

namespace ds4 {

constexpr uint32_t M2 = 0x03030303u;

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
template <int TT>
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
        const uint4 x0 = __ldg(xv), x1 = __ldg(xv + 1);
        const uint32_t g2 = __ldg((const uint32_t *)(ag + (size_t)tok[i] * (K >> 4) + 2 * blk));
        const int gs0 = (int)(int16_t)(g2 & 0xFFFFu), gs1 = (int)(int16_t)(g2 >> 16);
        const int A = sc0 * grp_dot(w0, x0) + sc1 * grp_dot(w1, x1);
        const int B = mn0 * gs0 + mn1 * gs1;
        acc[i] = __fadd_rn(acc[i], q2s_term(__ldg(ad + (size_t)tok[i] * nb + blk), d, dmin, A, B));
      }
    }
  }
}

// One Q8 tile (32 rows x 64 K = 2 blocks) against TT activation rows.
template <int TT>
__device__ __forceinline__ void q8_tile(uint32_t tile, int lane, int s, int K, const int *tok,
                                        const int8_t *__restrict__ aq, const float *__restrict__ ad, float *acc) {
  const uint32_t dd = ld_shared_u32(tile + 4 * lane);
  const int nb = K >> 5;
#pragma unroll
  for (int bb = 0; bb < 2; bb++) {
    const float d = half_bits_to_float(bb ? dd >> 16 : dd);
    const uint4 q0 = ld_shared_v4(tile + Q8_Q + 512 * (2 * bb) + 16 * lane);
    const uint4 q1 = ld_shared_v4(tile + Q8_Q + 512 * (2 * bb + 1) + 16 * lane);
    const int blk = 2 * s + bb;
#pragma unroll
    for (int i = 0; i < TT; i++) {
      const uint4 *xv = (const uint4 *)(aq + (size_t)tok[i] * K + 32 * blk);
      const int I = dot16(q1, __ldg(xv + 1), dot16(q0, __ldg(xv), 0));
      acc[i] = __fadd_rn(acc[i], q8_term(d, __ldg(ad + (size_t)tok[i] * nb + blk), I));
    }
  }
}

// Q8 RG8x4 tile: 8 rows x one K-step of 64 (two Q8_0 blocks), 544 bytes:
//   [0,32)    fp16 d of (row r, block bb) at 4r + 2bb
//   [32,544)  lane l = 4r + c -> 16 bytes: row r, block c>>1, elements
//             16*(c&1) .. 16*(c&1)+15 of that block.
// Four lanes share a row: the two halves of a block are added as exact ints
// (one shuffle), then every lane of the row adds the two block terms to its
// copy of the row sum in block order (CAS step 4, S = 1).
constexpr int Q8X4_TILE = 544, Q8X4_Q = 32, Q8X4_KSTEP = 64;

template <int TT>
__device__ __forceinline__ void q8x4_tile(uint32_t tile, int lane, int s, int K, const int *tok,
                                          const int8_t *__restrict__ aq, const float *__restrict__ ad, float *acc) {
  const int r = lane >> 2, c = lane & 3, bb = c >> 1;
  const uint32_t dd = ld_shared_u32(tile + 4 * r);
  const float d = half_bits_to_float(bb ? dd >> 16 : dd);
  const uint4 q = ld_shared_v4(tile + Q8X4_Q + 16 * lane);
  const int nb = K >> 5, blk = 2 * s + bb;
  const int src0 = lane & ~3, src1 = src0 | 2;
#pragma unroll
  for (int i = 0; i < TT; i++) {
    const uint4 x = __ldg((const uint4 *)(aq + (size_t)tok[i] * K + 64 * s + 16 * c));
    int I = dot16(q, x, 0);
    I += __shfl_xor_sync(0xffffffffu, I, 1);
    const float p = q8_term(d, __ldg(ad + (size_t)tok[i] * nb + blk), I);
    const float p0 = __shfl_sync(0xffffffffu, p, src0);
    const float p1 = __shfl_sync(0xffffffffu, p, src1);
    acc[i] = __fadd_rn(__fadd_rn(acc[i], p0), p1);
  }
}

}  // namespace ds4

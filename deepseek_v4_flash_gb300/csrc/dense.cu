// dense.cu -- y = W x for a dense Q8_0 matrix beside the MoE (the output head,
// the attention projections) at decode-sized token counts.
//
// Two kernels, chained with programmatic dependent launch:
//   k_dense_quant  CAS step 1 on x: one warp per 32-block of a token;
//   k_dense<TT,MMA,NW> persistent, one block per SM, NW warps (16 for matrices
//                  of more 32-row items than 8-warp blocks have warps, else
//                  8). The work is cut
//                  into units: 32 output rows (two 16-row tiles per K step,
//                  the layout of an expert's down matrix) times a run of
//                  whole CAS segments of K. A warp streams its units' tiles
//                  through its own ring of 1-D bulk copies; lane l owns row
//                  l of the unit and keeps, per token, the row's segment chain
//                  (CAS step 3: (d * dx) * I, added in block order).
//                  Calls of two or more tokens take the block dots I of 16
//                  rows x 8 tokens from two fp16 tensor-core instructions
//                  (mma.sync m16n8k16, f32 accumulation): the int8 codes are
//                  exact in fp16 and every partial sum is an integer below
//                  2^24, so I comes out exact. (The int8 form, m16n8k32,
//                  would give the same bits but runs at a quarter of the
//                  fp16 form's rate here: 68 against 8.5 cycles per
//                  instruction and sub-partition, measured.) The tokens'
//                  codes are staged as fp16; the weights' codes are widened
//                  in registers after ldmatrix. Lane (g, t) then keeps the
//                  chains of rows g, g + 8 of both tiles for tokens 2t,
//                  2t + 1.
//                  Unsplit rows (one unit covers all S segments) add each
//                  finished segment to the row sum in order (CAS step 4) and
//                  store y. Split rows store their segment sums.
//                  The tokens' codes sit in shared memory once per pass of up
//                  to TT tokens (int8, or fp16 for the tensor-core step), TT
//                  chosen per call from n_tok.
//   k_dense_fix    (split calls only) adds each split row's S segment sums
//                  in segment order and stores y.
// Units go to warps SM-first (unit u to warp u / G of block u % G), so that a
// small matrix still spreads over every SM; rows are split where that evens
// out the units per warp. Nothing in the streaming kernel waits on another
// warp.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "common.cuh"
#include "internal.h"

struct ds4moe_dense {
  int N, K, N_pad, max_tokens, part_tokens, device, n_sm;
  int dbg_ks, dbg_nst, dbg_ns;  // launch geometry overrides, 0 = automatic
  int dbg_tc;                   // 0 automatic, 1 dp4a path only, 2 tensor-core path where it fits
  int nw;                       // warps per block
  uint8_t *w;        // [N_pad/32][K/32][2][Q8 tile], row halves swizzled (k_repack_q8 swz)
  int8_t *xq;        // [max_tokens][K]
  float *dx;         // [max_tokens][K/32]
  float *part;       // [S][part_tokens][N_pad] segment sums of split rows
  uint32_t *err;     // device error flags
  uint64_t bytes, launches;
};

namespace ds4 {

constexpr int DN_KB = 2 * Q8_TILE;       // one K step of a unit: two 16-row tiles, 1088 bytes
constexpr int DN_MAX_KS = 8;             // K steps per ring stage, at most
constexpr int DN_MAX_NST = 6;            // ring stages per warp, at most
constexpr int DN_TT_MAX = 8;             // tokens per pass, at most
constexpr size_t DN_SMEM_LIMIT = 227 * 1024;
constexpr size_t DN_STATIC = 1024;       // kept for the static barriers

struct DnArgs {
  int N, N_pad, K, T;
  int ks, nst, ns;    // K steps per stage, ring stages per warp, units per row
  const uint8_t *w;
  const int8_t *xq;
  const float *dx;
  float *y;
  float *part;
  uint32_t *err;
};

// One warp per 32-block (lane = element) of token blockIdx.y.
__global__ void __launch_bounds__(256) k_dense_quant(const float *x, int K, int8_t *xq, float *dx, uint32_t *err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * 8 + warp, t = blockIdx.y;
  pdl_launch_dependents();
  pdl_wait();
  if (b >= K / 32) return;
  const float v = x[(size_t)t * K + 32 * b + lane];
  if (__any_sync(0xffffffffu, !isfinite(v)) && lane == 0) raise_flag(err, DS4MOE_DEVERR_NONFINITE);
  const float d = __fdiv_rn(warp_max(fabsf(v)), 127.0f);
  xq[(size_t)t * K + 32 * b + lane] = (int8_t)cas_code(v, d);
  if (lane == 0) dx[(size_t)t * (K / 32) + b] = d;
}

// 32-element integer dot of a row block and an activation block.
__device__ __forceinline__ int dn_dot32(const uint4 &q0, const uint4 &q1, const uint4 &x0, const uint4 &x1) {
  int I = __dp4a((int)q0.x, (int)x0.x, 0);
  I = __dp4a((int)q0.y, (int)x0.y, I);
  I = __dp4a((int)q0.z, (int)x0.z, I);
  I = __dp4a((int)q0.w, (int)x0.w, I);
  I = __dp4a((int)q1.x, (int)x1.x, I);
  I = __dp4a((int)q1.y, (int)x1.y, I);
  I = __dp4a((int)q1.z, (int)x1.z, I);
  return __dp4a((int)q1.w, (int)x1.w, I);
}

__device__ __forceinline__ uint32_t dn_lds_u16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// ldmatrix: four 8x8 b16 matrices; lane i gives the address of row i % 8 of
// matrix i / 8 and receives, from each matrix, bytes 4*(i%4)..+3 of row i/4.
__device__ __forceinline__ void dn_ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Four int8 codes (one word, element j in byte j) -> the same integers as
// fp16 pairs: lo = (e0, e1), hi = (e2, e3). Each half is built as
// 1024 + 128 + q (the byte q ^ 0x80 under the exponent byte 0x64) and 1152
// is subtracted: exact, as every value involved is an integer below 2^11.
__device__ __forceinline__ void dn_i8x4_to_h(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u, E = 0x64646464u, C = 0x64806480u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(E));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(E));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(C));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(C));
}

// D += A B for A 16x16 (rows, K) and B 16x8 (K, tokens) of fp16, D f32.
// Lane (g, t) = (lane / 4, lane % 4) holds A rows g, g + 8 at K slots 2t,
// 2t + 1 (a0, a1) and 8 + 2t, 9 + 2t (a2, a3), B token g at the same slots,
// and D rows g, g + 8 for tokens 2t, 2t + 1. The K order inside one
// instruction is free (a sum): slot pairs (2t, 2t + 1) and (8 + 2t, 9 + 2t)
// carry the codes 4t, 4t + 1 and 4t + 2, 4t + 3 of the 16-code half, so that
// one 32-bit word of codes feeds both pairs of a lane.
__device__ __forceinline__ void dn_mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The terms (d_r * dx_k) * I of one row r for the lane's two tokens (I the
// exact block dots as floats), added to the row's packed pair of chains; the
// second products are scalar (a packed product whose only use is a packed
// add would be fused into one rounding).
__device__ __forceinline__ void dn_mma_terms(unsigned long long &acc, float d, unsigned long long dx2, float i0,
                                             float i1) {
  float dd0, dd1;
  f2_unpack(f2_mul(f2_pack(d, d), dx2), dd0, dd1);
  acc = f2_add(acc, f2_pack(__fmul_rn(dd0, i0), __fmul_rn(dd1, i1)));
}

// MMA = false: lane l owns row l of the unit and a chain per token (TT
// tokens per pass, dp4a dots). MMA = true: eight tokens per pass on the
// tensor cores (mma.sync m16n8k16, fp16 codes), lane (g, t) owns rows g,
// g + 8 of both tiles for tokens 2t, 2t + 1.
template <int TT, bool MMA, int NW>
__global__ void __launch_bounds__(NW * 32, 1) k_dense(DnArgs a) {
  static_assert(!MMA || TT == 8, "the tensor-core step takes eight tokens");
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = a.K >> 5, S = expert_segs(DS4MOE_Q8_0, a.K), per = nb / S;
  const int ks = a.ks, ns = a.ns, nst = a.nst;
  const int sbytes = ks * DN_KB;
  const int nbu = nb / ns, ust = nbu / ks;  // blocks and ring stages of one unit
  const int sst = per / ks;                 // ring stages of one segment
  const int n_units = (a.N_pad >> 5) * ns;
  const int G = gridDim.x, W = G * NW, gw = warp * G + blockIdx.x;
  const int my_units = gw < n_units ? (n_units - 1 - gw) / W + 1 : 0;
  const int n_pass = (a.T + TT - 1) / TT;
  // shared memory: the pass's codes [TT][K + 16] int8 (dp4a step) or
  // [TT][K + 16] fp16 (tensor-core step) and scales [TT][K/32 + 4], then the
  // rings; the rows' padding puts the tensor-core step's loads of eight
  // tokens' rows in different banks
  constexpr int CB = MMA ? 2 : 1;  // bytes per staged code
  const int xrow = CB * (a.K + 16), drow = nb + 4;
  int8_t *xs = (int8_t *)smem;
  float *ds = (float *)(smem + TT * xrow);
  const int ring_off = (TT * xrow + TT * drow * 4 + 127) & ~127;
  if constexpr (MMA) {  // rows of a short last pass stay defined (zero)
    for (int i = threadIdx.x; i < (TT * xrow + TT * drow * 4) / 16; i += blockDim.x)
      *(uint4 *)(smem + 16 * i) = make_uint4(0, 0, 0, 0);
    __syncthreads();
  }
  const uint32_t ring = smem_u32(smem + ring_off + warp * nst * sbytes);
  __shared__ uint64_t bars[NW][DN_MAX_NST];
  const uint32_t bar = smem_u32(&bars[warp][0]);
  if (lane == 0) {
    for (int i = 0; i < nst; i++) mbar_init(bar + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const size_t item_bytes = (size_t)nb * DN_KB;
  // producer cursor over (pass, unit, stage) of this warp; every lane keeps
  // it, lane 0 issues the copies. A slot is refilled only after every lane
  // has used the values it loaded from it (the warp barrier at the end of a
  // stage), so the copy cannot overwrite bytes still to be read.
  int pp = 0, pu = 0, pst = 0;
  uint32_t g_prod = 0, g_cons = 0;
  auto fill = [&]() {
    while (pp < n_pass && g_prod - g_cons < (uint32_t)nst) {
      if (pu >= my_units) {
        pp++, pu = 0, pst = 0;
        continue;
      }
      const int u = gw + pu * W, item = u / ns, part = u - item * ns;
      const uint32_t slot = g_prod % nst;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar + 8 * slot, sbytes);
        bulk_g2s(ring + slot * sbytes, a.w + (size_t)item * item_bytes + ((size_t)part * nbu + (size_t)pst * ks) * DN_KB,
                 sbytes, bar + 8 * slot);
      }
      g_prod++;
      if (++pst == ust) pst = 0, pu++;
    }
  };
  fill();  // constant weights, before the codes of x exist
  pdl_launch_dependents();
  pdl_wait();
  // dp4a step: row rr of tile m; tensor-core step: g, t4 as above, and the
  // ldmatrix row address of this lane within a tile. Rows 4-7 and 12-15 of a
  // tile hold their two 16-byte halves swapped (bank-conflict-free reads).
  const int m = lane >> 4, rr = lane & 15, rsw = 16 * ((rr >> 2) & 1);
  const int g = lane >> 2, t4 = lane & 3;
  const int lr = ((lane >> 3) & 1) * 8 + (lane & 7);
  const uint32_t lm_off = Q8_Q + 32 * lr + 16 * ((lane >> 4) ^ ((lr >> 2) & 1));
  const uint32_t xs_s = smem_u32(xs);
  bool failed = false;
  for (int p = 0; p < n_pass; p++) {
    const int t0 = p * TT, nt = min(TT, a.T - t0);
    __syncthreads();  // the previous pass is done with the staged codes
    {
      const int qrow = a.K / 16, nq = nt * qrow, nd = nt * nb;
      const uint4 *src = (const uint4 *)(a.xq + (size_t)t0 * a.K);
      for (int i = threadIdx.x; i < nq; i += blockDim.x) {
        const int r = i / qrow;
        const uint4 v = __ldg(src + i);
        if constexpr (MMA) {
          uint4 lo, hi;
          dn_i8x4_to_h(v.x, lo.x, lo.y);
          dn_i8x4_to_h(v.y, lo.z, lo.w);
          dn_i8x4_to_h(v.z, hi.x, hi.y);
          dn_i8x4_to_h(v.w, hi.z, hi.w);
          uint4 *d = (uint4 *)(xs + r * xrow + 32 * (i - r * qrow));
          d[0] = lo, d[1] = hi;
        } else {
          *(uint4 *)(xs + r * xrow + 16 * (i - r * qrow)) = v;
        }
      }
      for (int i = threadIdx.x; i < nd; i += blockDim.x) {
        const int r = i / nb;
        ds[r * drow + (i - r * nb)] = __ldg(a.dx + (size_t)t0 * nb + i);
      }
    }
    __syncthreads();
    // a warp that gave up a wait skips its units but still meets every pass
    // barrier of its block
    for (int iu = 0; iu < my_units && !failed; iu++) {
      const int u = gw + iu * W, item = u / ns, part = u - item * ns;
      float acc[MMA ? 1 : TT], tot[MMA ? 1 : TT];
      unsigned long long macc[2][2], mtot[2][2];  // [tile][row g, g + 8]: tokens (2t4, 2t4 + 1)
      if constexpr (MMA) {
#pragma unroll
        for (int i = 0; i < 4; i++) macc[i >> 1][i & 1] = 0ull, mtot[i >> 1][i & 1] = 0ull;
      } else {
#pragma unroll
        for (int t = 0; t < TT; t++) acc[t] = 0.0f, tot[t] = 0.0f;
      }
      int seg = part * (nbu / per);
      for (int st = 0; st < ust; st++) {
        fill();
        const uint32_t slot = g_cons % nst;
        if (!mbar_wait_bounded(bar + 8 * slot, (g_cons / nst) & 1)) {
          failed = true;
          break;
        }
        const uint32_t stage = ring + slot * sbytes;
        const int bst = part * nbu + st * ks;
        // the K steps of the stage, unrolled so that their loads and integer
        // dots overlap; the float terms join each chain in block order
#pragma unroll
        for (int j = 0; j < DN_MAX_KS; j++) {
          if (j < ks) {
            const int b = bst + j;
            if constexpr (MMA) {
              // token g's codes 32b + 4t4 .. +3 (first half) and 32b + 16 + 4t4 .. +3
              const uint2 bl = ld_shared_v2(xs_s + g * xrow + 64 * b + 8 * t4);
              const uint2 bh = ld_shared_v2(xs_s + g * xrow + 64 * b + 32 + 8 * t4);
              const unsigned long long dx2 = f2_pack(ds[(2 * t4) * drow + b], ds[(2 * t4 + 1) * drow + b]);
#pragma unroll
              for (int mt = 0; mt < 2; mt++) {
                const uint32_t tb = stage + j * DN_KB + mt * Q8_TILE;
                // af: rows g, g + 8 at codes 4t4..+3 (af[0], af[1]) and 16 + 4t4..+3 (af[2], af[3])
                uint32_t af[4], al[4], ah[4];
                dn_ldsm_x4(tb + lm_off, af[0], af[1], af[2], af[3]);
#pragma unroll
                for (int q = 0; q < 4; q++) dn_i8x4_to_h(af[q], al[q], ah[q]);
                float dv[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                dn_mma_f16(dv, al[0], al[1], ah[0], ah[1], bl.x, bl.y);
                dn_mma_f16(dv, al[2], al[3], ah[2], ah[3], bh.x, bh.y);
                dn_mma_terms(macc[mt][0], half_bits_to_float(dn_lds_u16(tb + 2 * g)), dx2, dv[0], dv[1]);
                dn_mma_terms(macc[mt][1], half_bits_to_float(dn_lds_u16(tb + 2 * (g + 8))), dx2, dv[2], dv[3]);
              }
            } else {
              const uint32_t tb = stage + j * DN_KB + m * Q8_TILE;
              const float d = half_bits_to_float(dn_lds_u16(tb + 2 * rr));
              const uint4 q0 = ld_shared_v4(tb + Q8_Q + 32 * rr + rsw), q1 = ld_shared_v4(tb + Q8_Q + 32 * rr + (16 - rsw));
#pragma unroll
              for (int t = 0; t < TT; t++) {
                if (t < nt) {  // warp-uniform
                  const uint4 *xp = (const uint4 *)(xs + t * xrow + 32 * b);
                  const int I = dn_dot32(q0, q1, xp[0], xp[1]);
                  acc[t] = __fadd_rn(acc[t], __fmul_rn(__fmul_rn(d, ds[t * drow + b]), __int2float_rn(I)));
                }
              }
            }
          }
        }
        if ((st + 1) % sst == 0) {  // a segment is complete (stages never straddle one)
          if constexpr (MMA) {
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const int mt = i >> 1, h = i & 1;
              if (ns == 1) {
                mtot[mt][h] = f2_add(mtot[mt][h], macc[mt][h]);
              } else {
                const int row = 32 * item + 16 * mt + g + 8 * h;
                float v0, v1;
                f2_unpack(macc[mt][h], v0, v1);
                if (2 * t4 < nt) a.part[((size_t)seg * a.T + t0 + 2 * t4) * a.N_pad + row] = v0;
                if (2 * t4 + 1 < nt) a.part[((size_t)seg * a.T + t0 + 2 * t4 + 1) * a.N_pad + row] = v1;
              }
              macc[mt][h] = 0ull;
            }
          } else {
            const int row = 32 * item + 16 * m + rr;
#pragma unroll
            for (int t = 0; t < TT; t++) {
              if (t < nt) {
                if (ns == 1) tot[t] = __fadd_rn(tot[t], acc[t]);
                else a.part[((size_t)seg * a.T + t0 + t) * a.N_pad + row] = acc[t];
              }
              acc[t] = 0.0f;
            }
          }
          seg++;
        }
        __syncwarp();  // every lane is done with the slot before it is refilled
        g_cons++;
      }
      if (failed) break;
      if (ns == 1) {
        if constexpr (MMA) {
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const int mt = i >> 1, h = i & 1;
            const int row = 32 * item + 16 * mt + g + 8 * h;
            float v0, v1;
            f2_unpack(mtot[mt][h], v0, v1);
            if (row < a.N) {
              if (2 * t4 < nt) a.y[(size_t)(t0 + 2 * t4) * a.N + row] = v0;
              if (2 * t4 + 1 < nt) a.y[(size_t)(t0 + 2 * t4 + 1) * a.N + row] = v1;
            }
          }
        } else {
          const int row = 32 * item + 16 * m + rr;
#pragma unroll
          for (int t = 0; t < TT; t++)
            if (t < nt && row < a.N) a.y[(size_t)(t0 + t) * a.N + row] = tot[t];
        }
      }
    }
  }
  if (failed) {
    if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
    // the warp's own copies in flight land before the block may leave
    for (uint32_t gg = g_cons; gg < g_prod; gg++) (void)mbar_wait_bounded(bar + 8 * (gg % nst), (gg / nst) & 1);
  }
}

// Split rows: y[t][r] = the CAS row sum of the S stored segment sums, in
// segment order. One thread per (token, row).
__global__ void __launch_bounds__(256) k_dense_fix(const float *__restrict__ part, float *y, int N, int N_pad, int T,
                                                   int S) {
  pdl_launch_dependents();
  pdl_wait();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)T * N) return;
  const int t = (int)(i / N), r = (int)(i - (long long)t * N);
  float s = 0.0f;
  for (int sg = 0; sg < S; sg++) s = __fadd_rn(s, __ldcg(part + ((size_t)sg * T + t) * N_pad + r));
  y[i] = s;
}

// Tokens per pass, at most, for K: the codes of a pass take at most 64 KB.
static int dn_tt_cap(int K) {
  const size_t per_tok = (size_t)(K + 16) + (size_t)(K / 32 + 4) * 4;
  int tt = DN_TT_MAX;
  while (tt > 1 && (size_t)tt * per_tok > 65536) tt >>= 1;
  return tt;
}

// Tokens per pass for a call of T tokens: the smallest power of two that
// holds them, up to the cap.
static int dn_tt(int K, int T) {
  const int cap = dn_tt_cap(K);
  int tt = 1;
  while (tt < T && tt < cap) tt <<= 1;
  return tt;
}

// The pass's staged codes (int8, or fp16 for the tensor-core step) and scales.
static size_t dn_stage_smem(int TT, int K, bool mma) {
  return ((size_t)TT * (K + 16) * (mma ? 2 : 1) + (size_t)TT * (K / 32 + 4) * 4 + 127) & ~(size_t)127;
}

// Ring geometry: the largest K steps per stage (a divisor of a segment's
// blocks, at most 8) that still leaves every warp two stages, else one K
// step per stage; stages per warp from the shared memory left. Long stages
// win: a stage's K steps run unrolled, and each stage costs a wait.
static void dn_ring(int TT, int K, bool mma, int nw, int &ks, int &nst) {
  const int nb = K / 32, per = nb / expert_segs(DS4MOE_Q8_0, K);
  const size_t st = dn_stage_smem(TT, K, mma);
  if (st + (size_t)nw * 2 * DN_KB > DN_SMEM_LIMIT - DN_STATIC) {  // not even two one-step stages
    ks = 1, nst = 0;
    return;
  }
  const size_t left = DN_SMEM_LIMIT - DN_STATIC - st;
  for (ks = per < DN_MAX_KS ? per : DN_MAX_KS; ks > 1; ks--) {
    if (per % ks) continue;
    if (left / ((size_t)nw * ks * DN_KB) >= 2) break;
  }
  const size_t n = left / ((size_t)nw * ks * DN_KB);
  nst = n > DN_MAX_NST ? DN_MAX_NST : (int)n;
}

// Units per 32-row item: the split (a power of two dividing S) that best
// evens out the units per warp, the smallest one within 2 % of the best;
// only for a call of one pass that the segment-sum scratch holds. A split
// costs a store and a load of S sums per row and token, and the fix-up
// launch.
static int dn_split(const ds4moe_dense *h, int T, int TT) {
  if (T > TT || T > h->part_tokens || !h->part) return 1;
  const int S = expert_segs(DS4MOE_Q8_0, h->K);
  const long long items = h->N_pad / 32, W = (long long)h->n_sm * h->nw;
  auto eff = [&](int ns) {
    const long long u = items * ns, rounds = (u + W - 1) / W;
    return (double)u / (double)(rounds * W);
  };
  double best = 0.0;
  for (int ns = 1; ns <= S; ns <<= 1)
    if (S % ns == 0 && eff(ns) > best) best = eff(ns);
  for (int ns = 1; ns <= S; ns <<= 1)
    if (S % ns == 0 && eff(ns) >= best - 0.02) return ns;
  return 1;
}

}  // namespace ds4

using namespace ds4;

namespace {

bool dn_dev_ptr(const void *p) {
  if (!p) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

ds4moe_status dn_status(cudaError_t e) {
  if (e == cudaSuccess) return DS4MOE_OK;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? DS4MOE_ERR_OOM : DS4MOE_ERR_CUDA;
}

void dn_free(ds4moe_dense *h) {
  if (h->w) cudaFree(h->w);
  if (h->xq) cudaFree(h->xq);
  if (h->dx) cudaFree(h->dx);
  if (h->part) cudaFree(h->part);
  if (h->err) cudaFree(h->err);
}

template <int TT, bool MMA, int NW>
cudaError_t dn_launch_nw(ds4moe_dense *h, const DnArgs &a0, cudaStream_t s) {
  DnArgs a = a0;
  dn_ring(TT, h->K, MMA, NW, a.ks, a.nst);
  a.ns = dn_split(h, a.T, TT);
  if (h->dbg_ks || h->dbg_nst) {
    const int ks = h->dbg_ks ? h->dbg_ks : a.ks, nst = h->dbg_nst ? h->dbg_nst : a.nst;
    if (dn_stage_smem(TT, h->K, MMA) + (size_t)NW * nst * ks * DN_KB <= DN_SMEM_LIMIT - DN_STATIC)
      a.ks = ks, a.nst = nst;
  }
  if (h->dbg_ns) a.ns = (a.T <= TT && a.T <= h->part_tokens) ? h->dbg_ns : 1;
  void *args[] = {&a};
  const size_t smem = dn_stage_smem(TT, h->K, MMA) + (size_t)NW * a.nst * a.ks * DN_KB;
  cudaError_t e = launch_pdl((const void *)k_dense<TT, MMA, NW>, dim3(h->n_sm), dim3(NW * 32), smem, s, args, true);
  h->launches++;
  if (e == cudaSuccess && a.ns > 1) {
    int S = expert_segs(DS4MOE_Q8_0, h->K);
    const long long n = (long long)a.T * h->N;
    void *fargs[] = {(void *)&a.part, (void *)&a.y, (void *)&a.N, (void *)&a.N_pad, (void *)&a.T, (void *)&S};
    e = launch_pdl((const void *)k_dense_fix, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, fargs, true);
    h->launches++;
  }
  return e;
}

template <int TT, bool MMA>
cudaError_t dn_launch(ds4moe_dense *h, const DnArgs &a, cudaStream_t s) {
  return h->nw == 16 ? dn_launch_nw<TT, MMA, 16>(h, a, s) : dn_launch_nw<TT, MMA, 8>(h, a, s);
}

}  // namespace

extern "C" {

ds4moe_status ds4moe_dense_create(int32_t n_out, int32_t n_in, int32_t max_tokens, const void *w_q8,
                                  ds4moe_dense **out) {
  if (!out) return DS4MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_out < 1 || n_out > (1 << 24) || n_in < 32 || n_in > (1 << 16) || n_in % 32) return DS4MOE_ERR_INVALID_ARG;
  if ((n_in / 32) % expert_segs(DS4MOE_Q8_0, n_in)) return DS4MOE_ERR_INVALID_ARG;
  if (max_tokens < 1 || max_tokens > (1 << 16)) return DS4MOE_ERR_INVALID_ARG;
  if ((long long)max_tokens * n_out >= (1ll << 40)) return DS4MOE_ERR_INVALID_ARG;
  if (!dn_dev_ptr(w_q8)) return DS4MOE_ERR_INVALID_ARG;
  // Warps per block: 16 where every warp of 8-warp blocks would get more
  // than one 32-row item, else 8. Measured: the 129280 x 4096 head 1-4 %
  // faster with 16 (more warps hide the per-block latencies), a 4096 x 4096
  // projection 5 % slower (its units fit one 8-warp ring in flight).
  int n_sm = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_CUDA;
  }
  const int nw = (long long)((n_out + 31) / 32) > (long long)n_sm * 8 ? 16 : 8;
  {
    int ks, nst;
    dn_ring(dn_tt_cap(n_in), n_in, false, nw, ks, nst);
    if (nst < 2) return DS4MOE_ERR_UNSUPPORTED;
  }
  ds4moe_dense *h = new (std::nothrow) ds4moe_dense;
  if (!h) return DS4MOE_ERR_OOM;
  memset(h, 0, sizeof(*h));
  h->N = n_out, h->K = n_in, h->N_pad = (n_out + 31) / 32 * 32, h->max_tokens = max_tokens;
  h->part_tokens = max_tokens < DN_TT_MAX ? max_tokens : DN_TT_MAX;
  h->nw = nw;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->device);
  const size_t wb = (size_t)h->N_pad / 32 * (n_in / 32) * DN_KB;
  const size_t qb = (size_t)max_tokens * n_in, db = (size_t)max_tokens * (n_in / 32) * 4;
  const size_t pb = (size_t)expert_segs(DS4MOE_Q8_0, n_in) * h->part_tokens * h->N_pad * 4;
  for (const void *fn : {(const void *)k_dense<1, false, 8>, (const void *)k_dense<2, false, 8>,
                         (const void *)k_dense<4, false, 8>, (const void *)k_dense<8, false, 8>,
                         (const void *)k_dense<8, true, 8>, (const void *)k_dense<1, false, 16>,
                         (const void *)k_dense<2, false, 16>, (const void *)k_dense<4, false, 16>,
                         (const void *)k_dense<8, false, 16>, (const void *)k_dense<8, true, 16>})
    if (e == cudaSuccess)  // the static barriers take their part of the block's shared memory
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(DN_SMEM_LIMIT - DN_STATIC));
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->w, wb);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->xq, qb);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->dx, db);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->part, pb);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->err, 64);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->w, 0, wb, 0);  // padding rows stay zero
  if (e == cudaSuccess) e = cudaMemsetAsync(h->err, 0, 64, 0);
  if (e == cudaSuccess) e = repack_q8((const uint8_t *)w_q8, h->w, 1, n_out, n_in, 2, 0, 0, true);
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  if (e != cudaSuccess) {
    const ds4moe_status st = dn_status(e);
    cudaDeviceSynchronize();
    cudaGetLastError();
    dn_free(h);
    delete h;
    return st;
  }
  h->bytes = wb + qb + db + pb + 64;
  *out = h;
  return DS4MOE_OK;
}

void ds4moe_dense_destroy(ds4moe_dense *h) {
  if (!h) return;
  cudaDeviceSynchronize();
  dn_free(h);
  delete h;
}

ds4moe_status ds4moe_dense_forward(ds4moe_dense *h, const float *x, int32_t n_tok, float *y, void *stream) {
  if (!h || n_tok < 0 || n_tok > h->max_tokens) return DS4MOE_ERR_INVALID_ARG;
  if (n_tok == 0) return DS4MOE_OK;
  if (!dn_dev_ptr(x) || !dn_dev_ptr(y)) return DS4MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int K = h->K;
  cudaError_t e;
  {
    void *args[] = {(void *)&x, (void *)&K, (void *)&h->xq, (void *)&h->dx, (void *)&h->err};
    e = launch_pdl((const void *)k_dense_quant, dim3((K / 32 + 7) / 8, n_tok), dim3(256), 0, s, args, true);
  }
  if (e == cudaSuccess) {
    DnArgs a = {};
    a.N = h->N, a.N_pad = h->N_pad, a.K = K, a.T = n_tok;
    a.w = h->w, a.xq = h->xq, a.dx = h->dx, a.y = y, a.part = h->part, a.err = h->err;
    // two or more tokens: the tensor-core step (passes of eight tokens),
    // where eight tokens' fp16 codes leave room for the rings
    int tks, tnst;
    dn_ring(DN_TT_MAX, K, true, h->nw, tks, tnst);
    const bool fits = tnst >= 2;
    const bool tc = fits && (h->dbg_tc == 2 || (h->dbg_tc == 0 && n_tok >= 2));
    if (tc) {
      e = dn_launch<8, true>(h, a, s);
    } else {
      switch (dn_tt(K, n_tok)) {
        case 8: e = dn_launch<8, false>(h, a, s); break;
        case 4: e = dn_launch<4, false>(h, a, s); break;
        case 2: e = dn_launch<2, false>(h, a, s); break;
        default: e = dn_launch<1, false>(h, a, s); break;
      }
    }
  }
  h->launches++;  // the quantisation; dn_launch counts its own
  return dn_status(e);
}

ds4moe_status ds4moe_dense_get_device_error(ds4moe_dense *h, void *stream, uint32_t *flags_out) {
  if (!h) return DS4MOE_ERR_INVALID_ARG;
  uint32_t f = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemcpy(&f, h->err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, 4);
  if (e != cudaSuccess) return dn_status(e);
  if (flags_out) *flags_out = f;
  return f ? DS4MOE_ERR_DEVICE : DS4MOE_OK;
}

ds4moe_status ds4moe_dense_debug_config(ds4moe_dense *h, int32_t ks, int32_t nst, int32_t ns, int32_t tc) {
  if (!h || ks < 0 || nst < 0 || ns < 0 || tc < 0 || tc > 2) return DS4MOE_ERR_INVALID_ARG;
  const int S = expert_segs(DS4MOE_Q8_0, h->K), per = h->K / 32 / S;
  if (ks && (ks > DN_MAX_KS || per % ks)) return DS4MOE_ERR_INVALID_ARG;
  if (nst && (nst < 2 || nst > DN_MAX_NST)) return DS4MOE_ERR_INVALID_ARG;
  if (ns && S % ns) return DS4MOE_ERR_INVALID_ARG;
  h->dbg_ks = ks, h->dbg_nst = nst, h->dbg_ns = ns, h->dbg_tc = tc;
  return DS4MOE_OK;
}

uint64_t ds4moe_dense_device_bytes(const ds4moe_dense *h) { return h ? h->bytes : 0; }
uint64_t ds4moe_dense_launch_count(const ds4moe_dense *h) { return h ? h->launches : 0; }

}  // extern "C"

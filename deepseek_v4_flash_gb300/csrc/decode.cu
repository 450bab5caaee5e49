// decode.cu -- the decode-batch path (n_tok <= DEC_MAX_T): three kernels
// chained with programmatic dependent launch (PDL):
//
//   K1 k_route_dec  : int8 quantisation of x + router GEMV segment sums; the
//                     last CTA of each token tile runs sigmoid + bias top-k +
//                     renormalisation (or the hash lookup), and the last
//                     token tile buckets the (token, slot) pairs by expert.
//   K2 k_gateup_dec : gate/up of every (expert, row group) with in-register
//                     SwiGLU and the int8 requant of h.
//   K3 k_down_dec   : down of every (expert, row group); the last writer of
//                     each (token, 32 rows) adds the fixed-order combine into y.
//
// K2 and K3 are persistent: every warp is an independent streamer that
// claims work items from a global queue (largest items first: the shared
// expert), keeps DEC_NST stages of its item sequence in flight with 1-D bulk
// async copies into a shared-memory ring, and crosses item boundaries without
// draining the ring. Items of the shared expert are claimed before
// griddepcontrol.wait, so its weights stream while the previous kernel is
// still finishing. Queues and tickets reset themselves, so no per-call
// memset is needed and the whole forward can be captured in a CUDA graph.
//
// Prior art: the decode MoE kernels named in the ds4-rocm fork README
// (moe_gate_up_mid_decode_lut_qwarp32, moe_down_sum6_qwarp32) fuse the same
// steps on an RDNA iGPU; the work split, layouts and pipeline here are
// sm_103a-specific.
#include "bucket.cuh"
#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"

namespace ds4 {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ===========================================================================
// K1: routing.

constexpr int RD_RT = 8;      // tokens per token tile (one warp per token in top-k)
constexpr int RD_WARPS = 8;   // warps per CTA: one router row group each

struct RouteDecArgs {
  const float *x;
  const int32_t *tok;
  int T, H, E, E_pad, k, NS, n_shared, route, router_fmt, vocab;
  float scale;
  const uint8_t *W;            // router (Q8 RG32 or F32 [E][H])
  const float *bias;
  const int32_t *hash;
  int8_t *xq;
  float *dx;
  int16_t *gs;
  float *rpart;                // [T][8][E_pad]
  int32_t *ids;
  float *w;
  int32_t *cnt, *off, *active, *n_active, *list;
  int32_t *tick;               // [n_tiles + 1], self-resetting
  uint32_t *err;
};

// Quantise block b (32 values) of token t: lane = element.
__device__ __forceinline__ void quant_block(const float *x, int H, int t, int b, int lane, int8_t *xq_s,
                                            float *dx_s, int8_t *xq_g, float *dx_g, int16_t *gs_g, uint32_t *err) {
  const float v = __ldg(x + (size_t)t * H + 32 * b + lane);
  if (__any_sync(0xffffffffu, !isfinite(v)) && lane == 0) raise_flag(err, DS4MOE_DEVERR_NONFINITE);
  const float amax = warp_max(fabsf(v));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = cas_code(v, d);
  if (xq_s) xq_s[lane] = (int8_t)q;
  if (dx_s && lane == 0) *dx_s = d;
  if (xq_g) {
    const int s = half_warp_sum(q);
    xq_g[(size_t)t * H + 32 * b + lane] = (int8_t)q;
    if (lane == 0) dx_g[(size_t)t * (H >> 5) + b] = d;
    if ((lane & 15) == 0) gs_g[(size_t)t * (H >> 4) + 2 * b + (lane >> 4)] = (int16_t)s;
  }
}

// grid: (ceil(E_pad/32 / RD_WARPS), ROUTER_SEGS, n_tiles); block RD_WARPS*32.
// Each warp: router row group rg = blockIdx.x*RD_WARPS + warp, K segment seg,
// tokens of tile blockIdx.z. For hash routing the router part is skipped.
__global__ void __launch_bounds__(RD_WARPS * 32) k_route_dec(RouteDecArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.y, tile = blockIdx.z;
  const int t0 = tile * RD_RT, nt = min(RD_RT, a.T - t0);
  const int nb = a.H >> 5, per = nb / ROUTER_SEGS, b0 = seg * per;
  const bool learned = a.route == DS4MOE_ROUTE_LEARNED;
  const bool q8 = learned && a.router_fmt == DS4MOE_Q8_0;
  pdl_launch_dependents();

  // shared memory: [router tiles: RD_WARPS x seg_bytes][xq: RD_RT x per*32][dx: RD_RT x per][bar][misc]
  const int c0 = b0 >> 1, c1 = (b0 + per + 1) >> 1;  // Q8 2-block chunks covering the segment
  const int seg_bytes = q8 ? (c1 - c0) * Q8_TILE : 0;
  uint8_t *wsm = smem;
  int8_t *xq_s = (int8_t *)(smem + RD_WARPS * seg_bytes);
  float *dx_s = (float *)(xq_s + RD_RT * per * 32);
  uint64_t *bars = (uint64_t *)(dx_s + RD_RT * per + 2);
  int *misc = (int *)(bars + RD_WARPS);
  const int rg = blockIdx.x * RD_WARPS + warp;
  const bool row_ok = learned && rg < (a.E_pad >> 5);

  if (q8 && lane == 0) {
    const uint32_t bar = smem_u32(&bars[warp]);
    mbar_init(bar, 1);
    fence_mbar_init();
    if (row_ok) {
      mbar_arrive_expect_tx(bar, seg_bytes);
      bulk_g2s(smem_u32(wsm + warp * seg_bytes), a.W + ((size_t)rg * (a.H / Q8_KSTEP) + c0) * Q8_TILE, seg_bytes,
               bar);
    }
  }

  // Quantise this segment's blocks of the tile's tokens (all warps share it);
  // CTAs with blockIdx.x == 0 also publish the codes for the expert kernels.
  const bool publish = blockIdx.x == 0;
  for (int p = warp; p < nt * per; p += RD_WARPS) {
    const int i = p / per, b = b0 + p % per;
    quant_block(a.x, a.H, t0 + i, b, lane, xq_s + i * per * 32 + (b - b0) * 32, dx_s + i * per + (b - b0),
                publish ? a.xq : nullptr, a.dx, a.gs, a.err);
  }
  __syncthreads();

  if (row_ok) {
    float acc[RD_RT];
#pragma unroll
    for (int i = 0; i < RD_RT; i++) acc[i] = 0.0f;
    const int r = 32 * rg + lane;
    if (q8) {
      if (!mbar_wait_bounded(smem_u32(&bars[warp]), 0)) {
        if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
      } else {
        const uint32_t wt = smem_u32(wsm + warp * seg_bytes);
        for (int b = b0; b < b0 + per; b++) {
          const uint32_t tile = wt + ((b >> 1) - c0) * Q8_TILE;
          const uint32_t dd = ld_shared_u32(tile + 4 * lane);
          const float d = half_bits_to_float((b & 1) ? dd >> 16 : dd);
          const uint4 w0 = ld_shared_v4(tile + Q8_Q + 512 * (2 * (b & 1)) + 16 * lane);
          const uint4 w1 = ld_shared_v4(tile + Q8_Q + 512 * (2 * (b & 1) + 1) + 16 * lane);
#pragma unroll
          for (int i = 0; i < RD_RT; i++) {
            if (i < nt) {
              const uint4 *xv = (const uint4 *)(xq_s + i * per * 32 + (b - b0) * 32);
              const int I = dot16(w1, xv[1], dot16(w0, xv[0], 0));
              acc[i] = __fadd_rn(acc[i], q8_term(d, dx_s[i * per + (b - b0)], I));
            }
          }
        }
      }
    } else if (r < a.E) {  // fp32 router rows: fma chains over the segment (x unquantised)
      const int e0 = seg * (a.H / ROUTER_SEGS), e1 = e0 + a.H / ROUTER_SEGS;
      const float *wr = (const float *)a.W + (size_t)r * a.H;
      for (int i = 0; i < nt; i++) {
        const float *xv = a.x + (size_t)(t0 + i) * a.H;
        float s = 0.0f;
        for (int j = e0; j < e1; j++) s = __fmaf_rn(__ldg(wr + j), __ldg(xv + j), s);
        acc[i] = s;
      }
    }
#pragma unroll
    for (int i = 0; i < RD_RT; i++)
      if (i < nt) a.rpart[((size_t)(t0 + i) * ROUTER_SEGS + seg) * a.E_pad + r] = acc[i];
  }

  // ---- last CTA of this token tile: top-k (one warp per token)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) misc[0] = atomicAdd(&a.tick[tile], 1);
  __syncthreads();
  const int per_tile = gridDim.x * gridDim.y;
  if (misc[0] != per_tile - 1) return;
  __threadfence();
  if (warp < nt) {
    const int t = t0 + warp;
    if (learned) {
      // lane owns experts lane + 32 j
      float bk = 0.0f;
      const int nj = (a.E + 31) >> 5;
      int taken = 0;  // bit j: expert lane+32j taken (E <= 1024 -> nj <= 32)
      float *sv = (float *)(misc + 4) + warp * 2 * a.E_pad;  // s | key per warp (shared scratch)
      for (int j = 0; j < nj; j++) {
        const int e = lane + 32 * j;
        if (e < a.E) {
          float lg = 0.0f;
#pragma unroll
          for (int g = 0; g < ROUTER_SEGS; g++)
            lg = __fadd_rn(lg, __ldcg(a.rpart + ((size_t)t * ROUTER_SEGS + g) * a.E_pad + e));
          const float s = cas_sigmoid(lg);
          sv[e] = s;
          sv[a.E_pad + e] = __fadd_rn(s, __ldg(a.bias + e));
        }
      }
      __syncwarp();
      int sel[16];
      for (int j = 0; j < a.k; j++) {
        int bi = -1;
        for (int jj = 0; jj < nj; jj++) {
          const int e = lane + 32 * jj;
          if (e >= a.E || ((taken >> jj) & 1)) continue;
          const float ke = sv[a.E_pad + e];
          if (bi < 0 || ke > bk) bk = ke, bi = e;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (oi >= 0 && (bi < 0 || ok > bk || (ok == bk && oi < bi))) bk = ok, bi = oi;
        }
        sel[j] = bi;
        if (bi >= 0 && (bi & 31) == lane) taken |= 1 << (bi >> 5);
      }
      if (lane == 0) {
        float sum = 0.0f;
        for (int j = 0; j < a.k; j++) sum = __fadd_rn(sum, sel[j] >= 0 ? sv[sel[j]] : 0.0f);
        for (int j = 0; j < a.k; j++) {
          a.ids[(size_t)t * a.k + j] = sel[j];
          a.w[(size_t)t * a.k + j] = sel[j] >= 0 ? __fmul_rn(__fdiv_rn(sv[sel[j]], sum), a.scale) : 0.0f;
        }
      }
    } else if (lane == 0) {
      const int v = __ldg(a.tok + t);
      const bool ok = v >= 0 && v < a.vocab;
      if (!ok) raise_flag(a.err, DS4MOE_DEVERR_TOKEN_ID);
      const float wk = __fmul_rn(__fdiv_rn(1.0f, (float)a.k), a.scale);
      for (int j = 0; j < a.k; j++) {
        a.ids[(size_t)t * a.k + j] = ok ? __ldg(a.hash + (size_t)v * a.k + j) : -1;
        a.w[(size_t)t * a.k + j] = ok ? wk : 0.0f;
      }
    }
  }
  if (threadIdx.x == 0) a.tick[tile] = 0;  // reset for the next call
  // ---- last token tile: bucket every token
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) misc[1] = atomicAdd(&a.tick[gridDim.z], 1);
  __syncthreads();
  if (misc[1] != (int)gridDim.z - 1) return;
  __threadfence();
  bucket_block(a.ids, a.T, a.E, a.k, a.NS, a.n_shared, (int32_t *)(misc + 4), a.cnt, a.off, a.active, a.n_active,
               a.list, a.err);
  if (threadIdx.x == 0) a.tick[gridDim.z] = 0;
}

// ===========================================================================
// K2 / K3: persistent expert GEMV streamers.

constexpr int DEC_WARPS = 4;     // streamers per CTA
constexpr int DEC_NST = 8;       // ring stages per streamer
constexpr int DEC_STRIDE = 5376; // ring slot bytes (largest stage)
constexpr int DEC_SMEM = DEC_WARPS * (DEC_NST * DEC_STRIDE + DEC_NST * 8 + DEC_NST * 16);

enum { KIND_SH8 = 0, KIND_RG32_Q2S = 1, KIND_RG32_Q8 = 2 };

struct DecArgs {
  int H, F, E, k, NS, n_shared, rf, sf, down;
  int K;                         // reduction length: H (gate/up) or F (down)
  int rows;                      // output rows of the matrices: F (gate/up) or H (down)
  const uint8_t *w_r;            // routed weights, RG32
  const uint8_t *w_s;            // shared weights: RG8x4 if Q8 else RG32
  const int8_t *aq;              // activation codes: xq [T][H] or hq [T*NS][F]
  const float *ad;
  const int16_t *ag;
  const int32_t *cnt, *off, *active, *n_active, *list;
  const int32_t *ids;
  const float *w;
  int8_t *hq;
  float *dh;
  int16_t *gsh;
  float *hbuf;                   // [T*NS][F] h before requant (8-row items)
  int32_t *hticket;              // [T*NS][F/32]
  float *apart;                  // [T*NS][H]
  int32_t *cticket;              // [T][H/32]
  float *y;
  int32_t *queue;                // [2] claim counter, exited streamers
  uint32_t *err;
};

struct ItemDesc {
  const uint8_t *src;
  int kind, e, rg, nstages, sbytes, ksps;  // ksps: K-steps per stage
  int n_tok, list_off;
};

__device__ __forceinline__ int shared_items(const DecArgs &a) {
  if (!a.n_shared) return 0;
  return a.sf == DS4MOE_Q8_0 ? a.rows / 8 : a.rows / 32;
}

__device__ __forceinline__ int kstep_bytes(const DecArgs &a, int kind) {
  const int mats = a.down ? 1 : 2;
  return mats * (kind == KIND_SH8 ? Q8X4_TILE : kind == KIND_RG32_Q2S ? Q2S_TILE : Q8_TILE);
}

__device__ __forceinline__ int kstep_len(int kind) { return kind == KIND_RG32_Q2S ? Q2S_KSTEP : Q8_KSTEP; }

// K-steps per stage: as many as fit a ring slot, dividing the K-step count.
__device__ __forceinline__ int stage_ksteps(int kbytes, int nks) {
  int s = DEC_STRIDE / kbytes;
  if (s > nks) s = nks;
  while (s > 1 && nks % s) s--;
  return s < 1 ? 1 : s;
}

// Weight-side description of item i (valid for shared items before the
// dependency wait; routed items need the bucket).
__device__ ItemDesc item_desc(const DecArgs &a, int i, bool routing_known) {
  ItemDesc d;
  const int nsh = shared_items(a);
  const int nks_k = a.K;
  if (i < nsh) {
    d.kind = a.sf == DS4MOE_Q8_0 ? KIND_SH8 : KIND_RG32_Q2S;
    if (a.sf == DS4MOE_Q8_0) d.kind = KIND_SH8;
    d.e = a.E;
    d.rg = i;
  } else {
    const int RG = a.rows / 32;
    const int j = i - nsh;
    d.kind = a.rf == DS4MOE_Q2S ? KIND_RG32_Q2S : KIND_RG32_Q8;
    d.e = routing_known ? a.active[a.n_shared + j / RG] : -1;
    d.rg = j % RG;
  }
  const int nks = nks_k / kstep_len(d.kind);
  const int kb = kstep_bytes(a, d.kind);
  d.ksps = stage_ksteps(kb, nks);
  d.nstages = nks / d.ksps;
  d.sbytes = d.ksps * kb;
  const size_t item_bytes = (size_t)nks * kb;
  if (d.e == a.E) {
    d.src = a.w_s + (size_t)d.rg * item_bytes;
  } else if (d.e >= 0) {
    const int RG = a.rows / 32;
    d.src = a.w_r + ((size_t)d.e * RG + d.rg) * item_bytes;
  } else {
    d.src = nullptr;
  }
  d.n_tok = 0, d.list_off = 0;
  if (routing_known && d.e >= 0) {
    d.n_tok = a.cnt[d.e];
    d.list_off = a.off[d.e];
  }
  return d;
}

__device__ __forceinline__ int warp_claim(int32_t *q, int lane) {
  int v = 0;
  if (lane == 0) v = atomicAdd(q, 1);
  return __shfl_sync(0xffffffffu, v, 0);
}

// Token tile of pass p: activation rows (token index for gate/up, slot row
// for down) and slot rows for the outputs.
template <int TT>
__device__ __forceinline__ void load_tokens(const DecArgs &a, const ItemDesc &d, int pass, int *arow, int *srow,
                                            int *nt) {
  const int t0 = pass * TT;
  *nt = min(TT, d.n_tok - t0);
#pragma unroll
  for (int i = 0; i < TT; i++) {
    const int sr = __ldg(a.list + d.list_off + min(t0 + i, d.n_tok - 1));
    srow[i] = sr;
    arow[i] = a.down ? sr : sr / a.NS;
  }
}

template <int TT>
__device__ __forceinline__ void run_ksteps(const DecArgs &a, const ItemDesc &d, uint32_t st, int stage, int lane,
                                           const int *arow, float *acc0, float *acc1) {
  const int kb = kstep_bytes(a, d.kind), tb = a.down ? kb : kb / 2;
  for (int j = 0; j < d.ksps; j++) {
    const int s = stage * d.ksps + j;
    const uint32_t t = st + j * kb;
    if (d.kind == KIND_RG32_Q2S) {
      q2s_tile<TT>(t, lane, s, a.K, arow, a.aq, a.ad, a.ag, acc0);
      if (!a.down) q2s_tile<TT>(t + tb, lane, s, a.K, arow, a.aq, a.ad, a.ag, acc1);
    } else if (d.kind == KIND_RG32_Q8) {
      q8_tile<TT>(t, lane, s, a.K, arow, a.aq, a.ad, acc0);
      if (!a.down) q8_tile<TT>(t + tb, lane, s, a.K, arow, a.aq, a.ad, acc1);
    } else {
      q8x4_tile<TT>(t, lane, s, a.K, arow, a.aq, a.ad, acc0);
      if (!a.down) q8x4_tile<TT>(t + tb, lane, s, a.K, arow, a.aq, a.ad, acc1);
    }
  }
}

// CAS step 1 over 32 values held one per lane, written as the SwiGLU codes
// of h-block `blk` of slot row sr.
__device__ __forceinline__ void requant_store(const DecArgs &a, float h, int sr, int blk, int lane) {
  const float amax = warp_max(fabsf(h));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = cas_code(h, d);
  const int gsum = half_warp_sum(q);
  a.hq[(size_t)sr * a.F + 32 * blk + lane] = (int8_t)q;
  if (lane == 0) a.dh[(size_t)sr * (a.F >> 5) + blk] = d;
  if ((lane & 15) == 0) a.gsh[(size_t)sr * (a.F >> 4) + 2 * blk + (lane >> 4)] = (int16_t)gsum;
}

// CAS step 7 for rows 32*rg32 .. +31 of token t (lane = row).
__device__ __forceinline__ void combine_rows(const DecArgs &a, int t, int rg32, int lane) {
  if (__ldg(a.ids + (size_t)t * a.k) < 0) return;
  const int r = 32 * rg32 + lane;
  float acc = 0.0f;
  for (int j = 0; j < a.k; j++)
    acc = __fadd_rn(acc, __fmul_rn(__ldg(a.w + (size_t)t * a.k + j), __ldcg(a.apart + ((size_t)t * a.NS + j) * a.H + r)));
  if (a.n_shared) acc = __fadd_rn(acc, __ldcg(a.apart + ((size_t)t * a.NS + a.k) * a.H + r));
  float *yp = a.y + (size_t)t * a.H + r;
  *yp = __fadd_rn(*yp, acc);
}

__device__ __forceinline__ int valid_routed_slots(const DecArgs &a, int t) {
  int n = 0;
  for (int j = 0; j < a.k; j++) n += __ldg(a.ids + (size_t)t * a.k + j) >= 0;
  return n;
}

__device__ void item_epilogue(const DecArgs &a, const ItemDesc &d, int lane, const int *srow, int nt,
                              const float *acc0, const float *acc1) {
  const bool x4 = d.kind == KIND_SH8;
  for (int i = 0; i < nt; i++) {
    const int sr = srow[i];
    if (!a.down) {
      const float h = __fmul_rn(cas_silu(acc0[i]), acc1[i]);
      if (!x4) {
        requant_store(a, h, sr, d.rg, lane);
      } else {
        // 8 rows: stage h, the last of the 4 items of this 32-row block requantises.
        if ((lane & 3) == 0) a.hbuf[(size_t)sr * a.F + 8 * d.rg + (lane >> 2)] = h;
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(a.hticket + (size_t)sr * (a.F >> 5) + (d.rg >> 2), 1) == 3;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          const float hv = __ldcg(a.hbuf + (size_t)sr * a.F + 32 * (d.rg >> 2) + lane);
          requant_store(a, hv, sr, d.rg >> 2, lane);
          if (lane == 0) a.hticket[(size_t)sr * (a.F >> 5) + (d.rg >> 2)] = 0;
        }
      }
    } else {
      const int t = sr / a.NS;
      const int rg32 = x4 ? d.rg >> 2 : d.rg;
      if (!x4)
        a.apart[(size_t)sr * a.H + 32 * d.rg + lane] = acc0[i];
      else if ((lane & 3) == 0)
        a.apart[(size_t)sr * a.H + 8 * d.rg + (lane >> 2)] = acc0[i];
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        const int sh_arrivals = a.n_shared ? (a.sf == DS4MOE_Q8_0 ? 4 : 1) : 0;
        const int expect = valid_routed_slots(a, t) + sh_arrivals;
        last = atomicAdd(a.cticket + (size_t)t * (a.H >> 5) + rg32, 1) == expect - 1;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        combine_rows(a, t, rg32, lane);
        if (lane == 0) a.cticket[(size_t)t * (a.H >> 5) + rg32] = 0;
      }
    }
  }
}

template <int TT>
__global__ void __launch_bounds__(DEC_WARPS * 32, 1) k_expert_dec(DecArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *base = smem + warp * (DEC_NST * DEC_STRIDE + DEC_NST * 8 + DEC_NST * 16);
  const uint32_t buf = smem_u32(base);
  const uint32_t bar = buf + DEC_NST * DEC_STRIDE;
  int4 *meta = (int4 *)(base + DEC_NST * DEC_STRIDE + DEC_NST * 8);  // per slot: item, pass, stage, -
  pdl_launch_dependents();
  if (lane == 0) {
    for (int i = 0; i < DEC_NST; i++) mbar_init(bar + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int nsh = shared_items(a);
  uint32_t g_prod = 0, g_cons = 0;
  // producer cursor
  int p_item = warp_claim(a.queue, lane), p_pass = 0, p_stage = 0, p_npass = 0;
  ItemDesc pd;
  bool p_done = false;
  auto arm = [&](const ItemDesc &d) {
    const uint32_t slot = g_prod % DEC_NST;
    if (lane == 0) {
      meta[slot] = make_int4(p_item, p_pass, p_stage, 0);
      if (g_prod >= DEC_NST) fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar + 8 * slot, d.sbytes);
      bulk_g2s(buf + slot * DEC_STRIDE, d.src + (size_t)p_stage * d.sbytes, d.sbytes, bar + 8 * slot);
    }
    g_prod++;
    p_stage++;
  };
  // Shared-expert items do not depend on routing: start their weights now.
  if (p_item < nsh) {
    pd = item_desc(a, p_item, false);
    const int pre = min(DEC_NST, pd.nstages);
    for (int s = 0; s < pre; s++) arm(pd);
  }
  pdl_wait();
  const int n_items = nsh + (*a.n_active - a.n_shared) * (a.rows / 32);
  if (p_item >= n_items) {
    p_done = true;
  } else {
    pd = item_desc(a, p_item, true);
    p_npass = (pd.n_tok + TT - 1) / TT;
  }

  // consumer state
  ItemDesc cd;
  int c_item = -1, c_pass = -1, arow[TT], srow[TT], c_nt = 0;
  float acc0[TT], acc1[TT];
  bool failed = false;
  for (;;) {
    while (!p_done && g_prod - g_cons < DEC_NST) {
      if (p_stage == pd.nstages) {
        p_stage = 0;
        if (++p_pass >= p_npass) {
          p_item = warp_claim(a.queue, lane);
          p_pass = 0;
          if (p_item >= n_items) {
            p_done = true;
            break;
          }
          pd = item_desc(a, p_item, true);
          p_npass = (pd.n_tok + TT - 1) / TT;
        }
      }
      arm(pd);
    }
    if (g_cons == g_prod) break;
    const uint32_t slot = g_cons % DEC_NST;
    if (!mbar_wait_bounded(bar + 8 * slot, (g_cons / DEC_NST) & 1)) {
      failed = true;
      break;
    }
    __syncwarp();
    const int4 m = meta[slot];
    if (m.x != c_item || m.y != c_pass) {
      if (m.x != c_item) cd = item_desc(a, m.x, true);
      c_item = m.x, c_pass = m.y;
      load_tokens<TT>(a, cd, c_pass, arow, srow, &c_nt);
#pragma unroll
      for (int i = 0; i < TT; i++) acc0[i] = 0.0f, acc1[i] = 0.0f;
    }
    run_ksteps<TT>(a, cd, buf + slot * DEC_STRIDE, m.z, lane, arow, acc0, acc1);
    __syncwarp();
    g_cons++;
    if (m.z == cd.nstages - 1) item_epilogue(a, cd, lane, srow, c_nt, acc0, acc1);
  }
  if (failed) {
    if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
    for (uint32_t g = g_cons; g < g_prod; g++) (void)mbar_wait_bounded(bar + 8 * (g % DEC_NST), (g / DEC_NST) & 1);
  }
  // the last streamer to leave resets the queue for the next call
  if (lane == 0) {
    const int total = gridDim.x * DEC_WARPS;
    if (atomicAdd(a.queue + 1, 1) == total - 1) {
      atomicExch(a.queue, 0);
      atomicExch(a.queue + 1, 0);
    }
  }
}

// ===========================================================================
// Host launchers.

static cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args,
                              bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

size_t route_dec_smem(const ds4moe_layer *h) {
  const int H = h->d.hidden, nb = H / 32, per = nb / ROUTER_SEGS;
  const bool q8 = h->d.route == DS4MOE_ROUTE_LEARNED && h->d.router_fmt == DS4MOE_Q8_0;
  const int c0 = 0, c1 = (per + 1) / 2 + 1;
  const size_t seg_bytes = q8 ? (size_t)(c1 - c0) * Q8_TILE : 0;
  size_t bytes = RD_WARPS * seg_bytes + RD_RT * per * 32 + 4 * (RD_RT * per + 2) + 8 * RD_WARPS;
  bytes = (bytes + 15) & ~(size_t)15;
  const size_t scratch = 16 + sizeof(float) * (size_t)RD_WARPS * 2 * h->E_pad;
  const size_t bucket = 16 + sizeof(int) * (size_t)bucket_smem_ints(h->d.n_experts);
  return bytes + (scratch > bucket ? scratch : bucket);
}

cudaError_t launch_dec_route(const ds4moe_layer *h, const float *x, const int32_t *tok, int T, cudaStream_t s) {
  const ds4moe_layer_desc &d = h->d;
  Bucket b = bucket_view(h);
  RouteDecArgs r;
  r.x = x, r.tok = tok, r.T = T, r.H = d.hidden, r.E = d.n_experts, r.E_pad = h->E_pad, r.k = d.top_k;
  r.NS = h->NS, r.n_shared = d.n_shared, r.route = d.route, r.router_fmt = d.router_fmt, r.vocab = d.vocab;
  r.scale = d.route_scale, r.W = h->router, r.bias = h->bias, r.hash = h->hash;
  r.xq = h->xq, r.dx = h->dx, r.gs = h->gs, r.rpart = h->rpart, r.ids = h->ids, r.w = h->wts;
  r.cnt = b.cnt, r.off = b.off, r.active = b.active, r.n_active = b.n_active, r.list = b.list;
  r.tick = h->tick, r.err = h->err;
  const int n_tiles = (T + RD_RT - 1) / RD_RT;
  const int gx = d.route == DS4MOE_ROUTE_LEARNED ? (h->E_pad / 32 + RD_WARPS - 1) / RD_WARPS : 1;
  void *args[] = {&r};
  return launch_pdl((const void *)k_route_dec, dim3(gx, ROUTER_SEGS, n_tiles), dim3(RD_WARPS * 32),
                    route_dec_smem(h), s, args, false);
}

cudaError_t launch_dec_expert(const ds4moe_layer *h, int T, float *y, int down, cudaStream_t s) {
  const ds4moe_layer_desc &d = h->d;
  Bucket b = bucket_view(h);
  DecArgs a;
  a.H = d.hidden, a.F = d.ffn, a.E = d.n_experts, a.k = d.top_k, a.NS = h->NS, a.n_shared = d.n_shared;
  a.rf = d.routed_fmt, a.sf = d.n_shared ? d.shared_fmt : d.routed_fmt;
  a.cnt = b.cnt, a.off = b.off, a.active = b.active, a.n_active = b.n_active, a.list = b.list;
  a.ids = h->ids, a.w = h->wts, a.hq = h->hq, a.dh = h->dh, a.gsh = h->gsh, a.hbuf = h->hbuf;
  a.hticket = h->hticket, a.apart = h->apart, a.cticket = h->cticket, a.y = y, a.err = h->err;
  const bool sh8 = d.n_shared && d.shared_fmt == DS4MOE_Q8_0;
  a.down = down;
  if (!down) {
    a.K = d.hidden, a.rows = d.ffn, a.w_r = h->gu, a.w_s = sh8 ? h->sgu8 : h->sgu;
    a.aq = h->xq, a.ad = h->dx, a.ag = h->gs, a.queue = h->queue;
  } else {
    a.K = d.ffn, a.rows = d.hidden, a.w_r = h->dn, a.w_s = sh8 ? h->sdn8 : h->sdn;
    a.aq = h->hq, a.ad = h->dh, a.ag = h->gsh, a.queue = h->queue + 2;
  }
  void *args[] = {&a};
  const void *fn = T <= 1 ? (const void *)k_expert_dec<1>
                 : T <= 2 ? (const void *)k_expert_dec<2>
                 : T <= 4 ? (const void *)k_expert_dec<4> : (const void *)k_expert_dec<8>;
  return launch_pdl(fn, dim3(h->n_sm), dim3(DEC_WARPS * 32), DEC_SMEM, s, args, true);
}

cudaError_t decode_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(k_route_dec, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  const void *fns[] = {(const void *)k_expert_dec<1>, (const void *)k_expert_dec<2>,
                       (const void *)k_expert_dec<4>, (const void *)k_expert_dec<8>};
  for (const void *f : fns)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, DEC_SMEM);
  return e;
}

}  // namespace ds4

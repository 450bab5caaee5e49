// decode.cu -- the decode-batch path (n_tok <= DEC_MAX_T): three kernels
// chained with programmatic dependent launch (PDL):
//
//   K1 k_router_dec : int8 quantisation of x, the router GEMV segment sums,
//                     then (last block of each token) the token's routing --
//                     logits, sigmoid, bias top-k and renormalisation, or the
//                     hash lookup -- and (block of the last routed token) the
//                     per-expert bucketing of the call.
//   K2 k_expert_dec (gate/up): gate/up with in-register SwiGLU and the int8
//                     requant of h.
//   K3 k_expert_dec (down): down of every item; the last writer of each
//                     (token, 32 output rows) adds the fixed-order combine
//                     into y.
//
// K2 and K3 are persistent: every warp is an independent streamer that
// claims work items from a global queue (largest items first: the shared
// expert), keeps DEC_NST stages of its item sequence in flight with 1-D bulk
// async copies into a shared-memory ring, and crosses item boundaries without
// draining the ring. Items of the shared expert are claimed and their weights
// requested before griddepcontrol.wait, so they stream while the previous
// kernel (the router, or gate/up) finishes. Activations are staged in
// shared memory when they fit. Queues and tickets reset themselves, so no
// per-call memset is needed and the whole forward can be captured in a CUDA
// graph.
//
// Prior art: the decode MoE kernels named in the ds4-rocm fork README
// (moe_gate_up_mid_decode_lut_qwarp32, moe_down_sum6_qwarp32) fuse the same
// steps on an RDNA iGPU; the work split, layouts and pipeline here are
// sm_103a-specific.
#include "bucket.cuh"
#include "common.cuh"
#include "internal.h"
#include "route.cuh"
#include "tiles.cuh"

namespace ds4 {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ===========================================================================
// K1: quantisation, router segment sums, routing and bucketing.
//
// grid (ROUTER_SEGS, T), clusters of ROUTER_SEGS blocks: the cluster of
// token t has one block per K segment. Block seg quantises the token's
// 32-blocks of its segment (and publishes them), then sums every router row
// over the segment (warp w: row groups w, w + RC_WARPS, ...; lane = row) into
// its shared memory. After a cluster barrier, block 0 of the cluster adds the
// eight segment sums of each row in segment order, reading the other blocks'
// shared memory, and routes the token with all its threads (route.cuh; hash
// routing: the table lookup). When bucketing is asked for, the block that
// routed the call's last token (a self-resetting ticket; none for one token)
// buckets the call (bucket.cuh).

constexpr int RC_WARPS = 8;   // warps per block
constexpr int RC_HDR = 128;   // shared memory header: ticket flag, mbarriers
constexpr int RC_MAX_E = 1024;

struct RouteDecArgs {
  const float *x;
  int T, H, E, E_pad, k, NS, n_shared, learned, q8, vocab, A_cap;
  float scale;
  const uint8_t *W;     // router (RQ8 or F32 [E][H])
  const float *bias;
  const int32_t *hash, *tok;
  int8_t *xq;
  float *dx;
  int16_t *gs;
  int32_t *ids;         // [T][k] routing outputs
  float *w;
  int32_t *rticket;     // the call's ticket (self-resetting)
  int32_t *bucket;      // bucket table (null: no bucketing)
  uint32_t *err;
};

// Layout after the header: lgp [E_pad] f32 (this segment's row sums), dx_s
// [per] f32, xq_s [per*32] int8, then the 128-aligned work area (router
// tiles; afterwards the routing and bucketing scratch).
__host__ __device__ constexpr int rc_dx_off(int E_pad) { return RC_HDR + 4 * E_pad; }
__host__ __device__ constexpr int rc_xq_off(int E_pad, int per) { return rc_dx_off(E_pad) + ((4 * per + 15) & ~15); }
__host__ __device__ constexpr int rc_work_off(int E_pad, int per) {
  return (rc_xq_off(E_pad, per) + 32 * per + 127) & ~127;
}

// CAS step 1 for one value per lane of block b of token t, already loaded.
__device__ __forceinline__ void quant_value(float v, int H, int t, int b, int lane, int8_t *xq_s, float *dx_s,
                                            int8_t *xq_g, float *dx_g, int16_t *gs_g, uint32_t *err) {
  if (__any_sync(0xffffffffu, !isfinite(v)) && lane == 0) raise_flag(err, DS4MOE_DEVERR_NONFINITE);
  const float amax = warp_max(fabsf(v));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = cas_code(v, d);
  const int s = half_warp_sum(q);
  xq_s[lane] = (int8_t)q;
  if (lane == 0) *dx_s = d;
  xq_g[(size_t)t * H + 32 * b + lane] = (int8_t)q;
  if (lane == 0) dx_g[(size_t)t * (H >> 5) + b] = d;
  if ((lane & 15) == 0) gs_g[(size_t)t * (H >> 4) + 2 * b + (lane >> 4)] = (int16_t)s;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A float in the shared memory of block `rank` of this cluster.
__device__ __forceinline__ float ld_cluster_f32(const float *p, int rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// One arrival on a block-level ticket (thread 0); true in every thread of
// the block that completes it. The acquire-release atomic orders the block's
// earlier global writes (gathered by the barrier) before the completer's
// later reads; the completer resets the ticket.
__device__ __forceinline__ bool block_ticket_last(int32_t *tk, int expect, int *s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(tk) : "memory");
    const int last = old == expect - 1;
    if (last) *tk = 0;
    *s_flag = last;
  }
  __syncthreads();
  return *s_flag != 0;
}

__global__ void __cluster_dims__(ROUTER_SEGS, 1, 1) __launch_bounds__(RC_WARPS * 32, 1)
    k_router_dec(RouteDecArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x, t = blockIdx.y;
  const int nb = a.H >> 5, per = nb / ROUTER_SEGS, b0 = seg * per;
  const int c0 = b0 >> 1, c1 = (b0 + per + 1) >> 1;  // RQ8 2-block chunks covering the segment
  const int seg_bytes = a.q8 ? (c1 - c0) * RQ8_TILE : 0;
  const int nrg = a.learned ? (a.E_pad >> 5) : 0;
  int *s_flag = (int *)smem;
  uint64_t *bars = (uint64_t *)(smem + 64);
  float *lgp = (float *)(smem + RC_HDR);
  float *dx_s = (float *)(smem + rc_dx_off(a.E_pad));
  int8_t *xq_s = (int8_t *)(smem + rc_xq_off(a.E_pad, per));
  uint8_t *work = smem + rc_work_off(a.E_pad, per);
  pdl_launch_dependents();
  const uint32_t bar = smem_u32(&bars[warp]);
  const uint32_t wbuf = smem_u32(work + warp * seg_bytes);
  const size_t rg_stride = (size_t)(a.H / RQ8_KSTEP) * RQ8_TILE;
  if (a.q8 && lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    if (warp < nrg) {
      mbar_arrive_expect_tx(bar, seg_bytes);
      bulk_g2s(wbuf, a.W + (size_t)warp * rg_stride + (size_t)c0 * RQ8_TILE, seg_bytes, bar);
    }
  }
  // the routing block's bias values, requested early
  float bias_r[RC_MAX_E / (RC_WARPS * 32)];
#pragma unroll
  for (int i = 0; i < RC_MAX_E / (RC_WARPS * 32); i++) {
    const int e = threadIdx.x + i * RC_WARPS * 32;
    bias_r[i] = (seg == 0 && a.learned && e < a.E) ? __ldg(a.bias + e) : 0.0f;
  }
  // quantise the segment's blocks (warp w: blocks b0 + w + RC_WARPS*j), all
  // loads first
  if (a.x) {
    constexpr int QB = 4;
    for (int bb = warp; bb < per; bb += RC_WARPS * QB) {
      float v[QB];
#pragma unroll
      for (int j = 0; j < QB; j++) {
        const int b = bb + j * RC_WARPS;
        v[j] = b < per ? __ldg(a.x + (size_t)t * a.H + 32 * (b0 + b) + lane) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < QB; j++) {
        const int b = bb + j * RC_WARPS;
        if (b < per)
          quant_value(v[j], a.H, t, b0 + b, lane, xq_s + 32 * b, dx_s + b, a.xq, a.dx, a.gs, a.err);
      }
    }
  }
  __syncthreads();
  // segment sums of router rows 32*rg + lane
  for (int rg = warp, round = 0; rg < nrg; rg += RC_WARPS, round++) {
    float acc = 0.0f;
    const int r = 32 * rg + lane;
    if (a.q8) {
      if (round > 0 && lane == 0) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, seg_bytes);
        bulk_g2s(wbuf, a.W + (size_t)rg * rg_stride + (size_t)c0 * RQ8_TILE, seg_bytes, bar);
      }
      __syncwarp();
      if (!mbar_wait_bounded(bar, round & 1)) {
        if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
        break;
      }
      for (int b = b0; b < b0 + per; b++) {
        const uint32_t tile = wbuf + ((b >> 1) - c0) * RQ8_TILE;
        const uint32_t dd = ld_shared_u32(tile + 4 * lane);
        const float d = half_bits_to_float((b & 1) ? dd >> 16 : dd);
        const uint4 w0 = ld_shared_v4(tile + RQ8_Q + 512 * (2 * (b & 1)) + 16 * lane);
        const uint4 w1 = ld_shared_v4(tile + RQ8_Q + 512 * (2 * (b & 1) + 1) + 16 * lane);
        const uint4 *xv = (const uint4 *)(xq_s + (b - b0) * 32);
        const int I = dot16(w1, xv[1], dot16(w0, xv[0], 0));
        acc = __fadd_rn(acc, q8_term(d, dx_s[b - b0], I));
      }
    } else if (r < a.E) {  // fp32 router rows: fma chain over the segment (x unquantised)
      const int j0 = seg * (a.H / ROUTER_SEGS), j1 = j0 + a.H / ROUTER_SEGS;
      const float *wr = (const float *)a.W + (size_t)r * a.H;
      const float *xv = a.x + (size_t)t * a.H;
      for (int j = j0; j < j1; j++) acc = __fmaf_rn(__ldg(wr + j), __ldg(xv + j), acc);
    }
    lgp[r] = acc;
    __syncwarp();  // every lane is done with the tiles before the next copy
  }
  cluster_sync_all();
  // ---- routing of token t by block 0 of its cluster
  if (seg == 0) {
    if (a.learned) {
      const RouteScratch rs = route_scratch(work, a.E_pad, a.k);
#pragma unroll
      for (int i = 0; i < RC_MAX_E / (RC_WARPS * 32); i++) {
        const int e = threadIdx.x + i * RC_WARPS * 32;
        if (e < a.E_pad) {
          float lg = 0.0f;
          if (e < a.E)
            for (int g = 0; g < ROUTER_SEGS; g++) lg = __fadd_rn(lg, ld_cluster_f32(lgp + e, g));
          route_score(rs, e, a.E, lg, bias_r[i]);
        }
      }
      route_select(rs, a.E_pad, a.k, a.scale, a.ids + (size_t)t * a.k, a.w + (size_t)t * a.k);
    } else if (threadIdx.x < a.k) {
      const int v = __ldg(a.tok + t);
      const bool okv = v >= 0 && v < a.vocab;
      if (!okv && threadIdx.x == 0) raise_flag(a.err, DS4MOE_DEVERR_TOKEN_ID);
      a.ids[(size_t)t * a.k + threadIdx.x] = okv ? __ldg(a.hash + (size_t)v * a.k + threadIdx.x) : -1;
      a.w[(size_t)t * a.k + threadIdx.x] = okv ? __fmul_rn(__fdiv_rn(1.0f, (float)a.k), a.scale) : 0.0f;
    }
  }
  cluster_sync_all();  // the other blocks' segment sums stay until block 0 has read them
  if (seg != 0 || !a.bucket) return;
  // ---- bucketing of the call by the block that routed its last token
  if (a.T > 1 && !block_ticket_last(a.rticket, a.T, s_flag)) return;
  __syncthreads();
  int32_t *ids_s = (int32_t *)work;
  for (int i = threadIdx.x; i < a.T * a.k; i += blockDim.x) ids_s[i] = __ldcg(a.ids + i);
  __syncthreads();
  bucket_rank(ids_s, a.T, a.E, a.k, a.NS, a.n_shared, ids_s + ((a.T * a.k + 3) & ~3), a.bucket, a.A_cap, a.err);
}

// ===========================================================================
// K2 / K3: persistent expert GEMV streamers.
//
// Work items, largest first:
//   shared expert: (16-row group rg, K quarter q) for q = 0..3 -- the shared
//     expert's rows are summed in 4 segments (CAS step 4, S = 4), so each
//     quarter is an independent chain; the last quarter to finish adds the
//     four segment sums in order;
//   routed experts: (active expert, 16-row group), the whole K range.
// A gate/up item's SwiGLU values go to hbuf; the second 16-row item of each
// 32-row block requantises the block (CAS step 1 on h).

constexpr int DEC_WARPS = 8;     // streamers per CTA
constexpr int DEC_NST = 4;       // ring stages per streamer
constexpr int DEC_STRIDE = 5376; // ring slot bytes (largest stage)
constexpr int DEC_WARP_SMEM = DEC_NST * DEC_STRIDE + DEC_NST * 8 + DEC_NST * 16;
constexpr int DEC_RING = DEC_WARPS * DEC_WARP_SMEM;

struct DecArgs {
  int H, F, E, E_pad, k, NS, n_shared, rf, sf, down, T;
  int K;                         // reduction length: H (gate/up) or F (down)
  int rows;                      // output rows of the matrices: F (gate/up) or H (down)
  int act_smem;                  // activations staged in shared memory
  const uint8_t *w_r;            // routed weights, RG16
  const uint8_t *w_s;            // shared weights, RG16
  const int8_t *aq;              // activation codes: xq [T][H] or hq [T*NS][F]
  const float *ad;
  const int16_t *ag;
  // routing results (router kernel)
  int32_t *ids;
  float *w;
  const int32_t *bucket;         // bucket table (bucket.cuh)
  int A_cap;
  int8_t *hq;
  float *dh;
  int16_t *gsh;
  float *spart;                  // shared segment sums: [T][4][rows][mats]
  int32_t *sticket;              // [T][rows/16] shared merge tickets
  float *hbuf;                   // [T*NS][F] SwiGLU values before requant
  int32_t *hticket;              // [T*NS][F/32] requant tickets
  float *apart;                  // [T*NS][H]
  int32_t *cticket;              // [T][H/32] combine tickets
  float *y;
  int32_t *queue;                // [2] claim counter, exited streamers
  uint32_t *err;
};

// Routing view used by the streamers (shared memory).
struct Bk {
  const int4 *act;  // {expert, pairs, list offset, 0}
  const int32_t *list;
  int n_active;
};

struct ItemDesc {
  const uint8_t *src;
  int fmt, e, rg, quarter, nstages, sbytes, ksps, ks0;
  int n_tok, list_off;
};

__device__ __forceinline__ int shared_items(const DecArgs &a) {
  return a.n_shared ? SHARED_SEGS * (a.rows / TILE_ROWS) : 0;
}

// K-steps per stage: as many as fit a ring slot, dividing the K-step count.
__device__ __forceinline__ int stage_ksteps(int kbytes, int nks) {
  int s = DEC_STRIDE / kbytes;
  if (s > nks) s = nks;
  while (s > 1 && nks % s) s--;
  return s < 1 ? 1 : s;
}

// Item i. Shared items are fully described without the routing result, so
// their weights can stream before it exists.
__device__ ItemDesc item_desc(const DecArgs &a, const Bk *bk, int i) {
  ItemDesc d;
  const int nsh = shared_items(a), RG = a.rows / TILE_ROWS, mats = a.down ? 1 : 2;
  if (i < nsh) {
    d.fmt = a.sf, d.e = a.E, d.rg = i / SHARED_SEGS, d.quarter = i % SHARED_SEGS;
  } else {
    const int j = i - nsh;
    d.fmt = a.rf, d.e = bk ? bk->act[a.n_shared + j / RG].x : -1, d.rg = j % RG, d.quarter = -1;
  }
  const int kb = mats * tile_bytes(d.fmt);
  const int nks_all = a.K / kstep(d.fmt);
  const int nks = d.quarter >= 0 ? nks_all / SHARED_SEGS : nks_all;
  d.ks0 = d.quarter >= 0 ? d.quarter * nks : 0;
  d.ksps = stage_ksteps(kb, nks);
  d.nstages = nks / d.ksps;
  d.sbytes = d.ksps * kb;
  if (d.e == a.E)
    d.src = a.w_s + ((size_t)d.rg * nks_all + d.ks0) * kb;
  else if (d.e >= 0)
    d.src = a.w_r + ((size_t)d.e * RG + d.rg) * nks_all * kb;
  else
    d.src = nullptr;
  d.n_tok = 0, d.list_off = 0;
  if (bk && d.e >= 0) {
    const int4 en = bk->act[i < nsh ? 0 : a.n_shared + (i - nsh) / RG];
    d.n_tok = en.y, d.list_off = en.z;
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
__device__ __forceinline__ void load_tokens(const DecArgs &a, const Bk &bk, const ItemDesc &d, int pass, int *arow,
                                            int *srow, int *nt) {
  const int t0 = pass * TT;
  *nt = min(TT, d.n_tok - t0);
#pragma unroll
  for (int i = 0; i < TT; i++) {
    const int sr = bk.list[d.list_off + min(t0 + i, d.n_tok - 1)];
    srow[i] = sr;
    arow[i] = a.down ? sr : sr / a.NS;
  }
}

template <int TT, bool AS>
__device__ __forceinline__ void run_ksteps(const DecArgs &a, const ItemDesc &d, uint32_t st, int stage, int lane,
                                           const int *arow, const int8_t *aq, const float *ad, const int16_t *ag,
                                           float *acc0, float *acc1) {
  const int tb = tile_bytes(d.fmt), kb = a.down ? tb : 2 * tb;
  for (int j = 0; j < d.ksps; j++) {
    const int s = d.ks0 + stage * d.ksps + j;  // absolute K-step
    const uint32_t t = st + j * kb;
    if (d.fmt == DS4MOE_Q2S) {
      q2s_tile<TT, AS>(t, lane, s, a.K, arow, aq, ad, ag, acc0);
      if (!a.down) q2s_tile<TT, AS>(t + tb, lane, s, a.K, arow, aq, ad, ag, acc1);
    } else {
      q8_tile<TT, AS>(t, lane, s, a.K, arow, aq, ad, acc0);
      if (!a.down) q8_tile<TT, AS>(t + tb, lane, s, a.K, arow, aq, ad, acc1);
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

// CAS step 7 for rows 32*rg .. +31 of token t (lane = row).
__device__ __forceinline__ void combine_rows(const DecArgs &a, int t, int rg, int lane) {
  if (__ldg(a.ids + (size_t)t * a.k) < 0) return;
  const int r = 32 * rg + lane;
  float acc = 0.0f;
  for (int j = 0; j < a.k; j++)
    acc = __fadd_rn(acc,
                    __fmul_rn(__ldg(a.w + (size_t)t * a.k + j), __ldcg(a.apart + ((size_t)t * a.NS + j) * a.H + r)));
  if (a.n_shared) acc = __fadd_rn(acc, __ldcg(a.apart + ((size_t)t * a.NS + a.k) * a.H + r));
  float *yp = a.y + (size_t)t * a.H + r;
  *yp = __fadd_rn(*yp, acc);
}

__device__ __forceinline__ int valid_routed_slots(const DecArgs &a, int t) {
  int n = 0;
  for (int j = 0; j < a.k; j++) n += __ldg(a.ids + (size_t)t * a.k + j) >= 0;
  return n;
}

// Count one arrival on a ticket; true (on every lane) for the caller that
// completes it. The release/acquire atomic orders this warp's earlier global
// writes before the completer's later reads; the completer resets the ticket.
__device__ __forceinline__ bool ticket_last(int32_t *tk, int expect, int lane) {
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(tk) : "memory");
    last = old == expect - 1;
    if (last) *tk = 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();  // order lane 0's acquire before the other lanes' reads
  return last != 0;
}

// 16 rows (rg16) of the down output of slot row sr are in apart: count them
// towards the combine of token t, rows 32*(rg16/2)..; run it if complete.
__device__ __forceinline__ void down_done(const DecArgs &a, int sr, int rg16, int lane) {
  const int t = sr / a.NS, rg = rg16 >> 1;
  int expect = 0;
  if (lane == 0) expect = 2 * (valid_routed_slots(a, t) + a.n_shared);
  expect = __shfl_sync(0xffffffffu, expect, 0);
  if (ticket_last(a.cticket + (size_t)t * (a.H >> 5) + rg, expect, lane)) combine_rows(a, t, rg, lane);
}

// SwiGLU value h of row 16*rg16 + lane/2 of slot row sr (both lanes of a row
// hold it): stage it; the second 16-row half of the 32-row block requantises.
__device__ __forceinline__ void gateup_done(const DecArgs &a, float h, int sr, int rg16, int lane) {
  if ((lane & 1) == 0) a.hbuf[(size_t)sr * a.F + 16 * rg16 + (lane >> 1)] = h;
  const int blk = rg16 >> 1;
  if (ticket_last(a.hticket + (size_t)sr * (a.F >> 5) + blk, 2, lane))
    requant_store(a, __ldcg(a.hbuf + (size_t)sr * a.F + 32 * blk + lane), sr, blk, lane);
}

template <int TT>
__device__ void item_epilogue(const DecArgs &a, const ItemDesc &d, int lane, const int *srow, int nt,
                              const float *acc0, const float *acc1) {
  const int r = TILE_ROWS * d.rg + (lane >> 1);
  for (int i = 0; i < nt; i++) {
    const int sr = srow[i];
    if (d.quarter < 0) {  // routed: the whole chain is in this warp
      if (!a.down) {
        gateup_done(a, __fmul_rn(cas_silu(acc0[i]), acc1[i]), sr, d.rg, lane);
      } else {
        if ((lane & 1) == 0) a.apart[(size_t)sr * a.H + r] = acc0[i];
        down_done(a, sr, d.rg, lane);
      }
      continue;
    }
    // shared: publish this quarter's segment sums; the last quarter merges
    const int t = sr / a.NS, mats = a.down ? 1 : 2;
    float *sp = a.spart + ((size_t)t * SHARED_SEGS) * a.rows * mats;
    if ((lane & 1) == 0) {
      sp[((size_t)d.quarter * a.rows + r) * mats] = acc0[i];
      if (!a.down) sp[((size_t)d.quarter * a.rows + r) * mats + 1] = acc1[i];
    }
    if (!ticket_last(a.sticket + (size_t)t * (a.rows / TILE_ROWS) + d.rg, SHARED_SEGS, lane)) continue;
    float g = 0.0f, u = 0.0f;
#pragma unroll
    for (int q = 0; q < SHARED_SEGS; q++) {
      g = __fadd_rn(g, __ldcg(sp + ((size_t)q * a.rows + r) * mats));
      if (!a.down) u = __fadd_rn(u, __ldcg(sp + ((size_t)q * a.rows + r) * mats + 1));
    }
    if (!a.down) {
      gateup_done(a, __fmul_rn(cas_silu(g), u), sr, d.rg, lane);
    } else {
      if ((lane & 1) == 0) a.apart[(size_t)sr * a.H + r] = g;
      down_done(a, sr, d.rg, lane);
    }
  }
}

// Shared memory after the rings: [bucket ints][staged activations]. bucket:
// cnt[E+1] off[E+2] active[E+2] n_active[1] list[T*NS].
__host__ __device__ inline int dec_bucket_ints(int A_cap, int T, int NS) { return bucket_table_ints(A_cap, T, NS); }

template <int TT, bool AS>
__global__ void __launch_bounds__(DEC_WARPS * 32, 1) k_expert_dec(DecArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *base = smem + warp * DEC_WARP_SMEM;
  const uint32_t buf = smem_u32(base);
  const uint32_t bar = buf + DEC_NST * DEC_STRIDE;
  int4 *meta = (int4 *)(base + DEC_NST * DEC_STRIDE + DEC_NST * 8);  // per slot: item, pass, stage
  int32_t *bks = (int32_t *)(smem + DEC_RING);
  const int nbk = dec_bucket_ints(a.A_cap, a.T, a.NS);
  uint8_t *scratch = (uint8_t *)(bks + ((nbk + 31) & ~31));
  pdl_launch_dependents();
  if (lane == 0) {
    for (int i = 0; i < DEC_NST; i++) mbar_init(bar + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int nsh = shared_items(a);
  uint32_t g_prod = 0, g_cons = 0;
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
  // Shared-expert items do not depend on routing: request their weights now.
  if (p_item < nsh) {
    pd = item_desc(a, nullptr, p_item);
    const int pre = min(DEC_NST, pd.nstages);
    for (int s = 0; s < pre; s++) arm(pd);
  }
  pdl_wait();

  // ---- the routing result (bucketed by the router kernel) into shared memory
  for (int i = threadIdx.x; i < nbk; i += blockDim.x) bks[i] = __ldcg(a.bucket + i);
  __syncthreads();
  Bk bk;
  bk.act = (const int4 *)(bks + BKT_HDR), bk.list = bks + BKT_HDR + 4 * a.A_cap, bk.n_active = bks[0];

  // ---- activations into shared memory (when they fit)
  const int8_t *aq = a.aq;
  const float *ad = a.ad;
  const int16_t *ag = a.ag;
  if (AS) {
    const int rows = a.down ? a.T * a.NS : a.T;
    const size_t nq = (size_t)rows * a.K, nd = (size_t)rows * (a.K >> 5) * 4, ng = (size_t)rows * (a.K >> 4) * 2;
    uint8_t *dq = scratch, *dd = scratch + nq, *dg = dd + nd;
    for (size_t i = threadIdx.x; i < nq / 16; i += blockDim.x) ((uint4 *)dq)[i] = __ldg((const uint4 *)a.aq + i);
    for (size_t i = threadIdx.x; i < nd / 16; i += blockDim.x) ((uint4 *)dd)[i] = __ldg((const uint4 *)a.ad + i);
    for (size_t i = threadIdx.x; i < ng / 16; i += blockDim.x) ((uint4 *)dg)[i] = __ldg((const uint4 *)a.ag + i);
    aq = (const int8_t *)dq, ad = (const float *)dd, ag = (const int16_t *)dg;
    __syncthreads();
  }

  const int n_items = nsh + (bk.n_active - a.n_shared) * (a.rows / TILE_ROWS);
  if (p_item >= n_items) {
    p_done = true;
  } else {
    pd = item_desc(a, &bk, p_item);
    p_npass = (pd.n_tok + TT - 1) / TT;
  }

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
          pd = item_desc(a, &bk, p_item);
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
      if (m.x != c_item) cd = item_desc(a, &bk, m.x);
      c_item = m.x, c_pass = m.y;
      load_tokens<TT>(a, bk, cd, c_pass, arow, srow, &c_nt);
#pragma unroll
      for (int i = 0; i < TT; i++) acc0[i] = 0.0f, acc1[i] = 0.0f;
    }
    run_ksteps<TT, AS>(a, cd, buf + slot * DEC_STRIDE, m.z, lane, arow, aq, ad, ag, acc0, acc1);
    __syncwarp();
    g_cons++;
    if (m.z == cd.nstages - 1) item_epilogue<TT>(a, cd, lane, srow, c_nt, acc0, acc1);
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

static size_t router_dec_smem(const ds4moe_layer *h) {
  const ds4moe_layer_desc &d = h->d;
  const int H = d.hidden, nb = H / 32, per = nb / ROUTER_SEGS;
  const bool q8 = d.route == DS4MOE_ROUTE_LEARNED && d.router_fmt == DS4MOE_Q8_0;
  size_t work = q8 ? (size_t)RC_WARPS * ((per + 1) / 2 + 1) * RQ8_TILE : 0;
  const size_t route = route_block_smem(h->E_pad, d.top_k);
  const int n = h->Tc * d.top_k;
  const size_t bucket = (size_t)(((n + 3) & ~3) + bucket_rank_smem_ints(n)) * 4;
  if (route > work) work = route;
  if (bucket > work) work = bucket;
  return rc_work_off(h->E_pad, per) + work;
}

// Shared memory of the streamer kernel for n_tok tokens; act: with staged
// activations.
static size_t expert_dec_smem(const ds4moe_layer *h, int T, bool down, bool act) {
  const ds4moe_layer_desc &d = h->d;
  const size_t bucket = (size_t)((dec_bucket_ints(h->A_max, T, h->NS) + 31) & ~31) * 4;
  size_t scratch = 0;
  if (act) {
    const size_t rows = down ? (size_t)T * h->NS : (size_t)T;
    const size_t K = down ? d.ffn : d.hidden;
    scratch = rows * K + rows * (K / 32) * 4 + rows * (K / 16) * 2;
  }
  return DEC_RING + bucket + scratch;
}

size_t route_dec_smem(const ds4moe_layer *h) {
  // the decode path fits when its routing and both streamers fit at DEC_MAX_T
  size_t m = router_dec_smem(h);
  const size_t a = expert_dec_smem(h, DEC_MAX_T, false, false), b = expert_dec_smem(h, DEC_MAX_T, true, false);
  if (a > m) m = a;
  if (b > m) m = b;
  return m;
}

cudaError_t launch_dec_route(const ds4moe_layer *h, const float *x, const int32_t *tok, int T, int32_t *ids,
                             float *w, bool bucket, cudaStream_t s) {
  const ds4moe_layer_desc &d = h->d;
  RouteDecArgs r = {};
  r.x = x, r.T = T, r.H = d.hidden, r.E = d.n_experts, r.E_pad = h->E_pad, r.k = d.top_k, r.NS = h->NS;
  r.n_shared = d.n_shared, r.vocab = d.vocab, r.scale = d.route_scale, r.A_cap = h->A_max;
  r.learned = d.route == DS4MOE_ROUTE_LEARNED;
  r.q8 = r.learned && d.router_fmt == DS4MOE_Q8_0;
  r.W = h->router, r.bias = h->bias, r.hash = h->hash, r.tok = tok;
  r.xq = h->xq, r.dx = h->dx, r.gs = h->gs, r.err = h->err;
  r.ids = ids, r.w = w, r.rticket = h->rticket;
  r.bucket = bucket ? h->bucket : nullptr;
  void *args[] = {&r};
  return launch_pdl((const void *)k_router_dec, dim3(ROUTER_SEGS, T), dim3(RC_WARPS * 32), router_dec_smem(h), s,
                    args, false);
}

template <bool AS>
static const void *expert_fn(int T) {
  return T <= 1 ? (const void *)k_expert_dec<1, AS>
       : T <= 2 ? (const void *)k_expert_dec<2, AS>
       : T <= 4 ? (const void *)k_expert_dec<4, AS> : (const void *)k_expert_dec<8, AS>;
}

cudaError_t launch_dec_expert(const ds4moe_layer *h, const int32_t *tok, int T, float *y, int down,
                              cudaStream_t s) {
  const ds4moe_layer_desc &d = h->d;
  DecArgs a;
  a.H = d.hidden, a.F = d.ffn, a.E = d.n_experts, a.E_pad = h->E_pad, a.k = d.top_k, a.NS = h->NS;
  a.n_shared = d.n_shared, a.T = T;
  a.rf = d.routed_fmt, a.sf = d.n_shared ? d.shared_fmt : d.routed_fmt;
  (void)tok;
  a.bucket = h->bucket, a.A_cap = h->A_max;
  a.ids = h->ids, a.w = h->wts, a.hq = h->hq, a.dh = h->dh, a.gsh = h->gsh;
  a.apart = h->apart, a.cticket = h->cticket, a.y = y, a.err = h->err;
  a.down = down;
  if (!down) {
    a.K = d.hidden, a.rows = d.ffn, a.w_r = h->gu, a.w_s = h->sgu;
    a.aq = h->xq, a.ad = h->dx, a.ag = h->gs, a.queue = h->queue;
    a.spart = h->spart, a.sticket = h->sticket, a.hbuf = h->hbuf, a.hticket = h->hticket;
  } else {
    a.K = d.ffn, a.rows = d.hidden, a.w_r = h->dn, a.w_s = h->sdn;
    a.aq = h->hq, a.ad = h->dh, a.ag = h->gsh, a.queue = h->queue + 2;
    a.spart = h->spart_dn, a.sticket = h->sticket_dn, a.hbuf = h->hbuf, a.hticket = h->hticket;
  }
  const bool act = expert_dec_smem(h, T, down != 0, true) <= DEC_SMEM_LIMIT;
  a.act_smem = act;
  const size_t smem = expert_dec_smem(h, T, down != 0, act);
  void *args[] = {&a};
  const void *fn = act ? expert_fn<true>(T) : expert_fn<false>(T);
  return launch_pdl(fn, dim3(h->n_sm), dim3(DEC_WARPS * 32), smem, s, args, true);
}

cudaError_t decode_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(k_router_dec, cudaFuncAttributeMaxDynamicSharedMemorySize, DEC_SMEM_LIMIT);
  const void *fns[] = {expert_fn<true>(1), expert_fn<true>(2), expert_fn<true>(4), expert_fn<true>(8),
                       expert_fn<false>(1), expert_fn<false>(2), expert_fn<false>(4), expert_fn<false>(8)};
  for (const void *f : fns)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, DEC_SMEM_LIMIT);
  return e;
}

}  // namespace ds4

// decode.cu -- the router kernel of a decode-sized call (n_tok <= DEC_MAX_T)
// and the launch helper shared with the expert kernels (experts.cu):
//
//   k_router_dec : (optionally) the RMSNorm of x, its int8 quantisation,
//                  the router GEMV segment sums,
//                  then (block 0 of each token's cluster) the token's routing
//                  -- logits, sigmoid, bias top-k and renormalisation, or the
//                  hash lookup -- and (the block that routed the last token)
//                  the per-expert bucketing of the call.
//
// The forward is router -> gate/up -> down, chained with programmatic
// dependent launch (PDL) so that each kernel's launch and weight prefetch
// overlap the previous kernel. Tickets reset themselves, so no per-call
// memset is needed.
#include "bucket.cuh"
#include "common.cuh"
#include "internal.h"
#include "route.cuh"

namespace ds4 {


// ===========================================================================
// K1: quantisation, router segment sums, routing and bucketing.
//
// grid (ROUTER_SEGS, T), clusters of ROUTER_SEGS blocks: the cluster of
// token t has one block per K segment. The blocks pass one cluster barrier
// in their prologue, so no block's shared memory is written before it runs.
// When the call normalises its input, every block first needs the inverse
// RMS norm of each of its tokens (one warp over the whole row, the RMSNorm
// kernel's arithmetic): with one token per cluster each block takes it
// itself; with tg tokens block r takes token r's and stores it into every
// block of the cluster (one more cluster barrier). The block scales the
// values it reads by it. Block seg quantises the token's 32-blocks of its
// segment (and publishes them), then sums every router row over the segment
// (warp w: row groups w, w + RC_WARPS, ...; lane = row) into block 0's
// shared memory (distributed shared memory stores). After one cluster
// barrier the other blocks are done; block 0 adds the eight segment sums of
// each row in segment order from its own shared memory and routes the token
// with all its threads (route.cuh; hash routing: the table lookup). When
// bucketing is asked for, the block that routed the call's last token (a
// self-resetting ticket; none for one token) buckets the call (bucket.cuh).

constexpr int RC_WARPS = 8;   // warps per block
constexpr int RC_HDR = 128;   // shared memory header: ticket flag, mbarriers
constexpr int RC_MAX_E = 1024;

struct RouteDecArgs {
  const float *x;
  int T, H, E, E_pad, k, NS, n_shared, learned, q8, vocab, A_cap;
  int tg;               // tokens per cluster (1, or ROUTER_SEGS: block r routes token r)
  int norm;             // x is the un-normalised input: RMSNorm it first (eps)
  float scale, eps;
  const uint8_t *W;     // router (RQ8 or F32 [E][H])
  const float *bias;
  const int32_t *hash, *tok;
  int8_t *xq;
  float *dx;
  int16_t *gs;
  int32_t *ids;         // [T][k] routing outputs
  float *w;
  int32_t *rticket;     // the call's ticket (self-resetting)
  int32_t *xq_ready;    // decode forward: count of blocks whose codes of x are written, else null
  int32_t *bucket;      // bucket table (null: no bucketing)
  uint32_t *err;
};

// Layout after the header: lgp [ROUTER_SEGS][E_pad] f32 (in block 0: every
// segment's row sums, stored there by the cluster's blocks), dx_s [per] f32,
// xq_s [per*32] int8, then the 128-aligned work area (router tiles;
// afterwards the routing and bucketing scratch).
__host__ __device__ constexpr int rc_dx_off(int E_pad) { return RC_HDR + 4 * ROUTER_SEGS * E_pad; }
__host__ __device__ constexpr int rc_xq_off(int E_pad, int per, int tg) {
  return rc_dx_off(E_pad) + ((4 * per * tg + 15) & ~15);
}
__host__ __device__ constexpr int rc_work_off(int E_pad, int per, int tg) {
  return (rc_xq_off(E_pad, per, tg) + 32 * per * tg + 127) & ~127;
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

// CAS step 8 of one row v (H floats, 16-byte aligned, H a multiple of 256)
// by one warp: 1 / sqrt(mean(v^2) + eps). Lane l keeps the fma chain of the
// l-th of 32 contiguous segments in element order; the 32 segment sums are
// then added in order, as the RMSNorm kernel does. A segment of up to 128
// values is loaded in one round (one L2 round trip).
__device__ __forceinline__ float rms_inv_warp(const float *v, int H, float eps, int lane) {
  constexpr int RW = 32;  // float4 words per round
  const int n4 = H >> 7;  // float4 words of a segment
  const float4 *p = (const float4 *)(v + (size_t)lane * (H >> 5));
  float acc = 0.0f;
  for (int i = 0; i < n4; i += RW) {
    float4 r[RW];
#pragma unroll
    for (int j = 0; j < RW; j++) r[j] = i + j < n4 ? __ldg(p + i + j) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < RW; j++) {
      if (i + j < n4) {
        acc = __fmaf_rn(r[j].x, r[j].x, acc);
        acc = __fmaf_rn(r[j].y, r[j].y, acc);
        acc = __fmaf_rn(r[j].z, r[j].z, acc);
        acc = __fmaf_rn(r[j].w, r[j].w, acc);
      }
    }
  }
  float ss = 0.0f;
  for (int l = 0; l < 32; l++) ss = __fadd_rn(ss, __shfl_sync(0xffffffffu, acc, l));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores v at the address of p in the shared memory of block `rank` of this
// cluster.
__device__ __forceinline__ void st_cluster_f32(float *p, int rank, float v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
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
  const int seg = blockIdx.x, tg = a.tg, t0 = blockIdx.y * tg, ntg = min(tg, a.T - t0);
  const int nb = a.H >> 5, per = nb / ROUTER_SEGS, b0 = seg * per;
  const int c0 = b0 >> 1, c1 = (b0 + per + 1) >> 1;  // RQ8 2-block chunks covering the segment
  const int seg_bytes = a.q8 ? (c1 - c0) * RQ8_TILE : 0;
  const int nrg = a.learned ? (a.E_pad >> 5) : 0;
  int *s_flag = (int *)smem;
  float *ninv = (float *)(smem + 16);  // [tg] inverse RMS norms of the cluster's tokens (header bytes 16..47)
  uint64_t *bars = (uint64_t *)(smem + 64);
  float *lgp = (float *)(smem + RC_HDR);
  float *dx_s = (float *)(smem + rc_dx_off(a.E_pad));                  // [tg][per]
  int8_t *xq_s = (int8_t *)(smem + rc_xq_off(a.E_pad, per, tg));       // [tg][per * 32]
  uint8_t *work = smem + rc_work_off(a.E_pad, per, tg);
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
  // the routing blocks' bias values, requested early
  float bias_r[RC_MAX_E / (RC_WARPS * 32)];
#pragma unroll
  for (int i = 0; i < RC_MAX_E / (RC_WARPS * 32); i++) {
    const int e = threadIdx.x + i * RC_WARPS * 32;
    bias_r[i] = (seg < ntg && a.learned && e < a.E) ? __ldg(a.bias + e) : 0.0f;
  }
  // Every block of the cluster runs before any block stores into another's
  // shared memory: one cluster barrier, passed while the previous kernel of
  // the stream is still running (a barrier after the wait below measured
  // 0.3-0.5 us more per one-token layer).
  cluster_sync_all();
  // The router tiles and the bias above are constant: they are requested
  // before the previous kernel of the stream is done. Everything after reads
  // the call's inputs or writes scratch that kernel may still use.
  pdl_wait();
  // the gate/up kernel may launch now: it requests the shared expert's
  // weights while this kernel routes
  pdl_launch_dependents();
  // quantise the segment's blocks of the cluster's tokens (warp w: pairs
  // (token, block) w, w + RC_WARPS, ...), all loads of a round first; with
  // the RMSNorm, the first round's loads are issued before the norms
  if (a.x) {
    constexpr int QB = 4;
    const int np = ntg * per;
    float v[QB];
    auto load = [&](int pp) {
#pragma unroll
      for (int j = 0; j < QB; j++) {
        const int p = pp + j * RC_WARPS, i = p / per, b = p - i * per;
        v[j] = p < np ? __ldg(a.x + (size_t)(t0 + i) * a.H + 32 * (b0 + b) + lane) : 0.0f;
      }
    };
    load(warp);
    if (a.norm) {
      if (tg == 1) {
        if (warp == 0) {
          const float r = rms_inv_warp(a.x + (size_t)t0 * a.H, a.H, a.eps, lane);
          if (lane == 0) ninv[0] = r;
        }
        __syncthreads();
      } else {
        // clusters of tg tokens: block r takes token r's norm and stores it
        // into every block of the cluster (lane j: block j)
        if (warp == 0 && seg < ntg) {
          const float r = rms_inv_warp(a.x + (size_t)(t0 + seg) * a.H, a.H, a.eps, lane);
          if (lane < ROUTER_SEGS) st_cluster_f32(ninv + seg, lane, r);
        }
        cluster_sync_all();
      }
    }
    for (int pp = warp; pp < np; pp += RC_WARPS * QB) {
      if (pp != warp) load(pp);
#pragma unroll
      for (int j = 0; j < QB; j++) {
        const int p = pp + j * RC_WARPS, i = p / per, b = p - i * per;
        if (p < np)
          quant_value(a.norm ? __fmul_rn(v[j], ninv[i]) : v[j], a.H, t0 + i, b0 + b, lane, xq_s + 32 * p, dx_s + p,
                      a.xq, a.dx, a.gs, a.err);
      }
    }
  }
  __syncthreads();
  // The block's codes of x are written: the gate/up kernel starts the shared
  // expert on them while this kernel routes.
  if (a.xq_ready && threadIdx.x == 0) {
    __threadfence();
    red_release_gpu_add(a.xq_ready, 1);
  }
  // segment sums of router rows 32*rg + lane, for each of the cluster's
  // tokens (the row group's tiles once), into the table of the block that
  // routes the token
  for (int rg = warp, round = 0; rg < nrg; rg += RC_WARPS, round++) {
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
      for (int i = 0; i < ntg; i++) {
        float acc = 0.0f;
        for (int b = b0; b < b0 + per; b++) {
          const uint32_t tile = wbuf + ((b >> 1) - c0) * RQ8_TILE;
          const uint32_t dd = ld_shared_u32(tile + 4 * lane);
          const float d = half_bits_to_float((b & 1) ? dd >> 16 : dd);
          const uint4 w0 = ld_shared_v4(tile + RQ8_Q + 512 * (2 * (b & 1)) + 16 * lane);
          const uint4 w1 = ld_shared_v4(tile + RQ8_Q + 512 * (2 * (b & 1) + 1) + 16 * lane);
          const uint4 *xv = (const uint4 *)(xq_s + (i * per + b - b0) * 32);
          const int I = dot16(w1, xv[1], dot16(w0, xv[0], 0));
          acc = __fadd_rn(acc, q8_term(d, dx_s[i * per + b - b0], I));
        }
        st_cluster_f32(lgp + seg * a.E_pad + r, i, acc);
      }
    } else {
      for (int i = 0; i < ntg; i++) {
        float acc = 0.0f;
        if (r < a.E) {  // fp32 router rows: fma chain over the segment (x unquantised)
          const int j0 = seg * (a.H / ROUTER_SEGS), j1 = j0 + a.H / ROUTER_SEGS;
          const float *wr = (const float *)a.W + (size_t)r * a.H;
          const float *xv = a.x + (size_t)(t0 + i) * a.H;
          if (a.norm) {
            const float inv = ninv[i];
            for (int j = j0; j < j1; j++) acc = __fmaf_rn(__ldg(wr + j), __fmul_rn(__ldg(xv + j), inv), acc);
          } else {
            for (int j = j0; j < j1; j++) acc = __fmaf_rn(__ldg(wr + j), __ldg(xv + j), acc);
          }
        }
        st_cluster_f32(lgp + seg * a.E_pad + r, i, acc);
      }
    }
    __syncwarp();  // every lane is done with the tiles before the next copy
  }
  cluster_sync_all();  // block i has every segment's sums of token i
  if (seg >= ntg) return;
  const int t = t0 + seg;
  // ---- routing of token t by block seg of its cluster
  const RouteScratch rs = route_scratch(work, a.E_pad, a.k);
  int32_t *hash_ids = (int32_t *)(work + route_block_smem(a.E_pad, a.k));  // hash routing: this token's ids
  {
    if (a.learned) {
#pragma unroll
      for (int i = 0; i < RC_MAX_E / (RC_WARPS * 32); i++) {
        const int e = threadIdx.x + i * RC_WARPS * 32;
        if (e < a.E_pad) {
          float lg = 0.0f;
          if (e < a.E)
            for (int g = 0; g < ROUTER_SEGS; g++) lg = __fadd_rn(lg, lgp[g * a.E_pad + e]);
          route_score(rs, e, a.E, lg, bias_r[i]);
        }
      }
      route_select(rs, a.E_pad, a.k, a.scale, a.ids + (size_t)t * a.k, a.w + (size_t)t * a.k);
    } else if (threadIdx.x < a.k) {
      const int v = __ldg(a.tok + t);
      const bool okv = v >= 0 && v < a.vocab;
      if (!okv && threadIdx.x == 0) raise_flag(a.err, DS4MOE_DEVERR_TOKEN_ID);
      const int e = okv ? __ldg(a.hash + (size_t)v * a.k + threadIdx.x) : -1;
      hash_ids[threadIdx.x] = e;
      a.ids[(size_t)t * a.k + threadIdx.x] = e;
      a.w[(size_t)t * a.k + threadIdx.x] = okv ? __fmul_rn(__fdiv_rn(1.0f, (float)a.k), a.scale) : 0.0f;
    }
  }
  if (!a.bucket) return;
  // ---- bucketing of the call by the block that routed its last token (a
  // single token: from this block's own selection, still in shared memory)
  int32_t *scr = hash_ids + 16;
  if (a.T == 1) {  // the expert kernels build a single token's table from its ids
    if (threadIdx.x < a.k) {
      const int e = a.learned ? rs.sel[threadIdx.x] : hash_ids[threadIdx.x];
      if (e >= a.E) raise_flag(a.err, DS4MOE_DEVERR_INTERNAL);
    }
    return;
  }
  if (!block_ticket_last(a.rticket, a.T, s_flag)) return;
  int32_t *ids_s = scr;
  for (int i = threadIdx.x; i < a.T * a.k; i += blockDim.x) ids_s[i] = __ldcg(a.ids + i);
  __syncthreads();
  bucket_rank(ids_s, a.T, a.E, a.k, a.NS, a.n_shared, ids_s + ((a.T * a.k + 3) & ~3), a.bucket, a.A_cap, a.err);
}

// ===========================================================================
// Host launchers.

cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args,
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
  const int n = h->Tc * d.top_k;
  const size_t route = route_block_smem(h->E_pad, d.top_k) + 64 +
                       (size_t)(((n + 3) & ~3) + bucket_rank_smem_ints(n)) * 4;
  if (route > work) work = route;
  return rc_work_off(h->E_pad, per, ROUTER_SEGS) + work;
}

size_t route_dec_smem(const ds4moe_layer *h) {
  // the decode path fits when the router kernel and both expert kernels fit
  const size_t r = router_dec_smem(h), x = experts_smem(h);
  return r > x ? r : x;
}

cudaError_t launch_dec_route(const ds4moe_layer *h, const float *x, const int32_t *tok, int T, int32_t *ids,
                             float *w, bool bucket, cudaStream_t s, bool norm, float eps) {
  const ds4moe_layer_desc &d = h->d;
  RouteDecArgs r = {};
  r.x = x, r.T = T, r.H = d.hidden, r.E = d.n_experts, r.E_pad = h->E_pad, r.k = d.top_k, r.NS = h->NS;
  r.n_shared = d.n_shared, r.vocab = d.vocab, r.scale = d.route_scale, r.A_cap = bucket_cap(h, T);
  r.learned = d.route == DS4MOE_ROUTE_LEARNED;
  r.norm = norm && x, r.eps = eps;
  r.q8 = r.learned && d.router_fmt == DS4MOE_Q8_0;
  r.W = h->router, r.bias = h->bias, r.hash = h->hash, r.tok = tok;
  r.xq = h->xq, r.dx = h->dx, r.gs = h->gs, r.err = h->err;
  r.ids = ids, r.w = w, r.rticket = h->rticket;
  r.bucket = bucket ? h->bucket : nullptr;
  r.xq_ready = bucket && x ? h->xq_ready : nullptr;
  void *args[] = {&r};
  // without bucketing (prefill, ds4moe_route) and from 16 tokens on, a
  // cluster takes 8 tokens: its router tiles are read once for all of them
  r.tg = (!bucket && T >= 2 * ROUTER_SEGS) ? ROUTER_SEGS : 1;
  return launch_pdl((const void *)k_router_dec, dim3(ROUTER_SEGS, (T + r.tg - 1) / r.tg), dim3(RC_WARPS * 32),
                    router_dec_smem(h), s,
                    args, true);
}

cudaError_t decode_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(k_router_dec, cudaFuncAttributeMaxDynamicSharedMemorySize, DEC_SMEM_LIMIT);
  if (e == cudaSuccess) e = experts_set_attributes();
  return e;
}

}  // namespace ds4

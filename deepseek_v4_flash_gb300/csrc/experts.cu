// experts.cu -- gate/up and down of the routed and shared experts for a
// decode-sized call (n_tok <= DEC_MAX_T).
//
// Persistent: one block per SM (two for single-token calls), XC = 8 compute
// warps and XE = 4 epilogue warps (two for single-token calls). A work item
// is 16 rows of gate and up (interleaved per K-step) or 32 rows of down (two
// 16-row tiles per K-step) of one expert, for the
// tokens routed to that expert; a unit is an item with one pass over up to
// TT of those tokens. Every expert row is summed in 8 K-segments (CAS step
// 4), and compute warp w owns segment w of every unit: it streams that
// segment's tiles through a private ring of 1-D bulk async copies (mbarrier
// completion, bounded waits), keeps the segment chains for each token in
// registers, and leaves them in a shared-memory slot. An epilogue warp adds
// the segment sums in order and finishes the unit: SwiGLU and the int8
// requant of each 32-row block of h (gate/up), or the down output and the
// fixed-order combine into y (down). A 32-row block of h spans two gate/up
// items and the combine spans every slot of a token, so completion across
// blocks uses self-resetting tickets.
//
// Items are dealt to blocks round-robin in a fixed order (shared expert
// first, then the routed experts in bucket order); each block lists its items
// once in shared memory, so every warp walks the same unit sequence without
// any queue. The shared expert's weights are requested before the wait for
// the previous kernel; the routed items come after it. Gate/up with staged
// activations starts the shared expert's items as soon as the router blocks
// have written the codes of x (a release/acquire count), before the router
// has finished routing.
#include "bucket.cuh"
#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"

namespace ds4 {

constexpr int XC = EXPERT_SEGS;  // compute warps, one K-segment each
// Epilogue warps: 4, or 2 for single-token calls (a block has about three
// units then; two blocks per SM, and 10 warps instead of 12 leave the
// compute warps 96 registers instead of 80, with no spills).
__host__ __device__ constexpr int x_epi_warps(int TT) { return TT == 1 ? 2 : 4; }
__host__ __device__ constexpr int x_warps(int TT) { return XC + x_epi_warps(TT); }
// Ring per compute warp, 10.75 KB in flight per warp and 86 KB per SM, which
// covers the loaded HBM latency at full bandwidth: gate/up 2 slots of 5376
// bytes (two K-steps of a routed item, computed together for instruction-
// level parallelism), down 4 slots of 2688 bytes (one K-step of a routed
// 32-row item). Down at eight tokens: 2 slots, so that its activations
// (8 tokens x every slot) fit in shared memory beside the ring.
// With 4-bit routed experts a down K-step takes 4736 bytes: down then uses
// 2 slots of that size (about the same bytes in flight).
__host__ __device__ constexpr int x_ring_nst(int TT, bool down, bool wide) {
  return down ? (wide ? 2 : (TT >= 8 ? 2 : 4)) : 2;
}
__host__ __device__ constexpr int x_ring_stride(bool down, bool wide) { return down ? (wide ? 2 * Q4S_TILE : 2688) : 5376; }
__host__ __device__ constexpr int x_ring_bytes(int TT, bool down, bool wide) {
  return x_ring_nst(TT, down, wide) * x_ring_stride(down, wide);
}

struct XArgs {
  int H, F, E, k, NS, n_shared, T, A_cap;
  int rf, sf, down, K, rows;
  int wide;                      // a 4-bit matrix in the layer: the wider down ring
  int maxj;                      // item-table entries per block
  const uint8_t *w_r, *w_s;      // routed / shared weights (RG16)
  const int8_t *aq;              // activations in global memory: xq or hq
  const float *ad;
  const int16_t *ag;
  const int32_t *bucket;         // bucket table (bucket.cuh)
  int32_t *xq_ready;             // router blocks whose codes of x are written
  int xq_parts;                  // ... of this many (all of the call's)
  const int32_t *ids;            // routing [T][k]
  const float *w;
  int8_t *hq;                    // gate/up outputs
  float *dh;
  int16_t *gsh;
  float *hbuf;                   // [T*NS][F] SwiGLU values before requant
  int32_t *hticket;              // [T*NS][F/32]
  float *apart;                  // [T*NS][H] per-slot down outputs
  int32_t *cticket;              // [T][H/32]
  float *y;
  uint32_t *err;
  // bound of the hand-off waits (between the block's warps, and on the
  // router's count of quantised x); waits on the block's own copies keep
  // WAIT_LIMIT, so a block that gives up never leaves a copy in flight
  long long hlimit;
};

// Partial-sum slots between the compute and the epilogue warps (down at
// eight tokens: 4, for the same reason as its ring).
__host__ __device__ constexpr int x_slots(int TT, bool down) { return down && TT >= 8 ? 4 : 8; }

// Invariants of the items of one kind (shared or routed) for one warp.
struct XKind {
  int fmt, kb, nks, S, ksps, nst, sbytes, ks0;
  size_t item_bytes;  // one 16-row item over the whole K
};

__device__ __forceinline__ XKind x_kind(const XArgs &a, int fmt, int warp, int stride) {
  XKind k;
  k.fmt = fmt;
  k.kb = 2 * tile_bytes(fmt);  // a K-step of an item: two tiles
  k.nks = a.K / kstep(fmt);
  k.S = expert_segs(fmt, a.K);
  const int nseg = k.nks / k.S;
  int ks = stride / k.kb;  // K-steps per ring stage: as many as fit, dividing the segment
  if (ks > nseg) ks = nseg;
  while (ks > 1 && nseg % ks) ks--;
  k.ksps = ks < 1 ? 1 : ks;
  k.nst = warp < k.S ? nseg / k.ksps : 0;
  k.sbytes = k.ksps * k.kb;
  k.ks0 = warp * nseg;
  k.item_bytes = (size_t)k.nks * k.kb;
  return k;
}

// This block's items are c, c + G, c + 2G, ... of the fixed order (shared
// expert items first, then the routed experts' in bucket order). Entry j of
// the block's item table: {byte offset (lo, hi) into the routed or shared
// weights, tokens, list offset (-1: the shared expert, tokens 0..T-1)} and
// {routed, 16-row group, -, -}.
__device__ __forceinline__ void x_table_entry(const XArgs &a, int i, int nsh, int RG, const int4 *act,
                                              size_t ib_s, size_t ib_r, int4 *tab) {
  size_t off;
  int n_tok, list_off, routed, rg;
  if (i < nsh) {
    routed = 0, rg = i, n_tok = a.T, list_off = -1;
    off = (size_t)rg * ib_s;
  } else {
    const int j = i - nsh, aj = j / RG;
    const int4 en = act[a.n_shared + aj];
    routed = 1, rg = j % RG, n_tok = en.y, list_off = en.z;
    off = ((size_t)en.x * RG + rg) * ib_r;
  }
  tab[0] = make_int4((int)(off & 0xFFFFFFFFu), (int)(off >> 32), n_tok, list_off);
  tab[1] = make_int4(routed, rg, 0, 0);
}

// Slot row and activation row of token index idx of an item.
__device__ __forceinline__ void x_token(const XArgs &a, int list_off, const int32_t *list, int idx, int *sr,
                                        int *arow) {
  const int code = list_off < 0 ? (idx << 5) | a.k : list[list_off + idx];
  const int t = code >> 5;
  *sr = t * a.NS + (code & 31);
  *arow = a.down ? *sr : t;
}

// CAS step 1 over 32 values held one per lane, written as the SwiGLU codes
// of h-block `blk` of slot row sr.
__device__ __forceinline__ void x_requant(const XArgs &a, float h, int sr, int blk, int lane) {
  const float amax = warp_max(fabsf(h));
  const float d = __fdiv_rn(amax, 127.0f);
  const int q = cas_code(h, d);
  const int gsum = half_warp_sum(q);
  a.hq[(size_t)sr * a.F + 32 * blk + lane] = (int8_t)q;
  if (lane == 0) a.dh[(size_t)sr * (a.F >> 5) + blk] = d;
  if ((lane & 15) == 0) a.gsh[(size_t)sr * (a.F >> 4) + 2 * blk + (lane >> 4)] = (int16_t)gsum;
}

// CAS step 8 for rows 32*rg .. +31 of token t (lane = row).
// Every value is requested before the first is used (up to 8 routed slots;
// more take the plain loop).
__device__ __forceinline__ void x_combine(const XArgs &a, int t, int rg, int lane) {
  const int r = 32 * rg + lane;
  const float *ap = a.apart + (size_t)t * a.NS * a.H + r;
  const float *wp = a.w + (size_t)t * a.k;
  float *yp = a.y + (size_t)t * a.H + r;
  constexpr int KF = 8;
  if (a.k <= KF) {
    const int id0 = __ldg(a.ids + (size_t)t * a.k);
    float wv[KF], av[KF];
#pragma unroll
    for (int j = 0; j < KF; j++) {
      wv[j] = j < a.k ? __ldg(wp + j) : 0.0f;
      av[j] = j < a.k ? __ldcg(ap + (size_t)j * a.H) : 0.0f;
    }
    const float sh = a.n_shared ? __ldcg(ap + (size_t)a.k * a.H) : 0.0f;
    const float y0 = *yp;
    if (id0 < 0) return;  // an out-of-range hash token adds nothing
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < KF; j++)
      if (j < a.k) acc = __fadd_rn(acc, __fmul_rn(wv[j], av[j]));
    if (a.n_shared) acc = __fadd_rn(acc, sh);
    *yp = __fadd_rn(y0, acc);
    return;
  }
  if (__ldg(a.ids + (size_t)t * a.k) < 0) return;
  float acc = 0.0f;
  for (int j = 0; j < a.k; j++) acc = __fadd_rn(acc, __fmul_rn(__ldg(wp + j), __ldcg(ap + (size_t)j * a.H)));
  if (a.n_shared) acc = __fadd_rn(acc, __ldcg(ap + (size_t)a.k * a.H));
  *yp = __fadd_rn(*yp, acc);
}

// Shared-memory layout (bytes) for TT, staged activations of `act_bytes`,
// an item table of `maxj` entries.
struct XSmem {
  int ring, bars, ctrl, part, tab, valid, bkt, act, total;
};

__host__ __device__ inline XSmem x_smem(int TT, bool down, bool wide, int mats, int nbk, int act_bytes, int maxj,
                                        int T) {
  XSmem s;
  s.ring = 0;
  s.bars = XC * x_ring_bytes(TT, down, wide);
  s.ctrl = s.bars + XC * 8 * 8;
  s.part = s.ctrl + 256;  // bucket barrier, item count, then full[8] and empty[8] slot barriers
  s.tab = s.part + x_slots(TT, down) * XC * mats * TT * TILE_ROWS * 4;
  s.valid = s.tab + maxj * 32;
  s.bkt = s.valid + ((T * 4 + 127) & ~127);
  s.act = s.bkt + ((nbk * 4 + 127) & ~127);
  s.total = s.act + act_bytes;
  return s;
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// AS: activations staged in shared memory. DOWN: the down kernel (items of
// 32 rows), else gate/up (items of 16 rows, gate and up).
// The bucket table is loaded by one warp (the last epilogue warp, at its
// start, unless another gets there first), which publishes the routed items
// to the others; the compute warps meanwhile run the shared expert's items,
// which need no routing. The shared expert's weights are requested before
// the wait for the previous kernel.
// Q4: the 4-bit steps compiled in. The one-token kernels of layers without
// a 4-bit matrix leave them out (a smaller instruction footprint: 2 % faster
// at one token, measured; at eight tokens it measured slower, so only there).
template <int TT, bool AS, bool DOWN, bool Q4 = true>
__global__ void __launch_bounds__(x_warps(TT) * 32, TT == 1 ? 2 : 1) k_experts(XArgs a) {
  constexpr int XE = x_epi_warps(TT), X_WARPS = x_warps(TT);
  extern __shared__ __align__(128) uint8_t smem[];
  const int X_NST = x_ring_nst(TT, DOWN, a.wide != 0), X_STRIDE = x_ring_stride(DOWN, a.wide != 0);
  constexpr int PS = x_slots(TT, DOWN);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int mats = 2;       // gate and up (16 rows), or the two 16-row halves of 32 rows (down)
  constexpr int ROWS = DOWN ? 32 : 16;  // output rows of a work item
  const int nbk = bucket_table_ints(a.A_cap, a.T, a.NS);
  const int act_rows = DOWN ? a.T * a.NS : a.T;
  const int act_bytes = AS ? act_rows * (a.K + (a.K >> 5) * 4 + (a.K >> 4) * 2) : 0;
  const XSmem L = x_smem(TT, DOWN, a.wide != 0, mats, nbk, act_bytes, a.maxj, a.T);
  volatile int *s_nitems = (volatile int *)(smem + L.ctrl + 8);  // items of this block (after the bucket)
  int *s_claim = (int *)(smem + L.ctrl + 12);                     // the warp that loads the bucket
  const uint32_t full0 = smem_u32(smem + L.ctrl) + 64, empty0 = full0 + 64;  // slot barriers, 8 bytes apart
  float *part = (float *)(smem + L.part);  // [PS][XC][mats][TT][16]
  int4 *tab = (int4 *)(smem + L.tab);      // [maxj][2]
  int *valid = (int *)(smem + L.valid);    // down: routed slots with an expert, per token
  int32_t *bks = (int32_t *)(smem + L.bkt);
  const int4 *act = (const int4 *)(bks + BKT_HDR);
  const int32_t *list = bks + BKT_HDR + 4 * a.A_cap;
  const int8_t *aq = a.aq;
  const float *ad = a.ad;
  const int16_t *ag = a.ag;
  if (AS) {
    aq = (const int8_t *)(smem + L.act);
    ad = (const float *)(smem + L.act + act_rows * a.K);
    ag = (const int16_t *)(smem + L.act + act_rows * a.K + act_rows * (a.K >> 5) * 4);
  }
  pdl_launch_dependents();
  const uint32_t ring = smem_u32(smem + L.ring + warp * x_ring_bytes(TT, DOWN, a.wide != 0));
  const uint32_t bar = smem_u32(smem + L.bars + warp * 8 * 8);
  const int nsh = a.n_shared ? a.rows / ROWS : 0, RG = a.rows / ROWS;
  const int G = gridDim.x, c = blockIdx.x;
  const int n_sh_items = c < nsh ? (nsh - 1 - c) / G + 1 : 0;  // this block's shared items
  const XKind ks = x_kind(a, a.sf, warp < XC ? warp : 0, X_STRIDE), kr = x_kind(a, a.rf, warp < XC ? warp : 0, X_STRIDE);
  if (threadIdx.x == 0) {
    for (int i = 0; i < PS; i++) mbar_init(full0 + 8 * i, XC), mbar_init(empty0 + 8 * i, 1);
    *s_nitems = -1;  // no routed items known yet (read by the first prefetch pass)
    *s_claim = 0;
  }
  if (warp < XC && lane == 0)
    for (int i = 0; i < X_NST; i++) mbar_init(bar + 8 * i, 1);
  if (lane == 0) fence_mbar_init();
  // the shared-expert entries of the item table need no routing
  for (int j = threadIdx.x; j < n_sh_items; j += blockDim.x)
    x_table_entry(a, c + j * G, nsh, RG, act, ks.item_bytes, kr.item_bytes, tab + 2 * j);
  int n_items = -1;  // this block's items, once the bucket is known
  bool failed = false;
  __syncthreads();  // barriers and shared entries ready

  // Routed entries (after the bucket is in shared memory), by one warp.
  auto build_routed = [&]() {
    const int n_all = nsh + (bks[0] - a.n_shared) * RG;
    const int n = c < n_all ? (n_all - 1 - c) / G + 1 : 0;
    for (int j = n_sh_items + lane; j < n; j += 32)
      x_table_entry(a, c + j * G, nsh, RG, act, ks.item_bytes, kr.item_bytes, tab + 2 * j);
    __syncwarp();
    __threadfence_block();
    if (lane == 0) *s_nitems = n;
  };
  // the routed item count once published (n_items stays -1 before)
  auto poll_items = [&]() {
    if (n_items < 0) {
      const int v = *s_nitems;
      if (v >= 0) {
        __threadfence_block();
        n_items = v;
      }
    }
  };
  auto wait_items = [&]() -> bool {
    poll_items();
    if (n_items >= 0) return true;
    int mine = 0;
    if (lane == 0) mine = atomicCAS(s_claim, 0, 1) == 0;
    if (__shfl_sync(0xffffffffu, mine, 0)) {  // this warp loads the bucket for the block
      pdl_wait();
      if (a.T == 1) {  // a single token: the table from its routed ids
        const int e = lane < a.k ? __ldcg(a.ids + lane) : -1;
        bucket_one_token_ids(e, a.E, a.k, a.n_shared, bks, a.A_cap, nullptr, lane);
      } else
      // (loads of a round issued before its stores)
      for (int i0 = 0; i0 < nbk; i0 += 4 * 32) {
        int v[4];
#pragma unroll
        for (int j = 0; j < 4; j++) v[j] = i0 + lane + 32 * j < nbk ? __ldcg(a.bucket + i0 + lane + 32 * j) : 0;
#pragma unroll
        for (int j = 0; j < 4; j++)
          if (i0 + lane + 32 * j < nbk) bks[i0 + lane + 32 * j] = v[j];
      }
      if (DOWN)  // routed slots with an expert, per token (the combine's arrival count)
        for (int t = lane; t < a.T; t += 32) {
          int n = 0;
          for (int j0 = 0; j0 < a.k; j0 += 8) {
            int v[8];
#pragma unroll
            for (int j = 0; j < 8; j++) v[j] = j0 + j < a.k ? __ldg(a.ids + (size_t)t * a.k + j0 + j) : -1;
#pragma unroll
            for (int j = 0; j < 8; j++) n += v[j] >= 0;
          }
          valid[t] = n;
        }
      __syncwarp();
      build_routed();
    }
    const long long t0 = clock64();
    for (poll_items(); n_items < 0; poll_items()) {
      if (clock64() - t0 > a.hlimit) return false;
      __nanosleep(64);
    }
    return true;
  };

  // ---- compute warps: producer (ring) cursor
  int pj = 0, ppass = 0, pstage = 0, pnpass = 0, pnst = 0, psb = 0;
  bool p_ok = false, p_done = false;
  const uint8_t *psrc = nullptr;
  uint32_t g_prod = 0, g_cons = 0;
  auto fill = [&]() {
    while (!p_done && g_prod - g_cons < X_NST) {
      if (!p_ok) {
        if (pj >= n_sh_items) poll_items();
        if (pj >= n_sh_items && n_items < 0) return;  // routed items: after the previous kernel
        if (pj >= (pj < n_sh_items ? n_sh_items : n_items)) {
          p_done = true;
          return;
        }
        const int4 e0 = tab[2 * pj], e1 = tab[2 * pj + 1];
        const bool rt = e1.x != 0;
        pnst = rt ? kr.nst : ks.nst, psb = rt ? kr.sbytes : ks.sbytes;
        pnpass = (e0.z + TT - 1) / TT, ppass = 0, pstage = 0;
        psrc = (rt ? a.w_r : a.w_s) + ((size_t)(uint32_t)e0.x | ((size_t)(uint32_t)e0.y << 32)) +
               (size_t)(rt ? kr.ks0 * kr.kb : ks.ks0 * ks.kb);
        if (pnst == 0 || pnpass == 0) {  // no segment of this item for this warp
          pj++;
          continue;
        }
        p_ok = true;
      }
      // a slot is refilled only after the warp barrier that ends its use:
      // every lane has consumed the values it loaded from it
      const uint32_t slot = g_prod % X_NST;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar + 8 * slot, psb);
        bulk_g2s(ring + slot * X_STRIDE, psrc + (size_t)pstage * psb, psb, bar + 8 * slot);
      }
      g_prod++;
      if (++pstage == pnst) {
        pstage = 0;
        if (++ppass == pnpass) pj++, p_ok = false;
      }
    }
  };
  if (warp < XC) {
    __syncwarp();
    if (n_sh_items > 0) fill();  // shared-expert items need no routing: request them before the wait
  }

  {
    // ---- the staged activations (the bucket table is loaded by the first
    // warp that needs it, see wait_items). Gate/up with staged activations
    // waits only for the router blocks' codes of x (count with acquire
    // semantics, read through L2), so the shared expert runs while the
    // router is still routing; otherwise wait for the previous kernel. Down
    // clears the count: the gate/up grid, and with it the router grid (every
    // gate/up block waits for it before its routed items), is complete.
    constexpr bool EARLY = !DOWN && AS;
    if (EARLY) {
      if (threadIdx.x == 0 && !wait_count(a.xq_ready, a.xq_parts, a.hlimit)) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
      __syncthreads();
    } else {
      pdl_wait();
      if (DOWN && blockIdx.x == 0 && threadIdx.x == 0) a.xq_ready[0] = 0;
    }
    // Down with staged activations: the last warp loads the routed table
    // while the others stage (unstaged kernels load it after the barrier,
    // measured faster there; EARLY gate/up must wait for the router first).
    constexpr bool CLAIM = AS && !EARLY;
    const int nstage = CLAIM ? blockDim.x - 32 : blockDim.x;
    if (CLAIM && warp == X_WARPS - 1) {
      (void)wait_items();
    } else if (AS) {
      // the three arrays as one run of 16-byte words, every load of a
      // round issued before its stores
      uint4 *dst = (uint4 *)(smem + L.act);
      const size_t nq = (size_t)act_rows * a.K / 16, nd = (size_t)act_rows * (a.K >> 5) * 4 / 16,
                   ng = (size_t)act_rows * (a.K >> 4) * 2 / 16, n = nq + nd + ng;
      constexpr int SB = 4;
      for (size_t b0 = 0; b0 < n; b0 += (size_t)SB * nstage) {
        uint4 v[SB];
#pragma unroll
        for (int j = 0; j < SB; j++) {
          const size_t i = b0 + threadIdx.x + (size_t)j * nstage;
          if (i < n)
            v[j] = __ldcg(i < nq ? (const uint4 *)a.aq + i
                          : i < nq + nd ? (const uint4 *)a.ad + (i - nq) : (const uint4 *)a.ag + (i - nq - nd));
        }
#pragma unroll
        for (int j = 0; j < SB; j++) {
          const size_t i = b0 + threadIdx.x + (size_t)j * nstage;
          if (i < n) dst[i] = v[j];
        }
      }
    }
    __syncthreads();
  }

  if (warp < XC) {
    // ================= compute warp: segment `warp` of every unit
    int cj = 0, cpass = 0, cstage = 0, cnpass = 0, unit = 0, list_off = 0, n_tok = 0;
    int c_nst = 0, c_ksps = 1, c_kb = 0, c_ks0 = 0, c_fmt = 0;
    bool c_ok = false;
    int arow[TT], nt = 0;
    Chains<(TT > 1)> acc[TT];  // per token: the two tiles' row chains
    // units of eight tokens that hold at least MMA_MIN_NT of them: the int8
    // tensor-core steps (with fewer tokens most of the MMA's columns would
    // idle, and the dp4a steps skip the empty ones); this lane's rows of
    // activations: B token lane / 4, D tokens 2 (lane % 4) and + 1
    constexpr int MMA_MIN_NT = 3;
    bool mma = false;
    MChains macc;
    int ar_g = 0, ar0 = 0, ar1 = 0;
    for (;;) {
      if (!c_ok) {  // the consumer's next item
        if (cj >= n_sh_items && !wait_items()) {
          failed = true;
          break;
        }
        if (cj >= (cj < n_sh_items ? n_sh_items : n_items)) break;
        const int4 e0 = tab[2 * cj], e1 = tab[2 * cj + 1];
        const bool rt = e1.x != 0;
        c_nst = rt ? kr.nst : ks.nst, c_ksps = rt ? kr.ksps : ks.ksps, c_kb = rt ? kr.kb : ks.kb;
        c_ks0 = rt ? kr.ks0 : ks.ks0, c_fmt = rt ? kr.fmt : ks.fmt;
        n_tok = e0.z, list_off = e0.w, cnpass = (n_tok + TT - 1) / TT, cpass = 0, cstage = 0;
        c_ok = true;
        if (cnpass == 0) {
          cj++, c_ok = false;
          continue;
        }
      }
      if (cstage == 0) {  // a new unit: its tokens
        nt = min(TT, n_tok - cpass * TT);
        mma = TT == 8 && nt >= MMA_MIN_NT;
        if (mma) {
          int sr;
          const int u0 = cpass * TT, last = n_tok - 1;
          x_token(a, list_off, list, min(u0 + (lane >> 2), last), &sr, &ar_g);
          x_token(a, list_off, list, min(u0 + 2 * (lane & 3), last), &sr, &ar0);
          x_token(a, list_off, list, min(u0 + 2 * (lane & 3) + 1, last), &sr, &ar1);
          mchains_zero(macc);
        } else {
#pragma unroll
          for (int i = 0; i < TT; i++) {
            int sr;
            x_token(a, list_off, list, min(cpass * TT + i, n_tok - 1), &sr, &arow[i]);
            chains_zero(acc[i]);
          }
        }
      }
      if (c_nst > 0) {
        fill();
        const uint32_t slot = g_cons % X_NST;
        if (!mbar_wait_bounded(bar + 8 * slot, (g_cons / X_NST) & 1)) {
          failed = true;
          break;
        }
        __syncwarp();
        const uint32_t st = ring + slot * X_STRIDE;
        const int s0 = c_ks0 + cstage * c_ksps;
        if (TT == 8 && mma) {
          for (int j = 0; j < c_ksps; j++) {
            const uint32_t t = st + j * c_kb;
            if (c_fmt == DS4MOE_Q2S) sb_step_mma<AS, false>(t, lane, s0 + j, a.K, ar_g, ar0, ar1, aq, ad, ag, macc);
            else if (Q4 && c_fmt == DS4MOE_Q4S) sb_step_mma<AS, true>(t, lane, s0 + j, a.K, ar_g, ar0, ar1, aq, ad, ag, macc);
            else q8_step_mma<AS>(t, lane, s0 + j, a.K, ar_g, ar0, ar1, aq, ad, macc);
          }
        } else if (c_fmt == DS4MOE_Q2S && c_ksps == 2) {  // two K-steps in one block of code: their dots overlap
          q2s_step<TT, AS, (TT > 1)>(st, lane, s0, a.K, arow, nt, aq, ad, ag, acc);
          q2s_step<TT, AS, (TT > 1)>(st + c_kb, lane, s0 + 1, a.K, arow, nt, aq, ad, ag, acc);
        } else {
          for (int j = 0; j < c_ksps; j++) {
            const uint32_t t = st + j * c_kb;
            if (c_fmt == DS4MOE_Q2S) q2s_step<TT, AS, (TT > 1)>(t, lane, s0 + j, a.K, arow, nt, aq, ad, ag, acc);
            else if (Q4 && c_fmt == DS4MOE_Q4S) q4s_step<TT, AS, (TT > 1)>(t, lane, s0 + j, a.K, arow, nt, aq, ad, ag, acc);
            else q8_step<TT, AS, (TT > 1)>(t, lane, s0 + j, a.K, arow, nt, aq, ad, acc);
          }
        }
        __syncwarp();
        g_cons++;
      }
      if (c_nst == 0 || cstage == c_nst - 1) {
        // the unit's segment is done: partial sums into slot unit % PS
        const int ps = unit % PS, ph = unit / PS;
        if (ph > 0 && !mbar_wait_bounded(empty0 + 8 * ps, (ph - 1) & 1, a.hlimit)) {
          failed = true;
          break;
        }
        if (TT == 8 && mma && c_nst > 0) {
          // [tile][token][row]: rows g, g + 8 of both tiles, tokens 2t, 2t + 1
          float *dst = part + (size_t)(ps * XC + warp) * mats * TT * TILE_ROWS;
          const int g = lane >> 2, k0 = 2 * (lane & 3);
#pragma unroll
          for (int i = 0; i < 4; i++) {
            const int m = i >> 1, hh = i & 1;
            float v0, v1;
            f2_unpack(macc.v[m][hh], v0, v1);
            if (k0 < nt) dst[(m * TT + k0) * TILE_ROWS + g + 8 * hh] = v0;
            if (k0 + 1 < nt) dst[(m * TT + k0 + 1) * TILE_ROWS + g + 8 * hh] = v1;
          }
        } else if (c_nst > 0 && (lane & 1) == 0) {
          float *dst = part + (size_t)(ps * XC + warp) * mats * TT * TILE_ROWS;
#pragma unroll
          for (int i = 0; i < TT; i++) {
            if (i < nt) {
              float a0, a1;
              chains_get(acc[i], a0, a1);
              dst[i * TILE_ROWS + (lane >> 1)] = a0;
              dst[(TT + i) * TILE_ROWS + (lane >> 1)] = a1;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(full0 + 8 * ps);
        cstage = 0, unit++;
        if (++cpass == cnpass) cj++, c_ok = false;
      } else {
        cstage++;
      }
    }
    if (failed) {
      if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
      for (uint32_t g = g_cons; g < g_prod; g++) (void)mbar_wait_bounded(bar + 8 * (g % X_NST), (g / X_NST) & 1);
    }
    return;
  }

  // ================= epilogue warps: units u whose slot u % PS maps to this
  // warp ((u % PS) % XE == ew), so the units of one slot, which wait on the
  // same barriers in alternating phases, are always taken by the same warp
  const int ew = warp - XC;
  // the last epilogue warp loads the bucket table at once; in the down kernel
  // every epilogue warp needs it (arrival counts) before its first unit
  if ((ew == XE - 1 || DOWN) && !wait_items()) {
    if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
    return;
  }
  int unit = 0;
  for (int j = 0;; j++) {
    if (j >= n_sh_items && !wait_items()) {
      if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
      return;
    }
    if (j >= (j < n_sh_items ? n_sh_items : n_items)) break;
    const int4 e0 = tab[2 * j], e1 = tab[2 * j + 1];
    const int S = e1.x ? kr.S : ks.S, rg = e1.y, n_tok = e0.z, list_off = e0.w;
    const int npass = (n_tok + TT - 1) / TT;
    for (int p = 0; p < npass; p++, unit++) {
      if ((unit % PS) % XE != ew) continue;
      const int ps = unit % PS;
      if (!mbar_wait_bounded(full0 + 8 * ps, (unit / PS) & 1, a.hlimit)) {
        if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
        return;
      }
      const int nt = min(TT, n_tok - p * TT);
      const float *src = part + (size_t)ps * XC * mats * TT * TILE_ROWS;
      const int r = lane & 15;
      if (!DOWN) {  // 16 rows of gate and up: lanes 0-15 token i, 16-31 token i+1
        for (int i0 = 0; i0 < nt; i0 += 2) {
          const int i = i0 + (lane >> 4);
          if (i < nt) {
            float g = 0.0f, uu = 0.0f;  // segment sums in order (CAS step 4)
            for (int sg = 0; sg < S; sg++) {
              const float *pp = src + (size_t)sg * mats * TT * TILE_ROWS;
              g = __fadd_rn(g, pp[i * TILE_ROWS + r]);
              uu = __fadd_rn(uu, pp[(TT + i) * TILE_ROWS + r]);
            }
            int sr, arow;
            x_token(a, list_off, list, p * TT + i, &sr, &arow);
            a.hbuf[(size_t)sr * a.F + TILE_ROWS * rg + r] = __fmul_rn(cas_silu(g), uu);
          }
        }
      } else {  // 32 rows (lane = row) of each token
        const int m = lane >> 4;
        for (int i = 0; i < nt; i++) {
          float g = 0.0f;
          for (int sg = 0; sg < S; sg++) g = __fadd_rn(g, src[(size_t)sg * mats * TT * TILE_ROWS + (m * TT + i) * TILE_ROWS + r]);
          int sr, arow;
          x_token(a, list_off, list, p * TT + i, &sr, &arow);
          a.apart[(size_t)sr * a.H + 32 * rg + lane] = g;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * ps);  // the slot is free again
      // One ticket per token (lane i takes token i, all in flight at once):
      // gate/up: a 32-row block of h spans two items, requantised once both
      // are in; down: the fixed-order combine once every slot of the token
      // has these 32 rows. The acquire-release atomics order the other
      // item's (slot's) writes before this warp's reads; the completer resets
      // the ticket.
      {
        int last = 0;
        if (lane < nt) {
          int sr, arow;
          x_token(a, list_off, list, p * TT + lane, &sr, &arow);
          int32_t *tk;
          int expect;
          if (!DOWN) {
            tk = a.hticket + (size_t)sr * (a.F >> 5) + (rg >> 1);
            expect = 2;
          } else {
            const int t = sr / a.NS;
            tk = a.cticket + (size_t)t * (a.H >> 5) + rg;
            expect = valid[t] + a.n_shared;
          }
          int old;
          asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(tk) : "memory");
          last = old == expect - 1;
          if (last) *tk = 0;
        }
        unsigned done = __ballot_sync(0xffffffffu, last);
        __syncwarp();
        while (done) {
          const int i = __ffs(done) - 1;
          done &= done - 1;
          int sr, arow;
          x_token(a, list_off, list, p * TT + i, &sr, &arow);
          if (!DOWN) {
            const int blk = rg >> 1;
            x_requant(a, __ldcg(a.hbuf + (size_t)sr * a.F + 32 * blk + lane), sr, blk, lane);
          } else {
            x_combine(a, sr / a.NS, rg, lane);
          }
        }
      }
    }
  }
}

// ===========================================================================
// Host side.

static size_t x_act_bytes(const ds4moe_layer *h, int T, bool down) {
  const ds4moe_layer_desc &d = h->d;
  const size_t rows = down ? (size_t)T * h->NS : (size_t)T;
  const size_t K = down ? d.ffn : d.hidden;
  return rows * (K + (K / 32) * 4 + (K / 16) * 2);
}

// Tokens per unit: one for calls of one or two tokens (a unit per token; at two
// tokens only the shared expert's weights are read twice, and the one-token
// kernels run two blocks per SM without spills: measured 11 % faster), else
// up to 4 or 8.
static int x_tt(int T) { return T <= 2 ? 1 : T <= 4 ? 4 : 8; }

// Item-table entries per block: the call's items over the blocks.
// Blocks per SM: two for one-token units (registers capped to fit), so
// twice the warps hide the latency of the short per-item chains.
static int x_blocks(const ds4moe_layer *h, int T) { return (T <= 2 ? 2 : 1) * h->n_sm; }

static int x_maxj(const ds4moe_layer *h, int T, bool down) {
  const ds4moe_layer_desc &d = h->d;
  const int RG = down ? d.hidden / 32 : d.ffn / TILE_ROWS;
  const long long routed = (long long)T * d.top_k < d.n_experts ? (long long)T * d.top_k : d.n_experts;
  const long long n = (d.n_shared ? RG : 0) + routed * RG;
  const int G = x_blocks(h, T);
  return (int)((n + G - 1) / G);
}

// A 4-bit matrix anywhere in the layer: the down kernel's wider ring slots.
static bool x_wide(const ds4moe_layer *h) {
  return h->d.routed_fmt == DS4MOE_Q4S || (h->d.n_shared && h->d.shared_fmt == DS4MOE_Q4S);
}

static size_t x_smem_bytes(const ds4moe_layer *h, int T, bool down, bool as) {
  const int nbk = bucket_table_ints(bucket_cap(h, T), T, h->NS);
  return (size_t)x_smem(x_tt(T), down, x_wide(h), 2, nbk, as ? (int)x_act_bytes(h, T, down) : 0, x_maxj(h, T, down), T)
      .total;
}

size_t experts_smem(const ds4moe_layer *h) {
  // both kernels must fit at DEC_MAX_T with activations in global memory
  const size_t a = x_smem_bytes(h, DEC_MAX_T, false, false), b = x_smem_bytes(h, DEC_MAX_T, true, false);
  return a > b ? a : b;
}

// q4: the layer holds a 4-bit matrix (the one-token kernels then keep the
// 4-bit steps; the others always do)
template <bool AS, bool DOWN>
static const void *x_fn(int T, bool q4) {
  return T <= 2 ? (q4 ? (const void *)k_experts<1, AS, DOWN> : (const void *)k_experts<1, AS, DOWN, false>)
       : T <= 4 ? (const void *)k_experts<4, AS, DOWN> : (const void *)k_experts<8, AS, DOWN>;
}

cudaError_t launch_experts(const ds4moe_layer *h, int T, float *y, int down, cudaStream_t s) {
  const ds4moe_layer_desc &d = h->d;
  XArgs a = {};
  a.H = d.hidden, a.F = d.ffn, a.E = d.n_experts, a.k = d.top_k, a.NS = h->NS, a.n_shared = d.n_shared, a.T = T;
  a.A_cap = bucket_cap(h, T), a.rf = d.routed_fmt, a.sf = d.n_shared ? d.shared_fmt : d.routed_fmt, a.down = down;
  a.bucket = h->bucket, a.ids = h->ids, a.w = h->wts;
  a.xq_ready = h->xq_ready, a.xq_parts = ROUTER_SEGS * T;
  a.hq = h->hq, a.dh = h->dh, a.gsh = h->gsh, a.hbuf = h->hbuf, a.hticket = h->hticket;
  a.apart = h->apart, a.cticket = h->cticket, a.y = y, a.err = h->err;
  a.maxj = x_maxj(h, T, down != 0);
  a.wide = x_wide(h) ? 1 : 0;
  a.hlimit = h->wait_limit > 0 ? h->wait_limit : WAIT_LIMIT;
  if (!down) {
    a.K = d.hidden, a.rows = d.ffn, a.w_r = h->gu, a.w_s = h->sgu, a.aq = h->xq, a.ad = h->dx, a.ag = h->gs;
  } else {
    a.K = d.ffn, a.rows = d.hidden, a.w_r = h->dn, a.w_s = h->sdn, a.aq = h->hq, a.ad = h->dh, a.ag = h->gsh;
  }
  // activations staged in shared memory when they fit beside the rest (for
  // single-token calls: in half an SM, two blocks per SM)
  const size_t lim = T <= 2 ? (size_t)(228 * 1024 / 2 - 1024) : DEC_SMEM_LIMIT;
  const bool as = x_smem_bytes(h, T, down != 0, true) <= lim;

  const bool q4 = x_wide(h);  // a 4-bit matrix anywhere in the layer
  const void *fn = down ? (as ? x_fn<true, true>(T, q4) : x_fn<false, true>(T, q4))
                        : (as ? x_fn<true, false>(T, q4) : x_fn<false, false>(T, q4));
  void *args[] = {&a};
  return launch_pdl(fn, dim3(x_blocks(h, T)), dim3(x_warps(x_tt(T)) * 32), x_smem_bytes(h, T, down != 0, as), s, args,
                    true);
}

cudaError_t experts_set_attributes() {
  const void *fns[] = {x_fn<true, false>(1, true),  x_fn<true, false>(4, true),  x_fn<true, false>(8, true),
                       x_fn<false, false>(1, true), x_fn<false, false>(4, true), x_fn<false, false>(8, true),
                       x_fn<true, true>(1, true),   x_fn<true, true>(4, true),   x_fn<true, true>(8, true),
                       x_fn<false, true>(1, true),  x_fn<false, true>(4, true),  x_fn<false, true>(8, true),
                       x_fn<true, false>(1, false), x_fn<false, false>(1, false), x_fn<true, true>(1, false),
                       x_fn<false, true>(1, false)};
  cudaError_t e = cudaSuccess;
  for (const void *f : fns)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, DEC_SMEM_LIMIT);
  return e;
}

}  // namespace ds4

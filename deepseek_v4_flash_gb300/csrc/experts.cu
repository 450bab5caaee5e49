// experts.cu -- gate/up and down of the routed and shared experts for a
// decode-sized call (n_tok <= DEC_MAX_T).
//
// Persistent: one block per SM, XC = 8 compute warps and XE = 2 epilogue
// warps. A work item is 16 rows of one expert matrix (gate and up
// interleaved, or down) for the tokens routed to that expert; a unit is an
// item together with one pass over up to TT of those tokens. Every expert
// row is summed in S = 8 K-segments (CAS step 4), and compute warp w owns
// segment w of every unit: it streams that segment's tiles through a private
// ring of 1-D bulk async copies (mbarrier completion, bounded waits), keeps
// the segment chain of the 16 rows for each token in registers, and leaves
// it in a shared-memory slot. The epilogue warps add the S segment sums in
// order and finish the unit: SwiGLU, then the int8 requant of each 32-row
// block of h (gate/up); or the down output and the fixed-order combine into
// y (down). A 32-row block spans two items, so its completion across blocks
// uses self-resetting tickets.
//
// Items are dealt to blocks round-robin in a fixed order (shared expert
// first, then the routed experts in bucket order), so every warp of a block
// walks the same unit sequence without any queue. The gate/up kernel
// quantises x itself (when the activations fit shared memory), so the
// shared expert's units stream and compute before the router kernel ends;
// the routed units wait for its bucket table.
#include "bucket.cuh"
#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"

namespace ds4 {

constexpr int XC = EXPERT_SEGS;  // compute warps, one K-segment each
constexpr int XE = 2;            // epilogue warps
constexpr int X_WARPS = XC + XE;
constexpr int X_NST = 4;         // ring stages per compute warp
constexpr int X_STRIDE = 2688;   // ring slot bytes: one gate+up Q2S K-step

struct XArgs {
  int H, F, E, k, NS, n_shared, T, A_cap;
  int rf, sf, down, K, rows;
  const uint8_t *w_r, *w_s;      // routed / shared weights (RG16)
  const float *x;                // layer input (gate/up, quantised here when staged)
  const int8_t *aq;              // activations in global memory: xq or hq
  const float *ad;
  const int16_t *ag;
  const int32_t *bucket;         // bucket table (bucket.cuh)
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
};

__host__ __device__ constexpr int x_slots(int TT) { return TT <= 1 ? 8 : TT <= 2 ? 4 : 2; }

// Invariants of the items of one kind (shared or routed) for one warp.
struct XKind {
  int fmt, kb, nks, S, ksps, nst, sbytes, ks0;
  size_t item_bytes;  // one 16-row item over the whole K
};

__device__ __forceinline__ XKind x_kind(const XArgs &a, int fmt, int warp) {
  XKind k;
  const int mats = a.down ? 1 : 2;
  k.fmt = fmt;
  k.kb = mats * tile_bytes(fmt);
  k.nks = a.K / kstep(fmt);
  k.S = expert_segs(fmt, a.K);
  const int nseg = k.nks / k.S;
  int ks = X_STRIDE / k.kb;  // K-steps per ring stage: as many as fit, dividing the segment
  if (ks > nseg) ks = nseg;
  while (ks > 1 && nseg % ks) ks--;
  k.ksps = ks < 1 ? 1 : ks;
  k.nst = warp < k.S ? nseg / k.ksps : 0;
  k.sbytes = k.ksps * k.kb;
  k.ks0 = warp * nseg;
  k.item_bytes = (size_t)k.nks * k.kb;
  return k;
}

// Walks this block's items (c, c + G, c + 2G, ...; shared expert items
// first, then the routed experts' in bucket order), their token passes and
// this warp's stages, without divisions after the first routed item.
struct XCursor {
  int i;          // item index
  int routed;     // 0: shared item (rg = i), 1: routed
  int aj, rg;     // routed: act index (after the shared entry) and 16-row group
  int e, n_tok, list_off, npass;
  int pass, stage, unit;
  const uint8_t *src;  // this warp's segment of the item
};

// Sets up the item at c->i; false when the block has no more items. Routed
// items need the bucket (act, n_routed = active routed experts).
template <int TT>
__device__ __forceinline__ bool x_item_at(const XArgs &a, XCursor *c, int nsh, int RG, const int4 *act,
                                          int n_routed, const XKind &ks, const XKind &kr) {
  if (c->i < nsh) {
    c->routed = 0, c->rg = c->i, c->e = a.E, c->n_tok = a.T, c->list_off = -1;
    c->src = a.w_s + (size_t)c->rg * ks.item_bytes + (size_t)ks.ks0 * ks.kb;
  } else {
    if (!c->routed) {  // first routed item of this block
      const int j = c->i - nsh;
      c->aj = j / RG, c->rg = j % RG, c->routed = 1;
    }
    if (c->aj >= n_routed) return false;
    const int4 en = act[a.n_shared + c->aj];
    c->e = en.x, c->n_tok = en.y, c->list_off = en.z;
    c->src = a.w_r + ((size_t)c->e * RG + c->rg) * kr.item_bytes + (size_t)kr.ks0 * kr.kb;
  }
  c->npass = (c->n_tok + TT - 1) / TT;
  c->pass = 0, c->stage = 0;
  return true;
}

__device__ __forceinline__ void x_next_item(XCursor *c, int G, int RG) {
  c->i += G;
  if (c->routed) {
    c->rg += G;
    while (c->rg >= RG) c->rg -= RG, c->aj++;
  }
}

// Slot row and activation row of token index idx of the cursor's item.
__device__ __forceinline__ void x_token(const XArgs &a, const XCursor &c, const int32_t *list, int idx, int *sr,
                                        int *arow) {
  const int s = c.list_off < 0 ? idx * a.NS + a.k : list[c.list_off + idx];
  *sr = s;
  *arow = a.down ? s : s / a.NS;
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

// Count one arrival on a ticket; true (on every lane) for the caller that
// completes it. The acquire-release atomic orders this warp's earlier global
// writes before the completer's later reads; the completer resets it.
__device__ __forceinline__ bool x_ticket_last(int32_t *tk, int expect, int lane) {
  __syncwarp();
  int last = 0;
  if (lane == 0) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(tk) : "memory");
    last = old == expect - 1;
    if (last) *tk = 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  return last != 0;
}

// CAS step 8 for rows 32*rg .. +31 of token t (lane = row).
__device__ __forceinline__ void x_combine(const XArgs &a, int t, int rg, int lane) {
  if (__ldg(a.ids + (size_t)t * a.k) < 0) return;  // an out-of-range hash token adds nothing
  const int r = 32 * rg + lane;
  float acc = 0.0f;
  for (int j = 0; j < a.k; j++)
    acc = __fadd_rn(acc, __fmul_rn(__ldg(a.w + (size_t)t * a.k + j),
                                   __ldcg(a.apart + ((size_t)t * a.NS + j) * a.H + r)));
  if (a.n_shared) acc = __fadd_rn(acc, __ldcg(a.apart + ((size_t)t * a.NS + a.k) * a.H + r));
  float *yp = a.y + (size_t)t * a.H + r;
  *yp = __fadd_rn(*yp, acc);
}

// Shared-memory layout (bytes) for TT, staged activations of `act_bytes`.
struct XSmem {
  int ring, bars, ctrl, part, bkt, act, total;
};

__host__ __device__ inline XSmem x_smem(int TT, int mats, int nbk, int act_bytes) {
  XSmem s;
  s.ring = 0;
  s.bars = XC * X_NST * X_STRIDE;
  s.ctrl = s.bars + XC * X_NST * 8;
  s.part = s.ctrl + 256;  // bucket barrier, then full[8] and empty[8] slot barriers
  s.bkt = s.part + x_slots(TT) * XC * mats * TT * TILE_ROWS * 4;
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

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// early: gate/up with staged activations quantised here; the bucket comes
// later (epilogue warp 0 waits for the router kernel). Otherwise every
// thread waits for the previous kernel first.
template <int TT, bool AS, bool EARLY>
__global__ void __launch_bounds__(X_WARPS * 32, 1) k_experts(XArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int PS = x_slots(TT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mats = a.down ? 1 : 2;
  const int nbk = bucket_table_ints(a.A_cap, a.T, a.NS);
  const int act_rows = a.down ? a.T * a.NS : a.T;
  const int act_bytes = AS ? act_rows * (a.K + (a.K >> 5) * 4 + (a.K >> 4) * 2) : 0;
  const XSmem L = x_smem(TT, mats, nbk, act_bytes);
  const uint32_t bkt_bar = smem_u32(smem + L.ctrl);
  const uint32_t full0 = bkt_bar + 64, empty0 = bkt_bar + 128;  // slot barriers, 8 bytes apart
  float *part = (float *)(smem + L.part);  // [PS][XC][mats][TT][16]
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
  const uint32_t ring = smem_u32(smem + L.ring + warp * X_NST * X_STRIDE);
  const uint32_t bar = smem_u32(smem + L.bars + warp * X_NST * 8);
  if (threadIdx.x == 0) {
    mbar_init(bkt_bar, 1);
    for (int i = 0; i < PS; i++) mbar_init(full0 + 8 * i, XC), mbar_init(empty0 + 8 * i, 1);
  }
  if (warp < XC && lane == 0)
    for (int i = 0; i < X_NST; i++) mbar_init(bar + 8 * i, 1);
  if (lane == 0) fence_mbar_init();
  const int nsh = a.n_shared ? a.rows / TILE_ROWS : 0, RG = a.rows / TILE_ROWS;
  const int G = gridDim.x;
  const XKind ks = x_kind(a, a.sf, warp < XC ? warp : 0), kr = x_kind(a, a.rf, warp < XC ? warp : 0);
  int n_routed = -1;  // active routed experts, once the bucket is known
  bool failed = false;
  __syncthreads();  // barriers initialised

  // ---- compute warps: producer cursor; request shared-expert stages now
  XCursor P;
  P.i = blockIdx.x, P.routed = 0, P.unit = 0;
  bool p_ok = false, p_done = false;
  uint32_t g_prod = 0, g_cons = 0;
  // Next (item, pass, stage) of this warp after the current one.
  auto p_advance = [&](const XKind &k) {
    if (++P.stage < k.nst) return;
    P.stage = 0, P.unit++;
    if (++P.pass < P.npass) return;
    x_next_item(&P, G, RG);
    p_ok = false;
  };
  // Fill the ring; stops early when the next item needs the bucket.
  auto fill = [&]() {
    while (!p_done && g_prod - g_cons < X_NST) {
      if (!p_ok) {
        if (P.i >= nsh && n_routed < 0) {
          if (!mbar_test(bkt_bar, 0)) return;
          n_routed = bks[0] - a.n_shared;
        }
        if (!x_item_at<TT>(a, &P, nsh, RG, act, n_routed, ks, kr)) {
          p_done = true;
          return;
        }
        p_ok = true;
        const XKind &k = P.routed ? kr : ks;
        if (k.nst == 0) {  // no segment of this item for this warp
          P.unit += P.npass;
          x_next_item(&P, G, RG);
          p_ok = false;
          continue;
        }
      }
      const XKind &k = P.routed ? kr : ks;
      const uint32_t slot = g_prod % X_NST;
      if (lane == 0) {
        if (g_prod >= X_NST) fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar + 8 * slot, k.sbytes);
        bulk_g2s(ring + slot * X_STRIDE, P.src + (size_t)P.stage * k.sbytes, k.sbytes, bar + 8 * slot);
      }
      g_prod++;
      p_advance(k);
    }
  };
  if (warp < XC) {
    __syncwarp();
    if (EARLY || P.i < nsh) fill();  // (not early: only shared items, which need no bucket)
  }

  // ---- activations (and, unless early, the bucket)
  if (EARLY) {
    // CAS step 1 on x into shared memory (the router kernel publishes the same
    // codes); every warp's loads are issued before any of its blocks is done
    int8_t *xq_s = (int8_t *)(smem + L.act);
    float *dx_s = (float *)(smem + L.act + act_rows * a.K);
    int16_t *gs_s = (int16_t *)(smem + L.act + act_rows * a.K + act_rows * (a.K >> 5) * 4);
    const int nb = a.K >> 5, nblk = a.T * nb;
    constexpr int QB = 8;
    for (int p0 = warp; p0 < nblk; p0 += X_WARPS * QB) {
      float v[QB];
#pragma unroll
      for (int j = 0; j < QB; j++) {
        const int p = p0 + j * X_WARPS;
        v[j] = p < nblk ? __ldg(a.x + (size_t)(p / nb) * a.K + 32 * (p % nb) + lane) : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < QB; j++) {
        const int p = p0 + j * X_WARPS;
        if (p < nblk) {
          const int t = p / nb, b = p % nb;
          const float d = __fdiv_rn(warp_max(fabsf(v[j])), 127.0f);
          const int q = cas_code(v[j], d);
          const int gsum = half_warp_sum(q);
          xq_s[(size_t)t * a.K + 32 * b + lane] = (int8_t)q;
          if (lane == 0) dx_s[(size_t)t * nb + b] = d;
          if ((lane & 15) == 0) gs_s[(size_t)t * (a.K >> 4) + 2 * b + (lane >> 4)] = (int16_t)gsum;
        }
      }
    }
    __syncthreads();
    if (warp == XC) {  // epilogue warp 0: the bucket, once the router kernel is done
      pdl_wait();
      for (int i = lane; i < nbk; i += 32) bks[i] = __ldcg(a.bucket + i);
      __syncwarp();
      if (lane == 0) mbar_arrive(bkt_bar);
    }
  } else {
    pdl_wait();
    for (int i = threadIdx.x; i < nbk; i += blockDim.x) bks[i] = __ldcg(a.bucket + i);
    if (AS) {
      uint8_t *dst = smem + L.act;
      const size_t nq = (size_t)act_rows * a.K, nd = (size_t)act_rows * (a.K >> 5) * 4,
                   ng = (size_t)act_rows * (a.K >> 4) * 2;
      for (size_t i = threadIdx.x; i < nq / 16; i += blockDim.x) ((uint4 *)dst)[i] = __ldcg((const uint4 *)a.aq + i);
      for (size_t i = threadIdx.x; i < nd / 16; i += blockDim.x)
        ((uint4 *)(dst + nq))[i] = __ldcg((const uint4 *)a.ad + i);
      for (size_t i = threadIdx.x; i < ng / 16; i += blockDim.x)
        ((uint4 *)(dst + nq + nd))[i] = __ldcg((const uint4 *)a.ag + i);
    }
    __syncthreads();
    n_routed = bks[0] - a.n_shared;
  }

  if (warp < XC) {
    // ================= compute warp: segment `warp` of every unit
    XCursor C;
    C.i = blockIdx.x, C.routed = 0, C.unit = 0;
    bool c_ok = false;
    int arow[TT], nt = 0;
    float acc[2][TT];
    for (;;) {
      if (!c_ok) {  // the consumer's next item
        if (C.i >= nsh && n_routed < 0) {
          if (!mbar_wait_bounded(bkt_bar, 0)) {
            failed = true;
            break;
          }
          n_routed = bks[0] - a.n_shared;
        }
        if (!x_item_at<TT>(a, &C, nsh, RG, act, n_routed, ks, kr)) break;
        c_ok = true;
      }
      const XKind &k = C.routed ? kr : ks;
      if (C.stage == 0) {  // a new unit: its tokens
        nt = min(TT, C.n_tok - C.pass * TT);
#pragma unroll
        for (int i = 0; i < TT; i++) {
          int sr;
          x_token(a, C, list, min(C.pass * TT + i, C.n_tok - 1), &sr, &arow[i]);
          acc[0][i] = 0.0f, acc[1][i] = 0.0f;
        }
      }
      if (k.nst > 0) {
        fill();
        const uint32_t slot = g_cons % X_NST;
        if (!mbar_wait_bounded(bar + 8 * slot, (g_cons / X_NST) & 1)) {
          failed = true;
          break;
        }
        __syncwarp();
        const uint32_t st = ring + slot * X_STRIDE;
        const int s0 = k.ks0 + C.stage * k.ksps;
        for (int j = 0; j < k.ksps; j++) {
          const uint32_t t = st + j * k.kb;
          if (k.fmt == DS4MOE_Q2S) {
            if (a.down) q2s_step<TT, 1, AS>(t, lane, s0 + j, a.K, arow, aq, ad, ag, *(float(*)[1][TT])acc);
            else q2s_step<TT, 2, AS>(t, lane, s0 + j, a.K, arow, aq, ad, ag, acc);
          } else {
            if (a.down) q8_step<TT, 1, AS>(t, lane, s0 + j, a.K, arow, aq, ad, *(float(*)[1][TT])acc);
            else q8_step<TT, 2, AS>(t, lane, s0 + j, a.K, arow, aq, ad, acc);
          }
        }
        __syncwarp();
        g_cons++;
      }
      if (k.nst == 0 || C.stage == k.nst - 1) {
        // the unit's segment is done: partial sums into slot unit % PS
        const int ps = C.unit % PS, ph = C.unit / PS;
        if (ph > 0 && !mbar_wait_bounded(empty0 + 8 * ps, (ph - 1) & 1)) {
          failed = true;
          break;
        }
        if (k.nst > 0 && (lane & 1) == 0) {
          float *dst = part + (size_t)(ps * XC + warp) * mats * TT * TILE_ROWS;
#pragma unroll
          for (int i = 0; i < TT; i++) {
            if (i < nt) {
              dst[i * TILE_ROWS + (lane >> 1)] = acc[0][i];
              if (!a.down) dst[(TT + i) * TILE_ROWS + (lane >> 1)] = acc[1][i];
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(full0 + 8 * ps);
        C.stage = 0, C.unit++;
        if (++C.pass == C.npass) x_next_item(&C, G, RG), c_ok = false;
      } else {
        C.stage++;
      }
    }
    if (failed) {
      if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
      for (uint32_t g = g_cons; g < g_prod; g++) (void)mbar_wait_bounded(bar + 8 * (g % X_NST), (g / X_NST) & 1);
    }
    return;
  }

  // ================= epilogue warps: units u with u % XE == ew
  const int ew = warp - XC;
  XCursor E;
  E.i = blockIdx.x, E.routed = 0, E.unit = 0;
  for (;;) {
    if (E.i >= nsh && n_routed < 0) {  // routed units need the bucket
      if (!mbar_wait_bounded(bkt_bar, 0)) {
        if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
        return;
      }
      n_routed = bks[0] - a.n_shared;
    }
    if (!x_item_at<TT>(a, &E, nsh, RG, act, n_routed, ks, kr)) break;
    const int S = E.routed ? kr.S : ks.S;
    for (; E.pass < E.npass; E.pass++, E.unit++) {
      if (E.unit % XE != ew) continue;
      const int ps = E.unit % PS;
      if (!mbar_wait_bounded(full0 + 8 * ps, (E.unit / PS) & 1)) {
        if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
        return;
      }
      const int nt = min(TT, E.n_tok - E.pass * TT);
      const float *src = part + (size_t)ps * XC * mats * TT * TILE_ROWS;
      const int r = lane & 15;
      for (int i0 = 0; i0 < nt; i0 += 2) {
        const int i = i0 + (lane >> 4);
        if (i < nt) {
          float g = 0.0f, uu = 0.0f;  // segment sums in order (CAS step 4)
          for (int sg = 0; sg < S; sg++) {
            const float *p = src + (size_t)sg * mats * TT * TILE_ROWS;
            g = __fadd_rn(g, p[i * TILE_ROWS + r]);
            if (!a.down) uu = __fadd_rn(uu, p[(TT + i) * TILE_ROWS + r]);
          }
          int sr, arow;
          x_token(a, E, list, E.pass * TT + i, &sr, &arow);
          if (!a.down) a.hbuf[(size_t)sr * a.F + TILE_ROWS * E.rg + r] = __fmul_rn(cas_silu(g), uu);
          else a.apart[(size_t)sr * a.H + TILE_ROWS * E.rg + r] = g;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * ps);  // the slot is free again
      // completion of 32-row blocks across the two items that cover them
      const int blk = E.rg >> 1;
      for (int i = 0; i < nt; i++) {
        int sr, arow;
        x_token(a, E, list, E.pass * TT + i, &sr, &arow);
        if (!a.down) {
          if (x_ticket_last(a.hticket + (size_t)sr * (a.F >> 5) + blk, 2, lane))
            x_requant(a, __ldcg(a.hbuf + (size_t)sr * a.F + 32 * blk + lane), sr, blk, lane);
        } else {
          const int t = sr / a.NS;
          int expect = 0;
          if (lane == 0) {
            for (int jj = 0; jj < a.k; jj++) expect += __ldg(a.ids + (size_t)t * a.k + jj) >= 0;
            expect = 2 * (expect + a.n_shared);
          }
          expect = __shfl_sync(0xffffffffu, expect, 0);
          if (x_ticket_last(a.cticket + (size_t)t * (a.H >> 5) + blk, expect, lane)) x_combine(a, t, blk, lane);
        }
      }
    }
    x_next_item(&E, G, RG);
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

static int x_tt(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }

static size_t x_smem_bytes(const ds4moe_layer *h, int T, bool down, bool as) {
  const int nbk = bucket_table_ints(h->A_max, T, h->NS);
  return (size_t)x_smem(x_tt(T), down ? 1 : 2, nbk, as ? (int)x_act_bytes(h, T, down) : 0).total;
}

size_t experts_smem(const ds4moe_layer *h) {
  // both kernels must fit at DEC_MAX_T with activations in global memory
  const size_t a = x_smem_bytes(h, DEC_MAX_T, false, false), b = x_smem_bytes(h, DEC_MAX_T, true, false);
  return a > b ? a : b;
}

template <bool AS, bool EARLY>
static const void *x_fn(int T) {
  return T <= 1 ? (const void *)k_experts<1, AS, EARLY>
       : T <= 2 ? (const void *)k_experts<2, AS, EARLY>
       : T <= 4 ? (const void *)k_experts<4, AS, EARLY> : (const void *)k_experts<8, AS, EARLY>;
}

cudaError_t launch_experts(const ds4moe_layer *h, const float *x, int T, float *y, int down, cudaStream_t s) {
  const ds4moe_layer_desc &d = h->d;
  XArgs a = {};
  a.H = d.hidden, a.F = d.ffn, a.E = d.n_experts, a.k = d.top_k, a.NS = h->NS, a.n_shared = d.n_shared, a.T = T;
  a.A_cap = h->A_max, a.rf = d.routed_fmt, a.sf = d.n_shared ? d.shared_fmt : d.routed_fmt, a.down = down;
  a.bucket = h->bucket, a.ids = h->ids, a.w = h->wts;
  a.hq = h->hq, a.dh = h->dh, a.gsh = h->gsh, a.hbuf = h->hbuf, a.hticket = h->hticket;
  a.apart = h->apart, a.cticket = h->cticket, a.y = y, a.err = h->err, a.x = x;
  if (!down) {
    a.K = d.hidden, a.rows = d.ffn, a.w_r = h->gu, a.w_s = h->sgu, a.aq = h->xq, a.ad = h->dx, a.ag = h->gs;
  } else {
    a.K = d.ffn, a.rows = d.hidden, a.w_r = h->dn, a.w_s = h->sdn, a.aq = h->hq, a.ad = h->dh, a.ag = h->gsh;
  }
  const bool as = x_smem_bytes(h, T, down != 0, true) <= DEC_SMEM_LIMIT;
  const void *fn = as ? (down ? x_fn<true, false>(T) : x_fn<true, true>(T)) : x_fn<false, false>(T);
  void *args[] = {&a};
  return launch_pdl(fn, dim3(h->n_sm), dim3(X_WARPS * 32), x_smem_bytes(h, T, down != 0, as), s, args, true);
}

cudaError_t experts_set_attributes() {
  const void *fns[] = {x_fn<true, true>(1),  x_fn<true, true>(2),  x_fn<true, true>(4),  x_fn<true, true>(8),
                       x_fn<true, false>(1), x_fn<true, false>(2), x_fn<true, false>(4), x_fn<true, false>(8),
                       x_fn<false, false>(1), x_fn<false, false>(2), x_fn<false, false>(4), x_fn<false, false>(8)};
  cudaError_t e = cudaSuccess;
  for (const void *f : fns)
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, DEC_SMEM_LIMIT);
  return e;
}

}  // namespace ds4

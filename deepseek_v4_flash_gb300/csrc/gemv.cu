// gemv.cu -- expert gate/up (+ SiLU * up + int8 requant of h) and expert
// down GEMVs for decode-sized batches.
//
// The work item is (active expert, 32-row group). One warp owns an item; its
// lane r owns row r of the group for the whole K range, so every row sum is
// the CAS sequential chain (S = 1) with no cross-lane float reduction. The
// item's weight bytes are one contiguous stream in the RG32 layout; lane 0
// keeps a ring of stages in flight with 1-D bulk async copies
// (cp.async.bulk, completion on an mbarrier), and the warp computes each stage
// from shared memory: 512 contiguous bytes per 16-byte load, no bank
// conflicts. The tokens routed to the expert (up to TT per pass) reuse each
// unpacked weight word from registers.
//
// Prior art: the decode kernels of the ds4-rocm fork README ("Performance
// optimizations": moe_gate_up_mid_decode_lut_qwarp32 produces the SwiGLU
// "mid" from the routed gate/up, moe_down_sum6_qwarp32 the down projection;
// wide 128-bit weight loads in the q8_0/IQ2 inner loops). Those were tuned
// for a 40-CU RDNA iGPU; here the layout, the bulk-copy ring and the
// lane-per-row split are chosen for sm_103a.
#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"

namespace ds4 {

struct GemvArgs {
  int H, F, E, NS;
  const uint8_t *w;       // routed weights (gu or dn)
  const uint8_t *w_sh;    // shared weights (sgu or sdn)
  const int8_t *aq;       // activation codes: xq [T][H] (gate/up) or hq [T*NS][F] (down)
  const float *ad;        // activation scales
  const int16_t *ag;      // activation 16-group sums
  const int32_t *cnt, *off, *active, *n_active, *list;
  int8_t *hq;             // gate/up outputs
  float *dh;
  int16_t *gsh;
  float *apart;           // down output
  uint32_t *err;
};

template <int FMT, int TT>
__device__ __forceinline__ void tile_step(uint32_t tile, int lane, int s, int K, const int *tok,
                                          const GemvArgs &a, float *acc) {
  if (FMT == DS4MOE_Q2S)
    q2s_tile<TT>(tile, lane, s, K, tok, a.aq, a.ad, a.ag, acc);
  else
    q8_tile<TT>(tile, lane, s, K, tok, a.aq, a.ad, acc);
}

// Ring of NST stages of STRIDE bytes in dynamic shared memory, NST
// mbarriers after them. Lane 0 arms; all lanes wait.
template <int NST, int STRIDE>
struct Ring {
  uint32_t buf, bar;
  __device__ __forceinline__ void init(uint8_t *smem, int lane) {
    buf = smem_u32(smem);
    bar = buf + NST * STRIDE;
    if (lane == 0) {
      for (int i = 0; i < NST; i++) mbar_init(bar + 8 * i, 1);
      fence_mbar_init();
    }
    __syncwarp();
  }
  __device__ __forceinline__ void arm(uint32_t g, const uint8_t *src, uint32_t bytes) const {
    const uint32_t slot = g % NST;
    mbar_arrive_expect_tx(bar + 8 * slot, bytes);
    bulk_g2s(buf + slot * STRIDE, src, bytes, bar + 8 * slot);
  }
  __device__ __forceinline__ bool wait(uint32_t g) const {
    return mbar_wait_bounded(bar + 8 * (g % NST), (g / NST) & 1);
  }
  __device__ __forceinline__ uint32_t stage(uint32_t g) const { return buf + (g % NST) * STRIDE; }
  // After a timeout: wait (bounded) for every copy still in flight.
  __device__ __forceinline__ void drain(uint32_t g_next, uint32_t g_armed_end) const {
    for (uint32_t g = g_next; g < g_armed_end; g++) (void)wait(g);
  }
};

// Stream `nsteps` stages of `bytes` from `src` through the ring, calling
// body(stage_addr, s) for each. Returns false after a wait timeout.
template <int NST, int STRIDE, typename Body>
__device__ __forceinline__ bool stream_item(const Ring<NST, STRIDE> &ring, uint32_t &g, const uint8_t *src,
                                            int nsteps, uint32_t bytes, int lane, Body body) {
  const int pre = nsteps < NST ? nsteps : NST;
  if (lane == 0)
    for (int i = 0; i < pre; i++) ring.arm(g + i, src + (size_t)i * bytes, bytes);
  for (int s = 0; s < nsteps; s++) {
    if (!ring.wait(g + s)) {
      const int armed = (s + NST < nsteps) ? s + NST : nsteps;
      ring.drain(g + s, g + armed);
      g += nsteps;
      return false;
    }
    body(ring.stage(g + s), s);
    __syncwarp();
    if (lane == 0 && s + NST < nsteps) {
      fence_proxy_async_smem();
      ring.arm(g + s + NST, src + (size_t)(s + NST) * bytes, bytes);
    }
  }
  g += nsteps;
  return true;
}

constexpr int NST_GU = 4, STRIDE_GU = MAX_STAGE;
constexpr int NST_DN = 8, STRIDE_DN = MAX_STAGE / 2;

// Row sums in `segs` equal K segments (CAS step 4): the segment chain runs in
// acc[]; at each segment end it is added into tot[] and restarts at zero.
template <int TT>
__device__ __forceinline__ void fold_segment(int s, int seg_steps, float *acc, float *tot) {
  if ((s + 1) % seg_steps == 0) {
#pragma unroll
    for (int i = 0; i < TT; i++) tot[i] = __fadd_rn(tot[i], acc[i]), acc[i] = 0.0f;
  }
}

template <int FMT, int TT>
__device__ void gateup_item(const GemvArgs &a, const uint8_t *src, int rg, int n_e, const int32_t *lst, int segs,
                            Ring<NST_GU, STRIDE_GU> &ring, uint32_t &g, int lane) {
  const int H = a.H, F = a.F, NS = a.NS;
  const int KS = H / kstep(FMT), TB = tile_bytes(FMT), seg_steps = KS / segs;
  for (int t0 = 0; t0 < n_e; t0 += TT) {
    int tok[TT];
#pragma unroll
    for (int i = 0; i < TT; i++) tok[i] = lst[min(t0 + i, n_e - 1)] / NS;
    float acg[TT], acu[TT], tg[TT], tu[TT];
#pragma unroll
    for (int i = 0; i < TT; i++) acg[i] = 0.0f, acu[i] = 0.0f, tg[i] = 0.0f, tu[i] = 0.0f;
    const bool ok = stream_item(ring, g, src, KS, 2 * TB, lane, [&](uint32_t st, int s) {
      tile_step<FMT, TT>(st, lane, s, H, tok, a, acg);
      tile_step<FMT, TT>(st + TB, lane, s, H, tok, a, acu);
      fold_segment<TT>(s, seg_steps, acg, tg);
      fold_segment<TT>(s, seg_steps, acu, tu);
    });
    if (!ok) {
      if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
      return;
    }
    // h = silu(g) * u, then CAS step 1 over the 32 rows of this group
    // (= one 32-block of h).
#pragma unroll
    for (int i = 0; i < TT; i++) {
      if (t0 + i >= n_e) break;
      const int sr = lst[t0 + i];
      const float h = __fmul_rn(cas_silu(tg[i]), tu[i]);
      const float amax = warp_max(fabsf(h));
      const float d = __fdiv_rn(amax, 127.0f);
      const int q = cas_code(h, d);
      const int gsum = half_warp_sum(q);
      a.hq[(size_t)sr * F + 32 * rg + lane] = (int8_t)q;
      if (lane == 0) a.dh[(size_t)sr * (F >> 5) + rg] = d;
      if ((lane & 15) == 0) a.gsh[(size_t)sr * (F >> 4) + 2 * rg + (lane >> 4)] = (int16_t)gsum;
    }
  }
}

template <int FMT, int TT>
__device__ void down_item(const GemvArgs &a, const uint8_t *src, int rg, int n_e, const int32_t *lst, int segs,
                          Ring<NST_DN, STRIDE_DN> &ring, uint32_t &g, int lane) {
  const int H = a.H, F = a.F;
  const int KS = F / kstep(FMT), TB = tile_bytes(FMT), seg_steps = KS / segs;
  for (int t0 = 0; t0 < n_e; t0 += TT) {
    int sr[TT];
#pragma unroll
    for (int i = 0; i < TT; i++) sr[i] = lst[min(t0 + i, n_e - 1)];
    float acc[TT], tot[TT];
#pragma unroll
    for (int i = 0; i < TT; i++) acc[i] = 0.0f, tot[i] = 0.0f;
    const bool ok = stream_item(ring, g, src, KS, TB, lane, [&](uint32_t st, int s) {
      tile_step<FMT, TT>(st, lane, s, F, sr, a, acc);
      fold_segment<TT>(s, seg_steps, acc, tot);
    });
    if (!ok) {
      if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
      return;
    }
#pragma unroll
    for (int i = 0; i < TT; i++) {
      if (t0 + i >= n_e) break;
      a.apart[(size_t)sr[i] * H + 32 * rg + lane] = tot[i];
    }
  }
}

template <int TT, int RFMT, int SFMT>
__global__ void __launch_bounds__(32) k_gateup(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int rg = blockIdx.x, ai = blockIdx.y, lane = threadIdx.x;
  if (ai >= *a.n_active) return;
  const int e = a.active[ai];
  const int n_e = a.cnt[e];
  if (n_e == 0) return;
  const int32_t *lst = a.list + a.off[e];
  Ring<NST_GU, STRIDE_GU> ring;
  ring.init(smem, lane);
  uint32_t g = 0;
  const int RG = a.F >> 5;
  if (e == a.E) {
    const size_t item = (size_t)(a.H / kstep(SFMT)) * 2 * tile_bytes(SFMT);
    gateup_item<SFMT, TT>(a, a.w_sh + rg * item, rg, n_e, lst, SHARED_SEGS, ring, g, lane);
  } else {
    const size_t item = (size_t)(a.H / kstep(RFMT)) * 2 * tile_bytes(RFMT);
    gateup_item<RFMT, TT>(a, a.w + ((size_t)e * RG + rg) * item, rg, n_e, lst, 1, ring, g, lane);
  }
}

template <int TT, int RFMT, int SFMT>
__global__ void __launch_bounds__(32) k_down(GemvArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int rg = blockIdx.x, ai = blockIdx.y, lane = threadIdx.x;
  if (ai >= *a.n_active) return;
  const int e = a.active[ai];
  const int n_e = a.cnt[e];
  if (n_e == 0) return;
  const int32_t *lst = a.list + a.off[e];
  Ring<NST_DN, STRIDE_DN> ring;
  ring.init(smem, lane);
  uint32_t g = 0;
  const int RG = a.H >> 5;
  if (e == a.E) {
    const size_t item = (size_t)(a.F / kstep(SFMT)) * tile_bytes(SFMT);
    down_item<SFMT, TT>(a, a.w_sh + rg * item, rg, n_e, lst, SHARED_SEGS, ring, g, lane);
  } else {
    const size_t item = (size_t)(a.F / kstep(RFMT)) * tile_bytes(RFMT);
    down_item<RFMT, TT>(a, a.w + ((size_t)e * RG + rg) * item, rg, n_e, lst, 1, ring, g, lane);
  }
}

static GemvArgs base_args(const ds4moe_layer *h) {
  GemvArgs a;
  a.H = h->d.hidden, a.F = h->d.ffn, a.E = h->d.n_experts, a.NS = h->NS;
  Bucket b = bucket_view(h);
  a.cnt = b.cnt, a.off = b.off, a.active = b.active, a.n_active = b.n_active, a.list = b.list;
  a.hq = h->hq, a.dh = h->dh, a.gsh = h->gsh, a.apart = h->apart, a.err = h->err;
  return a;
}

static int pick_tt(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }

#define DS4_GEMV_DISPATCH(KERNEL, TT, R, S)                                                  \
  do {                                                                                     \
    if (r == R && sh == S) {                                                               \
      KERNEL<TT, R, S><<<grid, 32, smem, st>>>(a);                                         \
      return cudaGetLastError();                                                           \
    }                                                                                      \
  } while (0)

#define DS4_GEMV_ALL(KERNEL, TT)                                  \
  DS4_GEMV_DISPATCH(KERNEL, TT, DS4MOE_Q2S, DS4MOE_Q8_0);          \
  DS4_GEMV_DISPATCH(KERNEL, TT, DS4MOE_Q8_0, DS4MOE_Q8_0);         \
  DS4_GEMV_DISPATCH(KERNEL, TT, DS4MOE_Q2S, DS4MOE_Q2S);           \
  DS4_GEMV_DISPATCH(KERNEL, TT, DS4MOE_Q8_0, DS4MOE_Q2S)

static int active_max(const ds4moe_layer *h, int T) {
  const long long routed = (long long)T * h->d.top_k;
  return (int)(routed < h->d.n_experts ? routed : h->d.n_experts) + h->d.n_shared;
}

cudaError_t launch_gateup(const ds4moe_layer *h, int T, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  GemvArgs a = base_args(h);
  a.w = h->gu, a.w_sh = h->sgu, a.aq = h->xq, a.ad = h->dx, a.ag = h->gs;
  const int r = h->d.routed_fmt, sh = h->d.n_shared ? h->d.shared_fmt : h->d.routed_fmt;
  const dim3 grid(h->d.ffn / 32, active_max(h, T));
  const int smem = NST_GU * STRIDE_GU + 8 * NST_GU;
  switch (pick_tt(T)) {
    case 1: DS4_GEMV_ALL(k_gateup, 1); break;
    case 2: DS4_GEMV_ALL(k_gateup, 2); break;
    case 4: DS4_GEMV_ALL(k_gateup, 4); break;
    default: DS4_GEMV_ALL(k_gateup, 8); break;
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_down(const ds4moe_layer *h, int T, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  GemvArgs a = base_args(h);
  a.w = h->dn, a.w_sh = h->sdn, a.aq = h->hq, a.ad = h->dh, a.ag = h->gsh;
  const int r = h->d.routed_fmt, sh = h->d.n_shared ? h->d.shared_fmt : h->d.routed_fmt;
  const dim3 grid(h->d.hidden / 32, active_max(h, T));
  const int smem = NST_DN * STRIDE_DN + 8 * NST_DN;
  switch (pick_tt(T)) {
    case 1: DS4_GEMV_ALL(k_down, 1); break;
    case 2: DS4_GEMV_ALL(k_down, 2); break;
    case 4: DS4_GEMV_ALL(k_down, 4); break;
    default: DS4_GEMV_ALL(k_down, 8); break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace ds4

// dense.cu -- y = W x for a dense Q8_0 matrix beside the MoE (the output head,
// the attention projections) at decode-sized token counts.
//
// Two kernels, chained with programmatic dependent launch:
//   k_dense_quant  CAS step 1 on x: one warp per 32-block of a token;
//   k_dense<TT>    persistent, one block per SM: each warp owns whole items of
//                  32 output rows (two 16-row tiles per K step, the layout of
//                  an expert's down matrix) and streams an item's tiles through
//                  its own ring of 1-D bulk copies. The warp keeps a row's CAS
//                  segment chain and adds each finished segment to the row sum
//                  in order (CAS step 4, S = min(8, K/32) as for an expert row),
//                  so no other warp takes part in a row. The tokens' codes are
//                  staged in shared memory once per pass of up to TT tokens.
// Rows are independent, so nothing waits on another block: the weight stream
// is bounded only by the rings' bytes in flight.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "common.cuh"
#include "internal.h"
#include "tiles.cuh"

struct ds4moe_dense {
  int N, K, N_pad, max_tokens, device, n_sm;
  uint8_t *w;        // [N_pad/32][K/32][2][Q8 tile]
  int8_t *xq;        // [max_tokens][K]
  float *dx;         // [max_tokens][K/32]
  uint32_t *err;     // device error flags
  uint64_t bytes, launches;
};

namespace ds4 {

constexpr int DN_WARPS = 8;              // warps per block, each owning whole items
constexpr int DN_KB = 2 * Q8_TILE;       // one K step of an item: two 16-row tiles
constexpr int DN_MAX_KS = 4;             // K steps per ring stage, at most
constexpr size_t DN_SMEM_LIMIT = 227 * 1024;

// K steps per ring stage: the largest divisor of a segment's blocks up to 4,
// so that no stage straddles two segments.
__host__ __device__ inline int dn_ks(int K) {
  const int nb = K / 32, S = expert_segs(DS4MOE_Q8_0, K), per = nb / S;
  int ks = per < DN_MAX_KS ? per : DN_MAX_KS;
  while (ks > 1 && per % ks) ks--;
  return ks;
}

struct DnArgs {
  int N, K, T, nst;   // nst: ring stages per warp
  const uint8_t *w;
  const int8_t *xq;
  const float *dx;
  float *y;
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

template <int TT>
__global__ void __launch_bounds__(DN_WARPS * 32, 1) k_dense(DnArgs a) {
  constexpr bool PACK = TT > 1;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = a.K >> 5, S = expert_segs(DS4MOE_Q8_0, a.K), per = nb / S, ks = dn_ks(a.K);
  const int sbytes = ks * DN_KB, nstage = nb / ks;
  const int n_items = (a.N + 31) >> 5, wstride = gridDim.x * DN_WARPS;
  const int first = blockIdx.x * DN_WARPS + warp;
  const int my_items = first < n_items ? (n_items - 1 - first) / wstride + 1 : 0;
  const int n_pass = (a.T + TT - 1) / TT;
  // shared memory: the pass's codes [TT][K], scales [TT][K/32], then the rings
  int8_t *xs = (int8_t *)smem;
  float *ds = (float *)(smem + TT * a.K);
  const int ring_off = (TT * a.K + TT * (a.K >> 5) * 4 + 127) & ~127;
  const uint32_t ring = smem_u32(smem + ring_off + warp * a.nst * sbytes);
  __shared__ uint64_t bars[DN_WARPS][8];
  const uint32_t bar = smem_u32(&bars[warp][0]);
  if (lane == 0) {
    for (int i = 0; i < a.nst; i++) mbar_init(bar + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const size_t item_bytes = (size_t)nb * DN_KB;
  // producer cursor over (pass, item, stage) of this warp
  int pp = 0, pi = 0, pst = 0;
  uint32_t g_prod = 0, g_cons = 0;
  auto fill = [&]() {
    while (pp < n_pass && g_prod - g_cons < (uint32_t)a.nst) {
      if (pi >= my_items) {
        pp++, pi = 0, pst = 0;
        continue;
      }
      const uint32_t slot = g_prod % a.nst;
      if (lane == 0) {
        if (g_prod >= (uint32_t)a.nst) fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar + 8 * slot, sbytes);
        bulk_g2s(ring + slot * sbytes, a.w + (size_t)(first + pi * wstride) * item_bytes + (size_t)pst * sbytes,
                 sbytes, bar + 8 * slot);
      }
      g_prod++;
      if (++pst == nstage) pst = 0, pi++;
    }
  };
  fill();  // constant weights, before the codes of x exist
  pdl_launch_dependents();
  pdl_wait();
  bool failed = false;
  for (int p = 0; p < n_pass; p++) {
    const int t0 = p * TT, nt = min(TT, a.T - t0);
    __syncthreads();  // the previous pass is done with the staged codes
    {
      const int nq = nt * a.K / 16, nd = nt * (a.K >> 5);
      const uint4 *src = (const uint4 *)(a.xq + (size_t)t0 * a.K);
      for (int i = threadIdx.x; i < nq; i += blockDim.x) ((uint4 *)xs)[i] = __ldg(src + i);
      for (int i = threadIdx.x; i < nd; i += blockDim.x) ds[i] = __ldg(a.dx + (size_t)t0 * (a.K >> 5) + i);
    }
    __syncthreads();
    int arow[TT];
#pragma unroll
    for (int i = 0; i < TT; i++) arow[i] = i;
    // a warp that gave up a wait skips its items but still meets every pass
    // barrier of its block
    for (int it = 0; it < my_items && !failed; it++) {
      Chains<PACK> acc[TT], tot[TT];
#pragma unroll
      for (int i = 0; i < TT; i++) chains_zero(acc[i]), chains_zero(tot[i]);
      for (int st = 0; st < nstage; st++) {
        fill();
        const uint32_t slot = g_cons % a.nst;
        if (!mbar_wait_bounded(bar + 8 * slot, (g_cons / a.nst) & 1)) {
          failed = true;
          break;
        }
        __syncwarp();
        const uint32_t tile = ring + slot * sbytes;
        for (int j = 0; j < ks; j++) {
          const int s = st * ks + j;
          q8_step<TT, true, PACK>(tile + j * DN_KB, lane, s, a.K, arow, nt, xs, ds, acc);
          if ((s + 1) % per == 0) {  // a segment is complete: into the row sum, in order
#pragma unroll
            for (int i = 0; i < TT; i++) {
              if constexpr (PACK) tot[i].v = f2_add(tot[i].v, acc[i].v);
              else tot[i].c[0] = __fadd_rn(tot[i].c[0], acc[i].c[0]), tot[i].c[1] = __fadd_rn(tot[i].c[1], acc[i].c[1]);
              chains_zero(acc[i]);
            }
          }
        }
        __syncwarp();
        g_cons++;
      }
      if (failed) break;
      // lanes 2r hold rows r (tile 0) and 16 + r (tile 1) of the item
      if ((lane & 1) == 0) {
        const int r0 = 32 * (first + it * wstride) + (lane >> 1);
#pragma unroll
        for (int i = 0; i < TT; i++) {
          if (i < nt) {
            float v0, v1;
            chains_get(tot[i], v0, v1);
            if (r0 < a.N) a.y[(size_t)(t0 + i) * a.N + r0] = v0;
            if (r0 + 16 < a.N) a.y[(size_t)(t0 + i) * a.N + r0 + 16] = v1;
          }
        }
      }
    }
  }
  if (failed) {
    if (lane == 0) raise_flag(a.err, DS4MOE_DEVERR_TIMEOUT);
    // the warp's own copies in flight land before the block may leave
    for (uint32_t g = g_cons; g < g_prod; g++) (void)mbar_wait_bounded(bar + 8 * (g % a.nst), (g / a.nst) & 1);
  }
}

// Tokens per pass for K: the codes of a pass take at most 64 KB.
static int dn_tt(int K) {
  const size_t per_tok = (size_t)K + (size_t)(K / 32) * 4;
  return per_tok * 8 <= 65536 ? 8 : per_tok * 4 <= 65536 ? 4 : per_tok * 2 <= 65536 ? 2 : 1;
}

static size_t dn_stage_smem(int TT, int K) {
  return ((size_t)TT * K + (size_t)TT * (K / 32) * 4 + 127) & ~(size_t)127;
}

static int dn_nst(int TT, int K) {
  const size_t left = DN_SMEM_LIMIT - 1024 - dn_stage_smem(TT, K);  // 1 KB: the static barriers
  const size_t per_stage = (size_t)DN_WARPS * dn_ks(K) * DN_KB;
  const size_t n = left / per_stage;
  return n > 6 ? 6 : (int)n;
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
  if (h->err) cudaFree(h->err);
}

template <int TT>
cudaError_t dn_launch(ds4moe_dense *h, const DnArgs &a0, cudaStream_t s) {
  DnArgs a = a0;
  a.nst = dn_nst(TT, h->K);
  void *args[] = {&a};
  const size_t smem = dn_stage_smem(TT, h->K) + (size_t)DN_WARPS * a.nst * dn_ks(h->K) * DN_KB;
  return launch_pdl((const void *)k_dense<TT>, dim3(h->n_sm), dim3(DN_WARPS * 32), smem, s, args, true);
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
  if (dn_nst(dn_tt(n_in), n_in) < 2) return DS4MOE_ERR_UNSUPPORTED;
  ds4moe_dense *h = new (std::nothrow) ds4moe_dense;
  if (!h) return DS4MOE_ERR_OOM;
  memset(h, 0, sizeof(*h));
  h->N = n_out, h->K = n_in, h->N_pad = (n_out + 31) / 32 * 32, h->max_tokens = max_tokens;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->device);
  const size_t wb = (size_t)h->N_pad / 32 * (n_in / 32) * DN_KB;
  const size_t qb = (size_t)max_tokens * n_in, db = (size_t)max_tokens * (n_in / 32) * 4;
  for (const void *fn : {(const void *)k_dense<1>, (const void *)k_dense<2>, (const void *)k_dense<4>,
                         (const void *)k_dense<8>})
    if (e == cudaSuccess)  // the static barriers take their part of the block's shared memory
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DN_SMEM_LIMIT - 1024);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->w, wb);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->xq, qb);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->dx, db);
  if (e == cudaSuccess) e = cudaMalloc((void **)&h->err, 64);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->w, 0, wb, 0);  // padding rows stay zero
  if (e == cudaSuccess) e = cudaMemsetAsync(h->err, 0, 64, 0);
  if (e == cudaSuccess) e = repack_q8((const uint8_t *)w_q8, h->w, 1, n_out, n_in, 2, 0, 0);
  if (e == cudaSuccess) e = cudaStreamSynchronize(0);
  if (e != cudaSuccess) {
    const ds4moe_status st = dn_status(e);
    cudaDeviceSynchronize();
    cudaGetLastError();
    dn_free(h);
    delete h;
    return st;
  }
  h->bytes = wb + qb + db + 64;
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
    a.N = h->N, a.K = K, a.T = n_tok, a.w = h->w, a.xq = h->xq, a.dx = h->dx, a.y = y, a.err = h->err;
    switch (dn_tt(K)) {
      case 8: e = dn_launch<8>(h, a, s); break;
      case 4: e = dn_launch<4>(h, a, s); break;
      case 2: e = dn_launch<2>(h, a, s); break;
      default: e = dn_launch<1>(h, a, s); break;
    }
  }
  h->launches += 2;
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

uint64_t ds4moe_dense_device_bytes(const ds4moe_dense *h) { return h ? h->bytes : 0; }
uint64_t ds4moe_dense_launch_count(const ds4moe_dense *h) { return h ? h->launches : 0; }

}  // extern "C"

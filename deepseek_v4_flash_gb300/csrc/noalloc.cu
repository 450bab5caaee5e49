// noalloc.cu -- ds4moe_route_noalloc: routing (learned or hash) straight
// from the caller's canonical router buffers, with no layer handle and no
// device allocation. Its scratch -- the router segment sums of every token
// -- lives in one fixed device array of DS4MOE_NOALLOC_SCRATCH_BYTES bytes
// defined in this file.
//
// Two kernels:
//   k_na_router_part : int8 quantisation of each token's 32-blocks in one K
//                      segment (in shared memory) and that segment's sum of
//                      every router row, read from the canonical Q8_0 (or
//                      F32) rows with coalesced loads, written to the array;
//   k_na_route       : one block per token: logits, sigmoid, bias top-k and
//                      renormalisation from the segment sums (route.cuh);
//                      hash routing instead looks the table up.
// The arithmetic is the same binary32 sequence as ds4moe_route's.
#include <mutex>

#include "common.cuh"
#include "route.cuh"

using namespace ds4;

// The scratch of every ds4moe_route_noalloc call on this device:
// [n_tok][ROUTER_SEGS][E_pad] fp32 segment sums. No word of it has to start
// at zero: a call reads only what it wrote earlier in the same call.
static __device__ __align__(256) uint8_t na_scratch[DS4MOE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int NA_RT = 8;      // tokens per token tile of k_na_router_part
constexpr int NA_WARPS = 4;   // warps per block of k_na_router_part (32 router rows)
constexpr int NA_MAX_DEVICES = 64;
constexpr int NA_ROUTE_THREADS = 256;

struct NaArgs {
  const float *x;
  const uint8_t *W;        // router rows, canonical Q8_0 or F32 [E][H]
  const float *bias;       // [E]
  const int32_t *hash;     // [vocab][k]
  const int32_t *tok;      // [T]
  int T, H, E, E_pad, k, vocab, q8;
  float scale;
  float *part;             // na_scratch: [T][ROUTER_SEGS][E_pad]
  int32_t *ids;
  float *w;
  uint32_t *err;           // may be null
};

// grid (ceil(E_pad/32), ROUTER_SEGS, ceil(T / NA_RT)); block x handles
// router rows 32x .. 32x+31 over K segment y for the tokens of tile z, warp w
// the rows 32x + w, 32x + w + NA_WARPS, ... one at a time.
//
// A row's segment is `per` contiguous canonical Q8_0 blocks (34 bytes each,
// 2-byte aligned): the warp reads it with consecutive 16-bit loads into its
// shared-memory buffer (coalesced), then lane j computes the term of block j
// and the terms are added in block order (CAS step 4) by shuffles.
__global__ void __launch_bounds__(NA_WARPS * 32) k_na_router_part(NaArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.y, t0 = blockIdx.z * NA_RT, nt = min(NA_RT, a.T - t0);
  const int nb = a.H >> 5, per = nb / ROUTER_SEGS, b0 = seg * per;
  int8_t *xq_s = (int8_t *)sm;                         // [NA_RT][per * 32]
  float *dx_s = (float *)(sm + NA_RT * per * 32);      // [NA_RT][per]
  uint16_t *row_s = (uint16_t *)(sm + NA_RT * per * 36) + warp * (per * 17);  // this warp's row segment
  // CAS step 1 on the segment's blocks (lane = element); the F32 router uses
  // x unquantised and only needs the finiteness check
  for (int p = warp; p < nt * per; p += NA_WARPS) {
    const int i = p / per, bb = p % per;
    const float v = __ldg(a.x + (size_t)(t0 + i) * a.H + 32 * (b0 + bb) + lane);
    if (__any_sync(0xffffffffu, !isfinite(v)) && lane == 0 && blockIdx.x == 0)
      raise_flag(a.err, DS4MOE_DEVERR_NONFINITE);
    if (a.q8) {
      const float d = __fdiv_rn(warp_max(fabsf(v)), 127.0f);
      xq_s[i * per * 32 + bb * 32 + lane] = (int8_t)cas_code(v, d);
      if (lane == 0) dx_s[i * per + bb] = d;
    }
  }
  __syncthreads();
  for (int rr = warp; rr < 32; rr += NA_WARPS) {
    const int r = blockIdx.x * 32 + rr;
    if (r >= a.E) break;  // warp-uniform
    if (a.q8) {
      const uint16_t *src = (const uint16_t *)(a.W + ((size_t)r * nb + b0) * 34);
      for (int j = lane; j < per * 17; j += 32) row_s[j] = __ldg(src + j);
      __syncwarp();
      for (int i = 0; i < nt; i++) {
        float s = 0.0f;
        for (int c0 = 0; c0 < per; c0 += 32) {  // 32 blocks per round, lane = block
          const int bb = c0 + lane;
          float p = 0.0f;
          if (bb < per) {
            const uint16_t *blk = row_s + 17 * bb;
            const int *xv = (const int *)(xq_s + i * per * 32 + bb * 32);
            int I = 0;
#pragma unroll
            for (int m = 0; m < 8; m++)
              I = __dp4a((int)((uint32_t)blk[1 + 2 * m] | ((uint32_t)blk[2 + 2 * m] << 16)), xv[m], I);
            p = q8_term(half_bits_to_float(blk[0]), dx_s[i * per + bb], I);
          }
          const int nr = min(32, per - c0);
          for (int j = 0; j < nr; j++) s = __fadd_rn(s, __shfl_sync(0xffffffffu, p, j));
        }
        if (lane == 0) a.part[((size_t)(t0 + i) * ROUTER_SEGS + seg) * a.E_pad + r] = s;
      }
      __syncwarp();  // the buffer is read before the next row overwrites it
    } else {  // fp32 rows: lane i runs token i's fma chain over the segment
      const int j0 = seg * (a.H / ROUTER_SEGS), j1 = j0 + a.H / ROUTER_SEGS;
      const float *wr = (const float *)a.W + (size_t)r * a.H;
      if (lane < nt) {
        const float *xv = a.x + (size_t)(t0 + lane) * a.H;
        float s = 0.0f;
        for (int j = j0; j < j1; j++) s = __fmaf_rn(__ldg(wr + j), __ldg(xv + j), s);
        a.part[((size_t)(t0 + lane) * ROUTER_SEGS + seg) * a.E_pad + r] = s;
      }
    }
  }
}

// Learned routing: block t routes token t.
__global__ void __launch_bounds__(NA_ROUTE_THREADS) k_na_route(NaArgs a) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int t = blockIdx.x;
  route_token_block(a.part + (size_t)t * ROUTER_SEGS * a.E_pad, a.E, a.E_pad, a.k, a.bias, a.scale, sm,
                    a.ids + (size_t)t * a.k, a.w + (size_t)t * a.k);
}

// Hash routing: one thread per (token, slot).
__global__ void k_na_hash(NaArgs a) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)a.T * a.k) return;
  const int t = (int)(i / a.k), j = (int)(i % a.k);
  const int v = __ldg(a.tok + t);
  const bool ok = v >= 0 && v < a.vocab;
  if (!ok && j == 0) raise_flag(a.err, DS4MOE_DEVERR_TOKEN_ID);
  int e = ok ? __ldg(a.hash + (size_t)v * a.k + j) : -1;
  if (ok && (e < 0 || e >= a.E)) {
    raise_flag(a.err, DS4MOE_DEVERR_INTERNAL);
    e = -1;
  }
  a.ids[i] = e;
  a.w[i] = e >= 0 ? __fmul_rn(__fdiv_rn(1.0f, (float)a.k), a.scale) : 0.0f;
}

// Shared memory of k_na_router_part: codes and scales of the token tile's
// segment blocks, and one row segment (per * 34 bytes) per warp.
size_t na_router_smem(int per) { return (size_t)NA_RT * per * 36 + (size_t)NA_WARPS * per * 34; }

bool na_dev_ptr(const void *p) {
  if (!p) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

std::mutex na_mu;
void *na_addr[NA_MAX_DEVICES];

// Set-up, once per device, with that device current: the device address of
// na_scratch, and the shared-memory limit of k_na_router_part.
cudaError_t na_setup(int dev, void **out) {
  std::lock_guard<std::mutex> lock(na_mu);
  if (!na_addr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress((void **)&p, na_scratch);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_na_router_part, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    na_addr[dev] = p;
  }
  *out = na_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" ds4moe_status ds4moe_route_noalloc(const ds4moe_layer_desc *d, const ds4moe_weights *wt, const float *x,
                                              const int32_t *token_ids, int32_t n_tok, int32_t *ids_out,
                                              float *w_out, uint32_t *err_flags, void *stream) {
  if (!d || !wt || d->abi_version != DS4MOE_ABI_VERSION) return DS4MOE_ERR_INVALID_ARG;
  if (d->hidden <= 0 || d->hidden % 256 != 0 || d->hidden > (1 << 16)) return DS4MOE_ERR_INVALID_ARG;
  if (d->n_experts < 1 || d->n_experts > 1024) return DS4MOE_ERR_INVALID_ARG;
  if (d->top_k < 1 || d->top_k > 16 || d->top_k > d->n_experts) return DS4MOE_ERR_INVALID_ARG;
  if (!(d->route_scale == d->route_scale)) return DS4MOE_ERR_INVALID_ARG;
  const bool hash = d->route == DS4MOE_ROUTE_HASH;
  if (!hash && d->route != DS4MOE_ROUTE_LEARNED) return DS4MOE_ERR_INVALID_ARG;
  if (hash && d->vocab < 1) return DS4MOE_ERR_INVALID_ARG;
  if (!hash && d->router_fmt != DS4MOE_F32 && d->router_fmt != DS4MOE_Q8_0) return DS4MOE_ERR_INVALID_ARG;
  if (n_tok < 0) return DS4MOE_ERR_INVALID_ARG;
  const int E_pad = (d->n_experts + 31) & ~31;
  if (!hash && (size_t)n_tok * ROUTER_SEGS * E_pad * sizeof(float) > DS4MOE_NOALLOC_SCRATCH_BYTES)
    return DS4MOE_ERR_UNSUPPORTED;  // more tokens than the fixed scratch holds
  if (n_tok == 0) return DS4MOE_OK;
  if (!na_dev_ptr(ids_out) || !na_dev_ptr(w_out)) return DS4MOE_ERR_INVALID_ARG;
  if (err_flags && !na_dev_ptr(err_flags)) return DS4MOE_ERR_INVALID_ARG;
  if (hash ? (!na_dev_ptr(token_ids) || !na_dev_ptr(wt->hash_table))
           : (!na_dev_ptr(x) || !na_dev_ptr(wt->router_w) || !na_dev_ptr(wt->router_bias)))
    return DS4MOE_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEVICES) return DS4MOE_ERR_CUDA;
  void *scratch = nullptr;
  if (na_setup(dev, &scratch) != cudaSuccess) return DS4MOE_ERR_CUDA;

  NaArgs a = {};
  a.x = x, a.W = (const uint8_t *)wt->router_w, a.bias = wt->router_bias, a.hash = wt->hash_table;
  a.tok = token_ids, a.T = n_tok, a.H = d->hidden, a.E = d->n_experts, a.E_pad = E_pad, a.k = d->top_k;
  a.vocab = d->vocab, a.q8 = d->router_fmt == DS4MOE_Q8_0, a.scale = d->route_scale;
  a.part = (float *)scratch, a.ids = ids_out, a.w = w_out, a.err = err_flags;
  cudaStream_t s = (cudaStream_t)stream;
  // Each launch's own result decides the status (cudaLaunchKernel returns
  // it); an error left pending by unrelated earlier work is neither reported
  // as this call's nor cleared.
  void *args[] = {&a};
  cudaError_t e;
  if (hash) {
    const long long n = (long long)n_tok * a.k;
    e = cudaLaunchKernel((const void *)k_na_hash, dim3((unsigned)((n + 255) / 256)), dim3(256), args, 0, s);
  } else {
    const int per = (a.H >> 5) / ROUTER_SEGS;
    const dim3 grid(E_pad / 32, ROUTER_SEGS, (n_tok + NA_RT - 1) / NA_RT);
    e = cudaLaunchKernel((const void *)k_na_router_part, grid, dim3(NA_WARPS * 32), args,
                         na_router_smem(per), s);
    if (e == cudaSuccess)
      e = cudaLaunchKernel((const void *)k_na_route, dim3(n_tok), dim3(NA_ROUTE_THREADS), args,
                           route_block_smem(E_pad, a.k), s);
  }
  return e == cudaSuccess ? DS4MOE_OK : DS4MOE_ERR_CUDA;
}

// api.cu -- host side of the libds4moe C ABI: argument validation, device
// memory ownership, the create-time re-layout of the weights, and the
// per-call launch sequence
//   quantise x -> route (router GEMV + top-k, or hash) -> bucket by expert
//   -> gate/up (+ SwiGLU + requant) -> down -> fixed-order combine into y.
// Nothing here does arithmetic on the data; all of it runs in the kernels.
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <new>

#include "bucket.cuh"
#include "common.cuh"
#include "internal.h"

using namespace ds4;

namespace {

bool is_dev_ptr(const void *p) {
  if (!p) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

bool fmt_ok(int f) { return f == DS4MOE_Q8_0 || f == DS4MOE_Q2S || f == DS4MOE_Q4S; }

// K must be a whole number of K-steps of the format, split evenly into the
// row-sum segments of an expert row.
bool k_ok(int fmt, int K) { return K > 0 && K % kstep(fmt) == 0 && (K / kstep(fmt)) % expert_segs(fmt, K) == 0; }

ds4moe_status validate_desc(const ds4moe_layer_desc *d) {
  if (!d || d->abi_version != DS4MOE_ABI_VERSION) return DS4MOE_ERR_INVALID_ARG;
  if (d->hidden <= 0 || d->hidden % 256 != 0 || d->hidden > (1 << 16)) return DS4MOE_ERR_INVALID_ARG;
  if (d->ffn <= 0 || d->ffn % 64 != 0 || d->ffn > (1 << 16)) return DS4MOE_ERR_INVALID_ARG;
  if (d->n_experts < 1 || d->n_experts > 1024) return DS4MOE_ERR_INVALID_ARG;
  if (d->top_k < 1 || d->top_k > 16 || d->top_k > d->n_experts) return DS4MOE_ERR_INVALID_ARG;
  if (d->n_shared != 0 && d->n_shared != 1) return DS4MOE_ERR_INVALID_ARG;
  if (d->max_tokens < 1 || d->max_tokens > (1 << 20)) return DS4MOE_ERR_INVALID_ARG;
  if (!fmt_ok(d->routed_fmt)) return DS4MOE_ERR_INVALID_ARG;
  if (d->n_shared && !fmt_ok(d->shared_fmt)) return DS4MOE_ERR_INVALID_ARG;
  if (!k_ok(d->routed_fmt, d->hidden) || !k_ok(d->routed_fmt, d->ffn)) return DS4MOE_ERR_INVALID_ARG;
  if (d->n_shared && (!k_ok(d->shared_fmt, d->hidden) || !k_ok(d->shared_fmt, d->ffn))) return DS4MOE_ERR_INVALID_ARG;
  if (d->route == DS4MOE_ROUTE_LEARNED) {
    if (d->router_fmt != DS4MOE_F32 && d->router_fmt != DS4MOE_Q8_0) return DS4MOE_ERR_INVALID_ARG;
  } else if (d->route == DS4MOE_ROUTE_HASH) {
    if (d->vocab < 1) return DS4MOE_ERR_INVALID_ARG;
  } else {
    return DS4MOE_ERR_INVALID_ARG;
  }
  if (!(d->route_scale == d->route_scale)) return DS4MOE_ERR_INVALID_ARG;  // NaN
  // int32 index arithmetic bounds: T*NS*max(H,F) elements per scratch array
  const long long T = d->max_tokens, NS = d->top_k + d->n_shared;
  const long long big = d->hidden > d->ffn ? d->hidden : d->ffn;
  if (T * NS * big >= (1ll << 40)) return DS4MOE_ERR_INVALID_ARG;
  return DS4MOE_OK;
}

// Allocation-failure injection for tests: the n-th device allocation made by
// ds4moe_create after ds4moe_debug_fail_alloc(n) fails as if the device were
// out of memory (0: off). One process-wide countdown.
std::atomic<int> g_fail_alloc{0};

void free_all(ds4moe_layer *h) {
  for (int i = 0; i < h->n_allocs; i++) cudaFree(h->allocs[i]);
  h->n_allocs = 0;
}

template <typename T>
ds4moe_status alloc(ds4moe_layer *h, T **p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) return DS4MOE_OK;
  if (h->n_allocs >= (int)(sizeof(h->allocs) / sizeof(h->allocs[0]))) return DS4MOE_ERR_OOM;
  void *q = nullptr;
  int n = g_fail_alloc.load();
  while (n > 0 && !g_fail_alloc.compare_exchange_weak(n, n - 1)) {
  }
  if (n == 1) return DS4MOE_ERR_OOM;  // the injected failure
  if (cudaMalloc(&q, bytes) != cudaSuccess) {
    cudaGetLastError();
    return DS4MOE_ERR_OOM;
  }
  h->allocs[h->n_allocs++] = q;
  h->bytes += bytes;
  *p = (T *)q;
  return DS4MOE_OK;
}

ds4moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DS4MOE_OK;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? DS4MOE_ERR_OOM : DS4MOE_ERR_CUDA;
}

// Re-lay out a [n_mat][rows][K] expert tensor into the RG16 layout. pair 0:
// alone; 1: interleaved per K-step with a second tensor (which = 0, 1);
// 2: the two 16-row groups of every 32 rows interleaved per K-step.
cudaError_t repack(int fmt, const void *src, uint8_t *dst, int n_mat, int rows, int K, int pair, int which,
                   cudaStream_t s) {
  if (fmt == DS4MOE_Q2S) return repack_q2s((const uint8_t *)src, dst, n_mat, rows, K, pair, which, s);
  if (fmt == DS4MOE_Q4S) return repack_q4s((const uint8_t *)src, dst, n_mat, rows, K, pair, which, s);
  return repack_q8((const uint8_t *)src, dst, n_mat, rows, K, pair, which, s);
}

size_t rg16_bytes(int fmt, long long n_mat, long long rows, long long K) {
  return (size_t)(n_mat * (rows / TILE_ROWS) * (K / kstep(fmt)) * tile_bytes(fmt));
}

ds4moe_status build(ds4moe_layer *h, const ds4moe_weights *w) {
  const ds4moe_layer_desc &d = h->d;
  const int E = d.n_experts, H = d.hidden, F = d.ffn, k = d.top_k;
  const long long NS = h->NS;
  ds4moe_status st;
  cudaStream_t s = 0;

  // ---- weights
  if (d.route == DS4MOE_ROUTE_LEARNED) {
    if (!is_dev_ptr(w->router_w) || !is_dev_ptr(w->router_bias)) return DS4MOE_ERR_INVALID_ARG;
    if (d.router_fmt == DS4MOE_Q8_0) {
      const size_t nb = (size_t)(h->E_pad / 32) * (H / RQ8_KSTEP) * RQ8_TILE;
      if ((st = alloc(h, &h->router, nb)) != DS4MOE_OK) return st;
      if ((st = cuda_status(cudaMemsetAsync(h->router, 0, nb, s))) != DS4MOE_OK) return st;
      if ((st = cuda_status(repack_rq8((const uint8_t *)w->router_w, h->router, E, h->E_pad, H, s))) != DS4MOE_OK)
        return st;
    } else {
      const size_t nb = (size_t)E * H * 4;
      if ((st = alloc(h, &h->router, nb)) != DS4MOE_OK) return st;
      if ((st = cuda_status(cudaMemcpyAsync(h->router, w->router_w, nb, cudaMemcpyDeviceToDevice, s))) != DS4MOE_OK)
        return st;
    }
    if ((st = alloc(h, &h->bias, (size_t)E * 4)) != DS4MOE_OK) return st;
    if ((st = cuda_status(cudaMemcpyAsync(h->bias, w->router_bias, (size_t)E * 4, cudaMemcpyDeviceToDevice, s))) !=
        DS4MOE_OK)
      return st;
  } else {
    if (!is_dev_ptr(w->hash_table)) return DS4MOE_ERR_INVALID_ARG;
    const size_t nb = (size_t)d.vocab * k * 4;
    if ((st = alloc(h, &h->hash, nb)) != DS4MOE_OK) return st;
    if ((st = cuda_status(cudaMemcpyAsync(h->hash, w->hash_table, nb, cudaMemcpyDeviceToDevice, s))) != DS4MOE_OK)
      return st;
  }
  if (!is_dev_ptr(w->gate) || !is_dev_ptr(w->up) || !is_dev_ptr(w->down)) return DS4MOE_ERR_INVALID_ARG;
  const int rf = d.routed_fmt;
  if ((st = alloc(h, &h->gu, 2 * rg16_bytes(rf, E, F, H))) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->dn, rg16_bytes(rf, E, H, F))) != DS4MOE_OK) return st;
  if ((st = cuda_status(repack(rf, w->gate, h->gu, E, F, H, 1, 0, s))) != DS4MOE_OK) return st;
  if ((st = cuda_status(repack(rf, w->up, h->gu, E, F, H, 1, 1, s))) != DS4MOE_OK) return st;
  if ((st = cuda_status(repack(rf, w->down, h->dn, E, H, F, 2, 0, s))) != DS4MOE_OK) return st;
  if (d.n_shared) {
    if (!is_dev_ptr(w->sh_gate) || !is_dev_ptr(w->sh_up) || !is_dev_ptr(w->sh_down)) return DS4MOE_ERR_INVALID_ARG;
    const int sf = d.shared_fmt;
    if ((st = alloc(h, &h->sgu, 2 * rg16_bytes(sf, 1, F, H))) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->sdn, rg16_bytes(sf, 1, H, F))) != DS4MOE_OK) return st;
    if ((st = cuda_status(repack(sf, w->sh_gate, h->sgu, 1, F, H, 1, 0, s))) != DS4MOE_OK) return st;
    if ((st = cuda_status(repack(sf, w->sh_up, h->sgu, 1, F, H, 1, 1, s))) != DS4MOE_OK) return st;
    if ((st = cuda_status(repack(sf, w->sh_down, h->sdn, 1, H, F, 2, 0, s))) != DS4MOE_OK) return st;
  }

  // ---- scratch, sized for one chunk of either path (Ts = max(Tc, Tp) tokens)
  const long long Tc = h->Tc, Ts = h->Ts;
  if ((st = alloc(h, &h->xq, (size_t)Ts * H)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->dx, (size_t)Ts * (H / 32) * 4)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->gs, (size_t)Ts * (H / 16) * 2)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->ids, (size_t)Ts * k * 4)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->wts, (size_t)Ts * k * 4)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->bucket, (size_t)bucket_table_ints(h->A_max, (int)Tc, (int)NS) * 4)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->hq, (size_t)(Ts * NS) * F)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->dh, (size_t)(Ts * NS) * (F / 32) * 4)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->gsh, (size_t)(Ts * NS) * (F / 16) * 2)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->apart, (size_t)(Ts * NS) * H * 4)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->hbuf, (size_t)(Tc * NS) * F * 4)) != DS4MOE_OK) return st;
  if ((st = alloc(h, &h->xnorm, (size_t)H * 4)) != DS4MOE_OK) return st;
  if (h->Tp > 0) {
    if ((st = alloc(h, &h->pf_meta, (size_t)(E + 1) * 2 * 4)) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->pf_pass, (size_t)(E + 2) * 4)) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->pf_list, prefill_list_ints(h->Tp, k, d.n_shared) * 4)) != DS4MOE_OK) return st;
  }
  if ((st = alloc(h, &h->err, 64)) != DS4MOE_OK) return st;
  if ((st = cuda_status(cudaMemsetAsync(h->err, 0, 64, s))) != DS4MOE_OK) return st;
  {  // tickets start at zero and reset themselves
    const size_t n_ht = (size_t)(Tc * NS) * (F / 32) * 4, n_ct = (size_t)Tc * (H / 32) * 4;
    if ((st = alloc(h, &h->hticket, n_ht)) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->cticket, n_ct)) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->rticket, 16)) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->xq_ready, 16)) != DS4MOE_OK) return st;
    if ((st = cuda_status(cudaMemsetAsync(h->rticket, 0, 16, s))) != DS4MOE_OK) return st;
    if ((st = cuda_status(cudaMemsetAsync(h->xq_ready, 0, 16, s))) != DS4MOE_OK) return st;
    if ((st = cuda_status(cudaMemsetAsync(h->hticket, 0, n_ht, s))) != DS4MOE_OK) return st;
    if ((st = cuda_status(cudaMemsetAsync(h->cticket, 0, n_ct, s))) != DS4MOE_OK) return st;
  }

  if (d.route == DS4MOE_ROUTE_HASH) {
    // every table entry must name a routed expert
    if ((st = cuda_status(cudaMemsetAsync(h->bucket, 0, 4, s))) != DS4MOE_OK) return st;
    if ((st = cuda_status(check_hash_table(h->hash, (int64_t)d.vocab * k, E, h->bucket, s))) != DS4MOE_OK) return st;
    int32_t bad = 0;
    if ((st = cuda_status(cudaMemcpyAsync(&bad, h->bucket, 4, cudaMemcpyDeviceToHost, s))) != DS4MOE_OK) return st;
    if ((st = cuda_status(cudaStreamSynchronize(s))) != DS4MOE_OK) return st;
    if (bad) return DS4MOE_ERR_INVALID_ARG;
  }
  return cuda_status(cudaStreamSynchronize(s));
}

}  // namespace

extern "C" {

uint32_t ds4moe_abi_version(void) { return DS4MOE_ABI_VERSION; }

const char *ds4moe_status_string(ds4moe_status s) {
  switch (s) {
    case DS4MOE_OK: return "DS4MOE_OK";
    case DS4MOE_ERR_INVALID_ARG: return "DS4MOE_ERR_INVALID_ARG";
    case DS4MOE_ERR_UNSUPPORTED: return "DS4MOE_ERR_UNSUPPORTED";
    case DS4MOE_ERR_OOM: return "DS4MOE_ERR_OOM";
    case DS4MOE_ERR_CUDA: return "DS4MOE_ERR_CUDA";
    case DS4MOE_ERR_DEVICE: return "DS4MOE_ERR_DEVICE";
  }
  return "DS4MOE_ERR_UNKNOWN";
}

ds4moe_status ds4moe_create(const ds4moe_layer_desc *desc, const ds4moe_weights *w, ds4moe_layer **out) {
  if (!out) return DS4MOE_ERR_INVALID_ARG;
  *out = nullptr;
  ds4moe_status st = validate_desc(desc);
  if (st != DS4MOE_OK) return st;
  if (!w) return DS4MOE_ERR_INVALID_ARG;
  ds4moe_layer *h = new (std::nothrow) ds4moe_layer;
  if (!h) return DS4MOE_ERR_OOM;
  memset(h, 0, sizeof(*h));
  h->d = *desc;
  if (cudaGetDevice(&h->device) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return DS4MOE_ERR_CUDA;
  }
  h->E_pad = (desc->n_experts + 31) / 32 * 32;
  h->Tc = desc->max_tokens < DEC_MAX_T ? desc->max_tokens : DEC_MAX_T;
  h->pf_min = PF_MIN_T_DEFAULT;
  if (const char *v = getenv("DS4MOE_PREFILL_MIN_TOKENS")) {
    const long m = strtol(v, nullptr, 10);
    if (m >= 1 && m <= (1 << 20)) h->pf_min = (int)m;
  }
  h->Tp = 0;
  if (prefill_supported(*desc) && desc->max_tokens >= h->pf_min)
    h->Tp = desc->max_tokens < PF_MAX_T ? desc->max_tokens : PF_MAX_T;
  h->Ts = h->Tp > h->Tc ? h->Tp : h->Tc;
  if (cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return DS4MOE_ERR_CUDA;
  }
  h->NS = desc->top_k + desc->n_shared;
  {
    const long long routed = (long long)desc->max_tokens * desc->top_k;
    h->A_max = (int)(routed < desc->n_experts ? routed : desc->n_experts) + desc->n_shared;
  }
  if (route_dec_smem(h) > DEC_SMEM_LIMIT) {  // shapes whose kernels do not fit an SM
    delete h;
    return DS4MOE_ERR_UNSUPPORTED;
  }
  if (decode_set_attributes() != cudaSuccess || (h->Tp > 0 && prefill_set_attributes() != cudaSuccess)) {
    cudaGetLastError();
    delete h;
    return DS4MOE_ERR_CUDA;
  }
  st = build(h, w);
  if (st != DS4MOE_OK) {
    cudaDeviceSynchronize();
    cudaGetLastError();
    free_all(h);
    delete h;
    return st;
  }
  *out = h;
  return DS4MOE_OK;
}

void ds4moe_destroy(ds4moe_layer *h) {
  if (!h) return;
  cudaDeviceSynchronize();
  if (h->ev_made)
    for (int i = 0; i < 8; i++) cudaEventDestroy(h->ev[i]);
  for (int i = 0; i < DS4_HOST_GRAPHS; i++)
    if (h->host_graph[i]) cudaGraphExecDestroy(h->host_graph[i]);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->x_pin) cudaFreeHost(h->x_pin);
  if (h->y_pin) cudaFreeHost(h->y_pin);
  if (h->tok_pin) cudaFreeHost(h->tok_pin);
  free_all(h);
  delete h;
}

uint64_t ds4moe_device_bytes(const ds4moe_layer *h) { return h ? h->bytes : 0; }

static ds4moe_status check_call(ds4moe_layer *h, int32_t n_tok) {
  if (!h) return DS4MOE_ERR_INVALID_ARG;
  if (n_tok < 0 || n_tok > h->d.max_tokens) return DS4MOE_ERR_INVALID_ARG;
  return DS4MOE_OK;
}

ds4moe_status ds4moe_route(ds4moe_layer *h, const float *x, const int32_t *token_ids, int32_t n_tok,
                           int32_t *ids_out, float *w_out, void *stream) {
  ds4moe_status st = check_call(h, n_tok);
  if (st != DS4MOE_OK) return st;
  if (n_tok == 0) return DS4MOE_OK;
  if (!is_dev_ptr(ids_out) || !is_dev_ptr(w_out)) return DS4MOE_ERR_INVALID_ARG;
  const bool hash = h->d.route == DS4MOE_ROUTE_HASH;
  if (hash ? !is_dev_ptr(token_ids) : !is_dev_ptr(x)) return DS4MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const int H = h->d.hidden, k = h->d.top_k;
  cudaError_t e = cudaSuccess;
  for (int c0 = 0; c0 < n_tok && e == cudaSuccess; c0 += h->Tc) {
    const int nc = n_tok - c0 < h->Tc ? n_tok - c0 : h->Tc;
    e = launch_dec_route(h, hash ? nullptr : x + (size_t)c0 * H, hash ? token_ids + c0 : nullptr, nc,
                         ids_out + (size_t)c0 * k, w_out + (size_t)c0 * k, false, s);
    h->launches += 1;
  }
  return cuda_status(e);
}

// The launches of a forward call whose arguments are checked.
// norm: x is un-normalised; the router kernel applies the RMSNorm (eps).
static ds4moe_status forward_run(ds4moe_layer *h, const float *x, int32_t n_tok, const int32_t *token_ids, float *y,
                                 cudaStream_t s, bool norm = false, float eps = 0.0f) {
  const int H = h->d.hidden;
  const bool prof = h->prof_on != 0;
  auto mark = [&](int i) {
    if (prof) cudaEventRecord(h->ev[i], s);
  };
  // Tokens are independent: a prefill-sized call runs in chunks of at most Tp
  // tokens on the prefill path, anything else in chunks of at most Tc tokens
  // on the decode path.
  cudaError_t e = cudaSuccess;
  if (h->Tp > 0 && n_tok >= h->pf_min) {
    for (int c0 = 0; c0 < n_tok && e == cudaSuccess; c0 += h->Tp) {
      const int nc = n_tok - c0 < h->Tp ? n_tok - c0 : h->Tp;
      e = launch_prefill(h, x + (size_t)c0 * H, token_ids ? token_ids + c0 : nullptr, nc, y + (size_t)c0 * H, s,
                         prof ? h->ev : nullptr, norm, eps);
    }
    return cuda_status(e);
  }
  for (int c0 = 0; c0 < n_tok && e == cudaSuccess; c0 += h->Tc) {
    const int nc = n_tok - c0 < h->Tc ? n_tok - c0 : h->Tc;
    const float *xc = x + (size_t)c0 * H;
    const int32_t *tc = token_ids ? token_ids + c0 : nullptr;
    float *yc = y + (size_t)c0 * H;
    mark(0);
    mark(1);
    e = launch_dec_route(h, xc, tc, nc, h->ids, h->wts, true, s, norm, eps);
    mark(2);
    mark(3);
    if (e == cudaSuccess) e = launch_experts(h, nc, yc, 0, s);
    mark(4);
    if (e == cudaSuccess) e = launch_experts(h, nc, yc, 1, s);
    mark(5);
    mark(6);
    h->launches += 3;
  }
  // A call stopped between its router and its down kernel leaves the count
  // of quantised x that down clears; clear it here so that no later call
  // starts on it.
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaMemsetAsync(h->xq_ready, 0, sizeof(int32_t), s);
  }
  return cuda_status(e);
}

ds4moe_status ds4moe_forward(ds4moe_layer *h, const float *x, int32_t n_tok, const int32_t *token_ids, float *y,
                             void *stream) {
  ds4moe_status st = check_call(h, n_tok);
  if (st != DS4MOE_OK) return st;
  if (n_tok == 0) return DS4MOE_OK;
  if (!is_dev_ptr(x) || !is_dev_ptr(y) || x == y) return DS4MOE_ERR_INVALID_ARG;
  if (h->d.route == DS4MOE_ROUTE_HASH && !is_dev_ptr(token_ids)) return DS4MOE_ERR_INVALID_ARG;
  return forward_run(h, x, n_tok, token_ids, y, (cudaStream_t)stream);
}

// Every read of x is in the router kernel (or the RMSNorm kernel before
// it), and every write of y comes after it has completed (down waits for
// gate/up, which waits for the router; the prefill kernels are
// stream-ordered), so y may be x itself. A one-token call on the decode path
// runs the RMSNorm kernel into the handle's row buffer and the plain forward
// on it: there the separate kernel's run hides the router kernel's start
// (measured 0.5 us faster per layer than the folded norm, which is faster
// from two tokens on: 2.8 us per layer at eight).
ds4moe_status ds4moe_forward_rmsnorm(ds4moe_layer *h, const float *x, int32_t n_tok, const int32_t *token_ids,
                                     float eps, float *y, void *stream) {
  ds4moe_status st = check_call(h, n_tok);
  if (st != DS4MOE_OK) return st;
  if (n_tok == 0) return DS4MOE_OK;
  if (!is_dev_ptr(x) || !is_dev_ptr(y) || !(eps == eps) || ((uintptr_t)x & 15)) return DS4MOE_ERR_INVALID_ARG;
  const size_t n = (size_t)n_tok * h->d.hidden;
  if (x != y && x < y + n && y < x + n) return DS4MOE_ERR_INVALID_ARG;  // partial overlap
  if (h->d.route == DS4MOE_ROUTE_HASH && !is_dev_ptr(token_ids)) return DS4MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (n_tok == 1 && !(h->Tp > 0 && h->pf_min <= 1)) {
    const cudaError_t e = launch_rmsnorm(x, h->xnorm, 1, h->d.hidden, eps, s);
    h->launches++;
    if (e != cudaSuccess) return cuda_status(e);
    return forward_run(h, h->xnorm, 1, token_ids, y, s);
  }
  return forward_run(h, x, n_tok, token_ids, y, s, true, eps);
}

ds4moe_status ds4moe_profile_enable(ds4moe_layer *h, int32_t on) {
  if (!h) return DS4MOE_ERR_INVALID_ARG;
  if (on && !h->ev_made) {
    for (int i = 0; i < 8; i++) {
      cudaError_t e = cudaEventCreate(&h->ev[i]);
      if (e != cudaSuccess) return cuda_status(e);
    }
    h->ev_made = 1;
  }
  h->prof_on = on ? 1 : 0;
  if (!on) {
    for (int i = 0; i < 8; i++) h->prof_ms[i] = 0.0;
    h->prof_calls = 0;
  }
  return DS4MOE_OK;
}

ds4moe_status ds4moe_profile_collect(ds4moe_layer *h) {
  if (!h || !h->prof_on) return DS4MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaEventSynchronize(h->ev[DS4MOE_N_STAGES]);
  if (e != cudaSuccess) return cuda_status(e);
  for (int i = 0; i < DS4MOE_N_STAGES; i++) {
    float ms = 0.0f;
    e = cudaEventElapsedTime(&ms, h->ev[i], h->ev[i + 1]);
    if (e != cudaSuccess) return cuda_status(e);
    h->prof_ms[i] += ms;
  }
  h->prof_calls++;
  return DS4MOE_OK;
}

ds4moe_status ds4moe_profile_read(const ds4moe_layer *h, double *ms_out, int32_t n, int64_t *calls) {
  if (!h || n < 0 || (n > 0 && !ms_out)) return DS4MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n && i < DS4MOE_N_STAGES; i++) ms_out[i] = h->prof_ms[i];
  if (calls) *calls = h->prof_calls;
  return DS4MOE_OK;
}

uint64_t ds4moe_launch_count(const ds4moe_layer *h) { return h ? h->launches : 0; }

// A decode-sized forward_host call (n_tok <= Tc) runs on the handle's
// mapped pinned buffers: the kernels read x (and the token ids) and update y
// in host memory directly over the coherent CPU-GPU link, so no copy
// precedes or follows them; the launches are captured once per token count
// into a CUDA graph.
static cudaError_t host_sequence(ds4moe_layer *h, int n_tok, bool hash, cudaStream_t s) {
  float *xm = nullptr, *ym = nullptr;
  int32_t *tm = nullptr;
  cudaError_t e = cudaHostGetDevicePointer((void **)&xm, h->x_pin, 0);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer((void **)&ym, h->y_pin, 0);
  if (e == cudaSuccess) e = cudaHostGetDevicePointer((void **)&tm, h->tok_pin, 0);
  if (e != cudaSuccess) return e;
  return forward_run(h, xm, n_tok, hash ? tm : nullptr, ym, s) == DS4MOE_OK ? cudaSuccess : cudaErrorUnknown;
}

// The device address of pinned (page-locked, mapped) host memory, else null.
static void *mapped_ptr(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

static cudaGraphExec_t host_graph(ds4moe_layer *h, int n_tok, bool hash) {
  if (h->host_graph[n_tok]) return h->host_graph[n_tok];
  if (h->host_graph_off) return nullptr;
  if (!h->cap_stream && cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    h->cap_stream = nullptr;
    h->host_graph_off = 1;
    return nullptr;
  }
  const int64_t l0 = h->launches;
  cudaGraph_t g = nullptr;
  cudaGraphExec_t x = nullptr;
  if (cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaGetLastError();
    h->host_graph_off = 1;
    return nullptr;
  }
  const cudaError_t e = host_sequence(h, n_tok, hash, h->cap_stream);
  const cudaError_t e2 = cudaStreamEndCapture(h->cap_stream, &g);
  h->launches = l0;
  if (e == cudaSuccess && e2 == cudaSuccess && g && cudaGraphInstantiate(&x, g, 0) == cudaSuccess) {
    h->host_graph[n_tok] = x;
    h->host_graph_launches[n_tok] = 3 * ((n_tok + h->Tc - 1) / h->Tc);
  } else {  // not capturable here: the plain sequence from now on
    cudaGetLastError();
    h->host_graph_off = 1;
    x = nullptr;
  }
  if (g) cudaGraphDestroy(g);
  return x;
}

ds4moe_status ds4moe_forward_host(ds4moe_layer *h, const float *x_host, int32_t n_tok, const int32_t *token_ids_host,
                                  float *y_host, void *stream) {
  ds4moe_status st = check_call(h, n_tok);
  if (st != DS4MOE_OK) return st;
  if (n_tok == 0) return DS4MOE_OK;
  if (!x_host || !y_host) return DS4MOE_ERR_INVALID_ARG;
  const bool hash = h->d.route == DS4MOE_ROUTE_HASH;
  if (hash && !token_ids_host) return DS4MOE_ERR_INVALID_ARG;
  // device staging of one chunk (Ts tokens) for the copy path, on first use
  const size_t xb = (size_t)h->Ts * h->d.hidden * 4;
  if (!h->x_dev) {
    if ((st = alloc(h, &h->x_dev, xb)) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->y_dev, xb)) != DS4MOE_OK) return st;
    if ((st = alloc(h, &h->tok_dev, (size_t)h->Ts * 4)) != DS4MOE_OK) return st;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const size_t nb = (size_t)n_tok * h->d.hidden * 4;
  // Decode-sized calls on pinned caller buffers: the kernels read x (and the
  // token ids) and update y in them directly.
  if (n_tok <= h->Tc && !h->prof_on) {
    float *xm = (float *)mapped_ptr(x_host), *ym = (float *)mapped_ptr(y_host);
    int32_t *tm = hash ? (int32_t *)mapped_ptr(token_ids_host) : nullptr;
    if (xm && ym && xm != ym && (!hash || tm)) {
      st = forward_run(h, xm, n_tok, tm, ym, s);
      if (st != DS4MOE_OK) return st;
      return cuda_status(cudaStreamSynchronize(s));
    }
  }
  // Other decode-sized calls: the inputs into the handle's mapped pinned
  // buffers, one graph replay of the forward on them, the result back.
  if (n_tok <= h->Tc && !h->prof_on) {
    const size_t pb = (size_t)h->Tc * h->d.hidden * 4;
    if (!h->x_pin && (cudaHostAlloc(&h->x_pin, pb, cudaHostAllocMapped) != cudaSuccess ||
                      cudaHostAlloc(&h->y_pin, pb, cudaHostAllocMapped) != cudaSuccess ||
                      cudaHostAlloc(&h->tok_pin, (size_t)h->Tc * 4, cudaHostAllocMapped) != cudaSuccess)) {
      cudaGetLastError();
      return DS4MOE_ERR_OOM;
    }
    cudaGraphExec_t g = host_graph(h, n_tok, hash);
    if (g) {
      memcpy(h->x_pin, x_host, nb);
      memcpy(h->y_pin, y_host, nb);
      if (hash) memcpy(h->tok_pin, token_ids_host, (size_t)n_tok * 4);
      cudaError_t e = cudaGraphLaunch(g, s);
      if (e == cudaSuccess) e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return cuda_status(e);
      h->launches += h->host_graph_launches[n_tok];
      memcpy(y_host, h->y_pin, nb);
      return DS4MOE_OK;
    }
  }
  // Anything else: chunk by chunk through the device staging buffers.
  cudaError_t e = cudaSuccess;
  for (int c0 = 0; c0 < n_tok && e == cudaSuccess; c0 += h->Ts) {
    const int nc = n_tok - c0 < h->Ts ? n_tok - c0 : h->Ts;
    const size_t cb = (size_t)nc * h->d.hidden * 4, off = (size_t)c0 * h->d.hidden;
    e = cudaMemcpyAsync(h->x_dev, x_host + off, cb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->y_dev, y_host + off, cb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && hash)
      e = cudaMemcpyAsync(h->tok_dev, token_ids_host + c0, (size_t)nc * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) break;
    st = ds4moe_forward(h, h->x_dev, nc, hash ? h->tok_dev : nullptr, h->y_dev, stream);
    if (st != DS4MOE_OK) return st;
    e = cudaMemcpyAsync(y_host + off, h->y_dev, cb, cudaMemcpyDeviceToHost, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

ds4moe_status ds4moe_rmsnorm(const float *x, float *out, int32_t n_tok, int32_t hidden, float eps, void *stream) {
  if (n_tok < 0 || hidden <= 0 || hidden % 32 != 0 || !(eps == eps)) return DS4MOE_ERR_INVALID_ARG;
  if (n_tok == 0) return DS4MOE_OK;
  if (!is_dev_ptr(x) || !is_dev_ptr(out)) return DS4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_rmsnorm(x, out, n_tok, hidden, eps, (cudaStream_t)stream));
}

ds4moe_status ds4moe_get_device_error(ds4moe_layer *h, void *stream, uint32_t *flags_out) {
  if (!h) return DS4MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t f = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(&f, h->err, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, 4);
  // A block that gave up a wait left without its arrivals on the self-
  // resetting completion counters; zero them so that the next call starts
  // from a clean state.
  if (e == cudaSuccess && (f & DS4MOE_DEVERR_TIMEOUT)) {
    const long long Tc = h->Tc, NS = h->NS;
    e = cudaMemset(h->hticket, 0, (size_t)(Tc * NS) * (h->d.ffn / 32) * 4);
    if (e == cudaSuccess) e = cudaMemset(h->cticket, 0, (size_t)Tc * (h->d.hidden / 32) * 4);
    if (e == cudaSuccess) e = cudaMemset(h->rticket, 0, 16);
    if (e == cudaSuccess) e = cudaMemset(h->xq_ready, 0, 16);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
  }
  if (e != cudaSuccess) return cuda_status(e);
  if (flags_out) *flags_out = f;
  return f ? DS4MOE_ERR_DEVICE : DS4MOE_OK;
}

ds4moe_status ds4moe_debug_set_wait_limit(ds4moe_layer *h, int64_t cycles) {
  if (!h || cycles < 0) return DS4MOE_ERR_INVALID_ARG;
  h->wait_limit = cycles;
  return DS4MOE_OK;
}

ds4moe_status ds4moe_debug_fail_alloc(int32_t n) {
  if (n < 0) return DS4MOE_ERR_INVALID_ARG;
  g_fail_alloc.store(n);
  return DS4MOE_OK;
}

// Read-only views of the handle's scratch, for inspecting the intermediate
// results of the last call (integer codes, ids, weights).
ds4moe_status ds4moe_debug_scratch(ds4moe_layer *h, int32_t which, const void **ptr_out, uint64_t *bytes_out) {
  if (!h || !ptr_out || !bytes_out) return DS4MOE_ERR_INVALID_ARG;
  const long long T = h->Ts, NS = h->NS, H = h->d.hidden, F = h->d.ffn, k = h->d.top_k;
  const void *p = nullptr;
  uint64_t n = 0;
  switch (which) {
    case 0: p = h->xq, n = T * H; break;
    case 1: p = h->dx, n = T * (H / 32) * 4; break;
    case 2: p = h->gs, n = T * (H / 16) * 2; break;
    case 3: p = h->ids, n = T * k * 4; break;
    case 4: p = h->wts, n = T * k * 4; break;
    case 5: p = h->hq, n = T * NS * F; break;
    case 6: p = h->dh, n = T * NS * (F / 32) * 4; break;
    case 7: p = h->apart, n = T * NS * H * 4; break;
    default: return DS4MOE_ERR_INVALID_ARG;
  }
  *ptr_out = p;
  *bytes_out = n;
  return DS4MOE_OK;
}

}  // extern "C"

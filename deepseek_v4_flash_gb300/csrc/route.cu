// route.cu -- activation quantisation, router GEMV + sigmoid + bias top-k +
// renormalisation, hash routing, per-expert bucketing, the fixed-order
// combine into y, and RMSNorm.
//
// Routing follows "DeepSeek V4 Flash -- DFlash Integration" (Model
// Architecture: learned top-k with optional bias on layers >= 3, token-ID
// table on layers 0-2; Execution Modes: renormalise the kept weights). Every
// float operation is the CAS one (common.cuh), in the CAS order.
#include "common.cuh"
#include "internal.h"

namespace ds4 {

// ---------------------------------------------------------------------------
// CAS step 1 on x: one warp per 32-block.
__global__ void __launch_bounds__(256) k_quantize(const float *__restrict__ x, int H, int8_t *__restrict__ xq,
                                                  float *__restrict__ dx, int16_t *__restrict__ gs,
                                                  uint32_t *err) {
  const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = H >> 5;
  for (int b = warp; b < nb; b += blockDim.x >> 5) {
    const float v = x[(size_t)t * H + 32 * b + lane];
    if (__any_sync(0xffffffffu, !isfinite(v)) && lane == 0) raise_flag(err, DS4MOE_DEVERR_NONFINITE);
    const float amax = warp_max(fabsf(v));
    const float d = __fdiv_rn(amax, 127.0f);
    const int q = cas_code(v, d);
    const int s = half_warp_sum(q);
    xq[(size_t)t * H + 32 * b + lane] = (int8_t)q;
    if (lane == 0) dx[(size_t)t * nb + b] = d;
    if ((lane & 15) == 0) gs[(size_t)t * (H >> 4) + 2 * b + (lane >> 4)] = (int16_t)s;
  }
}

cudaError_t launch_quantize(const float *x, int T, int H, int8_t *xq, float *dx, int16_t *gs, uint32_t *err,
                            cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_quantize<<<T, 256, 0, s>>>(x, H, xq, dx, gs, err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Router GEMV, Q8_0 rows (CAS steps 2-4 with S = 8): one warp per
// (32 router rows, one of 8 K-segments, up to RT tokens); lane = row.
// Writes the segment sums rpart[t][seg][row].
constexpr int RT = 8;

__global__ void __launch_bounds__(32) k_router_q8(const uint8_t *__restrict__ W, int H, int E_pad,
                                                  const int8_t *__restrict__ xq, const float *__restrict__ dx,
                                                  int T, float *__restrict__ rpart) {
  const int rg = blockIdx.x, seg = blockIdx.y, t0 = blockIdx.z * RT, lane = threadIdx.x;
  const int nb = H >> 5, per = nb / ROUTER_SEGS, KS = H / RQ8_KSTEP;
  const int nt = min(RT, T - t0);
  float acc[RT];
#pragma unroll
  for (int i = 0; i < RT; i++) acc[i] = 0.0f;
  for (int b = seg * per; b < (seg + 1) * per; b++) {
    const uint8_t *tile = W + ((size_t)rg * KS + (b >> 1)) * RQ8_TILE;
    const uint32_t dd = *(const uint32_t *)(tile + 4 * lane);
    const float d = half_bits_to_float((b & 1) ? (dd >> 16) : dd);
    const uint4 w0 = *(const uint4 *)(tile + RQ8_Q + 512 * (2 * (b & 1)) + 16 * lane);
    const uint4 w1 = *(const uint4 *)(tile + RQ8_Q + 512 * (2 * (b & 1) + 1) + 16 * lane);
#pragma unroll
    for (int i = 0; i < RT; i++) {
      if (i < nt) {
        const int t = t0 + i;
        const uint4 *xv = (const uint4 *)(xq + (size_t)t * H + 32 * b);
        const int I = dot16(w1, __ldg(xv + 1), dot16(w0, __ldg(xv), 0));
        acc[i] = __fadd_rn(acc[i], q8_term(d, __ldg(dx + (size_t)t * nb + b), I));
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RT; i++)
    if (i < nt) rpart[((size_t)(t0 + i) * ROUTER_SEGS + seg) * E_pad + 32 * rg + lane] = acc[i];
}

// Router GEMV, fp32 rows (CAS step 4, F32 segments: fma chains).
__global__ void __launch_bounds__(32) k_router_f32(const float *__restrict__ W, int H, int E, int E_pad,
                                                   const float *__restrict__ x, float *__restrict__ rpart) {
  const int r = 32 * blockIdx.x + threadIdx.x, seg = blockIdx.y, t = blockIdx.z;
  const int per = H / ROUTER_SEGS;
  float acc = 0.0f;
  if (r < E) {
    const float *w = W + (size_t)r * H;
    const float *v = x + (size_t)t * H;
    for (int i = seg * per; i < (seg + 1) * per; i++) acc = __fmaf_rn(w[i], v[i], acc);
  }
  rpart[((size_t)t * ROUTER_SEGS + seg) * E_pad + r] = acc;
}

// CAS step 6: one warp per token. Segment sums -> logit -> sigmoid -> key;
// k rounds of warp arg-max (larger key, then lower index); renormalise.
__global__ void __launch_bounds__(32) k_topk(const float *__restrict__ rpart, const float *__restrict__ bias,
                                             int E, int E_pad, int k, float scale, int32_t *__restrict__ ids,
                                             float *__restrict__ w) {
  extern __shared__ float sh[];  // s[E] | key[E] | taken[E]
  float *s = sh, *key = sh + E;
  int *taken = (int *)(sh + 2 * E);
  __shared__ int sel[16];
  const int t = blockIdx.x, lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) {
    float lg = 0.0f;
#pragma unroll
    for (int g = 0; g < ROUTER_SEGS; g++) lg = __fadd_rn(lg, rpart[((size_t)t * ROUTER_SEGS + g) * E_pad + e]);
    const float se = cas_sigmoid(lg);
    s[e] = se;
    key[e] = __fadd_rn(se, bias[e]);
    taken[e] = 0;
  }
  __syncwarp();
  for (int j = 0; j < k; j++) {
    float bk = 0.0f;
    int bi = -1;
    for (int e = lane; e < E; e += 32) {
      if (taken[e]) continue;
      const float ke = key[e];
      if (bi < 0 || ke > bk) bk = ke, bi = e;  // ascending e: ties keep the lower index
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const bool better = oi >= 0 && (bi < 0 || ok > bk || (ok == bk && oi < bi));
      if (better) bk = ok, bi = oi;
    }
    if (lane == 0) {
      sel[j] = bi;
      if (bi >= 0) taken[bi] = 1;
    }
    __syncwarp();
  }
  if (lane == 0) {
    float sum = 0.0f;
    for (int j = 0; j < k; j++) sum = __fadd_rn(sum, sel[j] >= 0 ? s[sel[j]] : 0.0f);
    for (int j = 0; j < k; j++) {
      ids[(size_t)t * k + j] = sel[j];
      w[(size_t)t * k + j] = sel[j] >= 0 ? __fmul_rn(__fdiv_rn(s[sel[j]], sum), scale) : 0.0f;
    }
  }
}

// Hash routing: ids = table[token] in stored order, w = (1/k) * scale.
__global__ void k_hash(const int32_t *__restrict__ tok, const int32_t *__restrict__ table, int T, int k,
                       int vocab, float scale, int32_t *__restrict__ ids, float *__restrict__ w, uint32_t *err) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int v = tok[t];
  const bool ok = v >= 0 && v < vocab;
  if (!ok) raise_flag(err, DS4MOE_DEVERR_TOKEN_ID);
  const float wk = __fmul_rn(__fdiv_rn(1.0f, (float)k), scale);
  for (int j = 0; j < k; j++) {
    ids[(size_t)t * k + j] = ok ? table[(size_t)v * k + j] : -1;
    w[(size_t)t * k + j] = ok ? wk : 0.0f;
  }
}

cudaError_t launch_route(const ds4moe_layer *h, const float *x, const int32_t *tok, int T, int32_t *ids,
                         float *w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const ds4moe_layer_desc &d = h->d;
  if (d.route == DS4MOE_ROUTE_HASH) {
    k_hash<<<(T + 127) / 128, 128, 0, s>>>(tok, h->hash, T, d.top_k, d.vocab, d.route_scale, ids, w, h->err);
    return cudaGetLastError();
  }
  if (d.router_fmt == DS4MOE_Q8_0) {
    dim3 grid(h->E_pad / 32, ROUTER_SEGS, (T + RT - 1) / RT);
    k_router_q8<<<grid, 32, 0, s>>>(h->router, d.hidden, h->E_pad, h->xq, h->dx, T, h->rpart);
  } else {
    dim3 grid(h->E_pad / 32, ROUTER_SEGS, T);
    k_router_f32<<<grid, 32, 0, s>>>((const float *)h->router, d.hidden, d.n_experts, h->E_pad, x, h->rpart);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)d.n_experts * 12;
  k_topk<<<T, 32, smem, s>>>(h->rpart, h->bias, d.n_experts, h->E_pad, d.top_k, d.route_scale, ids, w);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bucketing (one CTA): per-expert counts and offsets, the (token, slot) list
// of every expert, and the active-expert list (shared expert first, then
// routed experts in ascending id). List order within an expert does not
// affect any result: every (token, slot) is computed on its own.
__global__ void __launch_bounds__(1024) k_bucket(const int32_t *__restrict__ ids, int T, int E, int k, int NS,
                                                 int n_shared, int32_t *cnt_g, int32_t *off_g, int32_t *act_g,
                                                 int32_t *nact_g, int32_t *list, uint32_t *err) {
  extern __shared__ int32_t smb[];
  int32_t *cnt = smb, *off = smb + (E + 1), *cur = off + (E + 2);
  const int tid = threadIdx.x, nth = blockDim.x;
  for (int e = tid; e <= E; e += nth) cnt[e] = 0, cur[e] = 0;
  __syncthreads();
  const int n = T * k;
  for (int i = tid; i < n; i += nth) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else if (e >= E) raise_flag(err, DS4MOE_DEVERR_INTERNAL);
  }
  __syncthreads();
  if (tid == 0) {
    cnt[E] = n_shared ? T : 0;
    int o = 0, na = 0;
    if (n_shared) act_g[na++] = E;
    for (int e = 0; e <= E; e++) {
      off[e] = o;
      o += cnt[e];
      if (e < E && cnt[e] > 0) act_g[na++] = e;
    }
    off[E + 1] = o;
    *nact_g = na;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += nth) cnt_g[e] = cnt[e], off_g[e] = off[e];
  if (tid == 0) off_g[E + 1] = off[E + 1];
  for (int i = tid; i < n; i += nth) {
    const int e = ids[i];
    if (e >= 0 && e < E) {
      const int p = atomicAdd(&cur[e], 1);
      list[off[e] + p] = (i / k) * NS + (i % k);
    }
  }
  if (n_shared)
    for (int t = tid; t < T; t += nth) list[off[E] + t] = t * NS + k;
}

cudaError_t launch_bucket(const ds4moe_layer *h, int T, cudaStream_t s) {
  const int E = h->d.n_experts;
  Bucket b = bucket_view(h);
  const size_t smem = sizeof(int32_t) * (size_t)(3 * E + 4);
  k_bucket<<<1, 1024, smem, s>>>(h->ids, T, E, h->d.top_k, h->NS, h->d.n_shared, b.cnt, b.off, b.active,
                                 b.n_active, b.list, h->err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// CAS step 7: y[r] = y[r] + ((sum_j w_j * a_j[r]) + a_shared[r]).
__global__ void __launch_bounds__(256) k_combine(const float *__restrict__ apart, const int32_t *__restrict__ ids,
                                                 const float *__restrict__ w, int H, int k, int NS, int n_shared,
                                                 float *__restrict__ y) {
  const int t = blockIdx.y, r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= H || ids[(size_t)t * k] < 0) return;
  float acc = 0.0f;
  for (int j = 0; j < k; j++)
    acc = __fadd_rn(acc, __fmul_rn(w[(size_t)t * k + j], apart[((size_t)t * NS + j) * H + r]));
  if (n_shared) acc = __fadd_rn(acc, apart[((size_t)t * NS + k) * H + r]);
  y[(size_t)t * H + r] = __fadd_rn(y[(size_t)t * H + r], acc);
}

cudaError_t launch_combine(const ds4moe_layer *h, int T, float *y, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 grid((h->d.hidden + 255) / 256, T);
  k_combine<<<grid, 256, 0, s>>>(h->apart, h->ids, h->wts, h->d.hidden, h->d.top_k, h->NS, h->d.n_shared, y);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// CAS step 8: one warp per row; lane l owns the l-th of 32 contiguous
// segments (fma chain), the 32 segment sums are then added in order.
__global__ void __launch_bounds__(32) k_rmsnorm(const float *x, float *out, int H, float eps) {
  const int t = blockIdx.x, lane = threadIdx.x, per = H >> 5;
  const float *v = x + (size_t)t * H;
  float acc = 0.0f;
  for (int i = lane * per; i < (lane + 1) * per; i++) acc = __fmaf_rn(v[i], v[i], acc);
  float ss = 0.0f;
  for (int l = 0; l < 32; l++) ss = __fadd_rn(ss, __shfl_sync(0xffffffffu, acc, l));
  const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
  __syncwarp();
  for (int i = lane; i < H; i += 32) out[(size_t)t * H + i] = __fmul_rn(v[i], inv);
}

cudaError_t launch_rmsnorm(const float *x, float *out, int T, int H, float eps, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_rmsnorm<<<T, 32, 0, s>>>(x, out, H, eps);
  return cudaGetLastError();
}

}  // namespace ds4

// internal.h -- the layer handle and the kernel launchers shared by the
// translation units of libds4moe.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "ds4moe.h"

constexpr int DS4_HOST_GRAPHS = 65;  // decode chunk sizes 1..64 (DEC_MAX_T) + 1

struct ds4moe_layer {
  ds4moe_layer_desc d;
  int device;
  int E_pad;   // router rows padded to a multiple of 32
  int NS;      // expert slots per token: top_k + n_shared
  int A_max;   // most active experts in one call: min(E, max_tokens*k) + n_shared
  int n_sm;    // streaming multiprocessors of the device
  int Tc;      // tokens per decode chunk: min(max_tokens, DEC_MAX_T)
  int Tp;      // tokens per prefill chunk: min(max_tokens, PF_MAX_T), 0 without the prefill path
  int Ts;      // scratch rows: max(Tc, Tp)
  int pf_min;  // calls with at least this many tokens take the prefill path

  // Weights in the library's layout (see common.cuh).
  uint8_t *router;       // Q8 RG32 [E_pad/32][H/64][tile], or F32 [E][H]
  float *bias;           // [E]
  int32_t *hash;         // [vocab][k]
  uint8_t *gu;           // routed gate+up [E][F/32][H/KSTEP][2][tile]
  uint8_t *dn;           // routed down    [E][H/32][F/KSTEP][2][tile] (16-row halves)
  uint8_t *sgu, *sdn;    // shared, same layouts with E = 1

  // Scratch for Ts tokens (one chunk of either path).
  int8_t *xq;            // [T][H]
  float *dx;             // [T][H/32]
  int16_t *gs;           // [T][H/16]
  int32_t *ids;          // [T][k]
  float *wts;            // [T][k]
  int32_t *bucket;       // per-expert table of the chunk (bucket.cuh): header, act[A_max], list[Tc*NS]
  int8_t *hq;            // [T*NS][F]
  float *dh;             // [T*NS][F/32]
  int16_t *gsh;          // [T*NS][F/16]
  float *apart;          // [T*NS][H]
  uint32_t *err;         // device error flags
  float *hbuf;           // [Tc*NS][F] SwiGLU values before requant
  int32_t *hticket;      // [Tc*NS][F/32] requant tickets (self-resetting)
  int32_t *cticket;      // [Tc][H/32] combine tickets (self-resetting)
  int32_t *rticket;      // router-kernel ticket of the call (self-resetting)
  int32_t *xq_ready;     // decode: router blocks whose codes of x are written (cleared by down)
  int32_t *pf_meta;      // prefill: [E+1][2] {pairs, list offset} per group (0 shared, 1+e routed)
  int32_t *pf_pass;      // prefill: [E+2] first pass of each group, then the total
  int32_t *pf_list;      // prefill: [Tp*k + Tp] pair codes (token << 5) | slot, grouped
  float *xnorm;          // [H] the normalised row of a one-token ds4moe_forward_rmsnorm call

  // Staging for ds4moe_forward_host.
  float *x_dev, *y_dev;
  int32_t *tok_dev;
  // Decode-sized ds4moe_forward_host calls replay one CUDA graph per token
  // count (the copies through these pinned buffers and the forward's
  // launches), captured on first use.
  float *x_pin, *y_pin;
  int32_t *tok_pin;
  cudaStream_t cap_stream;
  cudaGraphExec_t host_graph[DS4_HOST_GRAPHS];   // by token count, 1 .. decode chunk
  int64_t host_graph_launches[DS4_HOST_GRAPHS];   // kernels one replay launches
  int host_graph_off;                              // capture failed once: plain copies and launches

  // Profiling (ds4moe_profile_*) and launch counting.
  int prof_on;
  cudaEvent_t ev[8];
  int ev_made;
  double prof_ms[8];
  int64_t prof_calls;
  uint64_t launches;

  long long wait_limit;  // hand-off wait bound of the decode expert kernels (0: WAIT_LIMIT)

  uint64_t bytes;        // total device bytes owned
  void *allocs[40];
  int n_allocs;
};

namespace ds4 {

// repack.cu
cudaError_t repack_q2s(const uint8_t *src, uint8_t *dst, int n_mat, int rows, int K, int pair, int which,
                       cudaStream_t s);
cudaError_t repack_q8(const uint8_t *src, uint8_t *dst, int n_mat, int rows, int K, int pair, int which,
                      cudaStream_t s, bool swz = false);
cudaError_t repack_q4s(const uint8_t *src, uint8_t *dst, int n_mat, int rows, int K, int pair, int which,
                       cudaStream_t s);
cudaError_t repack_rq8(const uint8_t *src, uint8_t *dst, int rows, int rows_pad, int K, cudaStream_t s);
cudaError_t check_hash_table(const int32_t *table, int64_t n, int E, int32_t *bad_count, cudaStream_t s);

// rmsnorm.cu
cudaError_t launch_rmsnorm(const float *x, float *out, int T, int H, float eps, cudaStream_t s);

// decode.cu
constexpr int DEC_MAX_T = 64;  // largest n_tok served by the decode path
static_assert(DS4_HOST_GRAPHS == DEC_MAX_T + 1, "one forward_host graph per decode chunk size");
size_t route_dec_smem(const ds4moe_layer *h);
// Capacity of the bucket table's expert list for a decode call of T tokens:
// min(E, T*k) + n_shared (at most A_max). The router and both expert kernels
// of a call lay the table out with it, so a small call's table (and the
// expert kernels' shared-memory copy of it) stays small.
inline int bucket_cap(const ds4moe_layer *h, int T) {
  const long long routed = (long long)T * h->d.top_k;
  const int c = (int)(routed < h->d.n_experts ? routed : h->d.n_experts) + h->d.n_shared;
  return c < h->A_max ? c : h->A_max;
}
cudaError_t launch_dec_route(const ds4moe_layer *h, const float *x, const int32_t *tok, int T, int32_t *ids,
                             float *w, bool bucket, cudaStream_t s, bool norm = false, float eps = 0.0f);
cudaError_t launch_pdl(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args, bool pdl);

// prefill.cu
constexpr int PF_MAX_T = 4096;       // largest prefill chunk
constexpr int PF_MIN_T_DEFAULT = 65; // smallest call that takes the prefill path
bool prefill_supported(const ds4moe_layer_desc &d);
cudaError_t prefill_set_attributes();
size_t prefill_list_ints(int T, int k, int n_shared);
cudaError_t launch_prefill(ds4moe_layer *h, const float *x, const int32_t *tok, int T, float *y, cudaStream_t s,
                           cudaEvent_t *ev, bool norm = false, float eps = 0.0f);

// experts.cu
size_t experts_smem(const ds4moe_layer *h);
cudaError_t launch_experts(const ds4moe_layer *h, int T, float *y, int down, cudaStream_t s);
cudaError_t experts_set_attributes();
cudaError_t decode_set_attributes();
constexpr size_t DEC_SMEM_LIMIT = 227 * 1024;

}  // namespace ds4

// rmsnorm.cu -- RMSNorm with unit gain between stacked layers (the final norm
// of the "DeepSeek V4 Flash -- DFlash Integration" page, Forward Pass step 5,
// applied between layers of a stack of MoE FFNs).
#include "common.cuh"
#include "internal.h"

namespace ds4 {

constexpr int RN_THREADS = 256;
constexpr int RN_MAX_H = 8192;  // rows staged whole in shared memory up to this width

// CAS step 8: lane l of warp 0 owns the l-th of 32 contiguous segments (fma
// chain in element order), the 32 segment sums are then added in order.
// One block per row: the row is loaded coalesced into shared memory, each
// segment padded by one word so that the 32 chains read 32 different banks.
// Launched with programmatic dependent launch: the row is read only after
// the previous kernel of the stream has completed, and the next kernel may
// start launching at once.
__global__ void __launch_bounds__(RN_THREADS) k_rmsnorm(const float *x, float *out, int H, float eps) {
  __shared__ float row[RN_MAX_H + 32];
  __shared__ float s_inv;
  const int t = blockIdx.x, per = H >> 5;
  const float *v = x + (size_t)t * H;
  pdl_launch_dependents();
  pdl_wait();
  for (int i = threadIdx.x; i < H; i += RN_THREADS) row[i + i / per] = v[i];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const float *seg = row + lane * (per + 1);
    float acc = 0.0f;
    int i = 0;
    for (; i + 8 <= per; i += 8) {
      float r[8];
#pragma unroll
      for (int j = 0; j < 8; j++) r[j] = seg[i + j];
#pragma unroll
      for (int j = 0; j < 8; j++) acc = __fmaf_rn(r[j], r[j], acc);
    }
    for (; i < per; i++) acc = __fmaf_rn(seg[i], seg[i], acc);
    float ss = 0.0f;
    for (int l = 0; l < 32; l++) ss = __fadd_rn(ss, __shfl_sync(0xffffffffu, acc, l));
    if (lane == 0) s_inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)H), eps)));
  }
  __syncthreads();
  const float inv = s_inv;
  for (int i = threadIdx.x; i < H; i += RN_THREADS) out[(size_t)t * H + i] = __fmul_rn(row[i + i / per], inv);
}

// Rows wider than RN_MAX_H: one warp per row straight from global memory.
__global__ void __launch_bounds__(32) k_rmsnorm_wide(const float *x, float *out, int H, float eps) {
  const int t = blockIdx.x, lane = threadIdx.x, per = H >> 5;
  const float *v = x + (size_t)t * H;
  pdl_launch_dependents();
  pdl_wait();
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
  void *args[] = {(void *)&x, (void *)&out, (void *)&H, (void *)&eps};
  if (H <= RN_MAX_H) return launch_pdl((const void *)k_rmsnorm, dim3(T), dim3(RN_THREADS), 0, s, args, true);
  return launch_pdl((const void *)k_rmsnorm_wide, dim3(T), dim3(32), 0, s, args, true);
}

}  // namespace ds4

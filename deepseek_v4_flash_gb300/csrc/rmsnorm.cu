// rmsnorm.cu -- RMSNorm with unit gain between stacked layers (the final norm
// of the "DeepSeek V4 Flash -- DFlash Integration" page, Forward Pass step 5,
// applied between layers of a stack of MoE FFNs).
#include "common.cuh"
#include "internal.h"

namespace ds4 {

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

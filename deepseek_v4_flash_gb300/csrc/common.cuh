// common.cuh -- shared device helpers for libds4moe (sm_103a).
//
// 1. The canonical arithmetic spec (CAS) as device functions. Every binary32
//    operation on the numeric path goes through __fadd_rn / __fmul_rn /
//    __fmaf_rn / __fdiv_rn / __fsqrt_rn, which the compiler never contracts
//    or reorders, so results are bit-identical to a scalar CPU evaluation of
//    the same spec.
// 2. The library's internal weight layouts (16 rows per tile, two lanes per
//    row).
// 3. PTX wrappers for mbarriers and 1-D bulk async copies (cp.async.bulk)
//    with bounded waits.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ds4moe.h"

namespace ds4 {

// ---------------------------------------------------------------------------
// Internal layouts ("RG16": 16 rows per tile, two lanes per row; lane
// l = 2r + h serves row r with half h of the work, so a warp reads 512
// contiguous bytes per 16-byte load and the two lanes of a row add their
// exact integer partial dots with one shuffle).
//
// Q2S RG16 tile = 16 rows x one superblock (256 K), 1344 bytes. Lane
// l = 2r + h owns blocks h, h+2, h+4, h+6 of row r (both 16-weight groups of
// each block):
//   [0,256)     sm8: lane l -> 8 bytes: the scale/min nibble bytes of groups
//               2b, 2b+1 for b = h, h+2, h+4, h+6, in that order
//   [256,320)   dd:  row r -> 4 bytes at 4r (fp16 d, fp16 dmin)
//   [320,1344)  qs:  2 chunks c x 32 lanes x 16 bytes: lane l, chunk c holds
//               the group words of its blocks h+4c and h+4c+2 (groups 2b,
//               2b+1 each), each word's 2-bit fields transposed so that
//               ((W >> 2s) & 0x03030303) yields q[4s .. 4s+3] of the group
//               in element order (one dp4a against 4 consecutive int8 x).
// Q4S RG16 tile = 16 rows x one 4-bit superblock (256 K), 2368 bytes, the
// Q2S layout with 4-bit fields: [0,256) sm8 and [256,320) dd as for Q2S;
// [320,2368) qs: 4 chunks c x 32 lanes x 16 bytes: lane l, chunk c holds the
// four group words of its block h + 2c (group 2b: elements 0-7, 8-15; group
// 2b+1 the same), each word's nibbles transposed so that (W & 0x0F0F0F0F)
// yields elements 0-3 of its eight and ((W >> 4) & 0x0F0F0F0F) elements 4-7.
// Q8 RG16 tile = 16 rows x one Q8_0 block (32 K), 544 bytes:
//   [0,32)      d: row r -> fp16 at 2r
//   [32,544)    q: lane l -> 16 bytes: row r, elements 16h .. 16h+15
// Router Q8 rows use a 32-row, 2-block layout (RQ8): 32 rows x 64 K, 2176
// bytes: [0,128) d: lane l -> 4 bytes (fp16 d of block 0, block 1);
// [128,2176) q: 4 pieces m x 32 lanes x 16 bytes; piece m = block m/2,
// elements 16*(m%2) .. 16*(m%2)+15.
// Gate and up of the same expert are interleaved per K-step:
// [F/16][H/KSTEP][2][tile]; a down matrix interleaves the two 16-row halves
// of every 32 rows per K-step: [H/32][F/KSTEP][2][tile]. Either way one
// K-step of a work item is two consecutive tiles.
constexpr int TILE_ROWS = 16;
constexpr int Q2S_TILE = 1344, Q2S_SM = 0, Q2S_DD = 256, Q2S_QS = 320, Q2S_KSTEP = 256;
constexpr int Q4S_TILE = 2368, Q4S_SM = 0, Q4S_DD = 256, Q4S_QS = 320, Q4S_KSTEP = 256;
constexpr int Q8_TILE = 544, Q8_Q = 32, Q8_KSTEP = 32;
constexpr int RQ8_TILE = 2176, RQ8_Q = 128, RQ8_KSTEP = 64;

__host__ __device__ constexpr int tile_bytes(int fmt) {
  return fmt == DS4MOE_Q2S ? Q2S_TILE : fmt == DS4MOE_Q4S ? Q4S_TILE : Q8_TILE;
}
__host__ __device__ constexpr int kstep(int fmt) { return fmt == DS4MOE_Q8_0 ? Q8_KSTEP : Q2S_KSTEP; }

// Row-sum segments (CAS step 4): router rows 8; expert rows
// min(EXPERT_SEGS, K-steps of the row), a K-step being one superblock (Q2S,
// Q4S) or one block (Q8_0).
constexpr int ROUTER_SEGS = 8;
constexpr int EXPERT_SEGS = 8;
__host__ __device__ constexpr int expert_segs(int fmt, int K) {
  return K / kstep(fmt) < EXPERT_SEGS ? K / kstep(fmt) : EXPERT_SEGS;
}

// ---------------------------------------------------------------------------
// CAS device math.

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xFFFFu)));
}

// cas_exp: Cody & Waite reduction with ln2 split into a 16-bit head and a
// binary32 tail, then a degree-7 Taylor polynomial in fma Horner form, then
// scaling by 2^n built from exponent bits. Constants: log2(e), the head/tail
// of ln2, and 1/k! for k = 2..7, each rounded to binary32.
__device__ __forceinline__ float cas_exp(float z) {
  if (z != z) return z;
  z = z < -87.0f ? -87.0f : z;
  z = z > 88.0f ? 88.0f : z;
  const float n = rintf(__fmul_rn(z, 0x1.715476p+0f));
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, z);
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0x1p-1f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const float s = __int_as_float(((int)n + 127) << 23);
  return __fmul_rn(p, s);
}

__device__ __forceinline__ float cas_sigmoid(float z) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, cas_exp(-z)));
}

__device__ __forceinline__ float cas_silu(float g) {
  return __fdiv_rn(g, __fadd_rn(1.0f, cas_exp(-g)));
}

// int8 code of v for scale d (CAS step 1): round half away, clamp +-127.
__device__ __forceinline__ int cas_code(float v, float d) {
  if (d == 0.0f) return 0;
  float r = roundf(__fdiv_rn(v, d));
  r = r > 127.0f ? 127.0f : r;
  r = r < -127.0f ? -127.0f : r;
  return (r == r) ? (int)r : 0;
}

// Q2S block term (CAS step 3): dx * fma(d, A, -(dmin * B)).
__device__ __forceinline__ float q2s_term(float dx, float d, float dmin, int A, int B) {
  const float m = __fmul_rn(dmin, __int2float_rn(B));
  return __fmul_rn(dx, __fmaf_rn(d, __int2float_rn(A), -m));
}

// Q8_0 block term (CAS step 3): (d * dx) * I.
__device__ __forceinline__ float q8_term(float d, float dx, int I) {
  return __fmul_rn(__fmul_rn(d, dx), __int2float_rn(I));
}

// Two binary32 lanes per instruction (sm_100+ packed forms). Each lane is
// one correctly rounded operation, exactly as the scalar form: the packed
// forms change the instruction count, not the arithmetic.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float &lo, float &hi) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---------------------------------------------------------------------------
// Warp helpers.

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int half_warp_sum(int v) {
#pragma unroll
  for (int o = 8; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int dot16(uint4 w, uint4 x, int acc) {
  acc = __dp4a((int)w.x, (int)x.x, acc);
  acc = __dp4a((int)w.y, (int)x.y, acc);
  acc = __dp4a((int)w.z, (int)x.z, acc);
  acc = __dp4a((int)w.w, (int)x.w, acc);
  return acc;
}

// ---------------------------------------------------------------------------
// mbarrier + bulk async copy (global -> shared), non-multicast.

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One bounded test of the phase: try_wait without a suspend-time hint lets
// the hardware suspend the warp for its own short default interval only.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test with a suspend-time hint: the warp is parked (issuing
// nothing) until the phase completes or about MBAR_SUSPEND_NS pass.
constexpr uint32_t MBAR_SUSPEND_NS = 20000;
__device__ __forceinline__ bool mbar_try_wait_parked(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(MBAR_SUSPEND_NS)
      : "memory");
  return ok != 0;
}

// The bound of every on-chip wait: ~2^31 SM cycles (about a second).
constexpr long long WAIT_LIMIT = 1ll << 31;

// Bounded wait: gives up after `limit` SM cycles and returns false; callers
// then raise DS4MOE_DEVERR_TIMEOUT and leave. Between tests the warp is
// parked by the hardware, so waiting warps take no issue slots from the
// working ones and wake as soon as the phase completes.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit = WAIT_LIMIT) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_parked(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// Programmatic dependent launch: wait for the previous kernel's completion
// (and memory), and let the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// A count in global memory shared by the kernels of one call: arrivals with
// release semantics, a bounded wait with acquire semantics.
__device__ __forceinline__ void red_release_gpu_add(int32_t *p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Waits until *p >= target; false after `limit` cycles.
__device__ __forceinline__ bool wait_count(const int32_t *p, int target, long long limit = WAIT_LIMIT) {
  const long long t0 = clock64();
  while (ld_acquire_gpu(p) < target) {
    if (clock64() - t0 > limit) return false;
    __nanosleep(32);
  }
  return true;
}

__device__ __forceinline__ void raise_flag(uint32_t *err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 ld_shared_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

}  // namespace ds4

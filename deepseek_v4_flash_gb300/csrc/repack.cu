// repack.cu -- create-time conversion of the canonical weight bytes into the
// library's layouts (RG16 for expert matrices, RQ8 for the router; see
// common.cuh). Runs once per layer handle.
#include "common.cuh"
#include "internal.h"

namespace ds4 {

// Tile of 16-row group rg, K-step s of matrix m. npair 1: one matrix;
// npair 2: two matrices interleaved per K-step (gate, up: which = 0, 1);
// npair 3: the two 16-row groups of each 32-row group interleaved per K-step
// (which = rg & 1).
__device__ __forceinline__ int64_t tile_index(int m, int rows, int rg, int KS, int s, int npair, int which) {
  if (npair == 3) return ((((int64_t)m * (rows >> 5) + (rg >> 1)) * KS + s) * 2 + (rg & 1));
  return (((int64_t)m * (rows >> 4) + rg) * KS + s) * npair + which;
}

// One thread per canonical Q2S superblock (84 bytes) -> its two lanes'
// slices of an RG16 tile (common.cuh). Lane 2r + h owns blocks h + 2j
// (j = 0..3), both groups of each. The 2-bit fields of each 16-weight group
// are transposed: canonical element 4*s+j of the group (byte s of the group,
// bits 2j) moves to byte j, bits 2s of the group word, so (W >> 2s) &
// 0x03030303 gives 4 consecutive elements in byte order.
__global__ void k_repack_q2s(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int n_mat, int rows,
                             int KS, int npair, int which) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)n_mat * rows * KS;
  if (i >= total) return;
  const int s = (int)(i % KS);
  const int64_t mr = i / KS;
  const int r = (int)(mr % rows), m = (int)(mr / rows);
  const uint8_t *sb = src + i * 84;
  const int rg = r >> 4, rr = r & 15;
  uint8_t *tile = dst + tile_index(m, rows, rg, KS, s, npair, which) * Q2S_TILE;
  for (int j = 0; j < 4; j++) tile[Q2S_DD + 4 * rr + j] = sb[80 + j];
  for (int h = 0; h < 2; h++) {
    const int lane = 2 * rr + h;
    for (int j = 0; j < 4; j++) {
      const int b = h + 2 * j;
      for (int gi = 0; gi < 2; gi++) {
        const int g = 2 * b + gi;
        tile[Q2S_SM + 8 * lane + 2 * j + gi] = sb[g];
        uint32_t W = 0;
        for (int sbyte = 0; sbyte < 4; sbyte++) {
          const uint32_t v = sb[16 + 4 * g + sbyte];
          for (int e = 0; e < 4; e++) W |= ((v >> (2 * e)) & 3u) << (8 * e + 2 * sbyte);
        }
        uint8_t *o = tile + Q2S_QS + 512 * (j >> 1) + 16 * lane + 4 * (2 * (j & 1) + gi);
        o[0] = (uint8_t)W, o[1] = (uint8_t)(W >> 8), o[2] = (uint8_t)(W >> 16), o[3] = (uint8_t)(W >> 24);
      }
    }
  }
}

// One thread per canonical Q4S superblock (148 bytes) -> its two lanes'
// slices of a 4-bit RG16 tile (common.cuh). Lane 2r + h owns blocks h + 2c
// (c = 0..3), both groups of each; a group's 16 nibbles become two words,
// canonical element j (and j + 4) of each eight at byte j of the word, low
// (and high) nibble.
__global__ void k_repack_q4s(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int n_mat, int rows,
                             int KS, int npair, int which) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)n_mat * rows * KS;
  if (i >= total) return;
  const int s = (int)(i % KS);
  const int64_t mr = i / KS;
  const int r = (int)(mr % rows), m = (int)(mr / rows);
  const uint8_t *sb = src + i * 148;
  const int rg = r >> 4, rr = r & 15;
  uint8_t *tile = dst + tile_index(m, rows, rg, KS, s, npair, which) * Q4S_TILE;
  for (int j = 0; j < 4; j++) tile[Q4S_DD + 4 * rr + j] = sb[144 + j];
  for (int h = 0; h < 2; h++) {
    const int lane = 2 * rr + h;
    for (int c = 0; c < 4; c++) {
      const int b = h + 2 * c;
      for (int gi = 0; gi < 2; gi++) {
        const int g = 2 * b + gi;
        tile[Q4S_SM + 8 * lane + 2 * c + gi] = sb[g];
        for (int half = 0; half < 2; half++) {  // elements 8*half .. 8*half+7 of the group
          uint32_t W = 0;
          for (int j = 0; j < 4; j++) {
            const int e0 = 16 * g + 8 * half + j, e1 = e0 + 4;
            const uint32_t q0 = (sb[16 + (e0 >> 1)] >> (4 * (e0 & 1))) & 15u;
            const uint32_t q1 = (sb[16 + (e1 >> 1)] >> (4 * (e1 & 1))) & 15u;
            W |= (q0 | (q1 << 4)) << (8 * j);
          }
          uint8_t *o = tile + Q4S_QS + 512 * c + 16 * lane + 4 * (2 * gi + half);
          o[0] = (uint8_t)W, o[1] = (uint8_t)(W >> 8), o[2] = (uint8_t)(W >> 16), o[3] = (uint8_t)(W >> 24);
        }
      }
    }
  }
}

// Expert Q8_0 -> RG16: one thread per canonical block (34 bytes). swz: the
// two 16-byte halves of rows 4-7 and 12-15 of a tile trade places, so that
// eight consecutive rows' halves at a 32-byte row stride fall in 32
// different banks (ldmatrix and 16-byte loads without conflicts).
__global__ void k_repack_q8(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int n_mat, int rows,
                            int KS, int npair, int which, int swz) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)n_mat * rows * KS;
  if (i >= total) return;
  const int c = (int)(i % KS);
  const int64_t mr = i / KS;
  const int r = (int)(mr % rows), m = (int)(mr / rows);
  const uint8_t *b = src + i * 34;
  const int rg = r >> 4, rr = r & 15;
  uint8_t *tile = dst + tile_index(m, rows, rg, KS, c, npair, which) * Q8_TILE;
  tile[2 * rr + 0] = b[0], tile[2 * rr + 1] = b[1];
  const int hs = swz ? (rr >> 2) & 1 : 0;
  for (int h = 0; h < 2; h++)
    for (int j = 0; j < 16; j++) tile[Q8_Q + 16 * (2 * rr + (h ^ hs)) + j] = b[2 + 16 * h + j];
}

// Router Q8_0 -> RQ8: one thread per pair of canonical blocks (2 x 34 bytes);
// rows beyond `rows` (up to rows_pad) stay zero.
__global__ void k_repack_rq8(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst, int rows, int rows_pad,
                             int KS) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)rows * KS;
  if (i >= total) return;
  const int c = (int)(i % KS);
  const int r = (int)(i / KS);
  const uint8_t *b0 = src + (int64_t)r * ((int64_t)KS * 68) + (int64_t)c * 68;
  const uint8_t *b1 = b0 + 34;
  const int rg = r >> 5, lane = r & 31;
  uint8_t *tile = dst + ((int64_t)rg * KS + c) * RQ8_TILE;
  (void)rows_pad;
  tile[4 * lane + 0] = b0[0], tile[4 * lane + 1] = b0[1];
  tile[4 * lane + 2] = b1[0], tile[4 * lane + 3] = b1[1];
  for (int p = 0; p < 4; p++) {
    const uint8_t *q = (p < 2 ? b0 : b1) + 2 + 16 * (p & 1);
    uint8_t *o = tile + RQ8_Q + 512 * p + 16 * lane;
    for (int j = 0; j < 16; j++) o[j] = q[j];
  }
}

__global__ void k_check_table(const int32_t *__restrict__ t, int64_t n, int E, int32_t *bad) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n && (t[i] < 0 || t[i] >= E)) atomicAdd(bad, 1);
}

static unsigned blocks_for(int64_t n, int threads) { return (unsigned)((n + threads - 1) / threads); }

cudaError_t repack_q2s(const uint8_t *src, uint8_t *dst, int n_mat, int rows, int K, int pair, int which,
                       cudaStream_t s) {
  const int KS = K / Q2S_KSTEP;
  const int64_t n = (int64_t)n_mat * rows * KS;
  if (n == 0) return cudaSuccess;
  k_repack_q2s<<<blocks_for(n, 256), 256, 0, s>>>(src, dst, n_mat, rows, KS, pair == 2 ? 3 : pair ? 2 : 1, which);
  return cudaGetLastError();
}

cudaError_t repack_q4s(const uint8_t *src, uint8_t *dst, int n_mat, int rows, int K, int pair, int which,
                       cudaStream_t s) {
  const int KS = K / Q4S_KSTEP;
  const int64_t n = (int64_t)n_mat * rows * KS;
  if (n == 0) return cudaSuccess;
  k_repack_q4s<<<blocks_for(n, 256), 256, 0, s>>>(src, dst, n_mat, rows, KS, pair == 2 ? 3 : pair ? 2 : 1, which);
  return cudaGetLastError();
}

cudaError_t repack_q8(const uint8_t *src, uint8_t *dst, int n_mat, int rows, int K, int pair, int which,
                      cudaStream_t s, bool swz) {
  const int KS = K / Q8_KSTEP;
  const int64_t n = (int64_t)n_mat * rows * KS;
  if (n == 0) return cudaSuccess;
  k_repack_q8<<<blocks_for(n, 256), 256, 0, s>>>(src, dst, n_mat, rows, KS, pair == 2 ? 3 : pair ? 2 : 1, which,
                                                 swz ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t repack_rq8(const uint8_t *src, uint8_t *dst, int rows, int rows_pad, int K, cudaStream_t s) {
  const int KS = K / RQ8_KSTEP;
  const int64_t n = (int64_t)rows * KS;
  if (n == 0) return cudaSuccess;
  k_repack_rq8<<<blocks_for(n, 256), 256, 0, s>>>(src, dst, rows, rows_pad, KS);
  return cudaGetLastError();
}

cudaError_t check_hash_table(const int32_t *table, int64_t n, int E, int32_t *bad_count, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  k_check_table<<<blocks_for(n, 256), 256, 0, s>>>(table, n, E, bad_count);
  return cudaGetLastError();
}

}  // namespace ds4

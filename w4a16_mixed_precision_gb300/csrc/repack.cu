// repack.cu -- offline rewrite of GPTQ-order 4-bit codes, scales and zeros into
// the layouts the fused kernels stream, dense and 2:4-sparse ("Marlin /
// GPTQ-Marlin", section "Tiled layout et repacking"; "Marlin Project
// Overview", section "Key Techniques", item "Reshuffling for Access
// Patterns").  It runs once per weight, at load time.  The codes are laid out
// per lane fragment, so that one 16-byte shared load per lane feeds the MMA.
//
// Code layout: for every 128-column tile nt and 64-row block kb, one 4 KB chunk
// of 32-bit words [g = 0..7][l = 0..31][j = 0..3].  Word (g, l, j) carries the
// sixteen-by-sixteen fp16 operand fragment that lane l of a warp holds for
// columns 16g.. of the tile and rows 16j.. of the block: with r = l/4 and
// c = l%4, nibble p is column 16g + r + 8(p&1), row 16j + 4c + 2((p>>1)&1) + (p>>2).
// So one AND with 0x000F000F (after an optional 8-bit shift) yields the fp16
// pair of two consecutive rows of one column, and the four pairs of a word are,
// in order, the lane's fragment registers.  A lane reads its four words of a
// 64-row block as one 16-byte shared-memory load.
//
// Scales [G][N] -> [N/128][G][128] and zeros [G][N/8 words] -> [N/128][G][64
// bytes]: all groups of one column tile are contiguous, so a K-slice of a tile
// needs one copy for its scales and one for its zeros.
#include "kernels.h"

namespace w4a16 {

namespace {

// The multiply kernels may start reading the weights before their dependency
// wait (they treat the weights as constant), which a kernel that simply ends
// does not order against its own last stores.  Every repack thread therefore
// makes its stores visible device-wide before it exits, so a multiply enqueued
// right after a repack on the same stream reads the finished layout.
__device__ __forceinline__ void publish_before_exit() { __threadfence(); }

__global__ void repack_codes_kernel(const uint32_t* __restrict__ q, uint32_t* __restrict__ out, int K,
                                    int N, long long total) {
  const int KB = K / 64;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(t & 3);
    const int l = (int)((t >> 2) & 31);
    const int g = (int)((t >> 7) & 7);
    const long long chunk = t >> 10;
    const int kb = (int)(chunk % KB);
    const int nt = (int)(chunk / KB);
    const int n0 = nt * 128 + 16 * g + (l >> 2);
    const int k0 = kb * 64 + 16 * j + 4 * (l & 3);  // four consecutive rows k0..k0+3
    const size_t src_row = (size_t)(k0 >> 3) * N;
    const int shift = (k0 & 7) * 4;                  // 0 or 16
    const uint32_t a = (q[src_row + n0] >> shift) & 0xFFFFu;      // column n0, rows k0..k0+3
    const uint32_t b = (q[src_row + n0 + 8] >> shift) & 0xFFFFu;  // column n0 + 8
    // nibble p <- row offset 2((p>>1)&1) + (p>>2) of column n0 (p even) or n0+8 (p odd)
    uint32_t w = 0;
    w |= (a & 0xFu) | ((b & 0xFu) << 4);                    // p0, p1: row +0
    w |= ((a >> 8) & 0xFu) << 8 | ((b >> 8) & 0xFu) << 12;  // p2, p3: row +2
    w |= ((a >> 4) & 0xFu) << 16 | ((b >> 4) & 0xFu) << 20; // p4, p5: row +1
    w |= ((a >> 12) & 0xFu) << 24 | ((b >> 12) & 0xFu) << 28; // p6, p7: row +3
    out[t] = w;
  }
  publish_before_exit();
}

// Rows of `row_vec` 16-byte vectors: src [G][NT][row] -> dst [NT][G][row].
__global__ void tile_major_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int G, int NT,
                                  int row_vec) {
  const long long total = (long long)G * NT * row_vec;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int v = (int)(t % row_vec);
    const long long r = t / row_vec;
    const int nt = (int)(r % NT);
    const int gi = (int)(r / NT);
    dst[((long long)nt * G + gi) * row_vec + v] = src[t];
  }
  publish_before_exit();
}

// ---- 2:4 sparsity ("Marlin", section "支持 2:4 稀疏加速": two of every four
// weights zero at fixed positions) ----
//
// A weight is zero when its code equals the zero point.  In a group of four
// consecutive rows of a column the kept rows are those whose code differs
// from the zero point (the first two if there are more, which the caller is
// told through *bad), completed with the lowest remaining rows; their index
// pair i0 < i1 is the nibble i0 | i1 << 2, the metadata of a sparse
// tensor-core operand.
//
// Sparse tile layout, per 128-column tile nt and 64-row chunk kb (16 groups):
//   codes: word ((nt*KB + kb)*8 + gq)*64 + l*2 + s, nibble p: kept code
//          (p >> 2) of column 16gq + l/4 + 8(p&1), group 8s + l%4 + 4((p>>1)&1);
//   meta:  word ((nt*KB + kb)*8 + gq)*32 + (r*2 + h)*2 + s, nibble i: index pair
//          of column 16gq + r + 8(i>>2), group 8s + 4h + (i&3).
// So lane l = 4r + c of a warp holds, per 32-row step s, one code word whose
// four fp16 pairs are its sparse A fragment registers, and lanes c = 0, 1 hold
// the metadata words of the step's first and second 16 rows.

// Codes of rows 4j..4j+3 of column n (nibble i = row 4j+i) and their zero point.
__device__ __forceinline__ uint32_t group_codes(const uint32_t* q, int N, int j, int n) {
  return (q[(size_t)(j >> 1) * N + n] >> ((j & 1) * 16)) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t group_zero(const uint32_t* zeros, int N, int group, int j, int n) {
  if (!zeros) return 8u;
  return (zeros[(size_t)((4 * j) / group) * (N / 8) + n / 8] >> (4 * (n & 7))) & 0xFu;
}

// Kept-row mask of a group (two bits set) and whether it was 2:4.
__device__ __forceinline__ uint32_t kept_mask(uint32_t codes4, uint32_t z, bool* ok) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m |= (((codes4 >> (4 * i)) & 0xFu) != z ? 1u : 0u) << i;
  *ok = __popc(m) <= 2;
  if (!*ok) {
    const uint32_t lo = m & (0u - m);
    const uint32_t rest = m ^ lo;
    m = lo | (rest & (0u - rest));
  }
  while (__popc(m) < 2) m |= ~m & (m + 1u);  // lowest row not yet kept
  return m;
}

__global__ void sparse_codes_kernel(const uint32_t* __restrict__ q, const uint32_t* __restrict__ zeros,
                                    int K, int N, int group, uint32_t* __restrict__ out,
                                    long long total) {
  const int KB = K / 64;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int s = (int)(t & 1);
    const int l = (int)((t >> 1) & 31);
    const int gq = (int)((t >> 6) & 7);
    const long long chunk = t >> 9;
    const int kb = (int)(chunk % KB);
    const int nt = (int)(chunk / KB);
    uint32_t w = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {  // nibbles p (kept row 0) and p + 4 (kept row 1)
      const int n = nt * 128 + 16 * gq + (l >> 2) + 8 * (p & 1);
      const int j = kb * 16 + 8 * s + (l & 3) + 4 * ((p >> 1) & 1);
      const uint32_t c4 = group_codes(q, N, j, n);
      bool ok;
      const uint32_t m = kept_mask(c4, group_zero(zeros, N, group, j, n), &ok);
      const int i0 = __ffs(m) - 1;
      const int i1 = __ffs(m & (m - 1u)) - 1;
      w |= ((c4 >> (4 * i0)) & 0xFu) << (4 * p);
      w |= ((c4 >> (4 * i1)) & 0xFu) << (4 * (p + 4));
    }
    out[t] = w;
  }
  publish_before_exit();
}

__global__ void sparse_meta_kernel(const uint32_t* __restrict__ q, const uint32_t* __restrict__ zeros,
                                   int K, int N, int group, uint32_t* __restrict__ out, int* bad,
                                   long long total) {
  const int KB = K / 64;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int s = (int)(t & 1);
    const int h = (int)((t >> 1) & 1);
    const int r = (int)((t >> 2) & 7);
    const int gq = (int)((t >> 5) & 7);
    const long long chunk = t >> 8;
    const int kb = (int)(chunk % KB);
    const int nt = (int)(chunk / KB);
    uint32_t w = 0;
    int nbad = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int n = nt * 128 + 16 * gq + r + 8 * (i >> 2);
      const int j = kb * 16 + 8 * s + 4 * h + (i & 3);
      bool ok;
      const uint32_t m = kept_mask(group_codes(q, N, j, n), group_zero(zeros, N, group, j, n), &ok);
      nbad += ok ? 0 : 1;
      const uint32_t i0 = (uint32_t)(__ffs(m) - 1);
      const uint32_t i1 = (uint32_t)(__ffs(m & (m - 1u)) - 1);
      w |= (i0 | (i1 << 2)) << (4 * i);
    }
    out[t] = w;
    if (bad && nbad) atomicAdd(bad, nbad);
  }
  publish_before_exit();
}

int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  if (g > 152 * 16) g = 152 * 16;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t launch_repack(const uint32_t* q, uint32_t* out, int K, int N, cudaStream_t stream) {
  const long long total = (long long)K * N / 8;
  repack_codes_kernel<<<grid_for(total, 256), 256, 0, stream>>>(q, out, K, N, total);
  return cudaGetLastError();
}

cudaError_t launch_sparse_repack(const uint32_t* q, const uint32_t* zeros, int K, int N, int group,
                                 uint32_t* codes_out, uint32_t* meta_out, int* bad,
                                 cudaStream_t stream) {
  const long long chunks = (long long)(N / 128) * (K / 64);
  sparse_codes_kernel<<<grid_for(chunks * 512, 256), 256, 0, stream>>>(q, zeros, K, N, group, codes_out,
                                                                     chunks * 512);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sparse_meta_kernel<<<grid_for(chunks * 256, 256), 256, 0, stream>>>(q, zeros, K, N, group, meta_out,
                                                                    bad, chunks * 256);
  return cudaGetLastError();
}

cudaError_t launch_tile_major(const void* src, void* dst, int G, int N, int row_bytes,
                              cudaStream_t stream) {
  const int NT = N / 128;
  const int row_vec = row_bytes / 16;
  tile_major_kernel<<<grid_for((long long)G * NT * row_vec, 256), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), G, NT, row_vec);
  return cudaGetLastError();
}

}  // namespace w4a16

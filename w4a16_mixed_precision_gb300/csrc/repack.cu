// repack.cu -- offline rewrite of GPTQ-order 4-bit codes, scales and zeros into
// the layout the fused kernels stream ("Marlin / GPTQ-Marlin", section "Tiled
// layout et repacking": done once at load time; "Marlin Project Overview",
// section "Key Techniques", item "Reshuffling for Access Patterns": weights and scales rearranged
// offline into tensor-core operand order).
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

cudaError_t launch_tile_major(const void* src, void* dst, int G, int N, int row_bytes,
                              cudaStream_t stream) {
  const int NT = N / 128;
  const int row_vec = row_bytes / 16;
  tile_major_kernel<<<grid_for((long long)G * NT * row_vec, 256), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), G, NT, row_vec);
  return cudaGetLastError();
}

}  // namespace w4a16

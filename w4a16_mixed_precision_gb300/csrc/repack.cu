// repack.cu -- offline rewrite of GPTQ-order 4-bit codes into the tile layout
// the fused kernel streams ("Marlin / GPTQ-Marlin", section "Tiled layout et
// repacking": done once at load time; "Marlin Project Overview", section
// "Key Techniques", item "Reshuffling").
//
// Tile layout: for every 128-column tile nt and 64-row block kb, one 4 KB chunk
// [h = 0..1][nl = 0..127][i = 0..3] of 32-bit words; word (h, nl, i) carries the
// 8 codes of rows kb*64 + (h*4 + i)*8 .. +7 of column nt*128 + nl.  Inside the
// word the even rows of the 8 sit in nibbles 0..3 and the odd rows in nibbles
// 4..7, so one AND with 0x000F000F (after an optional 8-bit shift) isolates two
// consecutive rows, one per fp16 half.  Each dequantising thread owns one
// column and reads its 32 bytes per chunk as two conflict-free 16-byte loads.
#include "kernels.h"

namespace w4a16 {

namespace {

// GPTQ word (row 8r+i at nibble i) -> tile word (even rows in the low 16 bits,
// odd rows in the high 16 bits, each in ascending order).
__device__ __forceinline__ uint32_t split_even_odd_nibbles(uint32_t w) {
  uint32_t e = w & 0x0F0F0F0Fu;          // nibbles 0,2,4,6 in the low half of each byte
  uint32_t o = (w >> 4) & 0x0F0F0F0Fu;   // nibbles 1,3,5,7
  e = (e | (e >> 4)) & 0x00FF00FFu;
  o = (o | (o >> 4)) & 0x00FF00FFu;
  e = (e | (e >> 8)) & 0x0000FFFFu;
  o = (o | (o >> 8)) & 0x0000FFFFu;
  return e | (o << 16);
}

// One thread per (tile, block, h, column): 4 input words (rows of 8) -> one
// 16-byte output vector.  Consecutive threads take consecutive columns, so the
// reads of each GPTQ row and the 16-byte writes are both coalesced.
__global__ void repack_codes_kernel(const uint32_t* __restrict__ q, uint4* __restrict__ out, int K,
                                    int N, long long total) {
  const int KB = K / 64;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int nl = (int)(t & 127);
    const int h = (int)((t >> 7) & 1);
    const long long chunk = t >> 8;
    const int kb = (int)(chunk % KB);
    const int nt = (int)(chunk / KB);
    const int n = nt * 128 + nl;
    const size_t r0 = (size_t)kb * 8 + (size_t)h * 4;  // GPTQ row of the first word
    uint4 v;
    v.x = split_even_odd_nibbles(q[(r0 + 0) * N + n]);
    v.y = split_even_odd_nibbles(q[(r0 + 1) * N + n]);
    v.z = split_even_odd_nibbles(q[(r0 + 2) * N + n]);
    v.w = split_even_odd_nibbles(q[(r0 + 3) * N + n]);
    out[(chunk * 2 + h) * 128 + nl] = v;
  }
}

__global__ void copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  if (g > 152 * 16) g = 152 * 16;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t launch_repack(const uint32_t* q, uint32_t* out, int K, int N, cudaStream_t stream) {
  const long long total = (long long)(N / 128) * (K / 64) * 2 * 128;
  repack_codes_kernel<<<grid_for(total, 256), 256, 0, stream>>>(q, reinterpret_cast<uint4*>(out),
                                                                 K, N, total);
  return cudaGetLastError();
}

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  const long long n = (long long)(bytes / 16);
  if (n == 0) return cudaSuccess;
  copy16_kernel<<<grid_for(n, 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(src),
                                                      reinterpret_cast<uint4*>(dst), n);
  return cudaGetLastError();
}

}  // namespace w4a16

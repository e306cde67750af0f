// kernels.h -- internal interface between the C-ABI host layer (api.cu) and
// the device kernels (gemm.cu, small_m.cu, repack.cu).  Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

// Fixed geometry of the fused kernel.
constexpr int kThreads = 640;      // 20 warps: 2 producers, 2 MMA issuers (one owns TMEM), 16 dequant
constexpr int kTileN = 128;        // output columns per tile = UMMA M
constexpr int kChunkK = 64;        // K elements per dequantised A chunk
constexpr int kChunkCodeBytes = kTileN * kChunkK / 2;  // 4096
// 2:4-sparse layout: per 64-row chunk of a tile, the kept half of the codes
// and a 4-bit index pair per group of four rows
constexpr int kSpChunkCodeBytes = kTileN * kChunkK / 4;  // 2048
constexpr int kSpChunkMetaBytes = kTileN * kChunkK / 8;  // 1024
constexpr int kMaxWarpM = 32;      // largest M the warp-level kernel serves (4 blocks of 8 tokens)
constexpr int kAStages = 12;       // most A slots (one unit each) resident in TMEM
constexpr int kTmemCols = 512;
constexpr int kMaxStages = 16;
constexpr int kCtrlBytes = 1024;   // barriers and flags at the front of dynamic smem
constexpr int kMaxBn = 256;        // tokens per m-tile (UMMA N)

// Device status word bits (workspace offset 0).  The word at offset 4 holds
// the site of the first failed bounds check (debug builds only).
constexpr int kStatusTimeout = 1;
constexpr int kStatusBounds = 2;

struct GemmParams {
  const uint32_t* codes;    // tile-layout codes
  const uint32_t* meta;     // 2:4-sparse kernel: tile-layout index nibbles (else unused)
  const uint16_t* scales;   // fp16, tile-major [N/128][G][128]
  const uint8_t* zeros;     // zeros, tile-major bytes [N/128][G][64], or nullptr
  uint16_t* Y;              // fp16 [M][N]
  float* partials;          // [grid][bn][128] fp32: one partial tile per CTA
  int* counters;            // [m_tiles * n_tiles]
  int* status;              // status word
  int M, K, N, group, G;
  int bn;                   // tokens per m-tile, multiple of 16
  int m_tiles, n_tiles;
  int kt;                   // units per tile along K
  int cpu;                  // 64-wide chunks per unit (1 or 2)
  long long units;          // m_tiles * n_tiles * kt
  int stages;
  uint32_t stage_bytes;
  uint32_t x_chunk_bytes;   // bn * 128
  uint32_t off_codes, off_scales, off_zeros;  // byte offsets inside a stage
  uint32_t off_meta;        // 2:4-sparse kernel: index nibbles inside a stage
  int weights_reused;       // more than one m-tile reads the same weights
  int nacc;                 // tcgen05 kernel: MMA issuers, each with its own accumulator (1 or 2)
  int split_h;              // split_n: token columns of the first issuer (multiple of 16)
  int full_all;             // tcgen05 kernel: dequant warps wait on every stage (stage count not a multiple of 4)
  int split_n;              // tcgen05 kernel, bn > 128: the two issuers take token columns
                            // [0, 128) and [128, bn) of every unit (one accumulator of bn columns)
  uint32_t tx_w, tx_x;      // bytes landed per stage by the weights / activation producer
  int n_g;                  // scale/zero group rows per unit (2 only for group 128, 256-row units)
  int units_per_group;      // units per group row (>= 1)
  uint32_t off_xchg;        // small-M kernel: exchange buffer, bytes after stage 0
  int a_slots;              // tcgen05 kernel: A slots in TMEM (even, >= 4, <= kAStages)
  uint32_t a_base;          // tcgen05 kernel: TMEM column of A slot 0 (accumulators below it)
  int early_weights;        // stream the first ring of weights before the dependency wait
  int x3d;                  // X tensor map is [K/64][M][64] with a box of one unit's cpu chunks
  int even_split;           // every CTA holds the same whole number of units and every tile splits evenly
  unsigned long long timeout_ns;
  // Extents the bounds-checked (MARLIN_DEBUG) build checks addresses against,
  // in bytes: the logical sizes of the buffers the caller passed, and the
  // dynamic shared memory of the launch.
  unsigned long long codes_bytes, meta_bytes, scales_bytes, zeros_bytes, ws_bytes;
  uint32_t smem_bytes;
};

// Partition and resource plan of one marlin_gemm call.
enum KernelKind { kKernelTcgen05 = 0, kKernelSmallM = 1 };
struct GemmPlan {
  int kind;
  int bn, m_tiles, n_tiles, kt, cpu, stages, grid, n_g, upg, nacc, a_slots, split_n;
  uint32_t off_xchg;
  long long units;
  uint32_t stage_bytes, smem_bytes;
  size_t ws_counters_off, ws_partials_off, ws_bytes;
};

cudaError_t launch_gemm(const CUtensorMap& x_map, const GemmParams& p, int grid, uint32_t smem_bytes,
                        cudaStream_t stream);
cudaError_t gemm_set_smem_limit(int bytes);
// sparse: the 2:4 variant (p.codes / p.meta in the sparse tile layout)
cudaError_t launch_small_m(const CUtensorMap& x_map, const GemmParams& p, int grid,
                           uint32_t smem_bytes, bool sparse, cudaStream_t stream);
cudaError_t small_m_set_smem_limit(int bytes);

// Workspace bytes of the plan marlin_gemm uses for this call on the current
// device (not the worst case over kernels and smaller M that
// marlin_workspace_bytes reports); returns a marlin_status_t value.
int call_workspace_bytes(int M, int K, int N, int group, bool has_zeros, size_t* bytes);

cudaError_t launch_repack(const uint32_t* q, uint32_t* out, int K, int N, cudaStream_t stream);
// 2:4: GPTQ-order codes (+ zeros) -> kept codes and index nibbles in the sparse
// tile layout; *bad (if not null) += groups with more than two non-zero weights.
cudaError_t launch_sparse_repack(const uint32_t* q, const uint32_t* zeros, int K, int N, int group,
                                 uint32_t* codes_out, uint32_t* meta_out, int* bad,
                                 cudaStream_t stream);
// Rows of row_bytes (multiple of 16) from [G][N/128][row] to [N/128][G][row].
cudaError_t launch_tile_major(const void* src, void* dst, int G, int N, int row_bytes,
                              cudaStream_t stream);

}  // namespace w4a16

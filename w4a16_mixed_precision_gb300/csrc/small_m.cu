// small_m.cu -- the fused W4A16 matrix multiply for small batches (M <= 32; by
// default the library sends M <= 16 here and larger batches to gemm.cu; the
// 2:4-sparse instantiation serves every M, in m-tiles of 32 tokens):
// Y[M][N] = X[M][K] . dequant(W)[K][N] on the warp-level tensor-core path.
//
// At M <= 32 the multiply is bound by streaming the 4-bit weights from HBM, and
// the work per byte is the dequantisation ("Marlin", section "诞生背景": at
// batch 8-16 earlier kernels lost the 4x because dequantisation was not
// pipelined with the GEMM).  Here every consumer warp turns its own fragment
// words into fp16 tensor-core operands in registers and feeds them to
// mma.sync.m16n8k16 immediately ("Marlin", section "反量化与 GEMM 融合":
// dequantise in registers, then the tensor core, no intermediate in memory);
// no single thread issues MMAs for the whole SM and nothing is staged in TMEM.
//
//   * One persistent CTA per SM takes an equal stripe of (128-column tile,
//     K-slice) units ("Marlin Project Overview", section "Key Techniques",
//     item "Striped Partitioning"); tiles cut by a stripe boundary are summed by
//     the CTA that owns the tile's first unit, in a fixed order.
//   * Warp 0 streams the weights (codes, scales, zeros: one bulk copy each per
//     unit) and warp 1 streams X (tensor copies, 128-byte swizzle) into a ring
//     of mbarrier-guarded stages.
//   * Warps 2..17: consumer warp (g, h) owns columns 16g..16g+15 of the tile
//     and half h (the first or last 64 or 128 rows) of every unit ("Marlin
//     Project Overview", item "Warp Utilization": several warps compute partial
//     results of one output tile); the two halves are summed through shared
//     memory at the end of each tile.
//   * The MMA's k order is permuted consistently for both operands: lane l
//     holds rows 4(l%4)..4(l%4)+3 of every 16-row step (the repacked fragment
//     order), so its X operand is one 8-byte shared load per step and token
//     block.
//   * Every wait is bounded; on expiry the kernel records a timeout in the
//     status word and returns.
//   * The SP instantiation multiplies 2:4-sparse weights ("Marlin", section
//     "支持 2:4 稀疏加速"): a stage carries the kept half of the codes plus a
//     4-bit index pair per group of four rows, each consumer step covers 32
//     rows with one dequantised code word and one mma.sp per token block, and
//     X keeps its k order (no token permutation; one ldmatrix.x4 per token
//     block and step).
#include "common.cuh"

namespace w4a16 {

namespace {

constexpr int kSmConsumers = 16;
constexpr int kSmThreads = (2 + kSmConsumers) * 32;

struct SmCtrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t red_full;    // odd-half warps -> even-half warps: accumulators in smem
  uint64_t red_free;    // even-half warps -> odd-half warps: exchange buffer read
  uint64_t red_go;      // leader -> even-half warps: all partials published (reducer)
  int abort;
};
static_assert(sizeof(SmCtrl) <= kCtrlBytes, "control block too large");

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
  return v;
}

// Four 8x8 b16 matrices; lanes 8i..8i+7 give the row addresses of matrix i
// (16 bytes each), and lane l receives row l/4, elements 2(l%4), +1 of each.
__device__ __forceinline__ uint4 ldmatrix_x4(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// One 32-row step of the 2:4-sparse path ("Marlin / GPTQ-Marlin", section
// "4. Support de la sparsité 2:4 NVIDIA": dequantise, skip the zeros, sparse
// GEMM).  The lane's code word holds the kept weights of its two columns
// (r, r + 8) in two groups of four rows (c, c + 4 of the step); dequantised,
// its four fp16 pairs are the lane's registers of the compressed 16 x 16 A
// operand.  `e` is the step's index nibbles, supplied by lanes c = 0 (rows
// 0..15 of the step) and c = 1 (rows 16..31): sparsity selector 0.  One
// mma.sp per block of 8 tokens; b[nb] holds the lane's eight X values.
template <int NB>
__device__ __forceinline__ void dequant_mma_sp(float (&acc)[NB][4], uint32_t w, uint32_t e,
                                               uint32_t sub_r, uint32_t add_r8, uint32_t s_r,
                                               uint32_t s_r8, const uint4 (&b)[NB]) {
  const uint32_t k16 = 0x2C002C00u;  // 1/16 as an fp16 pair
  uint32_t a0, a1, a2, a3;
  asm volatile("{\n\t" W4A16_DEQ_PTX("%4", "%5", "%6", "%7", "%8", "%9")
               "mov.b32 %0, t0;\n\tmov.b32 %1, t1;\n\tmov.b32 %2, t2;\n\tmov.b32 %3, t3;\n\t}"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(w), "r"(sub_r), "r"(add_r8), "r"(s_r), "r"(s_r8), "r"(k16));
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
    asm volatile(
        "mma.sp::ordered_metadata.sync.aligned.m16n8k32.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9, %10, %11}, {%0, %1, %2, %3}, %12, 0x0;"
        : "+f"(acc[nb][0]), "+f"(acc[nb][1]), "+f"(acc[nb][2]), "+f"(acc[nb][3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b[nb].x), "r"(b[nb].y), "r"(b[nb].z),
          "r"(b[nb].w), "r"(e));
}

// NB: blocks of 8 tokens (M <= 8*NB).  JPW: 64-row chunks per consumer warp
// per unit (a unit has 2*JPW chunks; warp half h takes chunks h*JPW .. +JPW-1).
// ZP: explicit zero points (else the implicit zero 8 is a constant).
// SP: 2:4-sparse weights (kept codes + index nibbles, mma.sp).
template <int NB, int JPW, bool ZP, bool SP>
__global__ void __launch_bounds__(kSmThreads, 1)
    w4a16_small_m_kernel(const __grid_constant__ CUtensorMap x_map, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_addr - raw_addr);
  SmCtrl* ctrl = reinterpret_cast<SmCtrl*>(base);
  const uint32_t stage0 = base_addr + kCtrlBytes;
  float* xchg = reinterpret_cast<float*>(base + kCtrlBytes + p.off_xchg);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long U = p.units;
  const long long G = gridDim.x;
  const int u_begin = (int)stripe_begin(blockIdx.x, U, G);
  const int u_end = (int)stripe_begin(blockIdx.x + 1, U, G);
  const int KT = p.kt;
  const int S = p.stages;
  const int cpu = p.cpu;
  const int tile_begin = u_begin / KT;
  const int ku_begin = u_begin - tile_begin * KT;

  auto bar = [&](const uint64_t& b) { return smem_addr(&b); };

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(ctrl->full[s]), 2);
      mbar_init(bar(ctrl->empty[s]), kSmConsumers);
    }
    mbar_init(bar(ctrl->red_full), kSmConsumers / 2);
    mbar_init(bar(ctrl->red_free), kSmConsumers / 2);
    mbar_init(bar(ctrl->red_go), 1);
    ctrl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 1 && lane == 0) prefetch_tensormap(&x_map);
  __syncthreads();
  const WaitCtx wc{&ctrl->abort, p.status, p.timeout_ns};
  // Programmatic dependent launch: the next kernel in the stream may be
  // scheduled as soon as SMs free up, and this one waits, after its prologue,
  // until the previous kernel has finished and its writes are visible -- so
  // launch latency and set-up overlap the previous kernel.  The weights
  // (codes, index nibbles, scales, zeros) are constant inputs: with
  // early_weights the weight producer fills the ring with them before that
  // wait, so the previous kernel's tail overlaps this one's first HBM reads.
  // X, Y and the workspace are touched only after the wait.
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (warp != 0 || !p.early_weights) griddep_wait();

  if (warp == 0) {
    // ================= weights producer =================
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint8_t* codes = reinterpret_cast<const uint8_t*>(p.codes);
      const uint8_t* meta = reinterpret_cast<const uint8_t*>(p.meta);
      const int KB = p.K / kChunkK;
      constexpr uint32_t chunk_code = SP ? kSpChunkCodeBytes : kChunkCodeBytes;
      const uint32_t code_bytes = (uint32_t)cpu * chunk_code;
      const uint32_t meta_bytes = SP ? (uint32_t)cpu * kSpChunkMetaBytes : 0u;
      const uint32_t scale_bytes = (uint32_t)(p.n_g * kTileN * 2);
      const uint32_t zero_bytes = (uint32_t)(p.n_g * kTileN / 2);
      const uint32_t tx = code_bytes + meta_bytes + scale_bytes + (p.zeros ? zero_bytes : 0u);
      const int upg = p.units_per_group;
      // tiles are (column tile, m-tile) pairs, m-tile fastest: the m-tiles of
      // a column tile read the same weights one after the other (from L2)
      const int MT = p.m_tiles;
      int nt = tile_begin / MT, mt = tile_begin - (tile_begin / MT) * MT, ku = ku_begin;
      int g = (ku / upg) * p.n_g, ku_in_g = ku - (ku / upg) * upg;
      int s = 0, issued = 0;
      uint32_t ph = 0;
      // the first S stages need no wait; the dependency wait comes before the
      // first bounded wait (which would otherwise time the previous kernel)
      bool dep = !p.early_weights;
      for (int u = u_begin; u < u_end; ++u) {
        if (!dep && issued == S) { griddep_wait(); dep = true; }
        if (!wait_thread(bar(ctrl->empty[s]), ph ^ 1u, wc)) break;
        const uint32_t st = stage0 + (uint32_t)s * p.stage_bytes;
        const uint32_t fb = bar(ctrl->full[s]);
        mbar_arrive_expect_tx(fb, tx);
        const size_t chunk0 = (size_t)nt * KB + (size_t)ku * cpu;
        if (W4A16_IN_RANGE(p.status, chunk0 * chunk_code, code_bytes, p.codes_bytes, 1) &&
            W4A16_SMEM_OK(p, raw_addr, st + p.off_codes, code_bytes, 5))
          bulk_g2s(st + p.off_codes, codes + chunk0 * chunk_code, code_bytes, fb, pol);
        if (SP && W4A16_IN_RANGE(p.status, chunk0 * kSpChunkMetaBytes, meta_bytes, p.meta_bytes, 2) &&
            W4A16_SMEM_OK(p, raw_addr, st + p.off_meta, meta_bytes, 5))
          bulk_g2s(st + p.off_meta, meta + chunk0 * kSpChunkMetaBytes, meta_bytes, fb, pol);
        const size_t grow = (size_t)nt * p.G + g;
        if (W4A16_IN_RANGE(p.status, grow * kTileN * 2, scale_bytes, p.scales_bytes, 3) &&
            W4A16_SMEM_OK(p, raw_addr, st + p.off_scales, scale_bytes, 5))
          bulk_g2s(st + p.off_scales, p.scales + grow * kTileN, scale_bytes, fb, pol);
        if (p.zeros && W4A16_IN_RANGE(p.status, grow * (kTileN / 2), zero_bytes, p.zeros_bytes, 4) &&
            W4A16_SMEM_OK(p, raw_addr, st + p.off_zeros, zero_bytes, 5))
          bulk_g2s(st + p.off_zeros, p.zeros + grow * (kTileN / 2), zero_bytes, fb, pol);
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
        if (++ku_in_g == upg) { ku_in_g = 0; g += p.n_g; }
        if (++ku == KT) {
          ku = 0; g = 0; ku_in_g = 0;
          if (++mt == MT) { mt = 0; ++nt; }
        }
      }
      if (!dep) griddep_wait();
      const int first = issued > S ? issued - S : 0;
      for (int i = first; i < issued; ++i)
        wait_drain(bar(ctrl->full[i % S]), (uint32_t)((i / S) & 1), wc);
    }
  } else if (warp == 1) {
    // ================= activation producer =================
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();
      const uint32_t tx = (uint32_t)cpu * p.x_chunk_bytes;
      const int MT = p.m_tiles;
      int mt = tile_begin - (tile_begin / MT) * MT, ku = ku_begin;
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int u = u_begin; u < u_end; ++u) {
        if (!wait_thread(bar(ctrl->empty[s]), ph ^ 1u, wc)) break;
        const uint32_t st = stage0 + (uint32_t)s * p.stage_bytes;
        const uint32_t fb = bar(ctrl->full[s]);
        mbar_arrive_expect_tx(fb, tx);
        // one 3-D box: the unit's cpu chunks of 64 columns, bn token rows each
        if (W4A16_SMEM_OK(p, raw_addr, st, (uint32_t)cpu * p.x_chunk_bytes, 6))
          tma_load_3d(st, &x_map, 0, mt * p.bn, ku * cpu, fb, pol);
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
        if (++ku == KT) {
          ku = 0;
          if (++mt == MT) mt = 0;
        }
      }
      const int first = issued > S ? issued - S : 0;
      for (int i = first; i < issued; ++i)
        wait_drain(bar(ctrl->full[i % S]), (uint32_t)((i / S) & 1), wc);
    }
  } else {
    // ================= consumers =================
    const int cw = warp - 2;
    const int g = cw & 7;      // column group: tile columns 16g .. 16g + 15
    const int h = cw >> 3;     // K-half: chunks of parity h
    const int r = lane >> 2;   // fragment row / token column within a block of 8
    const int c = lane & 3;
    const int col_r = 16 * g + r;  // this lane's two tile columns: col_r, col_r + 8
    // X operand of k-step ks for token block nb: B column r reads token
    // xr = sigma(r) = 2(r%4) + r/4 of the block (so the four rows a half-warp
    // reads fall in four different 32-byte bank groups of the 128-byte
    // swizzle), rows k = 16ks + 4c .. +3 = 16-byte unit 2ks + c/2, swizzled by xr.
    // The sparse path keeps the k order: per 32-row step s, B register j of
    // lane (r, c) holds rows 32s + 8j + 2c, +1 of token r, which is what
    // ldmatrix.x4 delivers when lane l points at 16-byte unit 4s + l/8 of token
    // l%8's row (swizzled by the token; the eight rows of each matrix then fall
    // in eight different 16-byte columns).
    const int xr = SP ? (lane & 7) : (((r & 3) << 1) | (r >> 2));
    constexpr int kXo = SP ? 2 : 4;
    uint32_t xoff[JPW][kXo];  // stage-relative byte offsets, per chunk and k-step
#pragma unroll
    for (int jj = 0; jj < JPW; ++jj)
#pragma unroll
      for (int ks = 0; ks < kXo; ++ks) {
        const uint32_t row0 = (uint32_t)(h * JPW + jj) * p.x_chunk_bytes + (uint32_t)xr * 128;
        if constexpr (SP)
          xoff[jj][ks] = row0 + (uint32_t)(((4 * ks + (lane >> 3)) ^ xr) << 4);
        else
          xoff[jj][ks] = row0 + (uint32_t)(c & 1) * 8 + (uint32_t)(((2 * ks + (c >> 1)) ^ xr) << 4);
      }
    // stage-relative offsets of this lane's codes, scales and zeros; the
    // warp's chunks lie in one group row: row h of the unit when a unit spans
    // two groups (group 128, 256-row units), else row 0
    const int gsub = (p.n_g > 1) ? h : 0;
    constexpr uint32_t chunk_code = SP ? kSpChunkCodeBytes : kChunkCodeBytes;
    const uint32_t code_off = p.off_codes + (uint32_t)(h * JPW) * chunk_code +
                              (uint32_t)(g * 32 + lane) * (SP ? 8 : 16);
    // sparse: this lane's index words (both 32-row steps of a chunk), the
    // words of rows 0..15 (c even) or 16..31 (c odd) of each step
    const uint32_t meta_off = p.off_meta + (uint32_t)(h * JPW) * kSpChunkMetaBytes +
                              (uint32_t)((g * 8 + r) * 2 + (c & 1)) * 8;
    const uint32_t sc_off = p.off_scales + (uint32_t)(gsub * kTileN + col_r) * 2;
    const uint32_t zr_off = p.off_zeros + (uint32_t)(gsub * (kTileN / 2) + (col_r >> 1));
    const uint32_t z_shift = (uint32_t)(col_r & 1) * 4;
    // accumulator column 2c + e of a block is token sigma(2c + e) (sparse: 2c + e)
    const int tok0 = SP ? 2 * c : ((((2 * c) & 3) << 1) | ((2 * c) >> 2));
    const int tok1 = SP ? 2 * c + 1 : ((((2 * c + 1) & 3) << 1) | ((2 * c + 1) >> 2));
    // With two or more token blocks, odd k-steps accumulate into a second set
    // (acc2), so consecutive MMAs of a block do not wait on each other (measured:
    // M = 16 on 16384x19456, 46.1 -> 42.2 us; at NB = 1 it was 2% slower).
    constexpr bool kTwoChains = NB >= 2;
    float acc[NB][4], acc2[NB][4];
    int s = 0, seg = 0;
    uint32_t ph = 0;
    int u = u_begin, ku = ku_begin, tile = tile_begin;
    bool ok = true;
    while (ok && u < u_end) {
      const int seg_len = min(u_end - u, KT - ku);
      const bool whole = (ku == 0 && seg_len == KT);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int d = 0; d < 4; ++d) acc[nb][d] = acc2[nb][d] = 0.f;

      for (int i = 0; i < seg_len; ++i) {
        if (!wait_warp(bar(ctrl->full[s]), ph, wc)) { ok = false; break; }
        const uint32_t st = stage0 + (uint32_t)s * p.stage_bytes;
        uint4 wv[JPW];
        if constexpr (SP) {
          // x, y: code words of the chunk's two steps; z, w: their index words
#pragma unroll
          for (int jj = 0; jj < JPW; ++jj) {
            const uint32_t ca = st + code_off + (uint32_t)jj * kSpChunkCodeBytes;
            const uint32_t ma = st + meta_off + (uint32_t)jj * kSpChunkMetaBytes;
            const uint2 cw = W4A16_SMEM_OK(p, raw_addr, ca, 8, 7) ? lds64(ca) : make_uint2(0u, 0u);
            const uint2 mw = W4A16_SMEM_OK(p, raw_addr, ma, 8, 7) ? lds64(ma) : make_uint2(0u, 0u);
            wv[jj] = make_uint4(cw.x, cw.y, mw.x, mw.y);
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < JPW; ++jj) {
            const uint32_t ca = st + code_off + (uint32_t)jj * kChunkCodeBytes;
            wv[jj] = W4A16_SMEM_OK(p, raw_addr, ca, 16, 7) ? lds128(ca) : make_uint4(0u, 0u, 0u, 0u);
          }
        }
        // implicit zero 8: 1024 + 8 and -(64 + 8) as fp16 pairs
        uint32_t sub0 = 0x64086408u, add1 = 0xD480D480u;
        if constexpr (ZP) {
          const bool zok = W4A16_SMEM_OK(p, raw_addr, st + zr_off, 5, 8);
          const uint32_t zb0 = zok ? lds_u8(st + zr_off) : 0u, zb1 = zok ? lds_u8(st + zr_off + 4) : 0u;
          const ColConst k0 = col_const(0, (zb0 >> z_shift) & 0xFu);
          const ColConst k1 = col_const(0, (zb1 >> z_shift) & 0xFu);
          sub0 = k0.sub; add1 = k1.add;
        }
        const bool sok = W4A16_SMEM_OK(p, raw_addr, st + sc_off, 18, 8);
        const uint32_t sr = sok ? lds_u16(st + sc_off) : 0u, sr8 = sok ? lds_u16(st + sc_off + 16) : 0u;
        const uint32_t s0 = sr | (sr << 16), s1 = sr8 | (sr8 << 16);
        if constexpr (SP) {
#pragma unroll
          for (int jj = 0; jj < JPW; ++jj)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              uint4 b[NB];
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                const uint32_t xa = st + xoff[jj][ks] + (uint32_t)nb * 1024;
                b[nb] = W4A16_SMEM_OK(p, raw_addr, xa, 16, 9) ? ldmatrix_x4(xa) : make_uint4(0u, 0u, 0u, 0u);
              }
              const uint32_t w = ks ? wv[jj].y : wv[jj].x;
              const uint32_t e = ks ? wv[jj].w : wv[jj].z;
              if (kTwoChains && ks) dequant_mma_sp<NB>(acc2, w, e, sub0, add1, s0, s1, b);
              else dequant_mma_sp<NB>(acc, w, e, sub0, add1, s0, s1, b);
            }
        } else {
#pragma unroll
          for (int jj = 0; jj < JPW; ++jj) {
            const uint32_t wk[4] = {wv[jj].x, wv[jj].y, wv[jj].z, wv[jj].w};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              uint2 b[NB];
#pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                const uint32_t xa = st + xoff[jj][ks] + (uint32_t)nb * 1024;
                b[nb] = W4A16_SMEM_OK(p, raw_addr, xa, 8, 9) ? lds64(xa) : make_uint2(0u, 0u);
              }
              if (kTwoChains && (ks & 1)) dequant_mma<NB>(acc2, wk[ks], sub0, add1, s0, s1, b);
              else dequant_mma<NB>(acc, wk[ks], sub0, add1, s0, s1, b);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ctrl->empty[s]));
        if (++s == S) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;

      if (kTwoChains) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int d = 0; d < 4; ++d) acc[nb][d] += acc2[nb][d];
      }
      // ---- sum the two K-halves of each column group (fixed order: h0 + h1) ----
      if (h == 1) {
        if (seg > 0 && !wait_warp(bar(ctrl->red_free), (uint32_t)((seg - 1) & 1), wc)) break;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int d = 0; d < 4; ++d) {
            float* xp = &xchg[(nb * 4 + d) * 256 + g * 32 + lane];
            if (W4A16_SMEM_OK(p, raw_addr, smem_addr(xp), 4, 10)) *xp = acc[nb][d];
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ctrl->red_full));
      } else {
        if (!wait_warp(bar(ctrl->red_full), (uint32_t)(seg & 1), wc)) break;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int d = 0; d < 4; ++d) {
            const float* xp = &xchg[(nb * 4 + d) * 256 + g * 32 + lane];
            acc[nb][d] += W4A16_SMEM_OK(p, raw_addr, smem_addr(xp), 4, 10) ? *xp : 0.f;
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(ctrl->red_free));

        // ---- epilogue (even-half warps): fp16 Y, or fp32 partial + reduction ----
        // accumulator d of block nb: column col_r + 8*(d >> 1), token 8nb + tok[d & 1]
        const size_t y_col0 = (size_t)(tile / p.m_tiles) * kTileN + col_r;
        const int m_base = (tile - (tile / p.m_tiles) * p.m_tiles) * p.bn;   // first token of the m-tile
        if (whole) {
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int d = 0; d < 4; ++d) {
              const int m = 8 * nb + ((d & 1) ? tok1 : tok0);
              if (m_base + m < p.M &&
                  W4A16_IN_RANGE(p.status, (size_t)(m_base + m) * p.N + y_col0 + 8 * (d >> 1), 1,
                                 (size_t)p.M * p.N, 11))
                p.Y[(size_t)(m_base + m) * p.N + y_col0 + 8 * (d >> 1)] =
                    __half_as_ushort(__float2half_rn(acc[nb][d]));
            }
        } else {
          // The tile's reducer owns its first unit: it is this CTA exactly when
          // the segment starts there (ku == 0; a segment starting mid-tile is
          // the first of a contributor's stripe), so no division is needed to
          // tell; the reducer then finds its last contributor by one.
          const long long c_first = (long long)blockIdx.x;
          if (ku != 0) {
            // contributor (this is its first segment): publish the partial tile
            // word by word (tagged) and go on without waiting
            float* part = p.partials + (size_t)blockIdx.x * ((size_t)p.bn * kTileN);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int d = 0; d < 4; ++d) {
                const int m = 8 * nb + ((d & 1) ? tok1 : tok0);
                float* pw = part + (size_t)m * kTileN + col_r + 8 * (d >> 1);
                if (W4A16_IN_RANGE(p.status, (const char*)pw - (const char*)p.status, 4, p.ws_bytes, 12))
                  st_partial(pw, acc[nb][d]);
              }
          } else {
            // reducer (this is its last segment): every thread polls its own
            // words of the other contributors' partials (a word is final once
            // non-zero, so no arrival count is needed) and sums in stripe
            // order, own partial first.  The reducer warps meet at red_go
            // before writing Y; its leader arrives at once, except in a
            // MARLIN_DEBUG build, where it first waits (bounded) for the tile's
            // word in the workspace's counter block to be non-negative.  This
            // kernel never writes that word, so a test can hold the reduction
            // by presetting it negative and make the wait expire.  Measured,
            // release builds without the meeting point ran the main loop of the
            // two-block instantiations up to 6% slower (M = 16 on 8192 x 57344,
            // a code generation effect), and with it dropping the arrival
            // count saved 0.3-0.6 us per call at M <= 16 on 7B-sized shapes.
            const long long c_last = stripe_owner((long long)tile * KT + KT - 1, U, G);
            if (g == 0) {
              if (lane == 0) {
#ifdef MARLIN_DEBUG
                if (W4A16_IN_RANGE(p.status, (const char*)&p.counters[tile] - (const char*)p.status, 4,
                                   p.ws_bytes, 13))
                  wait_counter(&p.counters[tile], 0, wc);
#endif
                mbar_arrive(bar(ctrl->red_go));
              }
              __syncwarp();
            }
            bool got = true;
#pragma unroll
            for (int nb = 0; nb < NB && got; ++nb) {
              // the sums build up in acc (own partial first)
              uint32_t off[4];
#pragma unroll
              for (int d = 0; d < 4; ++d)
                off[d] = (uint32_t)((8 * nb + ((d & 1) ? tok1 : tok0)) * kTileN + col_r + 8 * (d >> 1));
              const size_t stride = (size_t)p.bn * kTileN;
              for (long long q0 = c_first + 1; q0 <= c_last && got; q0 += 4) {
                const int nq = (int)min(4LL, c_last - q0 + 1);
                float* base = p.partials + (size_t)q0 * stride;
                // the partial tiles of contributors q0 .. q0 + nq - 1 this thread polls
                if (!W4A16_IN_RANGE(p.status, (const char*)base - (const char*)p.status,
                                    4 * (size_t)nq * stride, p.ws_bytes, 12)) { got = false; break; }
                uint32_t raw[16];
                if (!poll_partials<4, 4>(base, stride, off, nq, raw, wc)) { got = false; break; }
#pragma unroll
                for (int jq = 0; jq < 4; ++jq)
                  if (jq < nq) {
#pragma unroll
                    for (int d = 0; d < 4; ++d) {
                      acc[nb][d] += partial_value(raw[jq * 4 + d]);
                      __stcg(base + jq * stride + off[d], 0.f);  // re-zero for the next call
                    }
                  }
              }
            }
            if (!wait_warp(bar(ctrl->red_go), 0, wc)) break;
            if (!got || *reinterpret_cast<volatile int*>(&ctrl->abort)) break;
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int d = 0; d < 4; ++d) {
                const int m = 8 * nb + ((d & 1) ? tok1 : tok0);
                if (m_base + m < p.M &&
                    W4A16_IN_RANGE(p.status, (size_t)(m_base + m) * p.N + y_col0 + 8 * (d >> 1), 1,
                                   (size_t)p.M * p.N, 11))
                  p.Y[(size_t)(m_base + m) * p.N + y_col0 + 8 * (d >> 1)] =
                      __half_as_ushort(__float2half_rn(acc[nb][d]));
              }
          }
        }
      }
      ++seg;
      u += seg_len;
      ku = 0;
      ++tile;
    }
  }
  __syncwarp();
  __syncthreads();
}

}  // namespace

#define W4A16_SMALL_M_KERNELS_SP(X, SP)                                                     \
  X(1, 1, false, SP) X(2, 1, false, SP) X(3, 1, false, SP) X(4, 1, false, SP)                \
  X(1, 2, false, SP) X(2, 2, false, SP) X(3, 2, false, SP) X(4, 2, false, SP)                \
  X(1, 1, true, SP) X(2, 1, true, SP) X(3, 1, true, SP) X(4, 1, true, SP)                    \
  X(1, 2, true, SP) X(2, 2, true, SP) X(3, 2, true, SP) X(4, 2, true, SP)
#define W4A16_SMALL_M_KERNELS(X) W4A16_SMALL_M_KERNELS_SP(X, false) W4A16_SMALL_M_KERNELS_SP(X, true)

cudaError_t small_m_set_smem_limit(int bytes) {
  cudaError_t e = cudaSuccess;
#define W4A16_SET(NB, JPW, ZP, SP)                                                           \
  if (e == cudaSuccess)                                                                      \
    e = cudaFuncSetAttribute(w4a16_small_m_kernel<NB, JPW, ZP, SP>,                          \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  W4A16_SMALL_M_KERNELS(W4A16_SET)
#undef W4A16_SET
  return e;
}

cudaError_t launch_small_m(const CUtensorMap& x_map, const GemmParams& p, int grid,
                           uint32_t smem_bytes, bool sparse, cudaStream_t stream) {
  const int nb = p.bn / 8, jpw = p.cpu / 2;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSmThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool zp = p.zeros != nullptr;
#define W4A16_LAUNCH(NB, JPW, ZP, SP)                                                      \
  if (nb == NB && jpw == JPW && zp == ZP && sparse == SP)                                  \
    return cudaLaunchKernelEx(&cfg, w4a16_small_m_kernel<NB, JPW, ZP, SP>, x_map, p);
  W4A16_SMALL_M_KERNELS(W4A16_LAUNCH)
#undef W4A16_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace w4a16

// gemm.cu -- the fused W4A16 matrix multiply for GB300 (sm_103a).
//
// Computes Y[M][N] = X[M][K] . dequant(W)[K][N], dequant(w) = fp16((q - z) * s)
// ("Marlin / GPTQ-Marlin", section "Le problème"; "Marlin" (dingiv.github.io),
// sections "Group size 为什么是 128" and "反量化精度权衡").
//
// Design (Blackwell-first; the pages' Ampere kernel is prior art only):
//   * Swapped operands: the tensor core computes D[n][m] = sum_k Wt[n][k] X[m][k]
//     with UMMA M = 128 output columns n and UMMA N = bn tokens m (16..256), so a
//     decode batch of 1..16 tokens still fills the 128-row MMA.
//   * One persistent CTA per SM walks a contiguous stripe of work units
//     (m-tile, n-tile, K-slice) -- the pages' "striped partitioning"
//     ("Marlin Project Overview", section "Key Techniques").  Column tiles cut by
//     a stripe boundary are summed through an fp32 workspace by the CTA owning
//     the tile's first unit, in a fixed order, so results are bit-reproducible.
//   * Warp roles: warp 0 streams packed codes, scales, zeros (bulk TMA) and
//     warp 3 streams X (tensor TMA, 128-byte swizzle) through a multi-stage
//     mbarrier ring in shared memory ("Marlin", sections "异步内存拷贝" and
//     "Striped 划分与流水线"); warps 4..19 (four warpgroups, taking whole
//     units in turn) turn 4-bit codes into fp16 with the 0x6400 exponent trick, scale them
//     with one fp16 multiply, and store the result straight into tensor memory
//     as the A operand; warps 1 and 2 issue tcgen05.mma (A from TMEM, B = X
//     from shared memory, fp32 accumulators in TMEM): for bn <= 128 on
//     alternate units, one accumulator each, and for bn > 128 on every unit,
//     splitting the token columns of one accumulator at 128; the dequant warps
//     then read the accumulators back with tcgen05.ld and write fp16 Y (or
//     tagged fp32 partial words).
//   * Every wait is bounded (global timer); on expiry the kernel records
//     kStatusTimeout in the status word, drains its own copies and MMAs, frees
//     TMEM and returns.
#include <cuda_fp16.h>

#include "common.cuh"

namespace w4a16 {

namespace {

struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t afull[kAStages];
  uint64_t aempty[kAStages];
  uint64_t dfull;
  uint64_t dempty;
  uint64_t drain[2];
  uint64_t red_go;      // leader -> dequant warps: the reducer may write Y
  uint64_t red_copy;    // the reducer's bulk copies of its contributors' partial tiles landed
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

constexpr int kNumDqWG = 4;                // dequant warpgroups
constexpr int kNumDqWarps = 4 * kNumDqWG;
constexpr int kFirstDqWarp = 4;
static_assert((kNumDqWG & (kNumDqWG - 1)) == 0, "unit residues need a power-of-two warpgroup count");
static_assert(kThreads == 32 * (kFirstDqWarp + kNumDqWarps), "block size");

// ---- the kernel -----------------------------------------------------------------
//
// Hot loops advance their ring positions and unit coordinates incrementally:
// the producer and the MMA issuer are single threads, so any integer division
// on their path sits directly on the critical path of the whole CTA.

// ZP: explicit zero points (else the implicit zero 8 folds into constants).
// BULK: bn > 32, where a warpgroup's epilogue covers several token chunks: a
// reducer may copy its contributors' partial tiles into the drained ring in
// bulk instead of polling them chunk by chunk (separate instantiation, so that
// the bn <= 32 plans keep the code generated without it).
template <bool ZP, bool BULK>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap x_map, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzled X tiles.
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_addr - raw_addr);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(base);
  const uint32_t stage0 = base_addr + kCtrlBytes;

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
  const WaitCtx wc{&ctrl->abort, p.status, p.timeout_ns};

  // ---- setup --------------------------------------------------------------------
  const int nacc = p.nacc;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(ctrl->full[s]), 2);                 // weights + activation producers
      // the unit's dequant warpgroup (every dequant warp when they all track
      // every stage) and its MMA issuer(s)
      mbar_init(bar(ctrl->empty[s]), (p.full_all ? kNumDqWarps : 4) + (p.split_n ? 2 : 1));
    }
    for (int a = 0; a < kAStages; ++a) {
      mbar_init(bar(ctrl->afull[a]), 4);
      mbar_init(bar(ctrl->aempty[a]), p.split_n ? 2 : 1);
    }
    mbar_init(bar(ctrl->dfull), nacc);
    mbar_init(bar(ctrl->dempty), kNumDqWarps);
    mbar_init(bar(ctrl->drain[0]), 1);
    mbar_init(bar(ctrl->drain[1]), 1);
    mbar_init(bar(ctrl->red_go), 1);
    mbar_init(bar(ctrl->red_copy), 1);
    ctrl->abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 3 && lane == 0) prefetch_tensormap(&x_map);
  if (warp == 2) {
    tmem_alloc(smem_addr(&ctrl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  // Programmatic dependent launch: the next kernel in the stream may be
  // scheduled as soon as SMs free up, and this one waits, after its prologue,
  // until the previous kernel has finished and its writes are visible -- so
  // launch latency and set-up overlap the previous kernel.  The weights are
  // constant inputs: with early_weights the weight producer fills the ring
  // with them before that wait; X, Y and the workspace are touched only after.
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (warp != 0 || !p.early_weights) griddep_wait();

  if (warp == 0) {
    // ================= weights producer: codes, scales, zeros =================
    if (lane == 0) {
      const uint64_t pol_w = p.weights_reused ? policy_evict_last() : policy_evict_first();
      const uint8_t* codes = reinterpret_cast<const uint8_t*>(p.codes);
      const int KB = p.K / kChunkK;
      const uint32_t code_bytes = (uint32_t)(cpu * kChunkCodeBytes);
      const int units_per_group = p.group / (cpu * kChunkK);
      int mt = tile_begin / p.n_tiles;
      int nt = tile_begin - mt * p.n_tiles;
      int ku = ku_begin;
      int g = ku / units_per_group, ku_in_g = ku - g * units_per_group;
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
        mbar_arrive_expect_tx(fb, p.tx_w);
        const size_t c_off = ((size_t)nt * KB + (size_t)ku * cpu) * kChunkCodeBytes;
        if (W4A16_IN_RANGE(p.status, c_off, code_bytes, p.codes_bytes, 21) &&
            W4A16_SMEM_OK(p, raw_addr, st + p.off_codes, code_bytes, 24))
          bulk_g2s(st + p.off_codes, codes + c_off, code_bytes, fb, pol_w);
        const size_t grow = (size_t)nt * p.G + g;  // tile-major group row
        if (W4A16_IN_RANGE(p.status, grow * kTileN * 2, kTileN * 2, p.scales_bytes, 22) &&
            W4A16_SMEM_OK(p, raw_addr, st + p.off_scales, kTileN * 2, 24))
          bulk_g2s(st + p.off_scales, p.scales + grow * kTileN, kTileN * 2, fb, pol_w);
        if (p.zeros && W4A16_IN_RANGE(p.status, grow * (kTileN / 2), kTileN / 2, p.zeros_bytes, 23) &&
            W4A16_SMEM_OK(p, raw_addr, st + p.off_zeros, kTileN / 2, 24))
          bulk_g2s(st + p.off_zeros, p.zeros + grow * (kTileN / 2), kTileN / 2, fb, pol_w);
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
        if (++ku_in_g == units_per_group) { ku_in_g = 0; ++g; }
        if (++ku == KT) {
          ku = 0; g = 0; ku_in_g = 0;
          if (++nt == p.n_tiles) { nt = 0; ++mt; }
        }
      }
      if (!dep) griddep_wait();
      // Wait for every copy still in flight before the CTA may exit.
      const int first = issued > S ? issued - S : 0;
      for (int i = first; i < issued; ++i)
        wait_drain(bar(ctrl->full[i % S]), (uint32_t)((i / S) & 1), wc);
    }
  } else if (warp == 3) {
    // ================= activation producer: X tiles =================
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_last();
      int mt = tile_begin / p.n_tiles;
      int nt = tile_begin - mt * p.n_tiles;
      int ku = ku_begin;
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int u = u_begin; u < u_end; ++u) {
        if (!wait_thread(bar(ctrl->empty[s]), ph ^ 1u, wc)) break;
        const uint32_t st = stage0 + (uint32_t)s * p.stage_bytes;
        const uint32_t fb = bar(ctrl->full[s]);
        mbar_arrive_expect_tx(fb, p.tx_x);
        if (p.x3d) {
          // one 3-D box: the unit's cpu chunks of 64 columns, bn token rows each
          if (W4A16_SMEM_OK(p, raw_addr, st, (uint32_t)cpu * p.x_chunk_bytes, 25))
            tma_load_3d(st, &x_map, 0, mt * p.bn, ku * cpu, fb, pol_x);
        } else {
          const int k0 = ku * cpu * kChunkK;
          for (int j = 0; j < cpu; ++j)
            if (W4A16_SMEM_OK(p, raw_addr, st + (uint32_t)j * p.x_chunk_bytes, p.x_chunk_bytes, 25))
              tma_load_2d(st + (uint32_t)j * p.x_chunk_bytes, &x_map, k0 + j * kChunkK, mt * p.bn, fb,
                          pol_x);
        }
        ++issued;
        if (++s == S) { s = 0; ph ^= 1u; }
        if (++ku == KT) {
          ku = 0;
          if (++nt == p.n_tiles) { nt = 0; ++mt; }
        }
      }
      const int first = issued > S ? issued - S : 0;
      for (int i = first; i < issued; ++i)
        wait_drain(bar(ctrl->full[i % S]), (uint32_t)((i / S) & 1), wc);
    }
  } else if (warp == 1 || warp == 2) {
    // ================= MMA issuers (one warp each) =================
    // For bn <= 128, issuer i takes the units i, i+2, ... of the stripe into
    // its own accumulator.  For bn > 128 (split_n), both take every unit:
    // issuer 0 the token columns [0, 128) of the accumulator, issuer 1 the
    // columns [128, bn), each with MMAs of N <= 128 reading its rows of X.  Every barrier ring is indexed
    // by the stripe's unit index, and each consumer of a ring takes a fixed
    // residue of it (issuer: unit mod 2, dequant warpgroup: unit mod 4; the
    // stage count is a multiple of 4 or the warpgroups wait on every stage;
    // the A slot count is even and at least 4, and each issuer's MMAs complete
    // in order), so a consumer is never more than one phase ahead of a barrier
    // it waits on.
    // The whole warp runs the loop; one elected lane issues each MMA and commit.
    const int iss = warp - 1;
    if (iss < nacc) {
      const bool split = p.split_n != 0;
      const uint32_t sh = (uint32_t)p.split_h;
      const uint32_t n_iss = split ? (iss == 0 ? sh : (uint32_t)p.bn - sh) : (uint32_t)p.bn;
      const uint32_t idesc = umma_idesc_f16_f32(n_iss);
      const uint32_t d_tmem = tmem + (split ? (uint32_t)iss * sh : (uint32_t)(iss * p.bn));
      const uint32_t x_rows = split ? (uint32_t)iss * sh * 128u : 0u;  // bytes: sh rows of 128 B
      const int a_slots = p.a_slots;
      const uint32_t a_cols = (uint32_t)cpu * (kChunkK / 2);
      // this issuer's units are r = first, first + stride, ... (r = unit index
      // in the stripe); (s, a) is the ring position of unit r
      const int stride = split ? 1 : nacc;
      int s = 0, a = 0, seg = 0;
      uint32_t ph = 0, aph = 0;
      auto advance = [&](int n) {
        s += n;
        while (s >= S) { s -= S; ph ^= 1u; }
        a += n;
        while (a >= a_slots) { a -= a_slots; aph ^= 1u; }
      };
      int r = split ? 0 : iss;
      advance(r);
      int u = u_begin, ku = ku_begin;
      bool ok = true;
      while (ok && u < u_end) {
        const int seg_len = min(u_end - u, KT - ku);
        const int r_end = u - u_begin + seg_len;  // first unit of the next segment
        if (seg > 0) {
          if (!wait_warp(bar(ctrl->dempty), (uint32_t)((seg - 1) & 1), wc)) break;
          tc_fence_after();
        }
        uint32_t acc = 0;
        for (; r < r_end; r += stride) {
          // the unit's A slot is filled only after its dequant warpgroup saw
          // the stage land, so its completion also covers the X tiles
          if (!wait_warp(bar(ctrl->afull[a]), aph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = stage0 + (uint32_t)s * p.stage_bytes;
          const uint32_t a_col = tmem + p.a_base + (uint32_t)a * a_cols;
          // the accumulator columns and the A slot lie in the allocation; B
          // (this issuer's X rows of every chunk) lies in the stage
          if (!W4A16_IN_RANGE(p.status, (d_tmem - tmem) & 0xFFFFu, n_iss, kTmemCols, 28) ||
              !W4A16_IN_RANGE(p.status, (a_col - tmem) & 0xFFFFu, a_cols, kTmemCols, 28) ||
              !W4A16_SMEM_OK(p, raw_addr, st + x_rows, (uint32_t)(cpu - 1) * p.x_chunk_bytes + n_iss * 128u, 27)) {
            ok = false;
            break;
          }
          for (int j = 0; j < cpu; ++j) {
            const uint64_t desc0 = umma_desc_sw128(st + (uint32_t)j * p.x_chunk_bytes + x_rows);
#pragma unroll
            for (int kk = 0; kk < kChunkK / 16; ++kk) {
              // +32 bytes per 16-row step = +2 in the descriptor's address field
              mma_f16_ts_elect(d_tmem, a_col + (uint32_t)(j * (kChunkK / 2) + kk * 8),
                               desc0 + (uint64_t)(2 * kk), idesc, acc);
              acc = 1;
            }
          }
          mma_commit_elect(bar(ctrl->aempty[a]));
          mma_commit_elect(bar(ctrl->empty[s]));
          advance(stride);
        }
        if (!ok) break;
        // an issuer without a unit in this segment has nothing in flight for it
        if (acc) mma_commit_elect(bar(ctrl->dfull));
        else if (lane == 0) mbar_arrive(bar(ctrl->dfull));
        ++seg;
        u += seg_len;
        ku = 0;
      }
      // Every issued MMA must finish before TMEM is released.
      mma_commit_elect(bar(ctrl->drain[iss]));
      wait_drain(bar(ctrl->drain[iss]), 0, wc);
    }
  } else if (warp >= kFirstDqWarp) {
    // ================= dequantisation + epilogue (16 warps) =================
    const int dq = warp - kFirstDqWarp;       // 0..15
    const int wg = dq >> 2;                   // warpgroup: takes every fourth unit
    const int quarter = warp & 3;             // TMEM lane quarter this warp may touch
    const int row = quarter * 32 + lane;      // epilogue: output column within the tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;

    // dequantisation: this thread holds fragment lane `lane` of the two 16-column
    // groups 2*quarter and 2*quarter+1, i.e. columns c0 + {0, 8, 16, 24}
    const int c0 = 32 * quarter + (lane >> 2);
    const uint32_t code_off = p.off_codes + (uint32_t)((2 * quarter) * 32 + lane) * 16;
    const uint32_t sc_off = p.off_scales + (uint32_t)c0 * 2;
    const uint32_t zr_off = p.off_zeros + (uint32_t)(c0 >> 1);
    const uint32_t z_shift = (uint32_t)(c0 & 1) * 4;
    const int a_slots = p.a_slots;
    const uint32_t a_cols = (uint32_t)cpu * (kChunkK / 2);
    // (s, a) are the stage and A slot of unit r (the unit's index in the
    // stripe), with their phases; advance(n) moves them n units on.  When the
    // stage count is a multiple of 4 each warpgroup visits only its own units
    // r = wg, wg + 4, ...: its stages and its A slots are then used by no
    // other warpgroup between two of its visits (the slot's next user after
    // unit r is unit r + a_slots, again after this warpgroup's own release),
    // so one phase of look-ahead is enough.  Otherwise (full_all) every warp
    // waits on and releases every stage, own or not.
    int s = 0, a = 0, seg = 0, r = 0;
    uint32_t ph = 0, aph = 0;
    auto advance = [&](int n) {
      s += n;
      while (s >= S) { s -= S; ph ^= 1u; }
      a += n;
      while (a >= a_slots) { a -= a_slots; aph ^= 1u; }
      r += n;
    };
    const int stride = p.full_all ? 1 : kNumDqWG;
    if (!p.full_all) advance(wg);
    int u = u_begin, ku = ku_begin, tile = tile_begin;
    bool ok = true;
    while (ok && u < u_end) {
      const int seg_len = min(u_end - u, KT - ku);
      const int r_end = u - u_begin + seg_len;  // first unit of the next segment
      const int mt = tile / p.n_tiles;
      const int nt = tile - mt * p.n_tiles;
      // ---- mainloop: dequantise this warpgroup's units into TMEM ----
      for (; r < r_end; advance(stride)) {
        const bool mine = (r & (kNumDqWG - 1)) == wg;
        if (!mine) {
          // full_all: track every stage: wait for it and release it, so that
          // the ring can neither run a phase ahead of this warp nor lap it
          if (!wait_warp(bar(ctrl->full[s]), ph, wc)) { ok = false; break; }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(ctrl->empty[s]));
        } else {
          if (!wait_warp(bar(ctrl->full[s]), ph, wc)) { ok = false; break; }
          const uint32_t st = stage0 + (uint32_t)s * p.stage_bytes;
          // a unit (cpu <= 2 chunks of 64 rows, group >= 128) lies in one group row
          const bool cok = W4A16_SMEM_OK(p, raw_addr, st + code_off, (cpu - 1) * kChunkCodeBytes + 512 + 16, 26);
          const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
          const uint4 w0 = cok ? lds128(st + code_off) : z4;        // chunk 0, group 2q
          const uint4 w1 = cok ? lds128(st + code_off + 512) : z4;  // chunk 0, group 2q+1
          uint32_t z0 = 8, z1 = 8, z2 = 8, z3 = 8;
          if (ZP && W4A16_SMEM_OK(p, raw_addr, st + zr_off, 13, 26)) {
            z0 = (lds_u8(st + zr_off) >> z_shift) & 0xFu;
            z1 = (lds_u8(st + zr_off + 4) >> z_shift) & 0xFu;
            z2 = (lds_u8(st + zr_off + 8) >> z_shift) & 0xFu;
            z3 = (lds_u8(st + zr_off + 12) >> z_shift) & 0xFu;
          }
          const bool sok = W4A16_SMEM_OK(p, raw_addr, st + sc_off, 50, 26);
          const ColConst k0 = col_const(sok ? (uint16_t)lds_u16(st + sc_off) : 0, z0);
          const ColConst k1 = col_const(sok ? (uint16_t)lds_u16(st + sc_off + 16) : 0, z1);
          const ColConst k2 = col_const(sok ? (uint16_t)lds_u16(st + sc_off + 32) : 0, z2);
          const ColConst k3 = col_const(sok ? (uint16_t)lds_u16(st + sc_off + 48) : 0, z3);
          // the first chunk is dequantised before waiting for the slot, so that
          // only its stores sit between the slot's release and its refill
          uint32_t d0[16], d1[16];
          dequant16(w0, k0.sub, k1.add, k0.s, k1.s, d0);
          dequant16(w1, k2.sub, k3.add, k2.s, k3.s, d1);
          if (!wait_warp(bar(ctrl->aempty[a]), aph ^ 1u, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t acol = tmem + p.a_base + (uint32_t)a * a_cols + lane_off;
          // this warp's 32 lanes and the slot's a_cols columns lie in the allocation
          if (!W4A16_IN_RANGE(p.status, (acol - tmem) & 0xFFFFu, a_cols, kTmemCols, 27) ||
              !W4A16_IN_RANGE(p.status, ((acol - tmem) >> 16) + 32u, 0, 128, 27)) {
            ok = false;
            break;
          }
          tmem_st_16x256b_x4(acol, d0);
          tmem_st_16x256b_x4(acol + (16u << 16), d1);
          if (cpu == 2) {
            const uint4 v0 = cok ? lds128(st + code_off + kChunkCodeBytes) : z4;
            const uint4 v1 = cok ? lds128(st + code_off + kChunkCodeBytes + 512) : z4;
            const uint32_t c1 = acol + (uint32_t)(kChunkK / 2);
            dequant_store_tmem(c1, v0, k0.sub, k1.add, k0.s, k1.s);
            dequant_store_tmem(c1 + (16u << 16), v1, k2.sub, k3.add, k2.s, k3.s);
          }
          // codes and scales read: the stage may be refilled once the MMA is done too
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(ctrl->empty[s]));
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(ctrl->afull[a]));
        }
      }
      if (!ok) break;

      // ---- epilogue: accumulators -> fp16 Y, or fp32 partial tile ----
      const bool whole = (ku == 0 && seg_len == KT);
      const int m_base = mt * p.bn;
      const size_t y_col = (size_t)nt * kTileN + row;
      const long long c_first = tile_reducer(tile, KT, U, G);
      const long long c_last = stripe_owner((long long)tile * KT + KT - 1, U, G);
      const bool reducer = !whole && (long long)blockIdx.x == c_first;
      const size_t part_stride = (size_t)p.bn * kTileN;
      // A reducer issues its loads of the first contributor's words of its
      // first token chunk before waiting for the accumulators, so that their
      // round trip (about 1.5 us while other CTAs stream weights) overlaps the
      // last MMAs (one contributor only: more pushed the kernel past its
      // register cap).
      uint32_t pre[8];
      bool preloaded = false;
      if (reducer && wg < p.bn / 8) {
        const float* base = p.partials + (size_t)(c_first + 1) * part_stride;
        if (W4A16_IN_RANGE(p.status, (const char*)base - (const char*)p.status, 4 * part_stride, p.ws_bytes,
                           31)) {
          uint32_t off[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) off[c] = (uint32_t)((wg * 8 + c) * kTileN + row);
          issue_partials<1, 8>(base, part_stride, off, 1, pre);
          preloaded = true;
        }
      }
      if (!wait_warp(bar(ctrl->dfull), (uint32_t)(seg & 1), wc)) break;
      tc_fence_after();
      if (reducer && dq == 0) {
        // reducer (this is its last segment): every thread polls its own words
        // of the contributors' partial tiles (a tagged word is final once
        // non-zero, so no arrival count is needed; measured 0.3-0.7 us less per
        // call at M = 32..128).  In a MARLIN_DEBUG build the leader first waits
        // (bounded) for the tile's word in the counter block to be
        // non-negative: nothing writes it, so a test can hold the reduction by
        // presetting it negative and make the wait expire.
        if (lane == 0) {
#ifdef MARLIN_DEBUG
          if (W4A16_IN_RANGE(p.status, (const char*)&p.counters[tile] - (const char*)p.status, 4, p.ws_bytes,
                             32))
            wait_counter(&p.counters[tile], 0, wc);
#endif
          mbar_arrive(bar(ctrl->red_go));
        }
        __syncwarp();
      }
      // BULK: a reducer whose warpgroups would otherwise wait for more than one
      // exposed round trip (about 1.5 us each while other CTAs stream weights:
      // one per token chunk and pair of contributors, the first hidden by the
      // load issued ahead) copies its contributors' partial tiles into the
      // ring, free now that the accumulators are final, with one bulk copy
      // each, and reads every chunk's words from there.  A word still zero in
      // the copy (its contributor not done) is polled from global memory.  Not
      // on an even split, where every contributor finishes its piece together
      // with the reducer (measured: the copy then mostly comes too early, and
      // 8192x8192 at M = 128 was 0.5 us slower with it).
      const uint32_t tile_bytes = (uint32_t)(part_stride * sizeof(float));
      int n_copy = 0;
      if constexpr (BULK) {
        if (reducer) {
          const long long nc = c_last - c_first;
          const long long cpw = (p.bn / 8 + kNumDqWG - 1) / kNumDqWG;  // token chunks per warpgroup
          const long long exposed = cpw * ((nc + 1) / 2) - (preloaded ? 1 : 0);
          const long long fit = (long long)((size_t)S * p.stage_bytes / tile_bytes);
          n_copy = (exposed > 1 && !p.even_split) ? (int)min(fit, nc) : 0;
          const float* src = p.partials + (size_t)(c_first + 1) * part_stride;
          if (n_copy > 0 &&
              (!W4A16_IN_RANGE(p.status, (const char*)src - (const char*)p.status,
                               (size_t)n_copy * tile_bytes, p.ws_bytes, 31) ||
               !W4A16_SMEM_OK(p, raw_addr, stage0, (uint32_t)n_copy * tile_bytes, 33)))
            n_copy = 0;
          if (n_copy > 0) {
            if (dq == 0 && lane == 0) {
              fence_proxy_async_smem();
              mbar_arrive_expect_tx(bar(ctrl->red_copy), (uint32_t)n_copy * tile_bytes);
              for (int i = 0; i < n_copy; ++i)
                bulk_g2s(stage0 + (uint32_t)i * tile_bytes, src + (size_t)i * part_stride, tile_bytes,
                         bar(ctrl->red_copy), policy_evict_first());
            }
            if (!wait_warp(bar(ctrl->red_copy), 0, wc)) {
              if (dq == 0 && lane == 0) wait_drain(bar(ctrl->red_copy), 0, wc);  // the copies land before exit
              break;
            }
          }
        }
      }
      float* part = p.partials + (size_t)blockIdx.x * ((size_t)p.bn * kTileN);
      // accumulators holding units of this tile: both, or the one of its only unit
      const bool alt = nacc == 2 && !p.split_n;
      const bool two = alt && seg_len >= 2;
      const uint32_t d_first = (alt && seg_len == 1) ? (uint32_t)(((u - u_begin) & 1) * p.bn) : 0u;
      bool got = true, go_seen = !reducer;
      for (int cc = wg; cc < p.bn / 8; cc += kNumDqWG) {
        uint32_t r[8], r1[8];
        if (!W4A16_IN_RANGE(p.status, d_first + (uint32_t)cc * 8, 8, kTmemCols, 29) ||
            (two && !W4A16_IN_RANGE(p.status, (uint32_t)(p.bn + cc * 8), 8, kTmemCols, 29))) {
          got = false;
          break;
        }
        tmem_ld_x8(tmem + lane_off + d_first + (uint32_t)cc * 8, r);
        if (two) tmem_ld_x8(tmem + lane_off + (uint32_t)(p.bn + cc * 8), r1);
        tmem_wait_ld();
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          acc[c] = two ? __uint_as_float(r[c]) + __uint_as_float(r1[c]) : __uint_as_float(r[c]);
        if (reducer) {
          // own partial first, then the others' in stripe order (fixed order,
          // bit-reproducible); each word is re-zeroed once read
          uint32_t off[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) off[c] = (uint32_t)((cc * 8 + c) * kTileN + row);
          long long q0 = c_first + 1;
          if (cc == wg && preloaded) {
            // the first contributor, loaded before the accumulator wait (its
            // range was checked then)
            float* base = p.partials + (size_t)q0 * part_stride;
            if (!poll_partials<1, 8>(base, part_stride, off, 1, pre, wc, true)) { got = false; break; }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              acc[c] += partial_value(pre[c]);
              __stcg(base + off[c], 0.f);
            }
            ++q0;
          }
          if constexpr (BULK) {
            for (; q0 <= c_first + n_copy; ++q0) {
              // a contributor copied in bulk: its words from the ring
              const uint32_t sb = stage0 + (uint32_t)(q0 - c_first - 1) * tile_bytes;
              float* base = p.partials + (size_t)q0 * part_stride;
              uint32_t raw[8];
#pragma unroll
              for (int c = 0; c < 8; ++c) raw[c] = lds_u32(sb + 4u * off[c]);
              if (!poll_partials<1, 8>(base, part_stride, off, 1, raw, wc, true)) { got = false; break; }
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                acc[c] += partial_value(raw[c]);
                __stcg(base + off[c], 0.f);
              }
            }
          }
          if constexpr (BULK) {
            for (; q0 <= c_last && got; ++q0) {
              // contributors beyond the ring's room: polled from global memory
              float* base = p.partials + (size_t)q0 * part_stride;
              if (!W4A16_IN_RANGE(p.status, (const char*)base - (const char*)p.status, 4 * part_stride,
                                  p.ws_bytes, 31)) { got = false; break; }
              uint32_t raw[8];
              if (!poll_partials<1, 8>(base, part_stride, off, 1, raw, wc)) { got = false; break; }
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                acc[c] += partial_value(raw[c]);
                __stcg(base + off[c], 0.f);
              }
            }
          } else {
            for (; q0 <= c_last && got; q0 += 2) {
              const int nq = (int)min(2LL, c_last - q0 + 1);
              float* base = p.partials + (size_t)q0 * part_stride;
              // the partial tiles of contributors q0 .. q0 + nq - 1 this thread polls
              if (!W4A16_IN_RANGE(p.status, (const char*)base - (const char*)p.status,
                                  4 * (size_t)nq * part_stride, p.ws_bytes, 31)) { got = false; break; }
              uint32_t raw[16];
              if (!poll_partials<2, 8>(base, part_stride, off, nq, raw, wc)) { got = false; break; }
#pragma unroll
              for (int j = 0; j < 2; ++j)
                if (j < nq) {
#pragma unroll
                  for (int c = 0; c < 8; ++c) {
                    acc[c] += partial_value(raw[j * 8 + c]);
                    __stcg(base + j * part_stride + off[c], 0.f);
                  }
                }
            }
          }
          if (!got) break;
          if (!go_seen) {
            if (!wait_warp(bar(ctrl->red_go), 0, wc) || *reinterpret_cast<volatile int*>(&ctrl->abort)) {
              got = false;
              break;
            }
            go_seen = true;
          }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int m = cc * 8 + c;
          if (whole || reducer) {
            if (m_base + m < p.M &&
                W4A16_IN_RANGE(p.status, (size_t)(m_base + m) * p.N + y_col, 1, (size_t)p.M * p.N, 30))
              p.Y[(size_t)(m_base + m) * p.N + y_col] = __half_as_ushort(__float2half_rn(acc[c]));
          } else if (W4A16_IN_RANGE(p.status, (const char*)(part + (size_t)m * kTileN + row) - (const char*)p.status,
                                    4, p.ws_bytes, 31)) {
            st_partial(part + (size_t)m * kTileN + row, acc[c]);
          }
        }
      }
      if (!got) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(ctrl->dempty));
      ++seg;
      u += seg_len;
      ku = 0;
      ++tile;
    }
  }

  // ---- teardown -------------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t gemm_set_smem_limit(int bytes) {
  cudaError_t e = cudaFuncSetAttribute(w4a16_gemm_kernel<false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(w4a16_gemm_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(w4a16_gemm_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(w4a16_gemm_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

cudaError_t launch_gemm(const CUtensorMap& x_map, const GemmParams& p, int grid, uint32_t smem_bytes,
                        cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool bulk = p.bn > 32;
  if (p.zeros)
    return bulk ? cudaLaunchKernelEx(&cfg, w4a16_gemm_kernel<true, true>, x_map, p)
                : cudaLaunchKernelEx(&cfg, w4a16_gemm_kernel<true, false>, x_map, p);
  return bulk ? cudaLaunchKernelEx(&cfg, w4a16_gemm_kernel<false, true>, x_map, p)
              : cudaLaunchKernelEx(&cfg, w4a16_gemm_kernel<false, false>, x_map, p);
}

}  // namespace w4a16

// common.cuh -- device helpers shared by the fused kernels: bounded mbarrier
// waits, the striped partition arithmetic, and the exact 4-bit -> fp16
// dequantisation of one operand fragment.
#pragma once

#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace w4a16 {

// Where a CTA records that it gave up: a shared abort flag (so the other roles
// stop quickly), the device status word, and the per-wait time limit.
struct WaitCtx {
  int* abort;
  int* status;
  unsigned long long timeout_ns;
};

// ---- bounded waits ----------------------------------------------------------
// Each wait sleeps inside mbarrier.try_wait (woken when the phase completes)
// and checks the abort flag and the global timer between sleeps.  The loops
// are kept small and not unrolled: the kernel's roles run different code and
// share one instruction cache.

static __device__ __noinline__ void raise_timeout(const WaitCtx& c) {
  *reinterpret_cast<volatile int*>(c.abort) = 1;
  atomicOr(c.status, kStatusTimeout);
}

// Slow path of a wait: returns false when the CTA is aborting or the wait expired.
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const WaitCtx& c) {
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(c.abort)) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      raise_timeout(c);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool wait_thread(uint32_t bar, uint32_t parity, const WaitCtx& c) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, c);
}

// Whole-warp wait with a warp-uniform outcome.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& c) {
  return __all_sync(0xffffffffu, wait_thread(bar, parity, c));
}

// Wait used while tearing down: ignores the abort flag, still bounded.
static __device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, const WaitCtx& c) {
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > c.timeout_ns) {
      atomicOr(c.status, kStatusTimeout);
      return;
    }
  }
}

// ---- bounds checks (MARLIN_DEBUG builds) --------------------------------------------
// W4A16_IN_RANGE(status, off, len, size, site) is true when [off, off + len)
// lies inside [0, size).  In a MARLIN_DEBUG build a failing check sets
// kStatusBounds in the status word, records `site` in the word after it (the
// first failure wins) and returns false, and the caller skips the access; a
// copy that is skipped leaves its barrier incomplete, so the waits expire
// (bounded) and the kernel returns.  Nothing traps.  In other builds the macro
// is the constant true and its arguments are not evaluated.
#ifdef MARLIN_DEBUG
static __device__ __noinline__ void bounds_fail(int* status, int site) {
  atomicCAS(status + 1, 0, site);
  atomicOr(status, kStatusBounds);
}
__device__ __forceinline__ bool in_range_dbg(int* status, unsigned long long off, unsigned long long len,
                                             unsigned long long size, int site) {
  if (off + len <= size) return true;
  bounds_fail(status, site);
  return false;
}
#define W4A16_IN_RANGE(status, off, len, size, site)                                          \
  ::w4a16::in_range_dbg((status), (unsigned long long)(off), (unsigned long long)(len),       \
                        (unsigned long long)(size), (site))
#else
#define W4A16_IN_RANGE(status, off, len, size, site) true
#endif

// Shared-memory extent check: `addr` is a shared-window address, `raw` the
// address of the dynamic shared memory's first byte.
#define W4A16_SMEM_OK(p, raw, addr, len, site) \
  W4A16_IN_RANGE((p).status, (addr) - (raw), (len), (p).smem_bytes, (site))

// ---- striped partition --------------------------------------------------------

// First unit of CTA c's stripe: floor(c * U / G).
__device__ __forceinline__ long long stripe_begin(long long c, long long U, long long G) {
  return (c * U) / G;
}

// CTA whose stripe holds unit u (every stripe is non-empty because G <= U).
__device__ __forceinline__ long long stripe_owner(long long u, long long U, long long G) {
  return ((u + 1) * G - 1) / U;
}

// ---- split-tile reduction across CTAs ----------------------------------------------
// A column tile cut by stripe boundaries is finished by its reducer: the CTA
// that owns the tile's first unit.  For that CTA the tile is always its last
// segment (its stripe ends inside the tile), and for every other contributor
// the tile is its first segment (its stripe starts inside the tile).  So each
// CTA publishes at most one partial tile (from its first segment, then goes on
// without waiting) and reduces at most one (at its very end), and no CTA ever
// waits for a CTA that is itself waiting: the wait graph has no cycles.
// Contributors publish their partial words tagged (st_partial); the reducer
// polls the words it needs with bounded waits and leaves them zeroed.  No
// arrival count is kept: the tags alone tell the reducer a word is final.  The
// workspace's counter block (one int per tile) is read only by bounds-checked
// (MARLIN_DEBUG) builds, whose reducers wait for their tile's word to be
// non-negative, so that a test can make that wait expire.

__device__ __forceinline__ long long tile_reducer(long long tile, long long KT, long long U,
                                                  long long G) {
  return stripe_owner(tile * KT, U, G);
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Partial tiles of split tiles are published element by element: a partial
// value v is stored as bits(v) ^ kPartTag, so that a zero word means "not
// written yet" (the workspace starts zeroed and the reducer re-zeroes what it
// read).  No fp32 result has the bits of kPartTag (a signalling-NaN payload
// that arithmetic never produces), so a written word is never zero, and the
// reducer needs no ordering between a contributor's stores: each word it
// polls is either absent or final.
constexpr uint32_t kPartTag = 0x7F800001u;

__device__ __forceinline__ void st_partial(float* p, float v) {
  __stcg(reinterpret_cast<unsigned int*>(p), __float_as_uint(v) ^ kPartTag);
}

// An L2 load (not cached in L1) of one tagged word.  Each word is written
// once per call and validates itself, so a plain cache-global load suffices;
// measured, strong (relaxed.gpu) loads of a batch of words took several times
// longer to come back.
__device__ __forceinline__ uint32_t ld_partial_raw(const float* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float partial_value(uint32_t raw) { return __uint_as_float(raw ^ kPartTag); }

// Loads of the words base[q * stride + off[i]] (q < nq, i < NO) into
// raw[q * NO + i] (0 for q >= nq), issued together; a reducer issues them
// ahead of other work so that their round trip overlaps it.
template <int NQ, int NO>
__device__ __forceinline__ void issue_partials(const float* base, size_t stride, const uint32_t (&off)[NO],
                                               int nq, uint32_t (&raw)[NQ * NO]) {
#pragma unroll
  for (int q = 0; q < NQ; ++q)
#pragma unroll
    for (int i = 0; i < NO; ++i) raw[q * NO + i] = q < nq ? ld_partial_raw(base + q * stride + off[i]) : 0u;
}

// Bounded poll until the words base[q * stride + off[i]] (q < nq, i < NO) are
// all written, into raw[q * NO + i]; returns false on timeout (recorded) or
// when the CTA is aborting.  With preloaded, raw already holds the words'
// values from issue_partials (a zero word is not written yet, and is loaded
// again); otherwise every word is loaded here.
template <int NQ, int NO>
__device__ __forceinline__ bool poll_partials(const float* base, size_t stride, const uint32_t (&off)[NO],
                                              int nq, uint32_t (&raw)[NQ * NO], const WaitCtx& c,
                                              bool preloaded = false) {
  if (!preloaded) {
#pragma unroll
    for (int i = 0; i < NQ * NO; ++i) raw[i] = 0u;
  }
  uint64_t t0 = 0;
#pragma unroll 1
  for (int attempt = 0;; ++attempt) {
    // issue every missing word's load first, then test them all: the loads
    // are in flight together (one round trip per attempt)
    if (attempt > 0 || !preloaded) {
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q < nq) {
#pragma unroll
          for (int i = 0; i < NO; ++i)
            if (raw[q * NO + i] == 0u) raw[q * NO + i] = ld_partial_raw(base + q * stride + off[i]);
        }
    }
    bool done = true;
#pragma unroll
    for (int q = 0; q < NQ; ++q)
      if (q < nq) {
#pragma unroll
        for (int i = 0; i < NO; ++i) done = done && raw[q * NO + i] != 0u;
      }
    if (done) return true;
    if (*reinterpret_cast<volatile int*>(c.abort)) return false;
    if (attempt == 0) {
      t0 = global_timer_ns();
    } else if (global_timer_ns() - t0 > c.timeout_ns) {
      raise_timeout(c);
      return false;
    }
    __nanosleep(64);
  }
}


// Bounded spin until *counter reaches `expected` (acquire).  Returns false on
// timeout (recorded in the status word) or when the CTA is aborting.
static __device__ __noinline__ bool wait_counter(const int* counter, int expected, const WaitCtx& c) {
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (ld_acquire_gpu(counter) < expected) {
    if (*reinterpret_cast<volatile int*>(c.abort)) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      raise_timeout(c);
      return false;
    }
    __nanosleep(100);
  }
  return true;
}

// ---- dequantisation -------------------------------------------------------------

// One 32-bit word of 8 codes -> the four fp16 pairs of a 16x16 operand
// fragment: h[0] = column r, rows k..k+1; h[1] = column r+8, rows k..k+1;
// h[2] = column r, rows k+2..k+3; h[3] = column r+8, rows k+2..k+3 (the
// nibble order the repack writes).  0x6400 | c is 1024 + c exactly (binary16
// ulp is 1 on [1024, 2048)); 0x6400 | (c << 4) is 1024 + 16c.  Subtracting
// 1024 + z (or scaling by 1/16 and adding -(64 + z)) gives q - z exactly; the
// single rounding of the dequantisation is the final multiply by the scale.
// Arguments are fp16 pairs in 32-bit registers.  The blocks of PTX below
// implement this for one word and feed the result straight to its consumer.

// This dequantisation fused with the tensor-core multiply-accumulates that
// consume it, as one block of PTX: the four fp16 pairs are produced directly in
// the registers the mma.sync A operand reads (written as separate statements,
// the compiler surrounds them with register moves).  NB mma.sync.m16n8k16 share
// the A fragment, one per block of 8 tokens: acc[nb] += A * B[nb].
#define W4A16_DEQ_PTX(W, SUB, ADD, S, S8, K16)                            \
  ".reg .b32 t0, t1, t2, t3, w8;\n\t"                                     \
  "lop3.b32 t0, " W ", 0x000F000F, 0x64006400, 0xEA;\n\t"                \
  "lop3.b32 t1, " W ", 0x00F000F0, 0x64006400, 0xEA;\n\t"                \
  "shr.u32 w8, " W ", 8;\n\t"                                             \
  "lop3.b32 t2, w8, 0x000F000F, 0x64006400, 0xEA;\n\t"                    \
  "lop3.b32 t3, w8, 0x00F000F0, 0x64006400, 0xEA;\n\t"                    \
  "sub.rn.f16x2 t0, t0, " SUB ";\n\t"                                     \
  "fma.rn.f16x2 t1, t1, " K16 ", " ADD ";\n\t"                           \
  "sub.rn.f16x2 t2, t2, " SUB ";\n\t"                                     \
  "fma.rn.f16x2 t3, t3, " K16 ", " ADD ";\n\t"                           \
  "mul.rn.f16x2 t0, t0, " S ";\n\t"                                       \
  "mul.rn.f16x2 t1, t1, " S8 ";\n\t"                                      \
  "mul.rn.f16x2 t2, t2, " S ";\n\t"                                       \
  "mul.rn.f16x2 t3, t3, " S8 ";\n\t"
#define W4A16_MMA_PTX(D0, D1, D2, D3, B0, B1)                                                     \
  "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {" D0 ", " D1 ", " D2 ", " D3 "}, "           \
  "{t0, t1, t2, t3}, {" B0 ", " B1 "}, {" D0 ", " D1 ", " D2 ", " D3 "};\n\t"

template <int NB>
__device__ __forceinline__ void dequant_mma(float (&acc)[NB][4], uint32_t w, uint32_t sub_r,
                                            uint32_t add_r8, uint32_t s_r, uint32_t s_r8,
                                            const uint2 (&b)[NB]) {
  const uint32_t k16 = 0x2C002C00u;  // 1/16 as an fp16 pair (an operand, so it is materialised once)
  if constexpr (NB == 1) {
    asm volatile("{\n\t" W4A16_DEQ_PTX("%4", "%5", "%6", "%7", "%8", "%11")
                 W4A16_MMA_PTX("%0", "%1", "%2", "%3", "%9", "%10") "}"
                 : "+f"(acc[0][0]), "+f"(acc[0][1]), "+f"(acc[0][2]), "+f"(acc[0][3])
                 : "r"(w), "r"(sub_r), "r"(add_r8), "r"(s_r), "r"(s_r8), "r"(b[0].x), "r"(b[0].y), "r"(k16));
  } else if constexpr (NB == 2) {
    asm volatile("{\n\t" W4A16_DEQ_PTX("%8", "%9", "%10", "%11", "%12", "%17")
                 W4A16_MMA_PTX("%0", "%1", "%2", "%3", "%13", "%14")
                 W4A16_MMA_PTX("%4", "%5", "%6", "%7", "%15", "%16") "}"
                 : "+f"(acc[0][0]), "+f"(acc[0][1]), "+f"(acc[0][2]), "+f"(acc[0][3]),
                   "+f"(acc[1][0]), "+f"(acc[1][1]), "+f"(acc[1][2]), "+f"(acc[1][3])
                 : "r"(w), "r"(sub_r), "r"(add_r8), "r"(s_r), "r"(s_r8), "r"(b[0].x), "r"(b[0].y),
                   "r"(b[1].x), "r"(b[1].y), "r"(k16));
  } else if constexpr (NB == 3) {
    asm volatile("{\n\t" W4A16_DEQ_PTX("%12", "%13", "%14", "%15", "%16", "%23")
                 W4A16_MMA_PTX("%0", "%1", "%2", "%3", "%17", "%18")
                 W4A16_MMA_PTX("%4", "%5", "%6", "%7", "%19", "%20")
                 W4A16_MMA_PTX("%8", "%9", "%10", "%11", "%21", "%22") "}"
                 : "+f"(acc[0][0]), "+f"(acc[0][1]), "+f"(acc[0][2]), "+f"(acc[0][3]),
                   "+f"(acc[1][0]), "+f"(acc[1][1]), "+f"(acc[1][2]), "+f"(acc[1][3]),
                   "+f"(acc[2][0]), "+f"(acc[2][1]), "+f"(acc[2][2]), "+f"(acc[2][3])
                 : "r"(w), "r"(sub_r), "r"(add_r8), "r"(s_r), "r"(s_r8), "r"(b[0].x), "r"(b[0].y),
                   "r"(b[1].x), "r"(b[1].y), "r"(b[2].x), "r"(b[2].y), "r"(k16));
  } else {
    static_assert(NB == 4, "NB must be 1..4");
    asm volatile("{\n\t" W4A16_DEQ_PTX("%16", "%17", "%18", "%19", "%20", "%29")
                 W4A16_MMA_PTX("%0", "%1", "%2", "%3", "%21", "%22")
                 W4A16_MMA_PTX("%4", "%5", "%6", "%7", "%23", "%24")
                 W4A16_MMA_PTX("%8", "%9", "%10", "%11", "%25", "%26")
                 W4A16_MMA_PTX("%12", "%13", "%14", "%15", "%27", "%28") "}"
                 : "+f"(acc[0][0]), "+f"(acc[0][1]), "+f"(acc[0][2]), "+f"(acc[0][3]),
                   "+f"(acc[1][0]), "+f"(acc[1][1]), "+f"(acc[1][2]), "+f"(acc[1][3]),
                   "+f"(acc[2][0]), "+f"(acc[2][1]), "+f"(acc[2][2]), "+f"(acc[2][3]),
                   "+f"(acc[3][0]), "+f"(acc[3][1]), "+f"(acc[3][2]), "+f"(acc[3][3])
                 : "r"(w), "r"(sub_r), "r"(add_r8), "r"(s_r), "r"(s_r8), "r"(b[0].x), "r"(b[0].y),
                   "r"(b[1].x), "r"(b[1].y), "r"(b[2].x), "r"(b[2].y), "r"(b[3].x), "r"(b[3].y), "r"(k16));
  }
}

// Dequantise the four fragment words of one 16-column group (k-steps 0..3 of a
// 64-row chunk) and store them to tensor memory as the A operand with one
// tcgen05.st.16x256b.x4, all in one block of PTX (so the 16 results are
// produced directly in the store's source registers).  Register order per
// repetition: (col r, k..k+1), (col r, k+2..k+3), (col r+8, k..k+1),
// (col r+8, k+2..k+3).
#define W4A16_DEQW_PTX(W, SUB, ADD, S, S8, X)                          \
  "shr.u32 w8, " W ", 8;\n\t"                                          \
  "lop3.b32 t0_" X ", " W ", 0x000F000F, 0x64006400, 0xEA;\n\t"        \
  "lop3.b32 t1_" X ", " W ", 0x00F000F0, 0x64006400, 0xEA;\n\t"        \
  "lop3.b32 t2_" X ", w8, 0x000F000F, 0x64006400, 0xEA;\n\t"           \
  "lop3.b32 t3_" X ", w8, 0x00F000F0, 0x64006400, 0xEA;\n\t"           \
  "sub.rn.f16x2 t0_" X ", t0_" X ", " SUB ";\n\t"                      \
  "fma.rn.f16x2 t1_" X ", t1_" X ", k16, " ADD ";\n\t"                 \
  "sub.rn.f16x2 t2_" X ", t2_" X ", " SUB ";\n\t"                      \
  "fma.rn.f16x2 t3_" X ", t3_" X ", k16, " ADD ";\n\t"                 \
  "mul.rn.f16x2 t0_" X ", t0_" X ", " S ";\n\t"                        \
  "mul.rn.f16x2 t1_" X ", t1_" X ", " S8 ";\n\t"                       \
  "mul.rn.f16x2 t2_" X ", t2_" X ", " S ";\n\t"                        \
  "mul.rn.f16x2 t3_" X ", t3_" X ", " S8 ";\n\t"

// The same dequantisation into registers, in the store's register order, for
// callers that store later (after waiting for a free tensor-memory slot).
__device__ __forceinline__ void dequant16(uint4 w, uint32_t sub_r, uint32_t add_r8, uint32_t s_r,
                                          uint32_t s_r8, uint32_t (&o)[16]) {
  asm volatile(
      "{\n\t.reg .b32 w8, k16, t0_0, t1_0, t2_0, t3_0, t0_1, t1_1, t2_1, t3_1, t0_2, t1_2, t2_2, "
      "t3_2, t0_3, t1_3, t2_3, t3_3;\n\t"
      "mov.b32 k16, 0x2C002C00;\n\t"
      W4A16_DEQW_PTX("%16", "%20", "%21", "%22", "%23", "0")
      W4A16_DEQW_PTX("%17", "%20", "%21", "%22", "%23", "1")
      W4A16_DEQW_PTX("%18", "%20", "%21", "%22", "%23", "2")
      W4A16_DEQW_PTX("%19", "%20", "%21", "%22", "%23", "3")
      "mov.b32 %0, t0_0;\n\tmov.b32 %1, t2_0;\n\tmov.b32 %2, t1_0;\n\tmov.b32 %3, t3_0;\n\t"
      "mov.b32 %4, t0_1;\n\tmov.b32 %5, t2_1;\n\tmov.b32 %6, t1_1;\n\tmov.b32 %7, t3_1;\n\t"
      "mov.b32 %8, t0_2;\n\tmov.b32 %9, t2_2;\n\tmov.b32 %10, t1_2;\n\tmov.b32 %11, t3_2;\n\t"
      "mov.b32 %12, t0_3;\n\tmov.b32 %13, t2_3;\n\tmov.b32 %14, t1_3;\n\tmov.b32 %15, t3_3;\n\t"
      "}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]), "=r"(o[4]), "=r"(o[5]), "=r"(o[6]),
        "=r"(o[7]), "=r"(o[8]), "=r"(o[9]), "=r"(o[10]), "=r"(o[11]), "=r"(o[12]), "=r"(o[13]),
        "=r"(o[14]), "=r"(o[15])
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(sub_r), "r"(add_r8), "r"(s_r), "r"(s_r8));
}

__device__ __forceinline__ void dequant_store_tmem(uint32_t taddr, uint4 w, uint32_t sub_r,
                                                   uint32_t add_r8, uint32_t s_r, uint32_t s_r8) {
  asm volatile(
      "{\n\t.reg .b32 w8, k16, t0_0, t1_0, t2_0, t3_0, t0_1, t1_1, t2_1, t3_1, t0_2, t1_2, t2_2, "
      "t3_2, t0_3, t1_3, t2_3, t3_3;\n\t"
      "mov.b32 k16, 0x2C002C00;\n\t"
      W4A16_DEQW_PTX("%1", "%5", "%6", "%7", "%8", "0")
      W4A16_DEQW_PTX("%2", "%5", "%6", "%7", "%8", "1")
      W4A16_DEQW_PTX("%3", "%5", "%6", "%7", "%8", "2")
      W4A16_DEQW_PTX("%4", "%5", "%6", "%7", "%8", "3")
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {t0_0, t2_0, t1_0, t3_0, t0_1, t2_1, t1_1, "
      "t3_1, t0_2, t2_2, t1_2, t3_2, t0_3, t2_3, t1_3, t3_3};\n\t"
      "}" ::"r"(taddr),
      "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(sub_r), "r"(add_r8), "r"(s_r), "r"(s_r8)
      : "memory");
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Per-column constants of the dequantisation: 1024 + z and -(64 + z) as fp16
// pairs, and the scale broadcast to both halves.
struct ColConst {
  uint32_t sub, add, s;
};

__device__ __forceinline__ ColConst col_const(uint16_t s_bits, uint32_t z) {
  const uint32_t sub_u = 0x6400u | z;
  const uint32_t add_u = 0xD400u | (z << 4);
  ColConst k;
  k.sub = sub_u | (sub_u << 16);
  k.add = add_u | (add_u << 16);
  k.s = (uint32_t)s_bits | ((uint32_t)s_bits << 16);
  return k;
}

}  // namespace w4a16

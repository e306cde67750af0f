// api.cu -- the C ABI declared in include/marlin.h: argument checks, the
// partition plan, the X tensor map, and the kernel launches.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "kernels.h"
#include "marlin.h"

using namespace w4a16;

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

struct DeviceState {
  bool init = false;
  int sms = 0;
  int smem_optin = 0;
  bool smem_set = false;
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

marlin_status_t device_state(int device, DeviceState** out) {
  if (device < 0 || device >= kMaxDevices) return MARLIN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_dev[device];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
            cudaSuccess)
      return MARLIN_ERR_CUDA;
    d.init = true;
  }
  *out = &d;
  return MARLIN_OK;
}

marlin_status_t get_encoder() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_encode) return MARLIN_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return MARLIN_ERR_CUDA;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return MARLIN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_shape(int K, int N) { return K > 0 && N > 0 && K % 128 == 0 && N % 128 == 0; }

// Shape and group check shared by every entry point.  group -1 means K.  A
// group that divides K but is not a multiple of 128 (32, 64: sizes some
// quantisers produce, which the pages say "may not run") is a valid request
// this library does not serve: MARLIN_ERR_UNSUPPORTED.  Anything else that is
// not a positive divisor of K, or a bad shape: MARLIN_ERR_INVALID_ARG.
marlin_status_t check_shape_group(int K, int N, int* group) {
  if (!valid_shape(K, N)) return MARLIN_ERR_INVALID_ARG;
  if (*group == -1) *group = K;
  if (*group <= 0 || K % *group != 0) return MARLIN_ERR_INVALID_ARG;
  return *group % 128 == 0 ? MARLIN_OK : MARLIN_ERR_UNSUPPORTED;
}

// Largest M served by the warp-level kernel (mma.sync fed from registers);
// larger M uses the tcgen05 kernel.  Measured crossover, each kernel forced,
// calls graph-replayed on rotating weights: the warp-level kernel is
// 1.04-1.11x faster at M = 16 (4096x12288, 8192x8192, 8192x57344), the tcgen05
// kernel 1.03-1.11x faster at M = 24.  (Launched alone and cold under ncu, the
// tcgen05 kernel already wins at M = 16 on 8192x8192, by 1.04x.)
// W4A16_SMALL_M_MAX overrides it (0..32, 0 disables the warp-level path), e.g.
// to test either kernel at any M.
int small_m_max() {
  static int v = [] {
    const char* e = getenv("W4A16_SMALL_M_MAX");
    int x = e ? atoi(e) : 16;
    return x < 0 ? 0 : (x > kMaxWarpM ? kMaxWarpM : x);
  }();
  return v;
}

// Whether the kernels read the first ring of weights before waiting for the
// previous kernel in the stream (programmatic dependent launch).  The weights
// are then treated as constant: they must not be written by a kernel that is
// still running when the multiply is enqueued.  W4A16_EARLY_WEIGHTS=0 turns
// it off.
bool early_weights() {
  static bool v = [] {
    const char* e = getenv("W4A16_EARLY_WEIGHTS");
    return !(e && atoi(e) == 0);
  }();
  return v;
}

// Recently encoded tensor maps of X, per host thread (direct-mapped).
struct XMapEntry {
  CUtensorMap map;
  const void* X;
  int M, K, bn;
  bool valid;
};
constexpr int kXMapSlots = 64;
thread_local XMapEntry t_xmaps[kXMapSlots];

int xmap_slot(const void* X, int M, int K, int bn) {
  uint64_t h = (uint64_t)reinterpret_cast<uintptr_t>(X) >> 8;
  h ^= (uint64_t)M * 0x9E3779B97F4A7C15ull ^ (uint64_t)K * 0xC2B2AE3D27D4EB4Full ^ (uint64_t)bn;
  h ^= h >> 29;
  return (int)(h & (kXMapSlots - 1));
}

// The partition plan.  A unit is one (m-tile, 128-column tile, K slice of
// cpu*64 rows); the grid is one CTA per SM (fewer if there are fewer units),
// each taking an equal contiguous stripe of units.
// kernel: MARLIN_KERNEL_AUTO picks by M (small_m_max); the others force one.
// sparse: 2:4 weights (the warp-level kernel; stages carry the kept codes and
// their index nibbles instead of the dense codes).
GemmPlan make_plan(int M, int K, int N, int group, int sms, int smem_optin, bool has_zeros,
                   int kernel = MARLIN_KERNEL_AUTO, bool sparse = false) {
  GemmPlan g{};
  g.n_tiles = N / kTileN;
  const int budget = smem_optin - kCtrlBytes - 1024;  // control block + alignment slack
  const bool warp_level =
      kernel == MARLIN_KERNEL_WARP || (kernel == MARLIN_KERNEL_AUTO && M <= small_m_max());
  if (warp_level) {
    // tokens in blocks of 8 (the mma.sync N dimension), at most 32 per m-tile;
    // larger batches (the 2:4 path only) take several m-tiles of 32
    g.kind = kKernelSmallM;
    g.bn = M <= kMaxWarpM ? 8 * ((M + 7) / 8) : kMaxWarpM;
    if (g.bn < 8) g.bn = 8;
    g.m_tiles = (M + g.bn - 1) / g.bn;
    // 256-row units wherever K and the group allow them.  Measured: also on
    // small problems, where 128-row units gave more units per SM but twice the
    // per-unit overhead per byte (4096x4096 M = 1: 6.57 -> 6.18 us; 2048x2048:
    // 5.50 -> 4.80 us; larger shapes unchanged).
    const bool can4 = K % 256 == 0 && (group == 128 || group % 256 == 0);
    g.cpu = can4 ? 4 : 2;
  } else {
    g.kind = kKernelTcgen05;
    g.bn = M <= kMaxBn ? (int)round_up((size_t)M, 16) : kMaxBn;
    g.m_tiles = (M + g.bn - 1) / g.bn;
    // two MMA issuers: for bn <= 128 on alternate units, each into its own
    // accumulator; above, on every unit, splitting the bn token columns of one
    // accumulator at 128 (so each issues MMAs of N <= 128)
    g.nacc = 2;
    g.split_n = g.bn > 128 ? 1 : 0;
    g.cpu = 2;
    // A slots (one unit of cpu*64 rows = cpu*32 columns each) fill the tensor
    // memory above the accumulators; an even count of at least 4 keeps every
    // waiter within one phase of the slot barriers
    const int a_cols = g.cpu * kChunkK / 2;
    int slots = (kTmemCols - (g.split_n ? 1 : g.nacc) * g.bn) / a_cols;
    if (slots > kAStages) slots = kAStages;
    g.a_slots = slots & ~1;
  }
  g.kt = K / (kChunkK * g.cpu);
  g.n_g = (g.cpu * kChunkK > group) ? (g.cpu * kChunkK) / group : 1;
  g.upg = (group > g.cpu * kChunkK) ? group / (g.cpu * kChunkK) : 1;
  g.units = (long long)g.m_tiles * g.n_tiles * g.kt;
  g.grid = (int)(g.units < sms ? g.units : sms);
  // Short stripes (under 240 KB of weight codes per SM): one SM in 19 is left
  // idle.  Measured with back-to-back calls on 152 SMs, 144 CTAs beat 152 by
  // 2-10% on 4096x4096, 4096x12288, 11008x4096, 2048x5632, 13824x5120 and
  // 8192x8192 (warp-level kernel at M = 1 and 16, tcgen05 kernel at M = 32..64)
  // and tied at 215-250 KB per SM; above that (4096x22016, 8192x10240) the
  // full grid is faster.
  // Very short stripes (at most 128 KB of codes per CTA): the largest grid of at
  // least 4/5 of the SMs that gives every CTA the same whole number of units
  // and splits every column tile evenly, if there is one.  Measured on
  // 4096x4096: 128 CTAs against 144, warp-level kernel M = 1 6.22 -> 5.85 us,
  // M = 16 7.98 -> 7.64 us, tcgen05 kernel M = 32 11.09 -> 9.71 us.  The
  // 128 KB bound holds for the warp-level kernel only: at 256 KB per CTA
  // (8192x8192) its even split was 2-4% slower than 144 CTAs, while the
  // tcgen05 kernel's was faster (8192x8192 at M = 32 / 64 / 128: 17.22 /
  // 20.10 / 28.31 -> 16.41 / 18.44 / 25.52 us), its epilogue per piece of a
  // split tile (accumulator read-back and partial write of bn x 128 fp32)
  // costing far more than the warp-level kernel's.
  {
    const long long unit_code_bytes =
        (long long)g.cpu * (sparse ? kSpChunkCodeBytes + kSpChunkMetaBytes : kChunkCodeBytes);
    const bool capped = g.kind == kKernelSmallM;
    if (g.grid == sms && g.units * unit_code_bytes < 240LL * 1024 * sms) {
      g.grid = sms - sms / 19;
      for (int G = sms; G * 5 >= sms * 4; --G) {
        const long long per = g.units / G;
        if (g.units % G == 0 && g.kt % per == 0 &&
            (!capped || per * unit_code_bytes <= 128LL * 1024)) {
          g.grid = G;
          break;
        }
      }
      // tcgen05 kernel without an even split: a tile can have up to
      // ceil(kt * G / units) contributors, which its reducer polls two at a
      // time, one L2 round trip (about 1.5 us under load) each.  Take the
      // largest grid (of at least 4/5 of the SMs) below the chosen one that
      // needs fewer rounds, if any.  Measured: 11008x4096 at M = 32, 144 -> 128
      // CTAs (three rounds -> two), 14.65 -> 13.26 us; every other measured
      // shape keeps its grid (4096x12288 M = 32: one round at 144 already).
      if (g.kind == kKernelTcgen05 && g.units % g.grid != 0) {
        auto rounds = [&](long long G) { return ((g.kt * G + g.units - 1) / g.units + 1) / 2; };
        const long long r0 = rounds(g.grid);
        for (int G = g.grid - 1; G * 5 >= sms * 4; --G)
          if (rounds(G) < r0) {
            g.grid = G;
            break;
          }
      }
    }
  }
  const size_t x_chunk = (size_t)g.bn * 128;
  const size_t chunk_w = sparse ? (size_t)(kSpChunkCodeBytes + kSpChunkMetaBytes) : kChunkCodeBytes;
  const size_t stage = g.cpu * (x_chunk + chunk_w) +
                       (size_t)g.n_g * (kTileN * 2 + (has_zeros ? kTileN / 2 : 0));
  g.stage_bytes = (uint32_t)round_up(stage, 1024);
  const size_t xchg = g.kind == kKernelSmallM ? (size_t)4 * (g.bn / 8) * 256 * sizeof(float) : 0;
  int stages = (int)((budget - (long long)xchg) / (long long)g.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  // Warp-level kernel: a ring of about 110 KB (at least 4 stages), not as many
  // stages as fit.  Every CTA keeps its whole ring of weight copies in flight
  // (at the start, before the dependency wait, too); 110 KB on 144 SMs is
  // still twice the bandwidth-latency product.  Measured, graph-replayed:
  // M = 1 on the 7B shapes 2.5-5% faster (4096x22016: 14.38 -> 13.80 us),
  // 8192x10240 M = 1..4 3-4%, 2:4 weights at M = 1 up to 10% (4096x22016:
  // 12.66 -> 11.38 us); M = 16 within 1% either way; 3 stages were slower
  // again.  The tcgen05 kernel keeps every stage that fits: fewer were slower
  // at M = 32..64.
  if (g.kind == kKernelSmallM) {
    const int ring = (int)((110 * 1024) / g.stage_bytes);
    const int cap = ring > 4 ? ring : 4;
    if (stages > cap) stages = cap;
  }
  // tcgen05 kernel: each dequant warpgroup takes a fixed residue of the unit
  // index mod 4.  With a stage count that is a multiple of 4 a warpgroup only
  // waits on its own stages.  Where rounding down would cost a large share of
  // a short ring (big X tiles at large bn), every stage that fits is kept and
  // the warpgroups track every stage's phase instead (measured: faster for
  // rings of 3..7 stages, slower for 9 -> 8).
  if (g.kind == kKernelTcgen05 && stages >= 8) stages &= ~3;
  g.stages = stages;
  g.off_xchg = (uint32_t)((size_t)stages * g.stage_bytes);
  g.smem_bytes = (uint32_t)(kCtrlBytes + 1024 + (size_t)stages * g.stage_bytes + xchg);
  // workspace: [status 256 B][counters][partials]
  g.ws_counters_off = 256;
  g.ws_partials_off = round_up(g.ws_counters_off + sizeof(int) * (size_t)g.m_tiles * g.n_tiles, 256);
  // one fp32 partial tile (bn x 128) per CTA: a CTA publishes at most one
  // (from its first segment); sized for #SMs CTAs, the most any plan launches
  g.ws_bytes = g.ws_partials_off + (size_t)sms * g.bn * kTileN * sizeof(float);
  return g;
}

marlin_status_t current_device(int* dev) {
  return cudaGetDevice(dev) == cudaSuccess ? MARLIN_OK : MARLIN_ERR_CUDA;
}

// The checks, the plan and the launch shared by marlin_gemm_ex and
// marlin_sparse_gemm.  meta != nullptr: the 2:4-sparse variant (packed and
// meta in the sparse tile layout; warp-level kernel only).
marlin_status_t run_gemm(const uint16_t* X, const void* packed, const void* meta,
                         const uint16_t* scales, const int32_t* zeros, uint16_t* Y, int M, int K,
                         int N, int group, void* workspace, size_t workspace_bytes, int kernel,
                         marlin_stream_t stream) {
  const bool sparse = meta != nullptr;
  if (M < 0) return MARLIN_ERR_INVALID_ARG;
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  if (!sparse && kernel == MARLIN_KERNEL_WARP && M > kMaxWarpM) return MARLIN_ERR_UNSUPPORTED;
  if (sparse) kernel = MARLIN_KERNEL_WARP;
  if (M == 0) return MARLIN_OK;
  if (!X || !packed || !scales || !Y || !workspace) return MARLIN_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(packed) || !aligned16(scales) || (zeros && !aligned16(zeros)) ||
      (meta && !aligned16(meta)) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(Y) & 1u))
    return MARLIN_ERR_MISALIGNED;
  int dev;
  marlin_status_t s = current_device(&dev);
  if (s != MARLIN_OK) return s;
  DeviceState* d;
  if ((s = device_state(dev, &d)) != MARLIN_OK) return s;
  if ((s = get_encoder()) != MARLIN_OK) return s;

  const GemmPlan g = make_plan(M, K, N, group, d->sms, d->smem_optin, zeros != nullptr, kernel, sparse);
  if (g.stages < 2 || g.units > 0x7FFFFFFFLL / 2) return MARLIN_ERR_UNSUPPORTED;
  if (g.kind == kKernelTcgen05 && g.a_slots < 4) return MARLIN_ERR_UNSUPPORTED;
  if (workspace_bytes < g.ws_bytes) return MARLIN_ERR_WORKSPACE_TOO_SMALL;

  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d->smem_set) {
      if (gemm_set_smem_limit(d->smem_optin) != cudaSuccess ||
          small_m_set_smem_limit(d->smem_optin) != cudaSuccess)
        return MARLIN_ERR_CUDA;
      d->smem_set = true;
    }
  }

  // X's tensor map depends only on (address, M, K, box rows): keep the last
  // few per host thread, so a decode loop over fixed buffers encodes each once
  // bn <= 64: X as [K/64][M][64] (the same bytes: row stride K * 2, chunk stride
  // 128 bytes) with a box of one unit's cpu chunks, so that one tensor copy
  // lands a whole unit's X exactly as cpu boxes of the 2-D map would.  Measured
  // against one copy per chunk: warp-level kernel 1-3% faster (8192x57344 M = 1:
  // 53.9 -> 52.5 us), tcgen05 kernel up to 3% faster at M = 32..64 (8192x57344
  // M = 64: 78.3 -> 75.8 us) but 1-4% slower at bn = 128 and 256.
  const bool x3 = g.bn <= 64;
  const int xkey = g.bn + (x3 ? 1000 * g.cpu : 0);
  XMapEntry& xe = t_xmaps[xmap_slot(X, M, K, xkey)];
  if (!(xe.valid && xe.X == X && xe.M == M && xe.K == K && xe.bn == xkey)) {
    const cuuint64_t dims[3] = {(cuuint64_t)(x3 ? kChunkK : K), (cuuint64_t)M, (cuuint64_t)(K / kChunkK)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)kChunkK * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kChunkK, (cuuint32_t)g.bn, (cuuint32_t)g.cpu};
    const cuuint32_t estr[3] = {1, 1, 1};
    xe.valid = false;
    if (g_encode(&xe.map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x3 ? 3 : 2, const_cast<uint16_t*>(X), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MARLIN_ERR_CUDA;
    xe.X = X;
    xe.M = M;
    xe.K = K;
    xe.bn = xkey;
    xe.valid = true;
  }
  const CUtensorMap& x_map = xe.map;

  GemmParams p{};
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.codes = static_cast<const uint32_t*>(packed);
  p.meta = static_cast<const uint32_t*>(meta);
  p.scales = scales;
  p.zeros = reinterpret_cast<const uint8_t*>(zeros);
  p.Y = Y;
  p.status = reinterpret_cast<int*>(ws);
  p.counters = reinterpret_cast<int*>(ws + g.ws_counters_off);
  p.partials = reinterpret_cast<float*>(ws + g.ws_partials_off);
  p.M = M;
  p.K = K;
  p.N = N;
  p.group = group;
  p.G = K / group;
  p.bn = g.bn;
  p.m_tiles = g.m_tiles;
  p.n_tiles = g.n_tiles;
  p.kt = g.kt;
  p.cpu = g.cpu;
  p.units = g.units;
  p.stages = g.stages;
  p.stage_bytes = g.stage_bytes;
  p.x_chunk_bytes = (uint32_t)g.bn * 128;
  p.off_codes = (uint32_t)g.cpu * p.x_chunk_bytes;
  p.off_meta = p.off_codes + (uint32_t)g.cpu * (sparse ? kSpChunkCodeBytes : kChunkCodeBytes);
  p.off_scales = sparse ? p.off_meta + (uint32_t)g.cpu * kSpChunkMetaBytes : p.off_meta;
  p.off_zeros = p.off_scales + (uint32_t)g.n_g * kTileN * 2;
  p.weights_reused = g.m_tiles > 1;
  p.nacc = g.nacc > 0 ? g.nacc : 1;
  p.split_n = g.split_n;
  p.split_h = g.bn > 128 ? 128 : (int)round_up((size_t)(g.bn / 2), 16);
  p.full_all = (g.stages % 4) != 0;
  p.a_slots = g.a_slots;
  p.a_base = (uint32_t)(kTmemCols - g.a_slots * g.cpu * (kChunkK / 2));
  p.tx_w = (uint32_t)g.cpu * kChunkCodeBytes + (uint32_t)g.n_g * (kTileN * 2 + (zeros ? kTileN / 2 : 0));
  p.tx_x = (uint32_t)g.cpu * p.x_chunk_bytes;
  p.n_g = g.n_g;
  p.units_per_group = g.upg;
  p.off_xchg = g.off_xchg;
  p.timeout_ns = kDefaultTimeoutNs;
  p.early_weights = early_weights() ? 1 : 0;
  p.x3d = g.bn <= 64 ? 1 : 0;
  p.even_split = (g.units % g.grid == 0 && g.kt % (g.units / g.grid) == 0) ? 1 : 0;
  // extents for the bounds-checked build: the logical sizes of the caller's buffers
  {
    const size_t Gr = (size_t)(K / group);
    p.codes_bytes = sparse ? (size_t)K * N / 4 : (size_t)K * N / 2;
    p.meta_bytes = sparse ? (size_t)K * N / 8 : 0;
    p.scales_bytes = Gr * N * 2;
    p.zeros_bytes = zeros ? Gr * N / 2 : 0;
    p.ws_bytes = workspace_bytes;
    p.smem_bytes = g.smem_bytes;
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = g.kind == kKernelSmallM
                            ? launch_small_m(x_map, p, g.grid, g.smem_bytes, sparse, st)
                            : launch_gemm(x_map, p, g.grid, g.smem_bytes, st);
  if (e != cudaSuccess) return MARLIN_ERR_CUDA;
  return MARLIN_OK;
}

}  // namespace

namespace w4a16 {

// Workspace bytes of the plan marlin_gemm (automatic kernel choice) uses for
// this call on the current device; a marlin_status_t value.
int call_workspace_bytes(int M, int K, int N, int group, bool has_zeros, size_t* bytes) {
  if (!bytes || M < 0) return MARLIN_ERR_INVALID_ARG;
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  int dev;
  marlin_status_t s = current_device(&dev);
  if (s != MARLIN_OK) return s;
  DeviceState* d;
  if ((s = device_state(dev, &d)) != MARLIN_OK) return s;
  *bytes = make_plan(M > 0 ? M : 1, K, N, group, d->sms, d->smem_optin, has_zeros).ws_bytes;
  return MARLIN_OK;
}

}  // namespace w4a16

extern "C" {

const char* marlin_status_string(marlin_status_t s) {
  switch (s) {
    case MARLIN_OK: return "MARLIN_OK";
    case MARLIN_ERR_INVALID_ARG: return "MARLIN_ERR_INVALID_ARG";
    case MARLIN_ERR_UNSUPPORTED: return "MARLIN_ERR_UNSUPPORTED";
    case MARLIN_ERR_MISALIGNED: return "MARLIN_ERR_MISALIGNED";
    case MARLIN_ERR_WORKSPACE_TOO_SMALL: return "MARLIN_ERR_WORKSPACE_TOO_SMALL";
    case MARLIN_ERR_CUDA: return "MARLIN_ERR_CUDA";
    case MARLIN_ERR_TIMEOUT: return "MARLIN_ERR_TIMEOUT";
    case MARLIN_ERR_BOUNDS: return "MARLIN_ERR_BOUNDS";
  }
  return "MARLIN_ERR_UNKNOWN";
}

marlin_status_t marlin_packed_layout(int K, int N, int group, int has_zeros, size_t* bytes,
                                     size_t* off_scales, size_t* off_zeros) {
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  const size_t G = (size_t)(K / group);
  const size_t codes = (size_t)K * N / 2;
  const size_t sc = round_up(codes, 256);
  const size_t zo = round_up(sc + G * N * 2, 256);
  const size_t total = has_zeros ? zo + G * N / 2 : zo;
  if (bytes) *bytes = total;
  if (off_scales) *off_scales = sc;
  if (off_zeros) *off_zeros = has_zeros ? zo : total;
  return MARLIN_OK;
}

marlin_status_t marlin_repack(const int32_t* q, const uint16_t* scales, const int32_t* zeros, int K,
                              int N, int group, void* out, marlin_stream_t stream) {
  if (!q || !scales || !out) return MARLIN_ERR_INVALID_ARG;
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  if (!aligned16(q) || !aligned16(scales) || !aligned16(out) || (zeros && !aligned16(zeros)))
    return MARLIN_ERR_MISALIGNED;
  size_t bytes, off_s, off_z;
  marlin_packed_layout(K, N, group, zeros != nullptr, &bytes, &off_s, &off_z);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* o = static_cast<uint8_t*>(out);
  const size_t G = (size_t)(K / group);
  if (launch_repack(reinterpret_cast<const uint32_t*>(q), reinterpret_cast<uint32_t*>(o), K, N, st) !=
      cudaSuccess)
    return MARLIN_ERR_CUDA;
  if (launch_tile_major(scales, o + off_s, (int)G, N, kTileN * 2, st) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  if (zeros && launch_tile_major(zeros, o + off_z, (int)G, N, kTileN / 2, st) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  return MARLIN_OK;
}

marlin_status_t marlin_workspace_bytes(int M, int K, int N, int group, int device, size_t* bytes) {
  if (!bytes || M < 0) return MARLIN_ERR_INVALID_ARG;
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  DeviceState* d;
  marlin_status_t s = device_state(device, &d);
  if (s != MARLIN_OK) return s;
  // the workspace must serve either kernel for every M' <= M (its size grows
  // with M' for each kernel; the warp-level one serves M' <= 32)
  const int m = M > 0 ? M : 1;
  size_t need = make_plan(m, K, N, group, d->sms, d->smem_optin, true, MARLIN_KERNEL_TCGEN05).ws_bytes;
  const GemmPlan w = make_plan(m < kMaxWarpM ? m : kMaxWarpM, K, N, group, d->sms, d->smem_optin, true,
                               MARLIN_KERNEL_WARP);
  if (w.ws_bytes > need) need = w.ws_bytes;
  if (m > kMaxWarpM) {
    // the 2:4 path at this M: m-tiles of 32 tokens, one int per (tile, m-tile)
    const GemmPlan sp = make_plan(m, K, N, group, d->sms, d->smem_optin, true, MARLIN_KERNEL_WARP, true);
    if (sp.ws_bytes > need) need = sp.ws_bytes;
  }
  *bytes = need;
  return MARLIN_OK;
}

marlin_status_t marlin_gemm(const uint16_t* X, const void* packed, const uint16_t* scales,
                            const int32_t* zeros, uint16_t* Y, int M, int K, int N, int group,
                            void* workspace, size_t workspace_bytes, marlin_stream_t stream) {
  return marlin_gemm_ex(X, packed, scales, zeros, Y, M, K, N, group, workspace, workspace_bytes,
                        MARLIN_KERNEL_AUTO, stream);
}

marlin_status_t marlin_gemm_ex(const uint16_t* X, const void* packed, const uint16_t* scales,
                               const int32_t* zeros, uint16_t* Y, int M, int K, int N, int group,
                               void* workspace, size_t workspace_bytes, marlin_kernel_t kernel,
                               marlin_stream_t stream) {
  if (kernel != MARLIN_KERNEL_AUTO && kernel != MARLIN_KERNEL_WARP && kernel != MARLIN_KERNEL_TCGEN05)
    return MARLIN_ERR_INVALID_ARG;
  return run_gemm(X, packed, nullptr, scales, zeros, Y, M, K, N, group, workspace, workspace_bytes,
                  kernel, stream);
}

marlin_status_t marlin_gemm_host(const uint16_t* X_host, uint16_t* X_dev, const void* packed,
                                 const uint16_t* scales, const int32_t* zeros, uint16_t* Y_dev,
                                 uint16_t* Y_host, int M, int K, int N, int group,
                                 void* workspace, size_t workspace_bytes, marlin_stream_t stream) {
  if (M < 0) return MARLIN_ERR_INVALID_ARG;
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  if (M == 0) return MARLIN_OK;
  if (!X_host || !Y_host || !X_dev || !Y_dev || !packed || !scales || !workspace)
    return MARLIN_ERR_INVALID_ARG;
  if (!aligned16(X_dev) || !aligned16(packed) || !aligned16(scales) || (zeros && !aligned16(zeros)) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(Y_dev) & 1u))
    return MARLIN_ERR_MISALIGNED;
  {
    int dev;
    DeviceState* d;
    marlin_status_t s = current_device(&dev);
    if (s != MARLIN_OK) return s;
    if ((s = device_state(dev, &d)) != MARLIN_OK) return s;
    const GemmPlan g = make_plan(M, K, N, group, d->sms, d->smem_optin, zeros != nullptr);
    if (workspace_bytes < g.ws_bytes) return MARLIN_ERR_WORKSPACE_TOO_SMALL;
  }
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(X_dev, X_host, (size_t)M * K * 2, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  const marlin_status_t s = marlin_gemm(X_dev, packed, scales, zeros, Y_dev, M, K, N, group, workspace,
                                        workspace_bytes, stream);
  if (s != MARLIN_OK) return s;
  if (cudaMemcpyAsync(Y_host, Y_dev, (size_t)M * N * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  return MARLIN_OK;
}

// ---- 2:4-sparse variant ----------------------------------------------------------

marlin_status_t marlin_sparse_packed_layout(int K, int N, int group, int has_zeros, size_t* bytes,
                                            size_t* off_meta, size_t* off_scales, size_t* off_zeros) {
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  const size_t G = (size_t)(K / group);
  const size_t codes = (size_t)K * N / 4;
  const size_t me = round_up(codes, 256);
  const size_t sc = round_up(me + (size_t)K * N / 8, 256);
  const size_t zo = round_up(sc + G * N * 2, 256);
  const size_t total = has_zeros ? zo + G * N / 2 : zo;
  if (bytes) *bytes = total;
  if (off_meta) *off_meta = me;
  if (off_scales) *off_scales = sc;
  if (off_zeros) *off_zeros = has_zeros ? zo : total;
  return MARLIN_OK;
}

marlin_status_t marlin_sparse_repack(const int32_t* q, const uint16_t* scales, const int32_t* zeros,
                                     int K, int N, int group, void* out, int* bad_groups,
                                     marlin_stream_t stream) {
  if (!q || !scales || !out) return MARLIN_ERR_INVALID_ARG;
  if (const marlin_status_t c = check_shape_group(K, N, &group)) return c;
  if (!aligned16(q) || !aligned16(scales) || !aligned16(out) || (zeros && !aligned16(zeros)) ||
      (reinterpret_cast<uintptr_t>(bad_groups) & 3u))
    return MARLIN_ERR_MISALIGNED;
  size_t bytes, off_m, off_s, off_z;
  marlin_sparse_packed_layout(K, N, group, zeros != nullptr, &bytes, &off_m, &off_s, &off_z);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* o = static_cast<uint8_t*>(out);
  const size_t G = (size_t)(K / group);
  if (launch_sparse_repack(reinterpret_cast<const uint32_t*>(q), reinterpret_cast<const uint32_t*>(zeros),
                           K, N, group, reinterpret_cast<uint32_t*>(o),
                           reinterpret_cast<uint32_t*>(o + off_m), bad_groups, st) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  if (launch_tile_major(scales, o + off_s, (int)G, N, kTileN * 2, st) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  if (zeros && launch_tile_major(zeros, o + off_z, (int)G, N, kTileN / 2, st) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  return MARLIN_OK;
}

marlin_status_t marlin_sparse_gemm(const uint16_t* X, const void* packed, const void* meta,
                                   const uint16_t* scales, const int32_t* zeros, uint16_t* Y, int M,
                                   int K, int N, int group, void* workspace, size_t workspace_bytes,
                                   marlin_stream_t stream) {
  if (!meta) return MARLIN_ERR_INVALID_ARG;
  return run_gemm(X, packed, meta, scales, zeros, Y, M, K, N, group, workspace, workspace_bytes,
                  MARLIN_KERNEL_WARP, stream);
}

marlin_status_t marlin_last_device_status(void* workspace, marlin_stream_t stream) {
  if (!workspace) return MARLIN_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MARLIN_ERR_CUDA;
  int status[2] = {0, 0};
  if (cudaMemcpy(status, workspace, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  if (status[0] != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpy(workspace, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MARLIN_ERR_CUDA;
    return (status[0] & kStatusBounds) ? MARLIN_ERR_BOUNDS : MARLIN_ERR_TIMEOUT;
  }
  return MARLIN_OK;
}

}  // extern "C"

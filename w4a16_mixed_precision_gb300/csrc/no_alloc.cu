// no_alloc.cu -- marlin_gemm_no_alloc: the fused W4A16 multiply for callers
// that cannot allocate device memory.  The scratch that marlin_gemm keeps in
// the caller's workspace (status word, one int per tile, fp32 partial tiles of
// the split reduction) lives here in a library-owned static device
// array instead; every GPU that loads the library holds it until the process
// exits.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "marlin.h"

namespace {

// Maximum scratch: 8 MiB.  On a 152-SM GB300 this covers every problem up to
// M = 96 tokens (one fp32 partial tile of 96 x 128 per SM, plus counters).
constexpr size_t kScratchBytes = (size_t)8 << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, so the address must come from the
// runtime: looked up once per device, with that device current.
marlin_status_t scratch_on(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return MARLIN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_lock);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MARLIN_ERR_CUDA;
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return MARLIN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" marlin_status_t marlin_gemm_no_alloc(const uint16_t* X, const void* packed,
                                                const uint16_t* scales, const int32_t* zeros,
                                                uint16_t* Y, int M, int K, int N, int group,
                                                marlin_stream_t stream) {
  if (M == 0) return MARLIN_OK;
  if (!X || !packed || !scales || !Y) return MARLIN_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(packed) || !aligned16(scales) || (zeros && !aligned16(zeros)) ||
      (reinterpret_cast<uintptr_t>(Y) & 1u))
    return MARLIN_ERR_MISALIGNED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MARLIN_ERR_CUDA;
  // the scratch this very call uses (its kernel and M), not the worst case
  size_t need = 0;
  marlin_status_t s = static_cast<marlin_status_t>(
      w4a16::call_workspace_bytes(M, K, N, group, zeros != nullptr, &need));
  if (s != MARLIN_OK) return s;
  if (need > kScratchBytes) return MARLIN_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if ((s = scratch_on(dev, &scratch)) != MARLIN_OK) return s;
  // The array keeps the previous call's contents.  Everything this call uses
  // must start at zero: the status word, the per-tile ints (which a
  // bounds-checked build's reducers wait on), and the partial-tile words (a
  // zero word means "not yet written").  A completed call
  // leaves them zeroed, but one whose kernel gave up on a bounded wait may not,
  // and this entry point does not report that; so clear this call's region.
  if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MARLIN_ERR_CUDA;
  return marlin_gemm(X, packed, scales, zeros, Y, M, K, N, group, scratch, kScratchBytes, stream);
}

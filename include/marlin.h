/*
 * marlin.h -- C ABI of the GB300 (sm_103a) W4A16 fused matrix multiply
 *
 *     Y[M][N] = X[M][K] . dequant(W)[K][N],   dequant(w) = fp16((q - z) * s)
 *
 * The operation is the one the Marlin pages define: "Marlin / GPTQ-Marlin"
 * (brain.gartu.xyz), section "Le problème": every linear layer computes
 * Y = X_fp16 x W_int4, the INT4 weights dequantised to FP16 on the fly;
 * "Marlin" (dingiv.github.io), section "Group size 为什么是 128": one fp16
 * scale (and one zero point) per group of 128 consecutive K elements of a
 * column; section "反量化精度权衡": FP16 operands, FP32 accumulation, FP16
 * output.
 *
 * Conventions for every entry point
 *   - Device pointers are CUDA device addresses on the current device; host
 *     pointers are marked "host".  The caller owns and allocates every buffer;
 *     the library allocates no device memory.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream) unless
 *     stated otherwise, and never synchronises, except
 *     marlin_last_device_status.
 *   - Argument errors are detected on the host before anything is launched; the
 *     call then returns the error code and touches nothing.
 *   - fp16 data is passed as raw 16-bit IEEE-754 binary16 (`uint16_t`).
 *
 * Data formats
 *   X       fp16 [M][K], row-major (K contiguous), 16-byte aligned base.
 *   q       GPTQ order: int32 [K/8][N]; bits 4i..4i+3 of word [r][n] hold the
 *           code q[8r+i][n], q in 0..15.
 *   scales  fp16 [K/group][N] (row j = group j).
 *   zeros   int32 [K/group][N/8]; bits 4j..4j+3 of word [g][c] hold z[g][8c+j]
 *           (stored literally, no offset).  NULL means z = 8 everywhere.
 *   group   128, any multiple of 128 that divides K, or K (or -1 meaning K)
 *           for one scale per column.  A group that divides K but is not a
 *           multiple of 128 (32, 64) -> MARLIN_ERR_UNSUPPORTED ("Marlin",
 *           section "Group size 为什么是 128": 64 and 256 run slower and 32
 *           may not run); any other group -> MARLIN_ERR_INVALID_ARG.
 *   Shapes  K % 128 == 0, N % 128 == 0, M >= 0 (M == 0 is a no-op).
 */
#ifndef W4A16_GB300_MARLIN_H
#define W4A16_GB300_MARLIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* marlin_stream_t; /* same type as cudaStream_t */

typedef enum {
  MARLIN_OK = 0,
  MARLIN_ERR_INVALID_ARG = 1,          /* bad shape, group, NULL pointer          */
  MARLIN_ERR_UNSUPPORTED = 2,          /* valid request this library cannot serve
                                          (group 32/64, M > 32 on the warp path)   */
  MARLIN_ERR_MISALIGNED = 3,           /* a pointer is not 16-byte aligned        */
  MARLIN_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace smaller than required        */
  MARLIN_ERR_CUDA = 5,                 /* a CUDA runtime call or launch failed    */
  MARLIN_ERR_TIMEOUT = 6,              /* a bounded wait inside a kernel gave up  */
  MARLIN_ERR_BOUNDS = 7                /* bounds-checked build only: a kernel
                                          formed an address outside its buffer    */
} marlin_status_t;

/* Human-readable name of a status code (static string, never NULL).  No page
 * passage: housekeeping of this library, not the method's arithmetic. */
const char* marlin_status_string(marlin_status_t status);

/*
 * Size and offsets of the single repacked weight buffer, laid out as
 * [codes | scales | zeros].  The pages fix no format for the repacked weights
 * ("Marlin / GPTQ-Marlin", section "Tiled layout et repacking", says only that
 * they are rewritten into a tiled layout); this is the size query for this
 * library's own layout:
 *   codes  K*N/2 bytes in this library's tile layout (see marlin_repack);
 *   scales fp16, K*N/group values, at *off_scales (tile-major, see marlin_repack);
 *   zeros  K*N/(2*group) bytes at *off_zeros (only if has_zeros; *off_zeros =
 *          *bytes otherwise), tile-major, see marlin_repack.
 * All offsets are multiples of 256 bytes.  Host-only, no CUDA call.
 * bytes, off_scales, off_zeros: host pointers, each may be NULL.
 */
marlin_status_t marlin_packed_layout(int K, int N, int group, int has_zeros, size_t* bytes,
                                     size_t* off_scales, size_t* off_zeros);

/*
 * Offline repack ("reshuffle" of the weights into a tile layout, done once at
 * load time): "Marlin / GPTQ-Marlin", section "Tiled layout et repacking";
 * "Marlin Project Overview" (vecbase.com), section "Key Techniques", item
 * "Reshuffling".
 *
 * q       device, int32 [K/8][N] GPTQ order (read only).
 * scales  device, fp16 [K/group][N] (read only).
 * zeros   device, int32 [K/group][N/8], or NULL for z = 8 (read only).
 * out     device, marlin_packed_layout(K, N, group, zeros != NULL) bytes,
 *         16-byte aligned, written.  Must not overlap the inputs.
 * Layout of `out` (the operand order of a 16x16 fp16 tensor-core fragment):
 *   codes   32-bit word ((nt*(K/64) + kb)*8 + g)*128 + l*4 + j, for nt < N/128,
 *           kb < K/64, g < 8, l < 32, j < 4, holds at bits 4p..4p+3 (p = 0..7)
 *           the code q[k][n] with n = nt*128 + 16g + l/4 + 8*(p & 1) and
 *           k = kb*64 + 16j + 4*(l % 4) + 2*((p >> 1) & 1) + (p >> 2);
 *   scales  fp16 [N/128][K/group][128] at off_scales: scale (gi, n) at
 *           ((n/128)*(K/group) + gi)*128 + n%128;
 *   zeros   bytes [N/128][K/group][64] at off_zeros: the 64-byte slice
 *           zeros[gi][16*(n/128) .. 16*(n/128)+15] at ((n/128)*(K/group) + gi)*64.
 * Errors: INVALID_ARG (shape/group/NULL), MISALIGNED, CUDA (launch).
 */
marlin_status_t marlin_repack(const int32_t* q, const uint16_t* scales, const int32_t* zeros, int K,
                              int N, int group, void* out, marlin_stream_t stream);

/*
 * Bytes of device workspace marlin_gemm needs for this problem on `device`
 * (its SM count sets the partition).  "Marlin Project Overview", section
 * "Key Techniques", item "Striped Partitioning", names the global reduction
 * this scratch serves; the size query itself has no page passage.
 * The workspace holds one fp32 partial tile per CTA for the striped
 * partition's global reduction, one int per output tile (read only by
 * bounds-checked MARLIN_DEBUG builds, whose reducers wait for it to be
 * non-negative; it must start at zero) and a status word.  A buffer sized for M also serves every smaller M with the
 * same K, N, group, with either kernel (marlin_gemm_ex).  Host-only; queries
 * the device attributes once.  bytes: host pointer, written.
 */
marlin_status_t marlin_workspace_bytes(int M, int K, int N, int group, int device, size_t* bytes);

/*
 * The fused W4A16 matrix multiply: Y = X . dequant(W) with fp32 accumulation
 * and fp16 output (round to nearest even; overflow gives +-inf).
 * "Marlin / GPTQ-Marlin", sections "Le problème" and "Architecture générale"
 * (one kernel fuses the dequantisation and the GEMM); "Marlin Project
 * Overview", section "Key Techniques", item "Striped Partitioning" (the SM
 * partition with global reduction).
 *
 * X          device, fp16 [M][K] row-major, 16-byte aligned (read only).
 * packed     device, the codes region of a marlin_repack output (offset 0).
 * scales     device, the scales region of the repacked buffer (packed + off_scales).
 * zeros      device, the zeros region (packed + off_zeros), or NULL for z = 8.
 * Y          device, fp16 [M][N] row-major, written; must not overlap inputs.
 * workspace  device, >= marlin_workspace_bytes(...) bytes, 16-byte aligned.
 *            Zero it once after allocating; every call leaves it zeroed again
 *            (after a call that reports MARLIN_ERR_TIMEOUT, zero it again).
 *            Calls that share a workspace must be ordered (same stream, or
 *            events): concurrent calls on one workspace race.
 * Result is deterministic: the same inputs give bit-identical Y on every run.
 * Weights (packed, scales, zeros) are treated as constant: the kernel may
 * start streaming them before the previous kernel on `stream` has finished
 * (programmatic dependent launch); X, Y and workspace are touched only after
 * it has.  So the weight buffers must not be written by a kernel that is
 * still running when this call is enqueued.  Writes by marlin_repack /
 * marlin_sparse_repack, by copies, or by any kernel that does not trigger
 * its dependents early are complete in time.  The environment variable
 * W4A16_EARLY_WEIGHTS=0 makes the kernels wait before reading anything.
 * Errors: INVALID_ARG, MISALIGNED, WORKSPACE_TOO_SMALL (host checks, nothing
 * launched); CUDA (launch failure).  A bounded wait that expires inside the
 * kernel is reported later by marlin_last_device_status.
 */
marlin_status_t marlin_gemm(const uint16_t* X, const void* packed, const uint16_t* scales,
                            const int32_t* zeros, uint16_t* Y, int M, int K, int N, int group,
                            void* workspace, size_t workspace_bytes, marlin_stream_t stream);

/*
 * Which fused kernel marlin_gemm_ex launches.  The pages' kernel is one
 * design; this library has two for the same operation: a warp-level one
 * (mma.sync fed from registers, M <= 32) and a tcgen05 one (operand in tensor
 * memory, any M).  MARLIN_KERNEL_AUTO picks by M (the warp-level kernel for
 * M <= 16, or the bound set by the environment variable W4A16_SMALL_M_MAX,
 * 0..32).
 */
typedef enum {
  MARLIN_KERNEL_AUTO = 0,
  MARLIN_KERNEL_WARP = 1,
  MARLIN_KERNEL_TCGEN05 = 2
} marlin_kernel_t;

/*
 * marlin_gemm with the kernel chosen by the caller (e.g. by a per-shape tuner
 * that times both).  Same arguments, results and errors as marlin_gemm; the
 * two kernels agree within the parity tolerance but not bit for bit (their
 * fp32 summation orders differ).  kernel: a marlin_kernel_t; other values ->
 * MARLIN_ERR_INVALID_ARG; MARLIN_KERNEL_WARP with M > 32 ->
 * MARLIN_ERR_UNSUPPORTED.  A workspace sized by marlin_workspace_bytes for M
 * serves either kernel.
 */
marlin_status_t marlin_gemm_ex(const uint16_t* X, const void* packed, const uint16_t* scales,
                               const int32_t* zeros, uint16_t* Y, int M, int K, int N, int group,
                               void* workspace, size_t workspace_bytes, marlin_kernel_t kernel,
                               marlin_stream_t stream);

/*
 * marlin_gemm without a caller-provided workspace.  The Marlin pages have no
 * counterpart to this entry point.
 *
 * For callers that cannot allocate device memory: an operator embedded in a
 * host framework whose memory planner owns all device memory and hands the
 * operator only its inputs and outputs, or code on a latency-critical path
 * where the implicit device synchronisation of cudaMalloc/cudaFree is not
 * acceptable.  The scratch that marlin_gemm keeps in `workspace` lives here in
 * a static device array of the library (8 MiB, held by every GPU that loads
 * the library until the process exits).  This call allocates nothing.
 *
 * Arguments as for marlin_gemm, without workspace.  Results are identical to
 * marlin_gemm's for the same inputs.
 * Limit: problems whose scratch exceeds 8 MiB (on a 152-SM GB300, M > 96)
 * return MARLIN_ERR_WORKSPACE_TOO_SMALL before anything is launched; other
 * argument errors as for marlin_gemm.
 * Set-up: the first call on a device looks up the array's device address
 * (once per device, with that device current); make that first call before
 * any stream capture.  Each call clears the part of the array it uses (status
 * word, tile counters, partial tiles) on `stream` before launching.
 * All calls share one array: calls that overlap on the GPU (different
 * streams, or different host threads on one device without ordering) race and
 * give wrong results.  A bounded wait that expires inside the kernel is
 * recorded only in the library's array and is not reported.
 */
marlin_status_t marlin_gemm_no_alloc(const uint16_t* X, const void* packed, const uint16_t* scales,
                                     const int32_t* zeros, uint16_t* Y, int M, int K, int N,
                                     int group, marlin_stream_t stream);

/*
 * marlin_gemm with X and Y in host memory, as an inference loop that keeps
 * activations on the host would call it.  The pages give no host-buffer form
 * of the call; this one only adds the two copies around marlin_gemm.
 *
 * On `stream`, in order: copy X_host (fp16 [M][K], M*K*2 bytes) into X_dev,
 * run marlin_gemm(X_dev, ..., Y_dev, ...), copy Y_dev (fp16 [M][N]) into
 * Y_host.  One cudaMemcpyAsync per copy.
 * X_host, Y_host  host; page-locked memory keeps the copies asynchronous
 *                 (pageable memory works but the copies then synchronise the
 *                 host).  They must stay valid until the stream has passed this
 *                 call; Y_host is complete only after the stream is synchronised.
 * X_dev, Y_dev    device staging buffers owned by the caller, with the
 *                 alignment marlin_gemm requires; overwritten.
 * Other arguments and errors as for marlin_gemm; a failed copy returns
 * MARLIN_ERR_CUDA.  Argument errors are detected before anything is enqueued.
 */
marlin_status_t marlin_gemm_host(const uint16_t* X_host, uint16_t* X_dev, const void* packed,
                                 const uint16_t* scales, const int32_t* zeros, uint16_t* Y_dev,
                                 uint16_t* Y_host, int M, int K, int N, int group,
                                 void* workspace, size_t workspace_bytes, marlin_stream_t stream);

/*
 * ---- 2:4-sparse variant ----------------------------------------------------
 *
 * "Marlin" (dingiv.github.io), section "支持 2:4 稀疏加速": the weights are
 * pruned ahead of time so that two of every four are zero, at fixed
 * positions; "Marlin / GPTQ-Marlin" (brain.gartu.xyz), section "4. Support de
 * la sparsité 2:4 NVIDIA": after dequantisation the zeros are skipped and the
 * sparse tensor core multiplies only the kept half.
 *
 * This library's reading: a weight is zero exactly when its code equals its
 * zero point (dequant = (q - z) * s), and the four weights of a group are four
 * consecutive rows k = 4j .. 4j+3 of one column (along K, the direction the
 * sparse tensor core compresses).  Inputs are the dense formats above (q,
 * scales, zeros); the product is the same Y = X . dequant(W) as marlin_gemm's.
 * In each group the kept rows are those whose code differs from z, in
 * ascending order, completed with the lowest remaining rows.
 */

/*
 * Size and offsets of the repacked 2:4 buffer, laid out as
 * [codes | meta | scales | zeros]:
 *   codes  K*N/4 bytes: the two kept codes of every group (tile layout below);
 *   meta   K*N/8 bytes at *off_meta: a 4-bit index pair i0 | i1 << 2 per group;
 *   scales, zeros as in marlin_packed_layout, at *off_scales / *off_zeros.
 * All offsets are multiples of 256 bytes.  Host-only, no CUDA call; each
 * output pointer may be NULL.  Errors: INVALID_ARG (shape/group).
 */
marlin_status_t marlin_sparse_packed_layout(int K, int N, int group, int has_zeros, size_t* bytes,
                                            size_t* off_meta, size_t* off_scales, size_t* off_zeros);

/*
 * Offline repack of 2:4-sparse weights into the sparse tile layout.
 *
 * q, scales, zeros  device, the dense input formats (read only); zeros NULL
 *                   means z = 8.
 * out               device, marlin_sparse_packed_layout(...) bytes, 16-byte
 *                   aligned, written; must not overlap the inputs.
 * bad_groups        device int or NULL.  The repack adds to it (atomically)
 *                   the number of groups of four rows in which more than two
 *                   codes differ from z, i.e. where the weights are not 2:4;
 *                   such a group keeps its first two non-zero rows and the
 *                   product no longer equals the dense one.  Zero it before
 *                   the call and check it after the stream is synchronised.
 * Layout of `out` (the operand order of the 16 x 32 sparse fp16 tensor-core
 * fragment), per 128-column tile nt < N/128 and 64-row chunk kb < K/64:
 *   codes  32-bit word ((nt*(K/64) + kb)*8 + gq)*64 + l*2 + s (gq < 8, l < 32,
 *          s < 2) holds at bits 4p..4p+3 the kept code number p >> 2 of
 *          column n = nt*128 + 16gq + l/4 + 8*(p & 1) in group
 *          j = kb*16 + 8s + l%4 + 4*((p >> 1) & 1) (rows 4j .. 4j+3);
 *   meta   word ((nt*(K/64) + kb)*8 + gq)*32 + (r*2 + h)*2 + s (r < 8, h < 2,
 *          s < 2) at off_meta holds at bits 4i..4i+3 the index pair of column
 *          n = nt*128 + 16gq + r + 8*(i >> 2) in group j = kb*16 + 8s + 4h + (i & 3);
 *   scales, zeros as for marlin_repack.
 * Errors: INVALID_ARG (shape/group/NULL), MISALIGNED (16-byte buffers,
 * 4-byte bad_groups), CUDA (launch).
 */
marlin_status_t marlin_sparse_repack(const int32_t* q, const uint16_t* scales, const int32_t* zeros,
                                     int K, int N, int group, void* out, int* bad_groups,
                                     marlin_stream_t stream);

/*
 * Y = X . dequant(W) for 2:4-sparse weights: dequantises only the kept half
 * of the codes and multiplies with mma.sp on the warp-level path, in m-tiles
 * of up to 32 tokens (every M; above 32 tokens each m-tile reads the same
 * weights again, from L2).
 *
 * packed     device, the codes region of a marlin_sparse_repack output.
 * meta       device, the meta region (packed + off_meta); NULL -> INVALID_ARG.
 * scales     device, packed + off_scales.  zeros: packed + off_zeros or NULL.
 * X, Y, workspace, stream, determinism, errors: as for marlin_gemm; a
 * workspace sized by marlin_workspace_bytes(M, K, N, group, ...) serves this
 * call too (it covers every M it was sized for).  Results agree with
 * marlin_gemm's on the expanded weights within the parity tolerance (the
 * fp32 summation orders differ).  Only the kept terms enter the sum, so for
 * an inf or NaN in X at a dropped row the result is not specified here (the
 * dense product gives NaN there; a sum over the kept terms stays finite).
 */
marlin_status_t marlin_sparse_gemm(const uint16_t* X, const void* packed, const void* meta,
                                   const uint16_t* scales, const int32_t* zeros, uint16_t* Y, int M,
                                   int K, int N, int group, void* workspace, size_t workspace_bytes,
                                   marlin_stream_t stream);

/*
 * No page passage: failure reporting of this library's bounded waits.
 * Synchronises `stream`, reads and clears the device status word that
 * marlin_gemm keeps in `workspace`, and returns MARLIN_OK,
 * MARLIN_ERR_TIMEOUT (a bounded wait in a kernel expired; that call's Y is
 * not valid) or, from a library built with -DMARLIN_DEBUG (which checks
 * every address its kernels form against the extent of its buffer and skips
 * the access instead of faulting), MARLIN_ERR_BOUNDS; the 32-bit word at byte
 * 4 of the workspace then names the first failed check (cleared too).
 * workspace: device, as passed to marlin_gemm.
 */
marlin_status_t marlin_last_device_status(void* workspace, marlin_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_GB300_MARLIN_H */

/*
 * nvfp4_group_gemm.h -- C ABI of the GB300 (sm_103a) NVFP4 grouped GEMM.
 *
 * The operation (kernelbot nvfp4-group-gemm, submissions 474067, 482269 and
 * 496386; the header comment of the CUDA source of 474067 names the formats,
 * tcgen05_mma_nvfp4 the block-16 scaling, and custom_kernel the per-group
 * (A, B, C) lists with (M, N, K) problem sizes):
 *
 *   for every group g:
 *     C_g[m][n] = fp16( sum_{k<K_g} a(m,k) * sfa(m, k/16) * b(n,k) * sfb(n, k/16) )
 *
 * a, b are FP4 E2M1 codes, sfa, sfb FP8 E4M3FN scale factors (one per 16
 * consecutive K-elements), accumulation is FP32 on the tensor cores, the
 * output is FP16 rounded to nearest even.  C is overwritten: there is no C
 * input, alpha, beta or per-tensor global scale (the first MMA of every tile
 * runs with the accumulator disabled: 474067, group_gemm_persistent_kernel,
 * MMA warp).
 *
 * Conventions for every entry point:
 *  - All data pointers are DEVICE pointers on the current CUDA device, owned
 *    by the caller; descriptor arrays are HOST memory, read completely before
 *    the call returns.  Nothing is allocated per call.
 *  - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *    stream).  Return codes report argument validation and launch errors
 *    only; a timeout inside a kernel is reported later through
 *    nvfp4_last_device_error().
 *  - Validation happens before any launch: an invalid argument launches
 *    nothing.
 *  - Thread safety: calls from several host threads are safe; calls that
 *    overlap on the GPU must not share output buffers.
 */
#ifndef NVFP4_GROUP_GEMM_H
#define NVFP4_GROUP_GEMM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define NVFP4_OK                    0
#define NVFP4_ERR_INVALID_ARGUMENT (-1) /* null pointer, bad size, K % 256 != 0, N % 8 != 0 ... */
#define NVFP4_ERR_MISALIGNED       (-2) /* a pointer is not 16-byte aligned                       */
#define NVFP4_ERR_UNSUPPORTED      (-3) /* current device is not compute capability 10.3        */
#define NVFP4_ERR_CUDA             (-4) /* a CUDA runtime / driver call failed                   */
#define NVFP4_ERR_TIMEOUT          (-5) /* a bounded wait inside a kernel expired                */
#define NVFP4_ERR_TOO_MANY         (-6) /* a size exceeds a documented limit                     */

/* One GEMM problem of a grouped call.
 *  A    [M][K/2] bytes: E2M1 codes, K-major, two per byte, element 2i in the
 *       low nibble of byte i.  16-byte aligned.
 *  B    [N][K/2] bytes, same encoding.  16-byte aligned.
 *  SFA  M-side scales in the TILED layout written by nvfp4_sf_relayout
 *       (rows = M): nvfp4_sf_tiled_bytes(M, K) bytes.  16-byte aligned.
 *  SFB  N-side scales, tiled (rows = N): nvfp4_sf_tiled_bytes(N, K) bytes.
 *  C    [M][N] FP16, row-major, leading dimension N.  16-byte aligned.
 *  Sizes: M >= 0 (M == 0 makes the group a no-op), N >= 8 with N % 8 == 0,
 *  K >= 256 with K % 256 == 0, M, N, K <= 2^20. */
typedef struct GroupDesc {
    const void *A;
    const void *B;
    const void *SFA;
    const void *SFB;
    void *C;
    int M, N, K;
} GroupDesc;

/* Grouped GEMM over `num_groups` problems (1 <= num_groups <= 4096) in one
 * persistent, warp-specialised tcgen05 kernel per chunk of up to 32 groups.
 * Groups may differ in M, N and K.  Output tiles of all groups are
 * flattened into one work list (kernelbot nvfp4-group-gemm 474067,
 * launch_gpu_implementation: per-group tile counts and prefix sums; 496386,
 * launch_group_gemm: the precomputed tile table).
 * Returns NVFP4_OK or a negative code; nothing is launched on error. */
int nvfp4_group_gemm(const GroupDesc *groups, int num_groups, cudaStream_t stream);

/* Fused epilogue options (an MoE layer's needs; the pages write plain FP16
 * A.B^T): C_g = alpha[g] * A_g . B_g^T, optionally through the SwiGLU of a
 * gate/up projection, stored as FP16 or BF16 (rounded to nearest even once,
 * from the FP32 accumulator).
 *  alpha     host array [num_groups] of per-group scales (the product of the
 *            per-tensor global scales of A_g and B_g), or NULL for 1.
 *  out_bf16  0: C elements FP16, 1: BF16.
 *  swiglu    0: C_g is [M_g][N_g].  1: every N_g is a multiple of 256 and
 *            the rows of B_g come in 256-row blocks, 128 gate rows followed
 *            by the 128 up rows of the same outputs; C_g is [M_g][N_g/2] with
 *            C[m][128 j + c] = silu(alpha g) * (alpha u), g = (A.B^T)[m][256 j
 *            + c], u = (A.B^T)[m][256 j + 128 + c], silu(x) = x / (1 + e^-x)
 *            in single precision. */
typedef struct GemmEpilogue {
    const float *alpha;
    int out_bf16;
    int swiglu;
} GemmEpilogue;

/* nvfp4_group_gemm with the fused epilogue options `epi` (NULL: plain FP16
 * as nvfp4_group_gemm).  The ldc of C_g is its output width (N_g or N_g/2).
 * Returns NVFP4_ERR_INVALID_ARGUMENT when swiglu is set and some non-empty
 * group has N % 256 != 0. */
int nvfp4_group_gemm_ex(const GroupDesc *groups, int num_groups, const GemmEpilogue *epi,
                        cudaStream_t stream);

/* Kernel configurations of the grouped GEMM (chosen per call from the
 * shapes; the environment variable NVFP4_GEMM_KIND forces one):
 *  STREAM  128 x 128 tiles, 512-K stages (any N): larger calls with an N
 *          that is not a multiple of 256
 *  WIDE    128 x 256 tiles, 256-K stages (every N a multiple of 256)
 *  COMPUTE 128 x 128 tiles, 256-K stages, 64-column stores (any N): calls
 *          whose 128 x 128 tiles fit one round of the grid
 *  WIDE512 128 x 256 tiles, 512-K stages
 *  WIDE_P2 / WIDE_P4  accepted for compatibility; the same as WIDE (every
 *          configuration spreads a stage's loads over four issuing warps)
 *  PAIR    256 x 256 tiles on CTA pairs (tcgen05 cta_group::2; N >= 256):
 *          chosen whenever pairing does not add a round of the grid (large
 *          M; calls of fewer tiles than SMs)
 *  WIDE_SK WIDE tiles with stream-K: the call's (tile, 256-K stage) units
 *          are cut into one equal contiguous range per SM, so a tile may be
 *          split between CTAs; the CTA holding a tile's first stages adds
 *          the FP32 partial sums of the others before its epilogue.  Only
 *          selected through NVFP4_GEMM_KIND=7: on GB300 whole tiles measured
 *          faster even with fewer tiles than SMs.  Needs a scratch area per
 *          stream (one 128 KiB partial-sum slot per SM and a few flag
 *          words), allocated on the first such call on that stream and kept
 *          until the process exits; when it cannot be allocated (e.g. the
 *          stream is being captured into a graph at that moment) the call
 *          runs as WIDE.  Sums of cut tiles are formed in a different order,
 *          so results may differ from WIDE in the last bits of FP32 before
 *          rounding.
 *  SWAP    the transposed product C^T = B . A^T on CTA pairs: 256 rows of B
 *          as the MMA's M side and a tile of <= 256 rows of A (a group's
 *          tokens; larger groups are split into tiles 128 or 256 rows
 *          apart) as its N side, rounded up to 16, so each B byte is staged
 *          once per token tile and no MMA work goes to padding rows beyond
 *          that rounding; the epilogue transposes through shared memory
 *          before its stores.  Any N; no SwiGLU (a forced SWAP call with
 *          SwiGLU runs as WIDE).  Only selected through NVFP4_GEMM_KIND=8:
 *          on GB300 it measured slower than WIDE on the MoE shapes it was
 *          built for (each stage's scale copies sit on the pair's critical
 *          path). */
enum {
    NVFP4_KIND_STREAM = 0,
    NVFP4_KIND_WIDE = 1,
    NVFP4_KIND_COMPUTE = 2,
    NVFP4_KIND_WIDE512 = 3,
    NVFP4_KIND_WIDE_P2 = 4,
    NVFP4_KIND_WIDE_P4 = 5,
    NVFP4_KIND_PAIR = 6,
    NVFP4_KIND_WIDE_SK = 7,
    NVFP4_KIND_SWAP = 8
};

/* The plan nvfp4_group_gemm would follow for these groups on the current
 * device, without launching anything: *kind (an NVFP4_KIND_* value) and
 * *launches (kernel launches of the call; 0 when every group is empty).
 * Validates like nvfp4_group_gemm; needs the device's SM count, so the
 * first call on a device does its one-time set-up (see nvfp4_group_gemm).
 * kind and launches: host pointers, written only on NVFP4_OK. */
int nvfp4_group_gemm_plan(const GroupDesc *groups, int num_groups, int *kind, int *launches);

/* The same plan for a device with sm_count SMs (152 on GB300), computed on
 * the host alone: no CUDA call is made, so it also answers on a machine
 * without a GPU.  The descriptors are validated like nvfp4_group_gemm's
 * (their pointers are checked, never read).  NVFP4_GEMM_KIND applies as in
 * nvfp4_group_gemm.  Returns NVFP4_ERR_INVALID_ARGUMENT for null kind or
 * launches or sm_count < 2; kind and launches are written only on
 * NVFP4_OK. */
int nvfp4_group_gemm_plan_for(const GroupDesc *groups, int num_groups, int sm_count, int *kind,
                              int *launches);

/* The grouped GEMM of nvfp4_group_gemm for callers that are not allowed to
 * allocate device memory: engines and plugins that receive every byte of
 * device memory from an arena planned ahead and may not allocate while they
 * run, and latency-critical loops that cannot afford the device-wide
 * synchronisation an allocation may bring.  nvfp4_group_gemm allocates a
 * 16-byte status word on its first call on a device; this entry point
 * allocates nothing, ever.  The pages have no counterpart of this entry
 * point.
 *
 * Arguments, layouts, limits and results are those of nvfp4_group_gemm, with
 * one more limit: the kernel's status record (two 32-bit words per kernel
 * launch; a call launches once per 32 non-empty groups) lives in a static
 * 256-byte array inside the library, enough for 32 launches, so a call with
 * more than 1024 non-empty groups returns NVFP4_ERR_TOO_MANY and launches
 * nothing.  Every GPU that loads the library holds that array until the
 * process exits.
 *
 * The first call on a device does a one-time set-up with that device current
 * (capability check, kernel attribute, the device address of the static
 * array); make that first call before any stream capture.  Each call clears
 * the status words it uses, on `stream`, before its launch.  All calls share
 * the one array: calls whose work overlaps on the GPU (different streams, or
 * several host threads) race on it, so serialise them.  A bounded wait that
 * expires inside this variant is recorded only in that array (the next call
 * clears it); use nvfp4_group_gemm and nvfp4_last_device_error where timeouts
 * must be observed.  The scales must already be in the tiled layout (run
 * nvfp4_sf_relayout where allocation is allowed, e.g. at load time; its first
 * call on a device allocates the library's status word). */
int nvfp4_group_gemm_noalloc(const GroupDesc *groups, int num_groups, cudaStream_t stream);

/* Scale-factor relayout: plain row-major E4M3FN scales [rows][K/16] (row
 * stride K/16 bytes) -> the tiled layout the GEMM reads.  The tiled buffer is
 * a sequence of 512-byte atoms, one per (128-row block rb, 64-element K
 * block kb), in the order [rb][kb] (474067, TMA producer warp: scale source
 * base + ((off_m/128) * (K/64) + off_k/64) * 512).  Inside an atom the scale
 * of row r (0..127 in the block) and 16-element sub-block j (0..3 in the K
 * block) is at byte (r % 32) * 16 + (r / 32) * 4 + j: the 32 x 16-byte shape
 * one tcgen05.cp 32x128b.warpx4 moves (474067, tcgen05_cp_nvfp4).  Rows
 * beyond `rows` in the last block are written as zero.
 *  src   device, rows * K/16 bytes, 16-byte aligned.
 *  dst   device, nvfp4_sf_tiled_bytes(rows, K) bytes, 16-byte aligned, must
 *        not overlap src.
 *  rows >= 0 (0 is a no-op), K % 256 == 0, K <= 2^20, rows <= 2^20. */
int nvfp4_sf_relayout(const void *src, void *dst, int rows, int K, cudaStream_t stream);

/* Several relayouts in one launch (for example SFA and SFB of every group of
 * a grouped call); each entry has the meaning and limits of
 * nvfp4_sf_relayout.  1 <= count <= 4096. */
typedef struct SfRelayoutDesc {
    const void *src;
    void *dst;
    int rows, K;
} SfRelayoutDesc;
int nvfp4_sf_relayout_group(const SfRelayoutDesc *descs, int count, cudaStream_t stream);

/* The whole path of one grouped call: the scale relayout of every group's
 * SFA and SFB (one nvfp4_sf_relayout_group launch) followed by the grouped
 * GEMM of nvfp4_group_gemm_ex on the tiled scales.  Because the library
 * launches the relayout itself, the GEMM's loads of A and B start while the
 * relayout is still finishing (A and B must therefore be complete before
 * this call's work begins in the stream, as for any stream-ordered call);
 * its scale loads, MMAs and C stores wait for the relayout.
 *  A, B, C, M, N, K  as in GroupDesc.
 *  SFA, SFB          device, row-major E4M3FN scales [M][K/16], [N][K/16]
 *                    (16-byte aligned; may be NULL when M == 0).
 *  SFA_tiled,        device, nvfp4_sf_tiled_bytes(M, K) and
 *  SFB_tiled           nvfp4_sf_tiled_bytes(N, K) bytes the relayout writes
 *                    and the GEMM reads; owned by the caller.
 * epi: NULL or the fused epilogue of nvfp4_group_gemm_ex.  Validation of
 * every group precedes both launches; an error after the relayout launch
 * (a CUDA launch failure) leaves the tiled scales written and C untouched. */
typedef struct StepDesc {
    const void *A;
    const void *B;
    const void *SFA;
    const void *SFB;
    void *SFA_tiled;
    void *SFB_tiled;
    void *C;
    int M, N, K;
} StepDesc;
int nvfp4_relayout_and_gemm(const StepDesc *steps, int num_groups, const GemmEpilogue *epi,
                            cudaStream_t stream);

/* NVFP4 quantisation of a 16-bit float matrix into the GEMM's operand
 * format (the step that produces A or B; the pages take quantised data as
 * given, so this follows the generator of their "quantized" configuration:
 * values quantised per 16-block to E2M1 with an absmax/6 scale rounded to
 * E4M3FN).  For every 16-element block of a row:
 *   scale = E4M3FN(absmax / 6)       round to nearest even, saturating at 448
 *   code  = E2M1(x / scale)          round to nearest even, saturating at 6
 * both on IEEE single-precision quotients rounded to nearest; a zero
 * magnitude is stored as code 0 (no sign bit) and a block whose scale rounds
 * to 0 (absmax < 6 * 2^-10, all zeros included) gets codes 0.
 *  x           device, [rows][K] FP16 (x_is_bf16 = 0) or BF16 (x_is_bf16 =
 *              1) elements, row stride K, finite values, 16-byte aligned.
 *  codes       device, [rows][K/2] bytes, element 2i in the low nibble of
 *              byte i (the GEMM's A / B layout), 16-byte aligned.
 *  sf_tiled    device, nvfp4_sf_tiled_bytes(rows, K) bytes: the scales in
 *              the tiled layout the GEMM reads (what nvfp4_sf_relayout
 *              writes), padding rows zero; 16-byte aligned.
 *  sf_rowmajor device [rows][K/16] bytes or NULL: the same scales row-major.
 *  rows >= 0 (0 is a no-op), K % 64 == 0, rows, K <= 2^20.  Outputs must not
 *  overlap the input.  Asynchronous on `stream`; returns NVFP4_OK or a
 *  negative code (nothing launched). */
int nvfp4_quantize(const void *x, int x_is_bf16, int rows, int K, void *codes, void *sf_tiled,
                   void *sf_rowmajor, cudaStream_t stream);

/* Bytes of the tiled scale buffer for a [rows][K/16] scale matrix:
 * ceil(rows / 128) * (K / 64) * 512; 0 for invalid sizes. */
size_t nvfp4_sf_tiled_bytes(int rows, int K);

/* Synchronises `stream`, then reads and clears the device error word that
 * kernels of this library on the current device set when a bounded wait
 * expires.  Returns NVFP4_OK, NVFP4_ERR_TIMEOUT, or NVFP4_ERR_CUDA (which
 * includes a sticky CUDA error from an earlier launch). */
int nvfp4_last_device_error(cudaStream_t stream);

/* Upper bound, in nanoseconds, for any single wait inside the GEMM kernel
 * (default 2e9).  A wait that expires sets the device error word, makes every
 * role of that CTA leave its loop, drains in-flight copies and returns.
 * Values below 1e6 are raised to 1e6. */
void nvfp4_set_wait_timeout_ns(uint64_t ns);

/* Test hook, not for production use: while enabled, the next GEMM launches
 * have CTA 0 skip the loads of its first pipeline stage, so the waits that
 * depend on it expire after the wait timeout and the kernel reports
 * NVFP4_ERR_TIMEOUT through nvfp4_last_device_error() (the outputs of that
 * call are then undefined).  No fault, trap or unbounded wait results. */
void nvfp4_debug_drop_first_stage(int enable);

/* Static description of the string for a return code (never NULL). */
const char *nvfp4_strerror(int code);

/* Library version, (major << 16) | (minor << 8) | patch. */
int nvfp4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GROUP_GEMM_H */

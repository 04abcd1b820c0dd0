/*
 * tern.h -- C ABI of libtern, the GB300 (sm_103a) ternary-g128 matrix product
 * and Walsh-Hadamard rotation library.
 *
 * The method (from the "prism-ml/Ternary-Bonsai-27B-mlx-2bit" Hugging Face
 * model card and the "Ternary-Bonsai-2-9B-2bit" article):
 *   - every weight is t * s_g, t in {-1, 0, +1}, with one FP16 scale s_g per
 *     128 consecutive weights along K (card, "Weight representation: ternary
 *     g128");
 *   - each t is stored in a 2-bit slot, 2.125 bits per weight with the scales
 *     (card, "Memory requirement");
 *   - the packed weights are used directly: codes are unpacked and scaled
 *     inside the matrix product, never expanded to a dense FP16 tensor (card,
 *     "CUDA (NVIDIA GPUs)");
 *   - where a layer uses it, the activation's last dimension is first rotated
 *     by the normalized Sylvester-Walsh-Hadamard transform, block 4096, with an
 *     explicit sign pattern (article, section 3 "Ternary weights and Hadamard
 *     rotation").
 *
 * Data layout (shared by every entry point):
 *   x       bf16 [M][K] row-major activations.
 *   codes   uint32 [N][K/16] row-major.  Weight (n, k) has code
 *           q = t + 1 in {0, 1, 2} in bits 2*(k%16) .. 2*(k%16)+1 of word
 *           codes[n][k/16] (little-endian uint32).  q = 3 is invalid.
 *   scales  fp16 [N][K/128] row-major: s[n][g] scales k in [128 g, 128 g + 128).
 *   y       [M][N] row-major, y[m][n] = sum_k x[m][k] * (q[n][k] - 1) * s[n][k/128].
 *   signs   int8 [K], each +1 or -1.
 *   Packed size: N*K/4 bytes of codes + N*K/64 bytes of scales.
 *   The 1-bit sibling format (tern_bin_*) keeps one bit per weight in uint32
 *   words [N][K/32]; an affine pack (tern_affine_*) adds fp16 biases
 *   [N][K/128] and allows code 3.  Their entry points describe them.
 *
 * Conventions:
 *   - Device entry points take device pointers owned by the caller, launch
 *     asynchronously on `stream` (NULL = the legacy default stream) and
 *     allocate nothing.  Where a kernel needs scratch memory the caller passes
 *     a device workspace of at least the size the matching *_workspace_bytes
 *     query returns, 256-byte aligned and zero-filled once before its first
 *     use (cudaMemset); every completed call leaves it ready for the next.
 *     Calls that share a workspace must be ordered (one stream, or events).
 *   - The return value reports host-side argument validation and launch
 *     errors only; on any error nothing is launched.  Device-side problems
 *     (a bounded wait that gave up) set a sticky device flag that
 *     tern_device_error() reads.
 *   - Pointers must be 16-byte aligned (TERN_ERR_ALIGN otherwise).
 *   - The product and rotation kernels use programmatic dependent launch.
 *     Those of the *gemv* and *fwht* entry points may begin reading `codes`,
 *     `scales` (and `biases`) while the previous tern_* kernel on the stream
 *     is still running, so these must not be outputs of the immediately
 *     preceding tern_* call (the packers and the scale conversion excepted:
 *     they never release their dependents early).  The *gemm* kernels start
 *     early too but read nothing before the previous kernel has finished.
 *     Activations, outputs and workspaces are always ordered.
 *   - Only sm_103 devices (GB300) are supported (TERN_ERR_ARCH otherwise).
 */
#ifndef TERN_H
#define TERN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *tern_stream_t;

typedef enum {
    TERN_OK = 0,
    TERN_ERR_NULL = 1,      /* a required pointer is NULL */
    TERN_ERR_SHAPE = 2,     /* M, N or K out of range or not a required multiple */
    TERN_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned */
    TERN_ERR_WORKSPACE = 4, /* workspace NULL or smaller than required */
    TERN_ERR_CUDA = 5,      /* a CUDA runtime/driver call or a launch failed */
    TERN_ERR_ARCH = 6,      /* the current device is not sm_103 */
    TERN_ERR_DEVICE = 7     /* a kernel reported a device-side error (bounded wait gave up) */
} tern_status;

/* A short English description of a status code (static storage). */
const char *tern_status_str(tern_status s);

/* Packed bytes of an N x K ternary-g128 matrix: N*K/4 + N*K/64. */
size_t tern_packed_bytes(int N, int K);

/* ---------------------------------------------------------------------- */
/* Packing and validation (card, "Memory requirement": 2-bit slots)        */
/* ---------------------------------------------------------------------- */

/* Device packer.  t: int8 [N][K] in {-1,0,+1}; codes: uint32 [N][K/16].
 * An entry outside {-1,0,+1} is written as the invalid code 3 and counted:
 * if bad_count (device int, nullable) is given, the number of invalid entries
 * is atomically ADDED to it (the caller zeroes it first).
 * K % 16 == 0 and N >= 0, K >= 0 (TERN_ERR_SHAPE otherwise); t 16-byte aligned. */
tern_status tern_pack(const int8_t *t, int N, int K, uint32_t *codes, int *bad_count,
                      tern_stream_t stream);

/* Host packer (loaders, tests): same layout and rules as tern_pack; the
 * number of invalid entries is stored in *bad_count (nullable). */
tern_status tern_pack_host(const int8_t *t, int N, int K, uint32_t *codes,
                           long long *bad_count);

/* Host unpacker: t[n][k] = q - 1; code 3 is written as 0 and counted. */
tern_status tern_unpack_host(const uint32_t *codes, int N, int K, int8_t *t,
                             long long *bad_count);

/* Host validator: counts code-3 slots in codes [N][K/16] into *bad_count. */
tern_status tern_validate_host(const uint32_t *codes, int N, int K, long long *bad_count);

/* The group-size-64 pack ([card] "Shipped components": the same g128
 * representation with each scale repeated in both 64-value halves of its
 * group, 7.59 GB against 7.17): its scales s64, fp16 [N][K/64], become the
 * g128 scales s128, fp16 [N][K/128], with s128[n][g] = s64[n][2g].  A group
 * whose halves differ bit for bit is counted (into *mismatch, a device int
 * the call ADDS to, for the device version; stored, for the host one) and
 * keeps its first half's scale.  The codes are taken to be in the layout
 * above; the pages give no other bit order for that pack.  K % 128 == 0,
 * N >= 0 (TERN_ERR_SHAPE otherwise); pointers 16-byte aligned. */
tern_status tern_scales_from_g64(const void *s64, int N, int K, void *s128, int *mismatch,
                                 tern_stream_t stream);
tern_status tern_scales_from_g64_host(const void *s64, int N, int K, void *s128, long long *mismatch);

/* ---------------------------------------------------------------------- */
/* The 1-bit sibling, binary g128 (card, "Highlights" and "Benchmarks":    */
/* 1-bit Bonsai at 1.125 bits per weight; "MLX packaging": s_mlx = 2 s_g,   */
/* bias = -s_g gives exactly +-s_g).  A weight is (2b - 1) * s_g, b the bit */
/* k%32 of little-endian uint32 word k/32 of its row (the pages fix no      */
/* order; the same reading as the 2-bit codes).  Scales as above.           */
/* ---------------------------------------------------------------------- */

/* Packed bytes of an N x K binary-g128 matrix: N*K/8 + N*K/64; 0 on bad input
 * (K % 128 != 0). */
size_t tern_bin_packed_bytes(int N, int K);

/* Device packer.  t: int8 [N][K] in {-1,+1}; words: uint32 [N][K/32].  An
 * entry other than +-1 is written as -1 and counted: if bad_count (device
 * int, nullable) is given, the count is atomically ADDED to it.  K % 32 == 0,
 * N >= 0, K >= 0 (TERN_ERR_SHAPE otherwise); t and words 16-byte aligned. */
tern_status tern_bin_pack(const int8_t *t, int N, int K, uint32_t *words, int *bad_count,
                          tern_stream_t stream);

/* Host packer and unpacker, same layout and rules (unpack writes 2b - 1). */
tern_status tern_bin_pack_host(const int8_t *t, int N, int K, uint32_t *words,
                               long long *bad_count);
tern_status tern_bin_unpack_host(const uint32_t *words, int N, int K, int8_t *t);

/* Native base-3 packing ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card,
 * "Weight representation: ternary g128" and "Memory requirement": a trit
 * carries log2 3 bits, 1.71 bits/weight with the scale, named there as future
 * work; the card gives no layout).  Five trits per byte: byte j < 25 of a
 * 128-weight group holds trits 5 j .. 5 j + 4 of the group as
 * q0 + 3 q1 + 9 q2 + 27 q3 + 81 q4 (q = t + 1, values 0..242); byte 25 holds
 * trits 125..127 as q0 + 3 q1 + 9 q2 (values 0..26).  Rows are
 * [N][26 K/128] bytes, so 1.75 bits per weight with the fp16 scales
 * [N][K/128] of the 2-bit format (18 % fewer bytes than the 2-bit slots). */

/* Bytes of a base-3 pack of an [N][K] matrix; 0 on bad input (K % 128 != 0). */
size_t tern_f3_packed_bytes(int N, int K);

/* Device packer.  t: int8 [N][K] in {-1,0,+1}; packed: uint8 [N][26 K/128],
 * owned by the caller.  An entry outside {-1,0,+1} is packed as -1 and
 * counted: if bad_count (device int, nullable) is given, the count is
 * atomically ADDED to it.  K % 128 == 0, N >= 0 (TERN_ERR_SHAPE otherwise).
 * One kernel launch (none for an empty matrix). */
tern_status tern_f3_pack(const int8_t *t, int N, int K, uint8_t *packed, int *bad_count,
                         tern_stream_t stream);

/* The decode product on a base-3 pack: y (fp32 [M][N]) = x W^T,
 * W[n][k] = (q[n][k] - 1) s[n][k/128].  x bf16 [M][K], packed as tern_f3_pack
 * writes it, scales fp16 [N][K/128]; x, packed, scales and y 16-byte aligned,
 * owned by the caller.  1 <= M <= 16, N >= 1, K >= 128 with K % 128 == 0.
 * One kernel launch, no workspace; every element of y is written.  With K a
 * multiple of 512 it runs on the tensor pipe: each byte's five trits become
 * 2-bit codes through a table, and the product is tern_gemv's, with its
 * accuracy statement (including the group term and the rule that a group
 * whose largest |x| is 2^100 or more, or not finite, is reported as
 * TERN_DEVERR_GEMV_ACTIVATION_RANGE through tern_device_error(), y then
 * undefined); its K-slices meet through flag words in a file-scope array
 * that every call on a device shares, so calls on different streams must be
 * ordered by the caller.  The words count back to 0 in every call; after a
 * call that reported a device error, tern_device_error() clears them as it
 * reads the error.  Otherwise it runs on the CUDA cores (fp32 FMAs, a
 * 243-entry table per byte) and agrees with the exact product to within
 * 1e-3 * sum_k |x w| + 1e-6 per element.  A byte above 242 (above 26 for a
 * group's last byte) is not a pack's; its weights are undefined. */
tern_status tern_f3_gemv(const void *x, const uint8_t *packed, const void *scales, float *y,
                         int M, int N, int K, tern_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Decode / small-batch product, M = 1..16 (card, "Cross-platform          */
/* throughput": tg128 is the memory-bandwidth-bound phase; "Speculative    */
/* decoding: DSpark": verify runs k + 1 tokens)                            */
/* ---------------------------------------------------------------------- */

/* Workspace bytes tern_gemv and tern_fwht_gemm need for (M, N, K); 0 on bad
 * input.  The size covers both calls (at least 256).  It holds one 32-bit flag
 * word per 16-row tile when K > 1024 (the K-slice sums of a row range are
 * added into y, and the flag orders the range's clearing before the
 * additions) and, for tern_fwht_gemm with M > 2, the rotated activation as the
 * product stages it (M * K fp16 values and one int32 exponent per token and
 * 128-group).
 * The workspace must be zero-filled once before its first use; every call
 * leaves its flags at zero again.  Calls that share a workspace must not run
 * concurrently (use one stream, or one workspace per stream).  After a device
 * error (tern_device_error) zero-fill it again. */
size_t tern_gemv_workspace_bytes(int M, int N, int K);

/* y (fp32 [M][N]) = x W^T with W given by (codes, scales).
 * 1 <= M <= 16, N >= 1, K >= 128 with K % 128 == 0.  One kernel launch.
 * For K <= 1024 the workspace may be NULL.  No pre-zeroing of y is needed (the
 * kernel clears what it adds into).
 * Results agree with the exact product to within 1e-3 * sum_k |x w| + 1e-6 per
 * element, plus 2^-22 * sum_g |s_g| * max_{k in g} |x_k|: the activation is
 * staged in fp16 with one exponent per token and group, so values far below
 * their group's largest lose bits (the term matters only when a group's
 * largest |x| meets a zero weight and the rest of the group is some 2^12 or
 * more below it).  A row of zero weights gives exactly 0.  When K spans more
 * than 8 groups (K > 1024) the K-slice sums are added into y with global float
 * reductions, and for M > 4 the group sums within a slice meet in shared-memory
 * atomics; in either case the last bits of y may vary from run to run.
 * Every |x| must be finite and below 2^100 (larger values would overflow the
 * fp16 staging): a group of 128 activations outside that range makes the call
 * report TERN_DEVERR_GEMV_ACTIVATION_RANGE through tern_device_error(), and
 * its y is then undefined. */
tern_status tern_gemv(const void *x, const uint32_t *codes, const void *scales, float *y,
                      int M, int N, int K, void *workspace, size_t workspace_bytes,
                      tern_stream_t stream);

/* Two products that read the same activation, in one launch (for example the
 * gate and up projections of a layer): y_a = x W_a^T (fp32 [M][N_a]) and
 * y_b = x W_b^T (fp32 [M][N_b]), each matrix as for tern_gemv.  The row
 * ranges are shared out between the two matrices in proportion to their rows,
 * so the fixed cost of a launch (the dependency wait and the tail) is paid once
 * for both.  y_a and y_b must not overlap.  The workspace is
 * tern_gemv_pair_workspace_bytes(M, N_a, N_b, K) bytes, zero-filled once, with
 * the rules of tern_gemv's.  Shapes, alignment and errors as for tern_gemv. */
size_t tern_gemv_pair_workspace_bytes(int M, int N_a, int N_b, int K);
tern_status tern_gemv_pair(const void *x, const uint32_t *codes_a, const void *scales_a, float *y_a, int N_a,
                           const uint32_t *codes_b, const void *scales_b, float *y_b, int N_b, int M, int K,
                           void *workspace, size_t workspace_bytes, tern_stream_t stream);

/* The same product for the 1-bit sibling format: y (fp32 [M][N]) = x W^T with
 * W[n][k] = (2 b[n][k] - 1) * s[n][k/128], words uint32 [N][K/32] as
 * tern_bin_pack writes them.  Shapes, alignment, workspace (the size
 * tern_gemv_workspace_bytes gives), ordering and error behaviour as for
 * tern_gemv.  Each weight costs the same tensor-core work as a 2-bit one, at
 * half the bytes. */
tern_status tern_bin_gemv(const void *x, const uint32_t *words, const void *scales, float *y,
                          int M, int N, int K, void *workspace, size_t workspace_bytes,
                          tern_stream_t stream);

/* The product on an affine pack: y (fp32 [M][N]) = x W^T with
 *     W[n][k] = s[n][k/128] * q[n][k] + b[n][k/128],
 * the scale-and-bias form of a group ("prism-ml/Ternary-Bonsai-27B-mlx-2bit"
 * model card, "MLX packaging").  codes uint32 [N][K/16] in the 2-bit slots of
 * tern_pack (code k in bits 2 (k % 16) of word k / 16), every code 0..3 valid;
 * scales and biases fp16 [N][K/128], 16-byte aligned, owned by the caller.
 * The ternary codes are the case b = -s; the card's own pair (2 s_g, -s_g) on
 * codes {0, 1} is the 1-bit format.  Shapes, alignment, workspace (the size
 * tern_gemv_workspace_bytes gives), ordering and error behaviour as for
 * tern_gemv; a NULL biases pointer is TERN_ERR_NULL.  Results agree with the
 * exact product to within 1e-3 * sum_k |x w| + 2^-23 * sum_k |x_k b_g(k)|
 * + 1e-6 per element (the second term covers the rounding of the bias part,
 * which the scale part may cancel). */
tern_status tern_affine_gemv(const void *x, const uint32_t *codes, const void *scales, const void *biases,
                             float *y, int M, int N, int K, void *workspace, size_t workspace_bytes,
                             tern_stream_t stream);

/* Fixed size of the library-owned scratch array behind tern_gemv_noalloc. */
#define TERN_NOALLOC_SCRATCH_BYTES (256u << 10)

/* The same product as tern_gemv, for callers that cannot allocate device
 * memory (code running inside an allocator's own callback, a caching
 * allocator that must not recurse into itself, a runtime that hands out all
 * device memory up front): it takes no workspace and allocates nothing.  The
 * pages describe no counterpart; this is a library convenience.
 *   - Its scratch (one flag word per 16-row tile, when K > 1024) is one
 *     file-scope device array of TERN_NOALLOC_SCRATCH_BYTES that every GPU
 *     loading the library holds until the process exits.  Shapes whose flags
 *     exceed it (N above 1,048,576 rows) are rejected with TERN_ERR_WORKSPACE
 *     and nothing is launched.
 *   - Every call looks up the array's device address on the current device
 *     (a host-side query; no stream work).  The first call on a device also
 *     loads the kernels and plans the shape: make it before any stream
 *     capture.
 *   - Each call clears the flags it uses with one cudaMemsetAsync on `stream`
 *     before the product kernel (tern_last_launch_count counts the kernel
 *     only).  All calls share the one array, so calls whose kernels overlap on
 *     the GPU (different streams) race: order them.
 * Arguments, layout, results and tolerance as for tern_gemv. */
tern_status tern_gemv_noalloc(const void *x, const uint32_t *codes, const void *scales, float *y,
                              int M, int N, int K, tern_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Rotation (article, section 3: normalized Sylvester-Walsh-Hadamard,      */
/* block 4096, last dimension, explicit signs)                             */
/* ---------------------------------------------------------------------- */

/* y (bf16 [M][K]) = H_4096 (signs (.) x) / 64 for each 4096-block of each row,
 * H in natural (Sylvester) order, computed in fp32 and rounded to nearest
 * even.  M >= 1, K >= 4096 with K % 4096 == 0.  x and y may not alias. */
tern_status tern_fwht(const void *x, const int8_t *signs, void *y, int M, int K,
                      tern_stream_t stream);

/* Rotation fused into the product: y (fp32 [M][N]) = rot(x) W^T.  The rotated
 * activation is computed in fp32 and staged as the product stages any
 * activation: per token and 128-group, fp16 values scaled by a power of two
 * chosen from the group's largest magnitude; it is never rounded to bf16.
 * For M <= 2 it is one kernel launch: each CTA of the product rebuilds the
 * 1024-wide slice of x' its K-slice reads in shared memory (H_4096 =
 * H_4 (x) H_1024: the signed sum of the 4096-block's four 1024-wide parts,
 * then a 1024-point transform).  For M > 2 a prologue kernel rotates x once
 * and stages it in the workspace (L2-resident) before the product (two
 * launches).  1 <= M <= 16, K % 4096 == 0; workspace as for tern_gemv
 * (required). */
tern_status tern_fwht_gemm(const void *x, const int8_t *signs, const uint32_t *codes,
                           const void *scales, float *y, int M, int N, int K,
                           void *workspace, size_t workspace_bytes, tern_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Prefill product (card, "Cross-platform throughput": pp512 is the        */
/* compute-bound phase)                                                    */
/* ---------------------------------------------------------------------- */

/* Workspace bytes tern_gemm needs; 0 on bad input.  It holds one counter per
 * (256-token x 128-row tile, 32-row quarter) and one 128 KB fp32 sum per tile
 * (for tiles whose K range is split between CTAs): 34 MB for a 512 x 17408
 * output.  It must be zero-filled once before its first use; every call
 * leaves its counters and sums at zero again.  Calls that share a workspace must not
 * run concurrently.  After a device error (tern_device_error) zero-fill it
 * again. */
size_t tern_gemm_workspace_bytes(int M, int N, int K);

/* y = x W^T on the tcgen05 tensor cores: each weight is unpacked on chip to
 * bf16 t * bf16(s_g) (the group scale rounded to nearest even bf16 and folded
 * in), the product accumulates in fp32 in tensor memory, and y is written as
 * fp32 (y_is_bf16 == 0) or bf16 rounded to nearest even (y_is_bf16 != 0).
 * On those operands the fp32 output is within 1e-3 * sum_k |x w| + 1e-6 and
 * the bf16 output within 8e-3 * max(|y|, (sum_k (x w)^2)^(1/2)); the rounding
 * of the scales moves y from the exact-scale product by at most
 * sum_g |bf16(s_g) - s_g| |sum_{k in g} x_k t_k|.
 * The (tile, K-stage) iterations are shared out evenly over the SMs
 * (stream-K); the parts of a tile split between CTAs are added in fp32 in no
 * fixed order, so the last bits of such tiles may vary from run to run.
 * M >= 1, N >= 1, K >= 128 with K % 128 == 0 (TERN_ERR_SHAPE otherwise). */
tern_status tern_gemm(const void *x, const uint32_t *codes, const void *scales, void *y,
                      int y_is_bf16, int M, int N, int K, void *workspace,
                      size_t workspace_bytes, tern_stream_t stream);

/* The same product for the 1-bit sibling format (words uint32 [N][K/32] as
 * tern_bin_pack writes them): each weight is unpacked to bf16
 * (2b - 1) * bf16(s_g).  Shapes, workspace (tern_gemm_workspace_bytes),
 * output types and error behaviour as for tern_gemm. */
tern_status tern_bin_gemm(const void *x, const uint32_t *words, const void *scales, void *y,
                          int y_is_bf16, int M, int N, int K, void *workspace,
                          size_t workspace_bytes, tern_stream_t stream);

/* The prefill product on an affine pack (W as for tern_affine_gemv): each
 * weight s q + b is formed in fp32 and rounded once to bf16 before the
 * tensor-core product, so the fp32 output differs from the exact product by at
 * most what those roundings explain, sum_g sum_q |d_q| |sum_{k in g, q_k = q}
 * x_k| with d_q = bf16(s q + b) - (s q + b), plus the fp32 accumulation.  Shapes, workspace
 * (tern_gemm_workspace_bytes), output types and error behaviour as for
 * tern_gemm; a NULL biases pointer is TERN_ERR_NULL and a misaligned one
 * TERN_ERR_ALIGN. */
tern_status tern_affine_gemm(const void *x, const uint32_t *codes, const void *scales, const void *biases,
                             void *y, int y_is_bf16, int M, int N, int K, void *workspace,
                             size_t workspace_bytes, tern_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Diagnostics                                                             */
/* ---------------------------------------------------------------------- */

/* Device-side error codes: which bounded wait gave up.  Every wait in the
 * kernels has a time limit (1 s for the waits below); the first wait to run
 * out stores its code, and the kernel returns with the call's output
 * incomplete. */
enum {
    TERN_DEVERR_GEMM_PRODUCER_WAIT = 0x101,  /* prefill: loader waited for a free stage */
    TERN_DEVERR_GEMM_UNPACK_WAIT = 0x102,    /* prefill: unpack warps waited for a tile or slot */
    TERN_DEVERR_GEMM_MMA_WAIT = 0x103,       /* prefill: MMA issuer waited for operands or TMEM */
    TERN_DEVERR_GEMM_EPILOGUE_WAIT = 0x104,  /* prefill: epilogue waited for an accumulator */
    TERN_DEVERR_GEMM_TEARDOWN_WAIT = 0x105,  /* prefill: teardown waited for work in flight */
    TERN_DEVERR_GEMV_RANGE_FLAG_WAIT = 0x202, /* decode: a K-slice waited for y's clearing */
    TERN_DEVERR_GEMV_ACTIVATION_RANGE = 0x203 /* decode: a group's largest |x| was >= 2^100 or not finite */
};

/* Reads and clears the sticky device-side error words of the current device
 * (synchronizes the device).  *code = 0 when no kernel reported an error;
 * otherwise the TERN_DEVERR_* code of the wait that gave up.  Returns TERN_OK
 * or TERN_ERR_CUDA. */
tern_status tern_device_error(int *code);

/* Self-test of the bounded waits (a diagnostic; the method has no counterpart).
 * Launches one small kernel that runs one of the products' own wait helpers on
 * something nothing ever completes, with a limit of limit_us microseconds
 * (1 .. 1,000,000):
 *   TERN_SELFTEST_RANGE_FLAG -- the decode K-slices' wait on a range flag word;
 *     reports TERN_DEVERR_GEMV_RANGE_FLAG_WAIT.
 *   TERN_SELFTEST_MBARRIER -- the prefill roles' mbarrier wait: one role's wait
 *     runs out, raises the CTA's abort flag and reports
 *     TERN_DEVERR_GEMM_MMA_WAIT; a second role in a 1 s wait sees the flag and
 *     returns early, so the kernel ends about limit_us after it starts.
 * The code is then read with tern_device_error, and the context stays usable.
 * Returns TERN_ERR_SHAPE for an unknown `which` or a limit out of range
 * (nothing launched), TERN_ERR_ARCH / TERN_ERR_CUDA as the products do. */
#define TERN_SELFTEST_RANGE_FLAG 0
#define TERN_SELFTEST_MBARRIER 1
tern_status tern_wait_selftest(int which, int limit_us, tern_stream_t stream);

/* The number of kernels the last entry point call launched (for launch
 * accounting in benchmarks); host-side, per process. */
int tern_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* TERN_H */

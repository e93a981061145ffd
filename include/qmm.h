/*
 * qmm.h -- C ABI of the GB300 group-quantized 4-bit-weight matmul library
 * (libqmm_gb300.so, built for sm_103a).
 *
 * The library computes the quantized linear layer of LLM inference,
 * y = W x, with W stored as 4-bit integers in groups of `group` consecutive
 * inputs (k), one fp16 scale per (output row n, group g), in two variants:
 *
 *   QMM_W4A8   symmetric weights q in [-8, 7]. Activations are optionally
 *              rotated by an in-group Walsh-Hadamard transform, quantized per
 *              row and per group to int8, contracted with the weights into
 *              exact int32 group partials, and rescaled in fp32:
 *                  Y[m][n] = sum_g sw[n][g] * sx[m][g] * P[m][n][g]
 *                  P[m][n][g] = sum_{k in g} q[n][k] * a[m][k]
 *              (cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill
 *              attention, and orthogonal embeddings": Summary, "Quantized
 *              matmul"; the per-group partials contract in its review thread;
 *              geistlib issue #500 "native W*A8 int8 GEMM for prefill":
 *              Design sketch.)
 *
 *   QMM_AFFINE unsigned weights q in [0, 15] with w = s*q + b per group. The
 *              bias term needs the per-row group sums of X, S[m][g]:
 *                  Y[m][n] = sum_g ( s[n][g] * sum_{k in g} q[n][k] x[m][k]
 *                                   + b[n][g] * S[m][g] )
 *              (TensorFold PR #3215 "simd_qmm on Metal: X's group sums and
 *              half operands from a prepass": What this changes.)
 *
 *   QMM_CQ4    codebook 4-bit weights: each weight is a 4-bit index i into
 *              one 16-entry int8 codebook C of the matrix, scaled by one fp32
 *              cb_scale per matrix and the per-group fp16 scale sw. The
 *              activation side is exactly the W4A8 one (same prepass), the
 *              partials stay integer and cb_scale folds into the rescale:
 *                  Y[m][n] = cb_scale * sum_g sw[n][g] * sx[m][g] * P[m][n][g]
 *                  P[m][n][g] = sum_{k in g} C[i[n][k]] * a[m][k]
 *              (cactus PR #697, Summary: 4-bit codebook expansion inside the
 *              GEMV leaf by table lookup; follow-up "single runtime weight
 *              format": the codebook scale is folded into the per-row norms.)
 *
 * Calls:  qmm_pack_weights / qmm_pack_weights_cq4 (once per weight) ->
 *         qmm_prep_act (per call) -> qmm_gemv (M == 1, W4A8 and CQ4) or
 *         qmm_gemm (any M, all variants); qmm_gemv_fused does the prepass and
 *         the GEMV in one launch.
 *
 * Conventions for every entry point:
 *   - All pointers named "device" are CUDA device pointers in the current
 *     device's context; the caller allocates and owns them. The library
 *     allocates no device memory.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). Outputs are valid once the stream reaches that
 *     point. Buffers passed to one call must not overlap one another.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and returned synchronously; nothing is written in that case.
 *   - A launch failure returns QMM_ERR_CUDA. There is no CPU fallback: a
 *     shape or device the kernels do not cover returns an error code.
 *   - Device pointers must be 16-byte aligned (QMM_ERR_MISALIGNED otherwise).
 *   - Kernels are launched with programmatic dependent launch: each kernel
 *     streams its packed weights before waiting on the previous kernel in the
 *     stream, and waits before it reads activations or writes outputs. The
 *     pack kernel lets the next kernel start only when it has finished, so a
 *     blob packed on the same stream is complete before it is read. A blob
 *     written by another producer must be complete before the call (any
 *     kernel that does not trigger its dependents early qualifies).
 *   - Not thread-safe per stream; distinct host threads may use distinct
 *     streams.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMM_OK = 0,
    QMM_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, bad enum */
    QMM_ERR_UNSUPPORTED_SHAPE = 2,  /* K % group != 0, group not supported, ... */
    QMM_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
    QMM_ERR_MISALIGNED = 4,         /* a device pointer is not 16-byte aligned */
    QMM_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
    QMM_ERR_TIMEOUT = 6,            /* a kernel gave up a bounded wait (qmm_device_status) */
    QMM_ERR_WORKSPACE = 7           /* workspace too small */
} qmm_status;

typedef enum { QMM_W4A8 = 0, QMM_AFFINE = 1, QMM_CQ4 = 2 } qmm_variant;

typedef enum { QMM_DTYPE_F32 = 0, QMM_DTYPE_F16 = 1, QMM_DTYPE_BF16 = 2 } qmm_dtype;

/* Which kernel a debug call goes through. */
typedef enum { QMM_PATH_GEMV = 0, QMM_PATH_GEMM = 1 } qmm_path;

/* Kernel identifiers reported by qmm_last_kernel_id(). */
typedef enum {
    QMM_KERNEL_NONE = 0,
    QMM_KERNEL_PACK = 1,
    QMM_KERNEL_PREP_W4A8 = 2,
    QMM_KERNEL_PREP_AFFINE = 3,
    QMM_KERNEL_GEMV_W4A8 = 4,
    QMM_KERNEL_GEMM_W4A8 = 5,
    QMM_KERNEL_GEMM_AFFINE = 6,
    QMM_KERNEL_GEMV_FUSED = 7,
    QMM_KERNEL_GEMM_ROWS = 8,
    QMM_KERNEL_GEMV_FUSED_SIBLINGS = 9,
    QMM_KERNEL_GEMV_CQ4 = 10,
    QMM_KERNEL_GEMM_CQ4 = 11,
    QMM_KERNEL_PREP_ROTATED = 12,
    QMM_KERNEL_GEMM_NARROW = 13,
    QMM_KERNEL_GEMM_NARROW_E4M3 = 14
} qmm_kernel_id;

typedef void* qmm_stream; /* cudaStream_t */

/* A quantized weight matrix W [N][K].
 *   variant: QMM_W4A8 or QMM_CQ4 (group 64 or 128), QMM_AFFINE (group 64).
 *   N >= 1, K >= group, K % group == 0. */
typedef struct {
    int32_t variant;
    int32_t N;
    int32_t K;
    int32_t group;
} qmm_weight_desc;

/*
 * Packed weight blob ("pack once, one runtime format"; cactus PR #697:
 * the packed weight cache is built once per weight and is the single runtime
 * format of both engines; geistlib issue #500, Design sketch item 2: repack at
 * resolve time).
 *
 * With T = ceil(N/128) row tiles, G = K/group groups and PP = group/32 pieces
 * per group, the blob is T*G chunks of CB bytes,
 *     CB = 64*group + 256            (QMM_W4A8, QMM_CQ4)
 *     CB = 64*group + 512            (QMM_AFFINE),
 * chunk (t, g) at byte (t*G + g)*CB. Inside a chunk:
 *     [0, 64*group)           nibbles: piece p (0..PP-1), row r (0..127) at
 *                             p*2048 + r*16; 16 bytes = 32 weights of row
 *                             n = 128t + r, k = g*group + 32p + 0..31, as four
 *                             little-endian 32-bit words j = 0..3 covering
 *                             k = 8j..8j+7 of the piece. In word j, nibble slot
 *                             s (bits 4s..4s+3) holds local k = 8j + 2s for
 *                             s < 4 and 8j + 2(s-4) + 1 for s >= 4.
 *                             Nibble value: q + 8 (QMM_W4A8), q (QMM_AFFINE),
 *                             the codebook index i (QMM_CQ4).
 *     [64*group, +256)        scales: 128 fp16, row r at 2r (sw[n][g]).
 *     [64*group+256, +256)    biases (QMM_AFFINE only): 128 fp16, row r at 2r.
 * QMM_CQ4 appends a 32-byte trailer at byte T*G*CB: the 16 codebook levels
 * (int8, level j at byte j), cb_scale (fp32, little-endian, bytes 16-19) and
 * 12 zero bytes.
 * Rows n >= N of the last tile hold q = 0 (index 0 for QMM_CQ4) and zero
 * scales and biases.
 * The blob depends only on the logical values of q, scales and biases.
 */
size_t qmm_packed_size(const qmm_weight_desc* w);

/*
 * Repack weights into the blob above (device kernel, on `stream`).
 *   q       device, [N][K/2] bytes, row-major. Byte j of row n holds k = 2j in
 *           its low nibble and k = 2j+1 in its high nibble (cactus PR #697,
 *           follow-up "single runtime weight format": low nibble first).
 *           QMM_W4A8: 4-bit two's complement q in [-8, 7]. QMM_AFFINE: q in [0, 15].
 *   scales  device, [N][G] fp16 (sw for W4A8, s for affine).
 *   biases  device, [N][G] fp16; QMM_AFFINE only (must be NULL for QMM_W4A8).
 *   packed  device, qmm_packed_size(w) bytes, written entirely.
 * K must be a multiple of 32 and of group. The sources may be freed once the
 * stream has passed this call. QMM_CQ4 weights need their codebook: they are
 * packed by qmm_pack_weights_cq4 (QMM_ERR_INVALID_ARG here).
 */
qmm_status qmm_pack_weights(const qmm_weight_desc* w, const uint8_t* q, const uint16_t* scales,
                            const uint16_t* biases, void* packed, qmm_stream stream);

/*
 * Repack QMM_CQ4 weights (device kernel, on `stream`).
 *   idx       device, [N][K/2] bytes of 4-bit codebook indices, low nibble
 *             first (the layout of qmm_pack_weights' q).
 *   codebook  HOST pointer, 16 int8 levels C[0..15] (read during the call).
 *   cb_scale  the matrix's codebook scale; must be finite (QMM_ERR_INVALID_ARG).
 *   scales    device, [N][G] fp16 sw.
 *   packed    device, qmm_packed_size(w) bytes (chunks + trailer), written
 *             entirely.
 * The codebook is the matrix's own: the integer partials use its levels as
 * given (no assumption of order or symmetry), so any relabelling of indices
 * and levels gives the same results.
 */
qmm_status qmm_pack_weights_cq4(const qmm_weight_desc* w, const uint8_t* idx, const int8_t* codebook,
                                float cb_scale, const uint16_t* scales, void* packed, qmm_stream stream);

/*
 * Repack weights given in 4-row panels (device kernel, on `stream`); any
 * variant. The blob is byte-identical to the one qmm_pack_weights (or
 * qmm_pack_weights_cq4) builds from the same weights in row-major order
 * (cactus PR #697: the packed weight cache builds from row-major or from the
 * production INTERLEAVED_4ROW layout with identical bytes; follow-up on the
 * orthogonal lm_head: rows in blocks of four, block nb at byte nb*2K, its
 * bytes ordered by k-chunk so that every 128-wide k range of a block is one
 * contiguous 256-byte sub-panel at nb*2K + g*256, and the per-row norms at
 * [(nb*G + g)*4 + ni]).
 *   chunk_k   weights per row in one k-chunk of a panel: 8, 16, 32, 64 or 128
 *             (the pages do not state the width; every divisor of 128 from 8
 *             up is accepted). K % chunk_k != 0: QMM_ERR_UNSUPPORTED_SHAPE.
 *   panels    device, ceil(N/4)*2K bytes. Row n = 4*nb + ni, weights
 *             k = c*chunk_k + 0..chunk_k-1 (c = k-chunk) are the chunk_k/2
 *             bytes at nb*2K + c*2*chunk_k + ni*chunk_k/2, low nibble = even k,
 *             nibble values as for qmm_pack_weights (indices for QMM_CQ4).
 *   scales    device, ceil(N/4)*G*4 fp16: row n, group g at ((n/4)*G + g)*4 + n%4.
 *   biases    device, the same layout; QMM_AFFINE only (NULL otherwise).
 *   codebook  HOST pointer, 16 int8 levels; QMM_CQ4 only (NULL otherwise).
 *   cb_scale  QMM_CQ4's codebook scale (finite); ignored otherwise.
 *   packed    device, qmm_packed_size(w) bytes, written entirely.
 * Rows of the last block beyond N are never read. Pointers must be 16-byte
 * aligned (QMM_ERR_MISALIGNED).
 */
qmm_status qmm_pack_weights_interleaved4(const qmm_weight_desc* w, int32_t chunk_k, const uint8_t* panels,
                                        const uint16_t* scales, const uint16_t* biases, const int8_t* codebook,
                                        float cb_scale, void* packed, qmm_stream stream);

/*
 * Activation prepass (device kernel, on `stream`).
 *
 * QMM_W4A8 and QMM_CQ4 (cactus PR #697, Summary: phase A rotates and quantizes
 * the activations to int8 in parallel; geistlib issue #500, Design sketch item 4: one
 * activation quantization shared by the GEMV and GEMM paths). For each row m
 * and group g, with v = x[m][g*group .. +group) in fp32:
 *   if hadamard == group: v <- H v, the unnormalised Sylvester-order
 *       Walsh-Hadamard transform, butterfly stages h = 1, 2, 4, .., group/2,
 *       each (v[i], v[i+h]) <- (v[i] + v[i+h], v[i] - v[i+h]) for (i & h) == 0,
 *       in fp32;
 *   amax = max |v|;  s = amax / 127 (fp32, IEEE division);
 *   a[m][k] = clamp(rint(v / s), -127, 127) (fp32 division, ties to even);
 *   sx[m][g] = s * c with c = fp32(1/sqrt(group)) when rotated, else 1;
 *   amax == 0 gives a = 0 and sx = 0;
 *   asum[m][g] = sum of the group's a.
 *   The orthonormal rotation H/sqrt(n) is carried by the scale, so the int8
 *   codes do not depend on its rounding.
 * Outputs (any may be NULL except sx):
 *   a     device int8  [M][K]   codes (GEMV operand)
 *   a16   device fp16  [M][K]   the same codes as fp16 (exact; GEMM operand)
 *   sx    device fp32  [M][G]
 *   asum  device int32 [M][G]
 * x: device [M][K], dtype x_dtype (F32, F16 or BF16; widened exactly to fp32).
 *
 * QMM_AFFINE (TensorFold PR #3215, What this changes: the group sums of X are
 * written once per call by a prepass, each with the tree
 * ((c0+c1)+(c2+c3))+((c4+c5)+(c6+c7)), c_j the left-to-right fp32 sum of
 * inputs 8j..8j+7 of the group). group must be 64, hadamard 0.
 *   gsum  device fp32 [M][G]    S[m][g] (required)
 *   x16   device fp16 [M][K]    fp16 image of x (RNE) when x_dtype is F32 or
 *                               BF16; may be NULL when x is already F16 (the
 *                               GEMM then reads x itself).
 *   S is summed from the fp32 values of x as given.
 * Pointers of the other variant must be NULL.
 */
qmm_status qmm_prep_act(int32_t variant, int32_t M, int32_t K, int32_t group, int32_t hadamard,
                        const void* x, int32_t x_dtype,
                        int8_t* a, uint16_t* a16, float* sx, int32_t* asum,
                        float* gsum, uint16_t* x16, qmm_stream stream);

/*
 * Activation prepass with a full K x K orthogonal rotation, for weights stored
 * rotated (QMM_W4A8 and QMM_CQ4 codes; device kernel, on `stream`).
 * cactus PR #697, Summary: the orthogonal-rotation CQ4 lm_head runs on the same
 * fused GEMV through an exact virtual 128-wide group view, the rotation applied
 * in phase A; "Orthogonal embedding dequantization": a K x K matvec with fp32
 * accumulation. For each row m:
 *   z[m][i] = sum_k R[i][k] * x[m][k], accumulated in fp32 with one fused
 *             multiply-add per term, k = 0, 1, ..., K-1 in that order;
 *   then per group g of z, as qmm_prep_act without an in-group transform:
 *   amax, s = amax/127, a = clamp(rint(z/s), -127, 127), sx = s (R is
 *   orthonormal: no further factor), asum = sum of a.
 * Weights W stored as W' = W R^T (one norm per row, the single group of
 * width K) are used through the virtual view: pack W' with group 128 (or 64)
 * and the row's norm repeated in every group; then W x = W' z, computed by
 * qmm_gemv / qmm_gemm on these codes.
 *   M >= 1; K % 128 == 0 (QMM_ERR_UNSUPPORTED_SHAPE); group 64 or 128.
 *   R      device, [K][K] fp32 row-major (a constant: it is read before the
 *          dependency wait on the previous kernel).
 *   x      device, [M][K] fp32 / fp16 / bf16 (x_dtype), widened exactly.
 *   a      device, [M][K] int8 codes, or NULL.
 *   a16    device, [M][K] fp16 image of the codes (the GEMM's operand), or NULL.
 *   sx     device, [M][G] fp32 (required).
 *   asum   device, [M][G] int32 code sums, or NULL.
 * Pointers 16-byte aligned (QMM_ERR_MISALIGNED).
 */
qmm_status qmm_prep_act_rotated(int32_t M, int32_t K, int32_t group, const float* R, const void* x,
                                int32_t x_dtype, int8_t* a, uint16_t* a16, float* sx, int32_t* asum,
                                qmm_stream stream);

/*
 * Bytes of workspace qmm_gemv wants for split-K over `w` (0 if none).
 * The workspace must be zero-filled before its first use; every completed
 * call leaves its counters at zero again, so it can be reused by later calls
 * on the same stream without clearing. Calls that may run concurrently need
 * separate workspaces.
 */
size_t qmm_gemv_workspace_size(const qmm_weight_desc* w);

/*
 * M = 1 decode GEMV, QMM_W4A8 or QMM_CQ4 (cactus PR #697, Summary: the hybrid
 * fused GEMV streams the packed nibbles, half the weight bytes, and is
 * DRAM-bound):
 *   y[n] = sum_g sw[n][g] * sx[g] * P[n][g],  P[n][g] = sum_{k in g} q[n][k] a[k]
 *   (QMM_CQ4: q[n][k] = C[i[n][k]] and y is multiplied by cb_scale)
 *   packed     device blob from qmm_pack_weights
 *   a          device int8 [K] (qmm_prep_act output a, row 0)
 *   sx         device fp32 [G]
 *   y          device fp32 [N]
 *   workspace  device, >= qmm_gemv_workspace_size(w) bytes, or NULL to run
 *              without split-K (fewer CTAs; the fp32 sum order differs).
 * Results are deterministic for a given shape and workspace choice: a fixed
 * reduction order, no atomics on data.
 */
qmm_status qmm_gemv(const qmm_weight_desc* w, const void* packed, const int8_t* a, const float* sx,
                    float* y, void* workspace, size_t workspace_bytes, qmm_stream stream);

/*
 * One-kernel M = 1 decode GEMV, QMM_W4A8 or QMM_CQ4: the activation prepass and the GEMV
 * in a single launch (cactus PR #697, Summary: the M = 1 path is one dispatch
 * whose phase A rotates and quantizes the activations and whose phase B
 * streams the packed nibbles through the integer partials).
 *   x         device [K], dtype x_dtype (F32, F16, BF16)
 *   hadamard  0 or w->group (as in qmm_prep_act)
 *   y         device fp32 [N]
 *   a_out     device int8 [K] or NULL: the codes (bit-identical to qmm_prep_act)
 *   sx_out    device fp32 [G] or NULL: the scales (bit-identical to qmm_prep_act)
 * y equals qmm_prep_act + qmm_gemv up to the fp32 summation order. The
 * K-slices of a 128-row tile run as one thread-block cluster and are summed
 * through distributed shared memory: no workspace, deterministic results.
 * QMM_ERR_UNSUPPORTED_SHAPE if a tile's K range does not fit the cluster's
 * shared memory (K > 16 x 44 x 64 for group 64, 16 x 22 x 128 for group 128).
 */
qmm_status qmm_gemv_fused(const qmm_weight_desc* w, const void* packed, const void* x, int32_t x_dtype,
                          int32_t hadamard, float* y, int8_t* a_out, float* sx_out, qmm_stream stream);

/*
 * Fused sibling GEMVs, QMM_W4A8 or QMM_CQ4: up to QMM_MAX_SIBLINGS weight matrices that
 * read the same input (q|k|v, gate|up) in one launch, x rotated and quantized
 * once per K-slice for all of them (cactus engine PR #750 "Metal Support":
 * sibling quantized GEMVs fused into one batched dispatch; geistlib issue #500,
 * Design sketch item 5: paired linears share one activation quantization).
 *   w[i], packed[i]  the matrices: one variant (all W4A8 or all CQ4, each CQ4
 *                    matrix with its own codebook), same K and group; any N[i]
 *   x, x_dtype, hadamard, a_out, sx_out   as qmm_gemv_fused
 *   y[i]             device fp32 [w[i].N]
 * Each y[i] matches qmm_gemv_fused on matrix i within the W4A8 tolerance (the
 * K-slice split, and with it the fp32 sum order, follows the launch's total
 * tile count); results are deterministic.
 * QMM_ERR_INVALID_ARG for count outside [1, QMM_MAX_SIBLINGS] or NULL
 * pointers; QMM_ERR_UNSUPPORTED_SHAPE for mismatched K, group or variant.
 */
#define QMM_MAX_SIBLINGS 8
qmm_status qmm_gemv_fused_siblings(int32_t count, const qmm_weight_desc* w, const void* const* packed,
                                   const void* x, int32_t x_dtype, int32_t hadamard, float* const* y,
                                   int8_t* a_out, float* sx_out, qmm_stream stream);

/*
 * M = 1 GEMV for callers that cannot allocate device memory. The pages have no
 * counterpart: it exists for code that runs inside a host program that owns
 * every device allocation and does not let it allocate, or on a latency-critical
 * path that must never reach cudaMalloc (which can synchronise the device).
 * Arguments, results and errors are those of qmm_gemv; instead of a caller's
 * workspace the split-K scratch is a fixed array inside the library of
 * QMM_GEMV_STATIC_SCRATCH_BYTES (1 MiB), held on every device that loads the
 * library until the process exits. A weight whose qmm_gemv_workspace_size
 * exceeds it is rejected with QMM_ERR_WORKSPACE. The call allocates nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call shares the array and finds the last call's contents in it; the
 *     call clears the part that must start at zero (the split-K counters) on
 *     `stream` before its kernel.
 *   - Calls whose work overlaps on the GPU (other streams, other host threads)
 *     race on the array: serialise them.
 */
#define QMM_GEMV_STATIC_SCRATCH_BYTES ((size_t)1 << 20)
qmm_status qmm_gemv_static_scratch(const qmm_weight_desc* w, const void* packed, const int8_t* a,
                                   const float* sx, float* y, qmm_stream stream);

/*
 * GEMM, any M >= 1, all variants, on the tcgen05 tensor cores
 * (cactus PR #697, Summary: fused GEMM with raw int32 partials and a separate
 * fp32 rescale; TensorFold PR #3215 for the affine tiles on the prepass sums).
 * A W4A8 or CQ4 call with M at or below the limit set by qmm_set_gemm_rows_max
 * (default 8) runs instead on the CUDA cores: exact int32 partials with dp4a,
 * each weight read once for all rows (qmm_last_kernel_id reports
 * QMM_KERNEL_GEMM_ROWS); same inputs, same outputs within the W4A8 tolerance.
 * With at least 512 row tiles (N > 65408) that kernel streams over the tiles
 * with all of K per block; with fewer it splits K over a cluster, and shapes
 * it cannot hold then (K above 1536 per 8-CTA cluster slice of 24 groups of
 * 64, or 12 of 128) go to the tensor cores. Of the calls on the tensor cores,
 * W4A8 ones with M <= 32 and at least 512 row tiles run the kernel that puts
 * the weights in the MMA's N slot, 256 weight rows per MMA
 * (QMM_KERNEL_GEMM_NARROW; see qmm_set_gemm_narrow), which performs the same
 * operations in the same order as the general tensor-core kernel. Those with
 * M <= 16 and group 128 (K at most 1792) run its e4m3 form
 * (QMM_KERNEL_GEMM_NARROW_E4M3): weight nibbles u = q + 8 and the two planes of
 * each activation code (16 floor(a/16) and a mod 16) are exact e4m3 numbers,
 * the kind::f8f6f4 MMA sums their products exactly, and the raw partial is
 * recovered as P = sum a u - 8 sum a; the rescale that follows is the general
 * kernel's, so the outputs are the same bits.
 *   QMM_W4A8:   act16 = qmm_prep_act a16 [M][K] fp16 codes, act_scale = sx [M][G]
 *               Y[m][n] = sum_g sw[n][g] * sx[m][g] * P[m][n][g]
 *   QMM_CQ4:    as QMM_W4A8, with q[n][k] = C[i[n][k]], times cb_scale
 *               (qmm_last_kernel_id: QMM_KERNEL_GEMM_CQ4 on the tensor cores)
 *   QMM_AFFINE: act16 = x as fp16 [M][K],     act_scale = S  [M][G]
 *               Y[m][n] = sum_g ( s[n][g] * sum_{k in g} q[n][k] x[m][k] + b[n][g] * S[m][g] )
 *   Y          device fp32 [M][N], row-major; rows m < M written, nothing else.
 * The weight operand is expanded from the nibbles to exact fp16 integers on
 * chip; group partials accumulate in fp32 in tensor memory (exact integers for
 * W4A8) and are rescaled in fp32 once per group.
 */
qmm_status qmm_gemm(const qmm_weight_desc* w, const void* packed, int32_t M, const uint16_t* act16,
                    const float* act_scale, float* Y, qmm_stream stream);

/*
 * Test hook (QMM_W4A8 and QMM_CQ4): run the GEMV or GEMM kernel of `path`
 * with its epilogue replaced by a store of the raw group partials
 *   P[m][n][g] = sum_{k in g} q[n][k] * a[m][k]   (int32, [M][N][G];
 *   QMM_CQ4: q[n][k] = C[i[n][k]], no cb_scale)
 * (the per-group partials contract of cactus PR #697: partials_out holds raw
 * dot products, the caller applies the scales).
 *   path QMM_PATH_GEMV: M must be 1, act = int8 a [K].
 *   path QMM_PATH_GEMM: act = fp16 a16 [M][K].
 */
qmm_status qmm_debug_partials(const qmm_weight_desc* w, const void* packed, int32_t M, int32_t path,
                              const void* act, int32_t* P, qmm_stream stream);

/* Static text for a status code. */
const char* qmm_status_string(qmm_status s);

/* The qmm_kernel_id of the last kernel this host thread enqueued (engagement check). */
int32_t qmm_last_kernel_id(void);

/*
 * Read and clear the device error word of the current device (synchronises
 * `stream`). Kernels that give up a bounded wait set it instead of hanging.
 * Returns QMM_OK, QMM_ERR_TIMEOUT, or QMM_ERR_CUDA; *flags (if non-NULL)
 * receives the raw word.
 */
qmm_status qmm_device_status(qmm_stream stream, int32_t* flags);

/* Enable (1, default) or disable (0) programmatic dependent launch for
 * launches made after the call (process-wide). */
void qmm_set_pdl(int32_t enable);

/*
 * Test-only fault injection (process-wide; 0 = off, the default). Point 1: the
 * next qmm_prep_act_rotated launches expect their first stage (the TMA box of R
 * and the rows of x) but never request it, so every CTA's bounded wait for it
 * runs out (one wait limit, about 2 s), the kernel sets the timeout bit of the
 * device error word and returns without writing its outputs (no CTA of a
 * cluster writes once any of them timed out); qmm_device_status then reports
 * QMM_ERR_TIMEOUT and the context stays usable. Other values turn injection off. (The pages have no
 * counterpart: it exercises the failure detection of the bounded waits.)
 */
void qmm_set_fault_injection(int32_t point);

/* Where qmm_gemm expands the 4-bit weights for the tensor cores (process-wide,
 * launches after the call): 0 (default) into tensor memory, read by
 * tcgen05.mma as its A operand; 1 into 128-byte-swizzled shared memory. Both
 * give the same partials; the choice only moves on-chip traffic. */
void qmm_set_gemm_weight_operand(int32_t in_shared_memory);

/* Largest M for which a W4A8 or CQ4 qmm_gemm runs on the CUDA-core (dp4a) kernel
 * (process-wide, launches after the call): 0 sends every call to the tensor
 * cores; values above 16 are treated as 16. Default 8 (above it the tensor
 * cores are as fast or faster on the measured shapes). */
void qmm_set_gemm_rows_max(int32_t max_rows);

/* When W4A8 and CQ4 qmm_gemm calls with M <= 32 (above the CUDA-core limit)
 * run the tensor-core kernel with the weights in the MMA's N slot
 * (process-wide, launches after the call): QMM_NARROW_OFF never;
 * QMM_NARROW_AUTO (default) for W4A8 with at least 512 row tiles, where it
 * measured faster (lm_head: 0.88x to 0.96x the time of the general kernel in
 * its fp16 form; codebook weights and few row tiles were slower);
 * QMM_NARROW_ALWAYS for every such call (tests); QMM_NARROW_F16 for every such
 * call, always in the fp16 form. Under AUTO and ALWAYS, W4A8 calls with
 * M <= 16 and group 128 take the e4m3 form when K fits its shared memory. The
 * outputs are the same bits whichever kernel runs; shapes whose activation
 * scales overflow the fp16 form's shared memory (K / group above about 300)
 * stay on the general kernel. */
enum { QMM_NARROW_OFF = 0, QMM_NARROW_AUTO = 1, QMM_NARROW_ALWAYS = 2, QMM_NARROW_F16 = 3 };
void qmm_set_gemm_narrow(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */

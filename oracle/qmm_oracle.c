/*
 * qmm_oracle.c -- plain CPU oracle of the group-quantized 4-bit matmul.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the CUDA path, with which it shares
 * no code. Build: gcc -O2 -std=c11 -ffp-contract=off (fp32 steps must be the
 * plain IEEE operations written here, never fused).
 *
 * Sources (the pages describing the method):
 *   [P1] cactus PR #697 "SME2 acceleration for CQ4 matmul, prefill attention,
 *        and orthogonal embeddings" (Summary; Quantized matmul; the per-group
 *        partials contract in its review thread; follow-up commits).
 *   [P2] geistlib issue #500 "cpu_neon: native W*A8 int8 GEMM for prefill,
 *        replacing dequant + BLAS sgemm" (Design sketch).
 *   [P3] TensorFold PR #3215 "simd_qmm on Metal: X's group sums and half
 *        operands from a prepass" (What this changes).
 *
 * Parity pins: every function here is checked by the non-GPU tests against
 * something other than itself (library routines, closed forms, brute force,
 * hand-computed fixtures). No function is "parity unpinned".
 */
#include "qmm_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------ binary16 */

/* IEEE 754 binary16 -> double (exact). */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* double -> IEEE 754 binary16, round to nearest, ties to even. */
uint16_t oracle_f64_to_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00;        /* rounds to infinity */
    if (a < ldexp(1.0, -14)) {                     /* subnormal range */
        double q = rint(a * ldexp(1.0, 24));       /* multiples of 2^-24 */
        return sign | (uint16_t)q;                 /* q == 1024 encodes 2^-14 */
    }
    int ex;
    frexp(a, &ex);                                 /* a = m * 2^ex, m in [0.5, 1) */
    int E = ex - 1;                                /* a in [2^E, 2^(E+1)) */
    double q = rint(ldexp(a, 10 - E));             /* significand * 1024, in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; E += 1; }
    if (E > 15) return sign | 0x7c00;
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0);
}

/* ------------------------------------------------------------ Hadamard */

/*
 * Unnormalised Walsh-Hadamard transform in Sylvester (natural) order, in fp32,
 * butterfly stages h = 1, 2, 4, ..., n/2 in that order:
 *     (v[i], v[i+h]) <- (v[i] + v[i+h], v[i] - v[i+h])   for (i & h) == 0.
 * [P1] Summary / Quantized matmul: the M=1 path applies a Hadamard transform to
 * the activations before their int8 quantization. The pages name neither the
 * ordering nor the stage order; this is the plain reading (natural order,
 * ascending stages).
 */
void oracle_fwht_f32(float* v, int n)
{
    for (int h = 1; h < n; h <<= 1)
        for (int i = 0; i < n; i++)
            if ((i & h) == 0) {
                float lo = v[i], hi = v[i + h];
                v[i] = lo + hi;
                v[i + h] = lo - hi;
            }
}

/* The same transform in fp64 (rotation-invariance checks). */
void oracle_fwht_f64(double* v, int n)
{
    for (int h = 1; h < n; h <<= 1)
        for (int i = 0; i < n; i++)
            if ((i & h) == 0) {
                double lo = v[i], hi = v[i + h];
                v[i] = lo + hi;
                v[i + h] = lo - hi;
            }
}

/* ------------------------------------------------------------ nibbles */

/*
 * [N][K/2] nibble bytes -> [N][K] values. Low nibble = even k ([P1] follow-up
 * "single runtime weight format": nibbles expand low nibble first).
 * W4A8: 4-bit two's complement, q in [-8, 7]. Affine: unsigned, q in [0, 15].
 */
int oracle_unpack_nibbles(int variant, int N, int K, const uint8_t* q_bytes, int8_t* q)
{
    if (N < 1 || K < 2 || (K & 1)) return 1;
    for (int n = 0; n < N; n++)
        for (int k = 0; k < K; k++) {
            uint8_t byte = q_bytes[(size_t)n * (K / 2) + k / 2];
            int u = (k & 1) ? (byte >> 4) : (byte & 0xf);
            if (variant == ORACLE_W4A8)
                q[(size_t)n * K + k] = (int8_t)(u >= 8 ? u - 16 : u);
            else
                q[(size_t)n * K + k] = (int8_t)u;
        }
    return 0;
}

/* ------------------------------------------------------------ packed blob */

/*
 * The packed weight blob, written from its index formula (the library's
 * header documents the same formula). [P1] Summary: the weight cache is built
 * once per weight and is byte-identical for every input layout; [P2] Design
 * sketch item 2: repack once at resolve time.
 *
 *   T = ceil(N/128) tiles, G = K/group, chunk (t, g) at (t*G + g)*CB,
 *   CB = 64*group + 256 (+256 for affine biases).
 *   nibble of (row r, local k) in piece p = k/32, word j = (k%32)/8,
 *   slot s = e/2 for even e = k%8, 4 + e/2 for odd e;
 *   byte offset p*2048 + r*16 + 4*j + s/2, high nibble when s is odd.
 *   Value stored: q + 8 (W4A8), q (affine). Scales at 64*group + 2r,
 *   biases at 64*group + 256 + 2r. Rows n >= N: q = 0, zero scales/biases.
 */
static int blob_ok(int variant, int N, int K, int group)
{
    if (N < 1 || K < 1) return 0;
    if (variant == ORACLE_W4A8 || variant == ORACLE_CQ4) return (group == 64 || group == 128) && K % group == 0;
    if (variant == ORACLE_AFFINE) return group == 64 && K % group == 0;
    return 0;
}

static size_t chunk_bytes(int variant, int group)
{
    return (size_t)64 * group + 256 + (variant == ORACLE_AFFINE ? 256 : 0);
}

size_t oracle_packed_size(int variant, int N, int K, int group)
{
    if (!blob_ok(variant, N, K, group)) return 0;
    size_t T = (size_t)(N + 127) / 128;
    return T * (size_t)(K / group) * chunk_bytes(variant, group) + (variant == ORACLE_CQ4 ? ORACLE_CQ4_TRAILER : 0);
}

static size_t nibble_offset(int r, int kl, int* high)
{
    int p = kl / 32, j = (kl % 32) / 8, e = kl % 8;
    int s = (e % 2 == 0) ? e / 2 : 4 + e / 2;
    *high = s & 1;
    return (size_t)p * 2048 + (size_t)r * 16 + 4 * j + s / 2;
}

/* Pack from logical values q_kn[n*K + k] (already unpacked). */
int oracle_pack_from_values(int variant, int N, int K, int group, const int8_t* q_nk,
                            const uint16_t* scales, const uint16_t* biases, uint8_t* blob)
{
    if (!blob_ok(variant, N, K, group)) return 1;
    if (variant == ORACLE_AFFINE && !biases) return 1;
    int G = K / group, T = (N + 127) / 128;
    size_t CB = chunk_bytes(variant, group);
    memset(blob, 0, oracle_packed_size(variant, N, K, group));
    for (int t = 0; t < T; t++)
        for (int g = 0; g < G; g++) {
            uint8_t* c = blob + ((size_t)t * G + g) * CB;
            for (int r = 0; r < 128; r++) {
                int n = t * 128 + r;
                for (int kl = 0; kl < group; kl++) {
                    int q = n < N ? q_nk[(size_t)n * K + g * group + kl] : 0;
                    int u = variant == ORACLE_W4A8 ? q + 8 : q;
                    int high;
                    size_t off = nibble_offset(r, kl, &high);
                    c[off] |= (uint8_t)(high ? (u & 0xf) << 4 : (u & 0xf));
                }
                uint16_t sv = n < N ? scales[(size_t)n * G + g] : 0;
                memcpy(c + 64 * group + 2 * r, &sv, 2);
                if (variant == ORACLE_AFFINE) {
                    uint16_t bv = n < N ? biases[(size_t)n * G + g] : 0;
                    memcpy(c + 64 * group + 256 + 2 * r, &bv, 2);
                }
            }
        }
    return 0;
}

/* Pack from the row-major nibble bytes (the library's input layout). */
int oracle_pack(int variant, int N, int K, int group, const uint8_t* q_bytes,
                const uint16_t* scales, const uint16_t* biases, uint8_t* blob)
{
    if (!blob_ok(variant, N, K, group)) return 1;
    int8_t* q = malloc((size_t)N * K);
    if (!q) return 2;
    oracle_unpack_nibbles(variant, N, K, q_bytes, q);
    int rc = oracle_pack_from_values(variant, N, K, group, q, scales, biases, blob);
    free(q);
    return rc;
}

/*
 * 4-row panels -> the row-major input of oracle_pack, from the panel's index
 * formula. [P1] Summary: the weight cache builds from row-major or from the
 * production INTERLEAVED_4ROW layout with byte-identical output; follow-up on
 * the orthogonal lm_head: rows come in blocks of four, block nb starting at
 * byte nb*2K (four rows of K/2 bytes), the block's bytes ordered by k-chunk so
 * that each 128-wide k range is one contiguous 256-byte sub-panel at
 * nb*2K + g*256, and the per-row norms at [(nb*G + g)*4 + ni].
 * The width of a k-chunk is not stated; it is the parameter chunk_k (8, 16,
 * 32, 64 or 128 weights, dividing K): chunk c of block nb holds the four rows'
 * chunk_k/2 bytes one row after the other. Row n = 4*nb + ni; rows of the last
 * block at or beyond N are not read. biases / pbiases may both be NULL.
 */
int oracle_interleaved4_to_rows(int N, int K, int group, int chunk_k, const uint8_t* panels,
                                const uint16_t* pscales, const uint16_t* pbiases, uint8_t* q_bytes,
                                uint16_t* scales, uint16_t* biases)
{
    if (N < 1 || K < 2 || group < 1 || K % group) return 1;
    if (chunk_k != 8 && chunk_k != 16 && chunk_k != 32 && chunk_k != 64 && chunk_k != 128) return 1;
    if (K % chunk_k) return 1;
    int G = K / group, cb = chunk_k / 2;
    for (int n = 0; n < N; n++) {
        int nb = n / 4, ni = n % 4;
        const uint8_t* block = panels + (size_t)nb * 2 * K;
        for (int c = 0; c < K / chunk_k; c++) {
            const uint8_t* piece = block + (size_t)c * 4 * cb + (size_t)ni * cb;
            for (int i = 0; i < cb; i++) q_bytes[(size_t)n * (K / 2) + (size_t)c * cb + i] = piece[i];
        }
        for (int g = 0; g < G; g++) {
            size_t at = ((size_t)nb * G + g) * 4 + ni;
            scales[(size_t)n * G + g] = pscales[at];
            if (biases && pbiases) biases[(size_t)n * G + g] = pbiases[at];
        }
    }
    return 0;
}

/* Inverse of the blob formula: recover values, scales and biases. */
int oracle_unpack_blob(int variant, int N, int K, int group, const uint8_t* blob,
                       int8_t* q, uint16_t* scales, uint16_t* biases)
{
    if (!blob_ok(variant, N, K, group)) return 1;
    int G = K / group;
    size_t CB = chunk_bytes(variant, group);
    for (int n = 0; n < N; n++) {
        int t = n / 128, r = n % 128;
        for (int g = 0; g < G; g++) {
            const uint8_t* c = blob + ((size_t)t * G + g) * CB;
            for (int kl = 0; kl < group; kl++) {
                int high;
                size_t off = nibble_offset(r, kl, &high);
                int u = high ? c[off] >> 4 : c[off] & 0xf;
                q[(size_t)n * K + g * group + kl] = (int8_t)(variant == ORACLE_W4A8 ? u - 8 : u);
            }
            memcpy(&scales[(size_t)n * G + g], c + 64 * group + 2 * r, 2);
            if (variant == ORACLE_AFFINE && biases)
                memcpy(&biases[(size_t)n * G + g], c + 64 * group + 256 + 2 * r, 2);
        }
    }
    return 0;
}

/* ------------------------------------------------------------ W4A8 prep */

/*
 * Activation prepass of the symmetric variant, per row m and group g
 * ([P1] Summary: "parallel Hadamard + int8 activation quantization" before the
 * GEMV's weight streaming; [P2] Design sketch item 4: one quantization shared
 * by GEMV and GEMM; per row and per group, rounding half to even, clamp to
 * [-127, 127]):
 *   1. v = x[m][g*group .. +group) in fp32;
 *   2. if hadamard == group: v <- unnormalised FWHT(v) (oracle_fwht_f32);
 *   3. amax = max |v|;
 *   4. amax == 0: a = 0, sx = 0;
 *   5. else s = amax / 127 (fp32 division); a = clamp(rint(v / s), -127, 127)
 *      (fp32 division, ties to even); sx = s * c, c = fp32(1/sqrt(group))
 *      with the rotation, c = 1 without.
 * The orthonormal rotation H/sqrt(n) is applied through its scale factor c,
 * so the codes do not depend on the rounding of the normalisation.
 */
int oracle_prep_w4a8(int M, int K, int group, int hadamard, const float* x,
                     int8_t* a, float* sx, int32_t* asum)
{
    if (M < 1 || group < 2 || K % group != 0) return 1;
    if (hadamard != 0 && hadamard != group) return 1;
    if (group & (group - 1)) return 1;
    int G = K / group;
    float c = hadamard ? (float)(1.0 / sqrt((double)group)) : 1.0f;
    float* v = malloc(sizeof(float) * group);
    if (!v) return 2;
    for (int m = 0; m < M; m++)
        for (int g = 0; g < G; g++) {
            const float* xg = x + (size_t)m * K + (size_t)g * group;
            for (int i = 0; i < group; i++) v[i] = xg[i];
            if (hadamard) oracle_fwht_f32(v, group);
            float amax = 0.0f;
            for (int i = 0; i < group; i++)
                if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
            int8_t* ag = a + (size_t)m * K + (size_t)g * group;
            int32_t sum = 0;
            if (amax == 0.0f) {
                for (int i = 0; i < group; i++) ag[i] = 0;
                sx[(size_t)m * G + g] = 0.0f;
            } else {
                float s = amax / 127.0f;
                for (int i = 0; i < group; i++) {
                    float r = rintf(v[i] / s);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    ag[i] = (int8_t)r;
                    sum += ag[i];
                }
                sx[(size_t)m * G + g] = s * c;
            }
            if (asum) asum[(size_t)m * G + g] = sum;
        }
    free(v);
    return 0;
}

/*
 * Activation prepass with a full K x K orthogonal rotation ([P1] Summary: the
 * orthogonal-rotation CQ4 lm_head runs on the same fused GEMV through an exact
 * virtual 128-wide group view, the rotation applied in phase A; [P1]
 * orthogonal embedding dequantization: the rotation is a K x K matvec with
 * fp32 accumulation). For each row m:
 *   1. z[i] = sum_k R[i][k] * x[m][k] in fp32: one fused multiply-add per
 *      term, k = 0, 1, ..., K-1 in that order (the pages fix no order; this
 *      is the plain one);
 *   2. the per-group quantization of oracle_prep_w4a8 on z with no in-group
 *      transform (R is orthonormal, so the scale carries no further factor).
 * z_out (nullable) receives z [M][K].
 */
int oracle_prep_rotated(int M, int K, int group, const float* R, const float* x,
                        int8_t* a, float* sx, int32_t* asum, float* z_out)
{
    if (M < 1 || K < 1 || group < 2 || K % group != 0) return 1;
    float* z = malloc(sizeof(float) * (size_t)M * K);
    if (!z) return 2;
    for (int m = 0; m < M; m++)
        for (int i = 0; i < K; i++) {
            const float* Ri = R + (size_t)i * K;
            const float* xm = x + (size_t)m * K;
            float acc = 0.0f;
            for (int k = 0; k < K; k++) acc = fmaf(Ri[k], xm[k], acc);
            z[(size_t)m * K + i] = acc;
        }
    int rc = oracle_prep_w4a8(M, K, group, 0, z, a, sx, asum);
    if (z_out) memcpy(z_out, z, sizeof(float) * (size_t)M * K);
    free(z);
    return rc;
}

/* ------------------------------------------------------------ W4A8 GEMM */

/*
 * Raw group partials ([P1] review thread, the per-group partials contract:
 * partials hold the plain integer dot product of one group of activations with
 * one channel's weights, and the caller applies the scales):
 *   P[m][n][g] = sum_{k in g} q[n][k] * a[m][k]   (exact, int64 then int32).
 */
int oracle_partials_w4a8(int M, int N, int K, int group, const uint8_t* q_bytes,
                         const int8_t* a, int32_t* P)
{
    if (M < 1 || N < 1 || K % group != 0) return 1;
    int G = K / group;
    int8_t* q = malloc((size_t)N * K);
    if (!q) return 2;
    oracle_unpack_nibbles(ORACLE_W4A8, N, K, q_bytes, q);
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++)
            for (int g = 0; g < G; g++) {
                int64_t acc = 0;
                for (int kl = 0; kl < group; kl++) {
                    int k = g * group + kl;
                    acc += (int64_t)q[(size_t)n * K + k] * a[(size_t)m * K + k];
                }
                P[((size_t)m * N + n) * G + g] = (int32_t)acc;
            }
    free(q);
    return 0;
}

/*
 * Symmetric output in fp64 ([P1] Summary: raw int32 partials with a separate
 * fp32 rescale; here the rescale is done exactly in fp64 as the reference):
 *   Y[m][n] = sum_g sw[n][g] * sx[m][g] * P[m][n][g]
 *   Ymag[m][n] = sum_g |sw[n][g] * sx[m][g] * P[m][n][g]|  (tolerance scale)
 * Only the output rows listed in `rows` are computed (all when rows == NULL);
 * Y and Ymag are [M][n_rows].
 */
int oracle_gemm_w4a8_rows(int M, int N, int K, int group, const uint8_t* q_bytes,
                          const uint16_t* sw, const int8_t* a, const float* sx,
                          int n_rows, const int32_t* rows, double* Y, double* Ymag)
{
    if (M < 1 || N < 1 || K % group != 0 || n_rows < 1) return 1;
    int G = K / group;
    int8_t* qrow = malloc((size_t)K);
    if (!qrow) return 2;
    for (int i = 0; i < n_rows; i++) {
        int n = rows ? rows[i] : i;
        if (n < 0 || n >= N) { free(qrow); return 1; }
        oracle_unpack_nibbles(ORACLE_W4A8, 1, K, q_bytes + (size_t)n * (K / 2), qrow);
        for (int m = 0; m < M; m++) {
            double y = 0.0, mag = 0.0;
            for (int g = 0; g < G; g++) {
                int64_t p = 0;
                for (int kl = 0; kl < group; kl++) {
                    int k = g * group + kl;
                    p += (int64_t)qrow[k] * a[(size_t)m * K + k];
                }
                double t = oracle_f16_to_f64(sw[(size_t)n * G + g]) * (double)sx[(size_t)m * G + g] * (double)p;
                y += t;
                mag += fabs(t);
            }
            Y[(size_t)m * n_rows + i] = y;
            if (Ymag) Ymag[(size_t)m * n_rows + i] = mag;
        }
    }
    free(qrow);
    return 0;
}

int oracle_gemm_w4a8(int M, int N, int K, int group, const uint8_t* q_bytes,
                     const uint16_t* sw, const int8_t* a, const float* sx,
                     double* Y, double* Ymag)
{
    return oracle_gemm_w4a8_rows(M, N, K, group, q_bytes, sw, a, sx, N, NULL, Y, Ymag);
}

/* ------------------------------------------------------------ affine */

/*
 * Group sums of X for the affine bias term, the tree of [P3] (What this
 * changes): for each row m and group g of 64 inputs, c_j is the left-to-right
 * fp32 sum of inputs 8j .. 8j+7 (j = 0..7), and
 *   S[m][g] = ((c0 + c1) + (c2 + c3)) + ((c4 + c5) + (c6 + c7))   in fp32.
 */
int oracle_group_sums_affine(int M, int K, int group, const float* x, float* S)
{
    if (M < 1 || group != 64 || K % group != 0) return 1;
    int G = K / group;
    for (int m = 0; m < M; m++)
        for (int g = 0; g < G; g++) {
            const float* xg = x + (size_t)m * K + (size_t)g * group;
            float c[8];
            for (int j = 0; j < 8; j++) {
                float acc = xg[8 * j];
                for (int i = 1; i < 8; i++) acc = acc + xg[8 * j + i];
                c[j] = acc;
            }
            S[(size_t)m * G + g] = ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));
        }
    return 0;
}

/*
 * Affine output in fp64 ([P3] What this changes: w = s*q + b per group, the
 * bias term through the group sums of X), from x's exact fp16 values:
 *   Y[m][n] = sum_g ( s[n][g] * sum_{k in g} q[n][k] x[m][k] + b[n][g] * sum_{k in g} x[m][k] )
 *   Ymag[m][n] = sum_k |(s q + b)[n][k] * x[m][k]|   (tolerance scale)
 * The group sums are exact here (fp64 sum of fp16 values), not the fp32 tree.
 * Only the output rows listed in `rows` are computed (all when rows == NULL).
 */
int oracle_gemm_affine_rows(int M, int N, int K, int group, const uint8_t* q_bytes,
                            const uint16_t* s, const uint16_t* b, const uint16_t* x16,
                            int n_rows, const int32_t* rows, double* Y, double* Ymag)
{
    if (M < 1 || N < 1 || group != 64 || K % group != 0 || n_rows < 1) return 1;
    int G = K / group;
    int8_t* qrow = malloc((size_t)K);
    double* xd = malloc(sizeof(double) * (size_t)M * K);
    if (!qrow || !xd) { free(qrow); free(xd); return 2; }
    for (size_t i = 0; i < (size_t)M * K; i++) xd[i] = oracle_f16_to_f64(x16[i]);
    for (int i = 0; i < n_rows; i++) {
        int n = rows ? rows[i] : i;
        if (n < 0 || n >= N) { free(qrow); free(xd); return 1; }
        oracle_unpack_nibbles(ORACLE_AFFINE, 1, K, q_bytes + (size_t)n * (K / 2), qrow);
        for (int m = 0; m < M; m++) {
            const double* xm = xd + (size_t)m * K;
            double y = 0.0, mag = 0.0;
            for (int g = 0; g < G; g++) {
                double sv = oracle_f16_to_f64(s[(size_t)n * G + g]);
                double bv = oracle_f16_to_f64(b[(size_t)n * G + g]);
                double qx = 0.0, sumx = 0.0;
                for (int kl = 0; kl < group; kl++) {
                    int k = g * group + kl;
                    qx += (double)qrow[k] * xm[k];
                    sumx += xm[k];
                    mag += fabs((sv * qrow[k] + bv) * xm[k]);
                }
                y += sv * qx + bv * sumx;
            }
            Y[(size_t)m * n_rows + i] = y;
            if (Ymag) Ymag[(size_t)m * n_rows + i] = mag;
        }
    }
    free(qrow);
    free(xd);
    return 0;
}

int oracle_gemm_affine(int M, int N, int K, int group, const uint8_t* q_bytes,
                       const uint16_t* s, const uint16_t* b, const uint16_t* x16,
                       double* Y, double* Ymag)
{
    return oracle_gemm_affine_rows(M, N, K, group, q_bytes, s, b, x16, N, NULL, Y, Ymag);
}

/* ------------------------------------------------------------ CQ4 */

/*
 * Codebook 4-bit weights (cactus PR #697 "SME2 acceleration for CQ4 matmul,
 * prefill attention, and orthogonal embeddings", Summary: in-engine 4-bit
 * codebook expansion in the GEMV leaf; follow-up "single runtime weight
 * format": codebook table lookup, a single fp32 rescale with the codebook
 * scale folded into the per-row norms).
 * Reading: each weight is a 4-bit index i (even k in the low nibble) into one
 * 16-entry int8 codebook C of the matrix; the weight is cb_scale * sw * C[i].
 * The partial stays integer, P[m][n][g] = sum_{k in g} C[i[n][k]] * a[m][k],
 * and the output is Y = sum_g (sw * cb_scale) * sx * P (here exactly, fp64).
 * Blob: the symmetric tile layout with the raw indices as nibbles, then a
 * 32-byte trailer: C[0..15] (int8), cb_scale (fp32), 12 zero bytes.
 */
int oracle_pack_cq4(int N, int K, int group, const uint8_t* idx_bytes, const int8_t* codebook, float cb_scale,
                    const uint16_t* scales, uint8_t* blob)
{
    if (!blob_ok(ORACLE_CQ4, N, K, group)) return 1;
    int8_t* q = malloc((size_t)N * K);
    if (!q) return 2;
    oracle_unpack_nibbles(ORACLE_CQ4, N, K, idx_bytes, q);
    int rc = oracle_pack_from_values(ORACLE_CQ4, N, K, group, q, scales, NULL, blob);
    free(q);
    if (rc) return rc;
    uint8_t* tr = blob + oracle_packed_size(ORACLE_CQ4, N, K, group) - ORACLE_CQ4_TRAILER;
    memcpy(tr, codebook, 16);
    memcpy(tr + 16, &cb_scale, 4);
    return 0;
}

int oracle_partials_cq4(int M, int N, int K, int group, const uint8_t* idx_bytes, const int8_t* codebook,
                        const int8_t* a, int32_t* P)
{
    if (M < 1 || N < 1 || K % group != 0) return 1;
    int G = K / group;
    int8_t* idx = malloc((size_t)N * K);
    if (!idx) return 2;
    oracle_unpack_nibbles(ORACLE_CQ4, N, K, idx_bytes, idx);
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++)
            for (int g = 0; g < G; g++) {
                int64_t acc = 0;
                for (int kl = 0; kl < group; kl++) {
                    int k = g * group + kl;
                    acc += (int64_t)codebook[idx[(size_t)n * K + k]] * a[(size_t)m * K + k];
                }
                P[((size_t)m * N + n) * G + g] = (int32_t)acc;
            }
    free(idx);
    return 0;
}

/* Y and Ymag (sum of |terms|, the tolerance scale) for the listed rows. */
int oracle_gemm_cq4_rows(int M, int N, int K, int group, const uint8_t* idx_bytes, const int8_t* codebook,
                         float cb_scale, const uint16_t* sw, const int8_t* a, const float* sx, int n_rows,
                         const int32_t* rows, double* Y, double* Ymag)
{
    if (M < 1 || N < 1 || K % group != 0 || n_rows < 1) return 1;
    int G = K / group;
    int8_t* idx = malloc((size_t)K);
    if (!idx) return 2;
    for (int i = 0; i < n_rows; i++) {
        int n = rows ? rows[i] : i;
        if (n < 0 || n >= N) { free(idx); return 1; }
        oracle_unpack_nibbles(ORACLE_CQ4, 1, K, idx_bytes + (size_t)n * (K / 2), idx);
        for (int m = 0; m < M; m++) {
            double y = 0.0, mag = 0.0;
            for (int g = 0; g < G; g++) {
                int64_t p = 0;
                for (int kl = 0; kl < group; kl++) {
                    int k = g * group + kl;
                    p += (int64_t)codebook[idx[k]] * a[(size_t)m * K + k];
                }
                double t = oracle_f16_to_f64(sw[(size_t)n * G + g]) * (double)cb_scale * (double)sx[(size_t)m * G + g] *
                           (double)p;
                y += t;
                mag += fabs(t);
            }
            Y[(size_t)m * n_rows + i] = y;
            if (Ymag) Ymag[(size_t)m * n_rows + i] = mag;
        }
    }
    free(idx);
    return 0;
}

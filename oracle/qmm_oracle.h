/*
 * qmm_oracle.h -- plain CPU oracle of the group-quantized 4-bit matmul.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code with
 * the CUDA path and the CUDA path never calls it.
 *
 * Each function states what it computes and the passage it follows. Where the
 * method reaches a result with a plain definition (partials, outputs, group
 * sums) the function is that definition written out; the activation prepass
 * follows the method's steps in order.
 */
#ifndef QMM_ORACLE_H
#define QMM_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#define ORACLE_W4A8 0
#define ORACLE_AFFINE 1
#define ORACLE_CQ4 2
#define ORACLE_CQ4_TRAILER 32

double oracle_f16_to_f64(uint16_t h);
uint16_t oracle_f64_to_f16(double v);

void oracle_fwht_f32(float* v, int n);
void oracle_fwht_f64(double* v, int n);

int oracle_unpack_nibbles(int variant, int N, int K, const uint8_t* q_bytes, int8_t* q);

size_t oracle_packed_size(int variant, int N, int K, int group);
int oracle_pack(int variant, int N, int K, int group, const uint8_t* q_bytes,
                const uint16_t* scales, const uint16_t* biases, uint8_t* blob);
int oracle_pack_from_values(int variant, int N, int K, int group, const int8_t* q_nk,
                            const uint16_t* scales, const uint16_t* biases, uint8_t* blob);
int oracle_interleaved4_to_rows(int N, int K, int group, int chunk_k, const uint8_t* panels,
                                const uint16_t* pscales, const uint16_t* pbiases, uint8_t* q_bytes,
                                uint16_t* scales, uint16_t* biases);
int oracle_unpack_blob(int variant, int N, int K, int group, const uint8_t* blob,
                       int8_t* q, uint16_t* scales, uint16_t* biases);

int oracle_prep_w4a8(int M, int K, int group, int hadamard, const float* x,
                     int8_t* a, float* sx, int32_t* asum);
int oracle_prep_rotated(int M, int K, int group, const float* R, const float* x,
                        int8_t* a, float* sx, int32_t* asum, float* z_out);
int oracle_partials_w4a8(int M, int N, int K, int group, const uint8_t* q_bytes,
                         const int8_t* a, int32_t* P);
int oracle_gemm_w4a8(int M, int N, int K, int group, const uint8_t* q_bytes,
                     const uint16_t* sw, const int8_t* a, const float* sx,
                     double* Y, double* Ymag);
int oracle_gemm_w4a8_rows(int M, int N, int K, int group, const uint8_t* q_bytes,
                          const uint16_t* sw, const int8_t* a, const float* sx,
                          int n_rows, const int32_t* rows, double* Y, double* Ymag);

int oracle_group_sums_affine(int M, int K, int group, const float* x, float* S);
int oracle_gemm_affine(int M, int N, int K, int group, const uint8_t* q_bytes,
                       const uint16_t* s, const uint16_t* b, const uint16_t* x16,
                       double* Y, double* Ymag);
int oracle_gemm_affine_rows(int M, int N, int K, int group, const uint8_t* q_bytes,
                            const uint16_t* s, const uint16_t* b, const uint16_t* x16,
                            int n_rows, const int32_t* rows, double* Y, double* Ymag);

int oracle_pack_cq4(int N, int K, int group, const uint8_t* idx_bytes, const int8_t* codebook, float cb_scale,
                    const uint16_t* scales, uint8_t* blob);
int oracle_partials_cq4(int M, int N, int K, int group, const uint8_t* idx_bytes, const int8_t* codebook,
                        const int8_t* a, int32_t* P);
int oracle_gemm_cq4_rows(int M, int N, int K, int group, const uint8_t* idx_bytes, const int8_t* codebook,
                         float cb_scale, const uint16_t* sw, const int8_t* a, const float* sx, int n_rows,
                         const int32_t* rows, double* Y, double* Ymag);

#endif

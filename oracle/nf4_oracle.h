/*
 * nf4_oracle.h -- CPU oracle for the NF4-dequant-fused backward-A GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path includes, links or
 * calls this code: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library; the NF4 codebook in nf4_oracle.c is typed a second time on
 * purpose.
 *
 * What it computes (page "aprender-gpu 0.32.0 -- src/kernels/backward/
 * nf4_tensor_core.rs", struct doc comment):
 *
 *     grad_A[M x K] = grad_out[M x N] @ dequant(B_nf4[K x N])^T
 *
 * in plain loops, with the operands rounded the way that page's kernel rounds
 * them (fp32 scale * codebook, then f32 -> f16; grad_out f32 -> f16) and the
 * sum taken in fp64 (double), sequentially over n.
 *
 * Layouts (same page, build_ptx, "PHASE 2: Dequant B_nf4"):
 *   scales  fp32 [N][K/64]              scale of (column n, 64-element K-block b)
 *   data    u8   [N][K/2]               byte of element (k, n) at n*(K/2) + k/2,
 *                                       low nibble = even k, high nibble = odd k
 *   B       fp32 [K][N] row-major       the dense weight that nf4o_quantize reads
 *   go      [M][N] row-major            fp32, or bf16 given as raw uint16 bits
 *   result  fp64 [rows][K]
 *
 * Every function returns 0 on success and a negative value on bad arguments.
 */
#ifndef NF4_ORACLE_H
#define NF4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { NF4O_F32 = 0, NF4O_BF16 = 1 };

/* The 16-value NormalFloat4 codebook, ascending. */
void nf4o_codebook(float out[16]);

/* IEEE 754 binary32 -> binary16, round to nearest even, gradual underflow,
 * overflow to infinity, NaN kept quiet.  Integer bit operations only. */
uint16_t nf4o_f32_to_f16(float x);
void nf4o_f32_to_f16_array(const float* x, long long count, uint16_t* out);
double nf4o_f16_to_f64(uint16_t h);
float nf4o_bf16_to_f32(uint16_t b);

/* Quantise B fp32 [K][N] (row-major) into packed NF4 codes and absmax scales.
 * K must be a positive multiple of 64, N positive. */
int nf4o_quantize(const float* B, int K, int N, uint8_t* data, float* scales);

/* The code of element (k, n), read back from the packed data. */
int nf4o_code_at(const uint8_t* data, int K, int k, int n);

/* deq(B)[k, n] = f16( fp32(scale[n][k/64] * codebook[code(k, n)]) ), written
 * transposed as raw f16 bits bt[n*K + k]. */
int nf4o_dequantize_f16(const float* scales, const uint8_t* data, int K, int N,
                        uint16_t* bt);

/* Round grad_out to the f16 operand the GEMM multiplies: f32 -> f16 (RNE), or
 * bf16 -> f32 (exact) -> f16 (RNE). */
int nf4o_round_operand(const void* go, int dtype, long long count, uint16_t* out);

/* ref[i][k] = sum_n f16(go)[rows[i], n] * deq(B)[k, n], in fp64, n ascending;
 * bound[i][k] = the same sum over absolute values of the products (may be
 * NULL).  go16 is [M][N] f16 bits, bt is [N][K] f16 bits. */
int nf4o_backward_a_rows(const uint16_t* go16, const uint16_t* bt,
                         int M, int N, int K, const int* rows, int nrows,
                         double* ref, double* bound);

/* Whole problem from raw inputs: rounds go, dequantises B, and computes every
 * row.  ref and bound are [M][K]; bound may be NULL. */
int nf4o_backward_a(const void* go, int dtype, const float* scales,
                    const uint8_t* data, int M, int N, int K,
                    double* ref, double* bound);

/* Sibling-projection fusion: the input gradient of a layer input shared by
 * `parts` projections, ref[i][k] = sum over parts p, then n < N[p], of
 * f16(go_p)[rows[i], n] * deq(B_p)[k, n], one fp64 sum per element (parts in
 * order, n ascending); bound the same over |products| (may be NULL).  go16[p]
 * is [M][N[p]] f16 bits, bt[p] is [N[p]][K] f16 bits. */
int nf4o_backward_a_fused_rows(int parts, const uint16_t* const* go16,
                               const uint16_t* const* bt, const int* N, int M, int K,
                               const int* rows, int nrows, double* ref, double* bound);

/* Forward product: ref[i][n] = sum_k f16(A)[rows[i], k] * deq(B)[k, n], in
 * fp64, k ascending; bound[i][n] the same over |products| (may be NULL).  a16
 * is [M][K] f16 bits, bt is deq(B) transposed, [N][K] f16 bits. */
int nf4o_forward_rows(const uint16_t* a16, const uint16_t* bt, int M, int N, int K,
                      const int* rows, int nrows, double* ref, double* bound);

/* Whole forward problem from raw inputs (A fp32 or bf16 bits, [M][K]); ref and
 * bound are [M][N]; bound may be NULL. */
int nf4o_forward(const void* a, int dtype, const float* scales, const uint8_t* data,
                 int M, int N, int K, double* ref, double* bound);

/* Dense weight gradient grad_B = A^T @ grad_C of C = A @ B (A [M][K], grad_C
 * [M][N], 16-bit floats as raw bits: dtype16 0 = f16, 1 = bf16): ref[i][n] =
 * sum_m A[m][rows[i]] * grad_C[m][n] in fp64, m ascending; bound the same over
 * |products| (may be NULL).  ref and bound are [nrows][N]. */
int nf4o_gemm_backward_b_rows(const uint16_t* a, const uint16_t* gc, int dtype16, int M, int K,
                              int N, const int* rows, int nrows, double* ref, double* bound);

/* OpenMP thread control for the row loops (1 when built without OpenMP). */
void nf4o_set_threads(int n);
int nf4o_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif

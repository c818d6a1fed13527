/*
 * nf4_oracle.c -- plain, slow CPU oracle for the NF4 backward-A GEMM.
 *
 * TEST INFRASTRUCTURE ONLY (see nf4_oracle.h).  Build with
 *     gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared
 * so that no a*b+c is fused and every float operation rounds as written.
 *
 * Sources followed, by page and section:
 *   [P3]  "trueno-gpu 0.4.17 -- src/kernels/backward/mod.rs", module list
 *         (GemmBackwardAKernel / GemmBackwardBKernel: gradients of both
 *         operands of a matrix product) and its parameter test.
 *   [P1]  "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs"
 *         struct doc comment: grad_A = grad_out @ dequant(B_nf4)^T, shared
 *         dimension N, output dimension K.
 *         build_ptx "PHASE 1": grad_out f32 -> f16 (cvt), out-of-range -> 0.
 *         build_ptx "PHASE 2": block = k/64, element = k%64, scale at
 *         scales[n*(K/64) + block], byte at data[n*(K/64)*32 + block*32 +
 *         element/2], nibble = (byte >> 4*(element%2)) & 0xF, weight =
 *         scale * codebook[nibble] in f32, then f32 -> f16.
 *         build_ptx "PHASE 3": f16 x f16 products accumulated over N.
 *   [QL]  Dettmers et al., "QLoRA: Efficient Finetuning of Quantized LLMs"
 *         (2023), the NormalFloat4 data type (quantiles of N(0,1), 7 negative
 *         values, zero, 8 positive values, normalised to [-1, 1]) and blockwise
 *         absmax quantisation.
 *
 * Readings where [P1] is silent (also listed in the design notes):
 *   - The quantiser is not on [P1].  Per block: s = max |x| (exact in f32);
 *     s == 0 gives scale 0 and code 7 everywhere; otherwise y = x / s (IEEE
 *     f32 division) and code = argmin_c |y - codebook[c]| with the differences
 *     in f32, ties to the lower code.
 *   - [P1]'s f32 -> f16 conversion does not show its rounding modifier; round
 *     to nearest even is taken (the only rounding a plain conversion has).
 *   - bf16 grad_out: widened exactly to f32, then rounded to f16 like f32.
 *   - The sum is the exact-up-to-fp64 reference: fp64 accumulation, n
 *     ascending, no reordering.
 */
#include "nf4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* [QL] NormalFloat4 values, ascending (the table printed with the NF4 type). */
static const float kNF4[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

void nf4o_codebook(float out[16]) {
    for (int i = 0; i < 16; ++i) out[i] = kNF4[i];
}

static uint32_t f32_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u;
}

/* IEEE 754-2008 binary32 -> binary16, roundTiesToEven. */
uint16_t nf4o_f32_to_f16(float x) {
    const uint32_t u = f32_bits(x);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    const uint32_t exp_field = (u >> 23) & 0xFFu;
    const uint32_t frac = u & 0x7FFFFFu;

    if (exp_field == 0xFFu) {                       /* inf or NaN */
        if (frac == 0) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | 0x7E00u | (frac >> 13));
    }
    if (exp_field == 0) {
        /* f32 zero or subnormal: magnitude < 2^-126, far below half of the
         * smallest f16 subnormal (2^-25), so the result is a signed zero. */
        return sign;
    }
    const int e = (int)exp_field - 127;            /* unbiased exponent */
    if (e > 15) return (uint16_t)(sign | 0x7C00u); /* >= 2^16: overflow */

    const uint32_t sig = frac | 0x800000u;          /* 24-bit significand */
    if (e >= -14) {
        /* Normal f16 range: keep 11 significant bits, drop 13. */
        uint32_t m = sig >> 13;                     /* includes the hidden bit */
        const uint32_t rem = sig & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (m & 1u))) ++m;
        int be = e + 15;
        if (m == 0x800u) {                          /* carried into next binade */
            m >>= 1;
            ++be;
        }
        if (be >= 31) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | ((uint32_t)be << 10) | (m & 0x3FFu));
    }
    /* Subnormal f16: the value is sig * 2^(e-23); in units of 2^-24 that is
     * sig * 2^(e+1), i.e. sig shifted right by -(e+1) >= 14 places. */
    const int shift = -(e + 1);
    if (shift > 25) return sign;                    /* < 2^-25: rounds to zero */
    uint32_t m = sig >> shift;
    const uint32_t rem = sig & ((1u << shift) - 1u);
    const uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (m & 1u))) ++m;
    /* m == 0x400 here is the smallest normal, which the encoding gives for free. */
    return (uint16_t)(sign | m);
}

void nf4o_f32_to_f16_array(const float* x, long long count, uint16_t* out) {
    for (long long i = 0; i < count; ++i) out[i] = nf4o_f32_to_f16(x[i]);
}

double nf4o_f16_to_f64(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int be = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    double v;
    if (be == 0) {
        v = ldexp((double)m, -24);
    } else if (be == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(m | 0x400), be - 25);
    }
    return sign ? -v : v;
}

float nf4o_bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Code of the codebook entry nearest to y, differences in f32, ties low. */
static int nearest_code(float y) {
    int best = 0;
    float best_d = fabsf(y - kNF4[0]);
    for (int c = 1; c < 16; ++c) {
        const float d = fabsf(y - kNF4[c]);
        if (d < best_d) {
            best_d = d;
            best = c;
        }
    }
    return best;
}

int nf4o_quantize(const float* B, int K, int N, uint8_t* data, float* scales) {
    if (!B || !data || !scales || K <= 0 || N <= 0 || K % 64 != 0) return -1;
    const int KB = K / 64;
    const long long half_k = K / 2;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < KB; ++b) {
            float s = 0.0f;
            for (int e = 0; e < 64; ++e) {
                const float a = fabsf(B[(long long)(b * 64 + e) * N + n]);
                if (a > s) s = a;
            }
            scales[(long long)n * KB + b] = s;
            for (int e = 0; e < 64; e += 2) {
                int code[2];
                for (int h = 0; h < 2; ++h) {
                    const int k = b * 64 + e + h;
                    if (s == 0.0f) {
                        code[h] = 7;
                    } else {
                        const float y = B[(long long)k * N + n] / s;
                        code[h] = nearest_code(y);
                    }
                }
                data[(long long)n * half_k + (b * 64 + e) / 2] =
                    (uint8_t)(code[0] | (code[1] << 4));
            }
        }
    }
    return 0;
}

int nf4o_code_at(const uint8_t* data, int K, int k, int n) {
    const int KB = K / 64;
    const int blk = k / 64;
    const int e = k % 64;
    const uint8_t byte = data[(long long)n * KB * 32 + (long long)blk * 32 + e / 2];
    return (byte >> (4 * (e % 2))) & 0xF;
}

int nf4o_dequantize_f16(const float* scales, const uint8_t* data, int K, int N,
                        uint16_t* bt) {
    if (!scales || !data || !bt || K <= 0 || N <= 0 || K % 64 != 0) return -1;
    const int KB = K / 64;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int k = 0; k < K; ++k) {
            const float s = scales[(long long)n * KB + k / 64];
            const float w = s * kNF4[nf4o_code_at(data, K, k, n)];
            bt[(long long)n * K + k] = nf4o_f32_to_f16(w);
        }
    }
    return 0;
}

int nf4o_round_operand(const void* go, int dtype, long long count, uint16_t* out) {
    if (!go || !out || count < 0) return -1;
    if (dtype == NF4O_F32) {
        const float* g = (const float*)go;
        for (long long i = 0; i < count; ++i) out[i] = nf4o_f32_to_f16(g[i]);
    } else if (dtype == NF4O_BF16) {
        const uint16_t* g = (const uint16_t*)go;
        for (long long i = 0; i < count; ++i)
            out[i] = nf4o_f32_to_f16(nf4o_bf16_to_f32(g[i]));
    } else {
        return -1;
    }
    return 0;
}

int nf4o_backward_a_rows(const uint16_t* go16, const uint16_t* bt,
                         int M, int N, int K, const int* rows, int nrows,
                         double* ref, double* bound) {
    if (!go16 || !bt || !rows || !ref || M < 0 || N <= 0 || K <= 0 || nrows < 0)
        return -1;
    for (int i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return -2;
    /* Every f16 value as a double, so the inner loop is a plain multiply-add. */
    double* f16v = (double*)malloc(sizeof(double) * 65536);
    if (!f16v) return -3;
    for (int h = 0; h < 65536; ++h) f16v[h] = nf4o_f16_to_f64((uint16_t)h);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        const long long m = rows[i];
        double* r = ref + (long long)i * K;
        double* a = bound ? bound + (long long)i * K : NULL;
        for (int k = 0; k < K; ++k) {
            r[k] = 0.0;
            if (a) a[k] = 0.0;
        }
        for (int n = 0; n < N; ++n) {
            const double g = f16v[go16[m * N + n]];
            const uint16_t* col = bt + (long long)n * K;
            for (int k = 0; k < K; ++k) {
                const double p = g * f16v[col[k]];
                r[k] += p;
                if (a) a[k] += fabs(p);
            }
        }
    }
    free(f16v);
    return 0;
}

int nf4o_backward_a(const void* go, int dtype, const float* scales,
                    const uint8_t* data, int M, int N, int K,
                    double* ref, double* bound) {
    if (!go || !scales || !data || !ref || M < 0 || N <= 0 || K <= 0 || K % 64 != 0)
        return -1;
    uint16_t* go16 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * (size_t)N + 2);
    uint16_t* bt = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)N * (size_t)K);
    int* rows = (int*)malloc(sizeof(int) * (size_t)M + sizeof(int));
    int rc = -3;
    if (go16 && bt && rows) {
        rc = nf4o_round_operand(go, dtype, (long long)M * N, go16);
        if (rc == 0) rc = nf4o_dequantize_f16(scales, data, K, N, bt);
        for (int i = 0; i < M; ++i) rows[i] = i;
        if (rc == 0) rc = nf4o_backward_a_rows(go16, bt, M, N, K, rows, M, ref, bound);
    }
    free(go16);
    free(bt);
    free(rows);
    return rc;
}

/* Sibling-projection fusion: the input gradient of a layer input x that feeds
 * several projections p (q, k and v; or gate and up), each with its own NF4
 * weight B_p [K x N_p] and output gradient go_p [M x N_p], is the sum of their
 * backward-A products ([P1] struct doc comment: 7 backward projections per
 * layer, q/k/v and gate/up sharing the layer's input width K):
 *     grad_x[m][k] = sum_p sum_n f16(go_p)[m][n] * deq(B_p)[k][n].
 * One fp64 accumulator per element, parts in order, n ascending within a part;
 * bound = the same sum over absolute values (may be NULL).  go16[p] is [M][N[p]]
 * f16 bits, bt[p] is deq(B_p) transposed, [N[p]][K] f16 bits. */
int nf4o_backward_a_fused_rows(int parts, const uint16_t* const* go16,
                               const uint16_t* const* bt, const int* N, int M, int K,
                               const int* rows, int nrows, double* ref, double* bound) {
    if (parts <= 0 || !go16 || !bt || !N || !rows || !ref || M < 0 || K <= 0 || nrows < 0)
        return -1;
    for (int p = 0; p < parts; ++p)
        if (!go16[p] || !bt[p] || N[p] <= 0) return -1;
    for (int i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return -2;
    double* f16v = (double*)malloc(sizeof(double) * 65536);
    if (!f16v) return -3;
    for (int h = 0; h < 65536; ++h) f16v[h] = nf4o_f16_to_f64((uint16_t)h);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        const long long m = rows[i];
        double* r = ref + (long long)i * K;
        double* a = bound ? bound + (long long)i * K : NULL;
        for (int k = 0; k < K; ++k) {
            r[k] = 0.0;
            if (a) a[k] = 0.0;
        }
        for (int p = 0; p < parts; ++p) {
            for (int n = 0; n < N[p]; ++n) {
                const double g = f16v[go16[p][m * N[p] + n]];
                const uint16_t* col = bt[p] + (long long)n * K;
                for (int k = 0; k < K; ++k) {
                    const double q = g * f16v[col[k]];
                    r[k] += q;
                    if (a) a[k] += fabs(q);
                }
            }
        }
    }
    free(f16v);
    return 0;
}

/* Forward product C[M x N] = A[M x K] @ deq(B)[K x N] (the module header of
 * [P1] names this forward kernel as the one the backward is the transposed
 * counterpart of; shared dimension K).  The operands are rounded as in the
 * backward ([P1] PHASE 1 and 2), and each C[m][n] is summed over k in order in
 * fp64.  bt = deq(B) transposed, f16 bits [N x K] (nf4o_dequantize_f16), so
 * C[m][n] is the dot product of row m of A16 with row n of bt. */
int nf4o_forward_rows(const uint16_t* a16, const uint16_t* bt, int M, int N, int K,
                      const int* rows, int nrows, double* ref, double* bound) {
    if (!a16 || !bt || !rows || !ref || M < 0 || N <= 0 || K <= 0 || nrows < 0)
        return -1;
    for (int i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return -2;
    double* f16v = (double*)malloc(sizeof(double) * 65536);
    if (!f16v) return -3;
    for (int h = 0; h < 65536; ++h) f16v[h] = nf4o_f16_to_f64((uint16_t)h);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        const uint16_t* arow = a16 + (long long)rows[i] * K;
        for (int n = 0; n < N; ++n) {
            const uint16_t* brow = bt + (long long)n * K;
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                const double p = f16v[arow[k]] * f16v[brow[k]];
                acc += p;
                mag += fabs(p);
            }
            ref[(long long)i * N + n] = acc;
            if (bound) bound[(long long)i * N + n] = mag;
        }
    }
    free(f16v);
    return 0;
}

int nf4o_forward(const void* a, int dtype, const float* scales, const uint8_t* data,
                 int M, int N, int K, double* ref, double* bound) {
    if (!a || !scales || !data || !ref || M < 0 || N <= 0 || K <= 0 || K % 64 != 0)
        return -1;
    uint16_t* a16 = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)M * (size_t)K + 2);
    uint16_t* bt = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)N * (size_t)K);
    int* rows = (int*)malloc(sizeof(int) * (size_t)M + sizeof(int));
    int rc = -3;
    if (a16 && bt && rows) {
        rc = nf4o_round_operand(a, dtype, (long long)M * K, a16);
        if (rc == 0) rc = nf4o_dequantize_f16(scales, data, K, N, bt);
        for (int i = 0; i < M; ++i) rows[i] = i;
        if (rc == 0) rc = nf4o_forward_rows(a16, bt, M, N, K, rows, M, ref, bound);
    }
    free(a16);
    free(bt);
    free(rows);
    return rc;
}

/* Dense weight gradient of C = A @ B ([P3] "trueno-gpu 0.4.17 --
 * src/kernels/backward/mod.rs": GemmBackwardBKernel, "matrix multiplication
 * gradients for A and B", kernel parameters a_ptr and grad_b_ptr):
 *     grad_B[k][n] = sum_m A[m][k] * grad_C[m][n]      (grad_B = A^T @ grad_C)
 * for the trainable (dense, 16-bit) weights next to the frozen NF4 base.  The
 * page does not print the kernel; this is the plain definition.  A [M][K] and
 * grad_C [M][N] are 16-bit floats given as raw bits (dtype16 0: f16, 1: bf16),
 * widened exactly; the sum runs over m ascending in fp64.  ref and bound are
 * [nrows][N] for the output rows k = rows[i]; bound (may be NULL) the same sum
 * over absolute values. */
static double half_to_f64(uint16_t h, int dtype16) {
    return dtype16 == 1 ? (double)nf4o_bf16_to_f32(h) : nf4o_f16_to_f64(h);
}

int nf4o_gemm_backward_b_rows(const uint16_t* a, const uint16_t* gc, int dtype16, int M, int K,
                              int N, const int* rows, int nrows, double* ref, double* bound) {
    if (!a || !gc || !rows || !ref || (dtype16 != 0 && dtype16 != 1) || M < 0 || K <= 0 ||
        N <= 0 || nrows < 0)
        return -1;
    for (int i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= K) return -2;
    double* v = (double*)malloc(sizeof(double) * 65536);
    if (!v) return -3;
    for (int h = 0; h < 65536; ++h) v[h] = half_to_f64((uint16_t)h, dtype16);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; ++i) {
        const int k = rows[i];
        double* r = ref + (long long)i * N;
        double* b = bound ? bound + (long long)i * N : NULL;
        for (int n = 0; n < N; ++n) {
            r[n] = 0.0;
            if (b) b[n] = 0.0;
        }
        for (int m = 0; m < M; ++m) {
            const double x = v[a[(long long)m * K + k]];
            const uint16_t* g = gc + (long long)m * N;
            for (int n = 0; n < N; ++n) {
                const double q = x * v[g[n]];
                r[n] += q;
                if (b) b[n] += fabs(q);
            }
        }
    }
    free(v);
    return 0;
}

void nf4o_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int nf4o_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

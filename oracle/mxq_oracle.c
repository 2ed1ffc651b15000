/*
 * f64 CPU checker for the affine group-wise quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * links it, includes it or calls it, and it shares no source with it.
 *
 * What it computes (mlxcel issue #1536, Baseline section: "affine 4-bit /
 * group 64" weights; PR #1562, What changed: "gather_mm against an f64 dense
 * per-expert reference"; issue #1538, 4-bit vs 8-bit section: dequantise,
 * then accumulate in float at every width):
 *
 *   q[n,k]   = code of weight (n, k), unpacked from the uint32 words
 *   w^[n,k]  = s[n, k/G] * q[n,k] + b[n, k/G]                (in f64)
 *   y[m,n]   = sum_k x[m,k] * w^[n,k]                        (in f64)
 *   bnd[m,n] = sum_k |x[m,k] * w^[n,k]|
 *
 * Packing: 4-bit codes eight per little-endian uint32, the lowest k in the
 * lowest nibble; 8-bit codes ("unsigned char weights", issue #1538, 4-bit vs
 * 8-bit section) four per uint32, the lowest k in the lowest byte.  Both are
 * one little-endian bit stream per row: code k holds bits [k*b, k*b + b) of
 * the row, word j bits [32j, 32j + 32).  The other widths (2, 3 and 6 bits;
 * the bit width is a parameter of the kernels in issue #1536, Diagnosis
 * item 3) are read with the same rule, so a 3- or 6-bit code may start in
 * one word and end in the next.
 *
 * The sorted-MoE variant (PR #1562, Summary: rows sorted by expert, B =
 * tokens * top_k) uses for sorted row r the expert e(r) and activation row
 * src(r).
 *
 * Plain loops, no blocking or reordering beyond the definition: a reader can
 * check each line against the formulas above.  Every function is pinned by
 * the CPU tests (hand-packed words, closed forms, exact brute force, the
 * constant-per-expert case).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double: the bf16 pattern is the upper half of an IEEE binary32. */
static double bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Code of weight (n, k): row n has K*bits/32 words; the code's bits start
 * at bit k*bits of the row and may continue into the next word. */
static unsigned code_at(const uint32_t* w, long long words_per_row, int n, int k, int bits) {
    const uint32_t* row = w + (long long)n * words_per_row;
    long long first = (long long)k * bits;       /* bit index of the code's lowest bit */
    long long j = first / 32;
    int off = (int)(first % 32);
    uint64_t v = row[j] >> off;
    if (off + bits > 32) v |= (uint64_t)row[j + 1] << (32 - off);
    return (unsigned)(v & ((1u << bits) - 1u));
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Unpack every code of an [N, K] matrix into q (uint8 [N, K]). */
void oracle_unpack(const uint32_t* w, int N, int K, int bits, uint8_t* q) {
    long long wpr = (long long)K * bits / 32;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            q[(long long)n * K + k] = (uint8_t)code_at(w, wpr, n, k, bits);
}

/* Dense f64 dequantised weights w^[N, K]. */
void oracle_dequant(const uint32_t* w, const uint16_t* scales, const uint16_t* biases,
                    int N, int K, int bits, int group, double* what) {
    long long wpr = (long long)K * bits / 32;
    int ng = K / group;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            double s = bf16_to_f64(scales[(long long)n * ng + k / group]);
            double b = bf16_to_f64(biases[(long long)n * ng + k / group]);
            what[(long long)n * K + k] = s * (double)code_at(w, wpr, n, k, bits) + b;
        }
}

/* One output row n for the activation rows listed: dequantise row n of one
 * expert's matrix into a scratch row, then take the f64 dot products. */
static void row_dot(const uint16_t* x, const uint32_t* w, const uint16_t* scales,
                    const uint16_t* biases, int K, int bits, int group, int n,
                    const int* xrows, int nrows, double* wrow,
                    double* y_out, double* bnd_out, long long ystride) {
    long long wpr = (long long)K * bits / 32;
    int ng = K / group;
    for (int k = 0; k < K; ++k) {
        double s = bf16_to_f64(scales[(long long)n * ng + k / group]);
        double b = bf16_to_f64(biases[(long long)n * ng + k / group]);
        wrow[k] = s * (double)code_at(w, wpr, n, k, bits) + b;
    }
    for (int i = 0; i < nrows; ++i) {
        const uint16_t* xr = x + (long long)xrows[i] * K;
        double acc = 0.0, bnd = 0.0;
        for (int k = 0; k < K; ++k) {
            double t = bf16_to_f64(xr[k]) * wrow[k];
            acc += t;
            bnd += fabs(t);
        }
        y_out[(long long)i * ystride] = acc;
        if (bnd_out) bnd_out[(long long)i * ystride] = bnd;
    }
}

/* y[M, N] = x[M, K] . w^[N, K]^T in f64; bound likewise (may be NULL). */
int oracle_qmm(const uint16_t* x, const uint32_t* w, const uint16_t* scales,
               const uint16_t* biases, int M, int K, int N, int bits, int group,
               double* y, double* bound) {
    int* rows = (int*)malloc(sizeof(int) * (M > 0 ? M : 1));
    if (!rows) return 1;
    for (int m = 0; m < M; ++m) rows[m] = m;
    int fail = 0;
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * (K > 0 ? K : 1));
        if (!wrow) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int n = 0; n < N; ++n)
                row_dot(x, w, scales, biases, K, bits, group, n, rows, M, wrow,
                        y + n, bound ? bound + n : NULL, N);
            free(wrow);
        }
    }
    free(rows);
    return fail;
}

/* qmv is qmm with one activation row. */
int oracle_qmv(const uint16_t* x, const uint32_t* w, const uint16_t* scales,
               const uint16_t* biases, int K, int N, int bits, int group,
               double* y, double* bound) {
    return oracle_qmm(x, w, scales, biases, 1, K, N, bits, group, y, bound);
}

/* The other operand layout (PR #1562, What changed: the grouped GEMM is
 * checked for both operand layouts): w is stored [K, N], row k holding the
 * codes of all N outputs as the same little-endian bit stream (code n of row
 * k in bits [n*b, n*b + b)), and the groups run along n:
 *
 *   w^[k,n] = s[k, n/G] * q[k,n] + b[k, n/G]      scales, biases [K, N/G]
 *   y[m,n]  = sum_k x[m,k] * w^[k,n]              (in f64, k in order)
 *
 * One output column at a time: dequantise column n into a scratch vector,
 * then the f64 dot products. */
int oracle_qmm_kn(const uint16_t* x, const uint32_t* w, const uint16_t* scales,
                  const uint16_t* biases, int M, int K, int N, int bits, int group,
                  double* y, double* bound) {
    long long wpr = (long long)N * bits / 32;  /* words per row k */
    int ng = N / group;
    int fail = 0;
#pragma omp parallel
    {
        double* wcol = (double*)malloc(sizeof(double) * (K > 0 ? K : 1));
        if (!wcol) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int n = 0; n < N; ++n) {
                for (int k = 0; k < K; ++k) {
                    double s = bf16_to_f64(scales[(long long)k * ng + n / group]);
                    double b = bf16_to_f64(biases[(long long)k * ng + n / group]);
                    wcol[k] = s * (double)code_at(w, wpr, k, n, bits) + b;
                }
                for (int m = 0; m < M; ++m) {
                    const uint16_t* xr = x + (long long)m * K;
                    double acc = 0.0, bnd = 0.0;
                    for (int k = 0; k < K; ++k) {
                        double t = bf16_to_f64(xr[k]) * wcol[k];
                        acc += t;
                        bnd += fabs(t);
                    }
                    y[(long long)m * N + n] = acc;
                    if (bound) bound[(long long)m * N + n] = bnd;
                }
            }
            free(wcol);
        }
    }
    return fail;
}

/* Sorted-MoE variant: y[B, N]; row r uses expert expert_ids[r] and activation
 * row row_src[r] (row_src NULL means row r).  w is [E, N, K*bits/32],
 * scales/biases [E, N, K/G].  Rows whose expert id is out of [0, E) get 0. */
int oracle_gather_qmm(const uint16_t* x, const uint32_t* w, const uint16_t* scales,
                      const uint16_t* biases, const int32_t* expert_ids,
                      const int32_t* row_src, int T, int B, int E, int K, int N,
                      int bits, int group, double* y, double* bound) {
    (void)T;
    long long wmat = (long long)N * K * bits / 32;
    long long smat = (long long)N * (K / group);
    int fail = 0;
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * (K > 0 ? K : 1));
        if (!wrow) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < B; ++r) {
                int e = expert_ids[r];
                int src = row_src ? row_src[r] : r;
                for (int n = 0; n < N; ++n) {
                    if (e < 0 || e >= E) {
                        y[(long long)r * N + n] = 0.0;
                        if (bound) bound[(long long)r * N + n] = 0.0;
                        continue;
                    }
                    row_dot(x, w + e * wmat, scales + e * smat, biases + e * smat, K, bits,
                            group, n, &src, 1, wrow, y + (long long)r * N + n,
                            bound ? bound + (long long)r * N + n : NULL, 1);
                }
            }
            free(wrow);
        }
    }
    return fail;
}

/* Selected outputs of the sorted-MoE variant (or of qmm with E = 1 and
 * expert_ids NULL): for each i, output (rows[i], cols[i]).  Used to check
 * full-size launches element by element on a sample. */
int oracle_points(const uint16_t* x, const uint32_t* w, const uint16_t* scales,
                  const uint16_t* biases, const int32_t* expert_ids,
                  const int32_t* row_src, int E, int K, int N, int bits, int group,
                  const int64_t* rows, const int64_t* cols, long long count,
                  double* y, double* bound) {
    long long wmat = (long long)N * K * bits / 32;
    long long smat = (long long)N * (K / group);
    int fail = 0;
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * (K > 0 ? K : 1));
        if (!wrow) {
#pragma omp atomic write
            fail = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (long long i = 0; i < count; ++i) {
                int r = (int)rows[i];
                int n = (int)cols[i];
                int e = expert_ids ? expert_ids[r] : 0;
                int src = row_src ? row_src[r] : r;
                if (e < 0 || e >= E) {
                    y[i] = 0.0;
                    if (bound) bound[i] = 0.0;
                    continue;
                }
                row_dot(x, w + e * wmat, scales + e * smat, biases + e * smat, K, bits,
                        group, n, &src, 1, wrow, y + i, bound ? bound + i : NULL, 1);
            }
            free(wrow);
        }
    }
    return fail;
}

/* ------------------------------------------------------------------ encoder
 *
 * The affine min/max encoder that produces the stored format (mlxcel issue
 * #1536, Baseline section: "affine 4-bit / group 64"; the affine map is read
 * in its plainest form: per (row, group) the bias is the group minimum and
 * the scale spreads the group's range over the 2^bits - 1 code steps).  Every
 * decision is taken in binary32, the precision the GPU encoder uses, so both
 * sides reach the same codes bit for bit:
 *
 *   mn, mx = min, max of the group's values (-0 read as +0)
 *   s      = bf16(RN(RN(mx - mn) / (2^bits - 1)))     bf16 rounding: RNE
 *   b      = bf16(mn)
 *   q      = 0 when s == 0, else clamp(rint(RN(RN(w - b) / s)), 0, 2^bits - 1)
 *
 * with s and b used as their stored bf16 values, rint rounding half to even.
 */
static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

void oracle_quantize(const float* W, int N, int K, int bits, int group, uint32_t* codes,
                     uint16_t* scales, uint16_t* biases) {
    const int levels = (1 << bits) - 1;
    const int groups = K / group;
    const long long words_per_row = (long long)K * bits / 32;
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (long long i = 0; i < words_per_row; ++i) codes[(long long)n * words_per_row + i] = 0;
        for (int g = 0; g < groups; ++g) {
            const float* v = W + (long long)n * K + (long long)g * group;
            float mn = v[0] + 0.0f, mx = v[0] + 0.0f;
            for (int j = 1; j < group; ++j) {
                const float t = v[j] + 0.0f;
                if (t < mn) mn = t;
                if (t > mx) mx = t;
            }
            const volatile float range = mx - mn;
            const volatile float step = range / (float)levels;
            const uint16_t sb = f32_to_bf16_rne(step);
            const uint16_t bb = f32_to_bf16_rne(mn);
            scales[(long long)n * groups + g] = sb;
            biases[(long long)n * groups + g] = bb;
            const float s = bf16_to_f32(sb), b = bf16_to_f32(bb);
            for (int j = 0; j < group; ++j) {
                unsigned q = 0;
                if (s != 0.0f) {
                    const volatile float d = v[j] - b;
                    const volatile float t = d / s;
                    float r = rintf(t);
                    if (r < 0.0f) r = 0.0f;
                    if (r > (float)levels) r = (float)levels;
                    q = (unsigned)r;
                }
                /* code k occupies bits [k*bits, k*bits + bits) of the row */
                uint32_t* row = codes + (long long)n * words_per_row;
                const long long first = (long long)(g * group + j) * bits;
                const int off = (int)(first % 32);
                row[first / 32] |= (uint32_t)q << off;
                if (off + bits > 32) row[first / 32 + 1] |= (uint32_t)q >> (32 - off);
            }
        }
    }
}

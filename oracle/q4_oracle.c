/*
 * q4_oracle.c -- TEST INFRASTRUCTURE ONLY: the plain, slow, obviously-correct fp64
 * CPU reference for the 4-bit group-symmetric weight-quantized linear.
 *
 * Nothing in the product library calls, links or includes this file.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it (through
 * oracle/__init__.py).  It shares no code, header, table or helper with the CUDA
 * library: it has its own binary16 decoder, its own nibble unpacking and its own
 * loops, written straight from the definition.
 *
 * What it computes (every function cites the passage it follows):
 *
 *   out[m,n] = bias[n] + sum_k x[m,k] * (nib(W)[n,k] - 8) * scale[k / group_size, n]
 *
 *   - "[ExecuTorch][WebGPU] Add linear_qcs4w op (et_vk.linear_qcs4w)", Solution and
 *     Constraints (2)-(3): the per-term formula acc += in[m,k] * (unpack_int4(w) - 8) *
 *     scale, the grouped scale index scales[(k / group_size) * N + n] (we read N, not a
 *     padded N, as the row stride), the +8-shifted signed int4, and the q4gsw packer's
 *     "(odd << 4) | even" byte, i.e. the LOW nibble holds the even k.
 *   - "[ExecuTorch][WebGPU] Add fp32 matmul ops ... (linear_q4gsw_backward)", #20943:
 *     dequant(W[n,k]) = (code - 8) * scale with [num_groups, N] scales.
 *   - "[ExecuTorch][WebGPU] Add optimized linear_fp32 op", Solution: the bias epilogue
 *     v = v + bias[n], applied once after the full sum, only when a bias is given.
 *   - The golden truth on those pages is an fp64 dequant-matmul; so is this file.
 *
 * Arithmetic: everything in IEEE double, k ascending.  (q - 8) has at most 4 significant
 * bits and a scale at most 24, so w = (q - 8) * s is exact in double; x has 24 bits, so
 * x * w (<= 52 bits) is exact too.  The only roundings are those of the running sums.
 *
 * Readings of points the pages leave open (the pages are silent on each):
 *   - Packed row stride is ceil(K/2) bytes; for odd K the last byte's high nibble is
 *     padding and is never read ("K_packed == ceil(K/2)" guard of the qcs4w page).
 *   - num_groups = ceil(K / group_size); a last partial group is indexed floor(k / gs).
 *   - A zero scale simply gives w = 0 (the zero-scale special case is requant-only).
 *   - NaN / Inf propagate by IEEE rules.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define Q4O_OK 0
#define Q4O_BAD_ARG 1

/* Threads an OpenMP loop of this library uses (1 without OpenMP). */
int q4o_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* IEEE 754 binary16 -> double, from the bit fields (1 sign, 5 exponent bias 15,
 * 10 fraction bits).  Written here so the oracle needs no half-precision library. */
double q4o_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 0x1F;
    int fraction = h & 0x3FF;
    double v;
    if (exponent == 0) {
        v = ldexp((double)fraction, -24); /* subnormal: 0.fraction * 2^-14 */
    } else if (exponent == 31) {
        v = (fraction == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + fraction), exponent - 25); /* 1.fraction * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* The stored nibble for (n, k).  Default order (the q4gsw packer): low nibble = even k.
 * even_high != 0 selects the qcs4w AOT packer's swapped order "(even << 4) | odd"
 * ("Add linear_qcs4w op", Constraints (2)). */
static int nibble_at(const uint8_t* qweight, int64_t row_bytes, int64_t n, int64_t k,
                     int even_high) {
    uint8_t byte = qweight[n * row_bytes + k / 2];
    int k_is_even = (k % 2) == 0;
    int take_low = even_high ? !k_is_even : k_is_even;
    return take_low ? (byte & 0x0F) : (byte >> 4);
}

static double scale_at(const void* scales, int scale_is_f16, int64_t N, int64_t g,
                       int64_t n) {
    if (scale_is_f16) return q4o_f16_to_f64(((const uint16_t*)scales)[g * N + n]);
    return (double)((const float*)scales)[g * N + n];
}

/* One output element by the definition, k ascending.  Writes the sum without bias and
 * the magnitude sum_k |x * w| (the tolerance denominator). */
static void element(const float* x, const uint8_t* qweight, const void* scales,
                    int scale_is_f16, int64_t N, int64_t K, int64_t group_size,
                    int even_high, int64_t m, int64_t n, double* acc_out,
                    double* mag_out) {
    int64_t row_bytes = (K + 1) / 2;
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        int q = nibble_at(qweight, row_bytes, n, k, even_high);
        double s = scale_at(scales, scale_is_f16, N, k / group_size, n);
        double w = (double)(q - 8) * s;
        double p = (double)x[m * K + k] * w;
        acc += p;
        mag += fabs(p);
    }
    *acc_out = acc;
    *mag_out = mag;
}

static int check_args(const float* x, const uint8_t* qweight, const void* scales,
                      int64_t M, int64_t N, int64_t K, int64_t group_size) {
    if (M < 0 || N < 0 || K < 1 || group_size < 1) return Q4O_BAD_ARG;
    if ((M > 0 && !x) || (N > 0 && (!qweight || !scales))) return Q4O_BAD_ARG;
    return Q4O_OK;
}

/* The full [M, N] output.  out = sum + bias (bias may be NULL); mag = sum_k |x * w|.
 * OpenMP (when compiled in) splits the independent (m, n) elements; each element's
 * k-loop stays sequential, so the result does not depend on the thread count. */
int q4o_linear(const float* x, const uint8_t* qweight, const void* scales,
               int scale_is_f16, const float* bias, int64_t M, int64_t N, int64_t K,
               int64_t group_size, int even_high, double* out, double* mag) {
    if (check_args(x, qweight, scales, M, N, K, group_size)) return Q4O_BAD_ARG;
    int64_t total = M * N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < total; ++i) {
        int64_t m = i / N, n = i % N;
        double acc, mg;
        element(x, qweight, scales, scale_is_f16, N, K, group_size, even_high, m, n,
                &acc, &mg);
        out[i] = acc + (bias ? (double)bias[n] : 0.0);
        mag[i] = mg;
    }
    return Q4O_OK;
}

/* Selected elements only, (ms[i], ns[i]) for i < count: for outputs too large to
 * compute in full.  Same per-element definition as q4o_linear. */
int q4o_linear_at(const float* x, const uint8_t* qweight, const void* scales,
                  int scale_is_f16, const float* bias, int64_t M, int64_t N, int64_t K,
                  int64_t group_size, int even_high, const int64_t* ms,
                  const int64_t* ns, int64_t count, double* out, double* mag) {
    if (check_args(x, qweight, scales, M, N, K, group_size)) return Q4O_BAD_ARG;
    for (int64_t i = 0; i < count; ++i)
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return Q4O_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        double acc, mg;
        element(x, qweight, scales, scale_is_f16, N, K, group_size, even_high, ms[i],
                ns[i], &acc, &mg);
        out[i] = acc + (bias ? (double)bias[ns[i]] : 0.0);
        mag[i] = mg;
    }
    return Q4O_OK;
}

/* Per-output-channel (qcs4w) linear, written separately from q4o_linear so that the
 * identity "qcs4w == q4gsw with group_size = K" can be checked between two independent
 * routines.  "Add linear_qcs4w op", Solution: acc += in[m,k] * (unpack_int4(w) - 8) *
 * scales[n] with a 1-D [N] scale and no group.  Here the channel scale is factored out
 * of the k-sum (one multiply at the end), the integer codes are summed against x, and
 * the nibble is taken with a shift by 4 * (k & 1) instead of a branch. */
int q4o_linear_qcs4w(const float* x, const uint8_t* qweight, const void* scales_n,
                     int scale_is_f16, const float* bias, int64_t M, int64_t N,
                     int64_t K, double* out, double* mag) {
    if (check_args(x, qweight, scales_n, M, N, K, 1)) return Q4O_BAD_ARG;
    int64_t row_bytes = (K + 1) / 2;
    for (int64_t n = 0; n < N; ++n) {
        double s = scale_is_f16 ? q4o_f16_to_f64(((const uint16_t*)scales_n)[n])
                                : (double)((const float*)scales_n)[n];
        const uint8_t* row = qweight + n * row_bytes;
        for (int64_t m = 0; m < M; ++m) {
            const float* xr = x + m * K;
            double dot = 0.0, absdot = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int code = (row[k >> 1] >> (4 * (k & 1))) & 0xF;
                double t = (double)xr[k] * (double)(code - 8);
                dot += t;
                absdot += fabs(t);
            }
            out[m * N + n] = dot * s + (bias ? (double)bias[n] : 0.0);
            mag[m * N + n] = absdot * fabs(s);
        }
    }
    return Q4O_OK;
}

/* ------------------------------------------------------------ training-path ops
 *
 * Input gradient of the linear (the frozen 4-bit base during adapter training):
 *
 *   d_x[m,k] = sum_n d_out[m,n] * (nib(W)[n,k] - 8) * scale[k / group_size, n]
 *
 * "[ExecuTorch][WebGPU] Add fp32 matmul ops ... (linear_q4gsw_backward)", #20943:
 * d_x[M,K] = d_out[M,N] @ dequant(W)[N,K], contracting over N, dequant(W[n,k]) =
 * (code - 8) * scale with [num_groups, N] scales, on the same packed weight and scale
 * layout as the forward.  n ascending, IEEE double; mag = sum_n |d_out * w| (the
 * tolerance denominator).  OpenMP over the independent (m, k) elements. */
int q4o_backward_dx(const float* d_out, const uint8_t* qweight, const void* scales,
                    int scale_is_f16, int64_t M, int64_t N, int64_t K, int64_t group_size,
                    int even_high, double* d_x, double* mag) {
    if (M < 0 || N < 0 || K < 1 || group_size < 1) return Q4O_BAD_ARG;
    if ((M > 0 && N > 0 && !d_out) || (N > 0 && (!qweight || !scales))) return Q4O_BAD_ARG;
    int64_t row_bytes = (K + 1) / 2;
    int64_t total = M * K;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < total; ++i) {
        int64_t m = i / K, k = i % K;
        double acc = 0.0, mg = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            int q = nibble_at(qweight, row_bytes, n, k, even_high);
            double w = (double)(q - 8) * scale_at(scales, scale_is_f16, N, k / group_size, n);
            double p = (double)d_out[m * N + n] * w;
            acc += p;
            mg += fabs(p);
        }
        d_x[i] = acc;
        mag[i] = mg;
    }
    return Q4O_OK;
}

/* Straight-through re-quantisation of fp32 latent weights [N, K] to the 4-bit codes with
 * frozen scales, packed in the forward's layout [N, ceil(K/2)]:
 *
 *   code[n,k] = clamp(round(latent[n,k] / scale[k / group_size, n]), -8, 7) + 8,
 *   a zero scale gives code 8.
 *
 * "[ExecuTorch][WebGPU] Add fp32 matmul ops ... (q4gsw_requant)", #20945 (the rule and
 * the zero-scale case) and #20946 (its golden: round / clamp, zero scale -> code 8).
 * Readings where the page is silent:
 *   - the quotient is an fp32 quotient (latents and scales are fp32 on the page, and the
 *     integer decision is taken at that precision): it is computed in double and rounded
 *     once to float, which for a division equals the IEEE fp32 quotient (53 >= 2*24 + 2);
 *   - round() rounds half to even (the page's tests avoid ties);
 *   - a NaN quotient gives code 8, like a zero scale;
 *   - for odd K the padding nibble of the last byte is 8, the bias-zero code the page
 *     writes for positions outside the matrix. */
int q4o_requant(const float* latent, const void* scales, int scale_is_f16, int64_t N,
                int64_t K, int64_t group_size, int even_high, uint8_t* qweight) {
    if (N < 0 || K < 1 || group_size < 1) return Q4O_BAD_ARG;
    if (N > 0 && (!latent || !scales || !qweight)) return Q4O_BAD_ARG;
    int64_t row_bytes = (K + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < row_bytes; ++b) {
            int codes[2] = {8, 8}; /* [even k, odd k] */
            for (int j = 0; j < 2; ++j) {
                int64_t k = 2 * b + j;
                if (k >= K) break;
                double s = scale_at(scales, scale_is_f16, N, k / group_size, n);
                if (s == 0.0) continue;
                float quotient = (float)((double)latent[n * K + k] / s);
                if (isnan(quotient)) continue;
                double r = rint((double)quotient);
                if (r < -8.0) r = -8.0;
                if (r > 7.0) r = 7.0;
                codes[j] = (int)r + 8;
            }
            int low = even_high ? codes[1] : codes[0];
            int high = even_high ? codes[0] : codes[1];
            qweight[n * row_bytes + b] = (uint8_t)(low | (high << 4));
        }
    }
    return Q4O_OK;
}

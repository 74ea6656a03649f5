/*
 * kt_mlp_oracle.c -- plain float64 CPU oracle for the fused transformer MLP.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file.  Its users are the tests, the smoke check and the timed CPU
 * baseline of the bench harness.  It shares no code, header or table with the
 * CUDA library: it has its own fp16/bf16 codecs, its own loops and uses the host
 * C library's erfc / exp in double precision.
 *
 * What it computes (all sums in natural index order, float64):
 *
 *   P[m,j]  = sum_k X[m,k] * W_up[k,j]  (+ b_up[j])                      j < F_up
 *   gelu    : H~[m,j] = gelu(P[m,j])                                     F_up = F
 *   none    : H~[m,j] = P[m,j]                                           F_up = F
 *   gelu_sigmoid / silu : H~ = P * sigmoid(1.702 P) / P * sigmoid(P)     F_up = F
 *   geglu   : H~[m,j] = P[m,j] * gelu_erf(P[m,F+j])                      F_up = 2F
 *   H[m,j]  = round_to_nearest_even_dt(H~[m,j])        (the single rounding of H)
 *   Yx[m,n] = sum_j H[m,j] * W_down[j,n]  (+ b_down[n])  (+ R[m,n])
 *   Y[m,n]  = round_to_nearest_even_dt(Yx[m,n])
 *
 * Options (oracle_mlp_rows_ex): a LayerNorm of each row of X before the up
 * projection, X' = round_dt((x - mean) / sqrt(var + eps) * gamma + beta) with the
 * mean and the biased variance over D in float64 (the GEMM reads 16-bit operands);
 * a residual R added before the final rounding; weights given in PyTorch
 * nn.Linear order ([out][in]) instead of [in][out].
 *
 * Sources on the pages:
 *   - "SDXL as a requirements inventory", section 1.3 (FeedForward): one
 *     projection to 2*4*dim, chunk in two along the last axis, the SECOND half is
 *     the gate, h * gelu(gate), then the projection back to dim.
 *   - same page, section 9.3: SDXL's gelu is the erf form; a sigmoid stand-in and
 *     gating on the wrong half are named traps.
 *   - "MLP layout sweep and remaining representation limits", opening paragraph:
 *     the F16 SigLIP MLP [1,729,1152] -> [1,729,4304] -> [1,729,1152], no biases,
 *     up GEMM, GELU, down GEMM; its "ISA review" section computes GELU with tanh.
 *   - "The software stack", section 2.3: the accumulator is a resident format and
 *     never a memory word; outputs are written in the 16-bit I/O format.
 *   - "SDXL as a requirements inventory", section 1.3 (BasicTransformerBlock): the
 *     feed-forward is applied as x = ff(norm(x)) + x, a LayerNorm before it and the
 *     residual after it; section 9.3: KohakuTPU's geglu lowers the sigmoid GELU
 *     x * sigmoid(1.702 x); section 1.3 (timestep embedding): Linear -> SiLU -> Linear;
 *     section 1.4: Linear weights are stored [out][in].
 *
 * Readings where the pages are silent (stated once more in the design notes):
 *   - tanh GELU uses the published constants sqrt(2/pi) and 0.044715
 *     (Hendrycks & Gimpel 2016).  It is evaluated through the exact identity
 *     (1 + tanh(u)) / 2 = 1 / (1 + exp(-2u)), and the erf form through
 *     (1 + erf(z/sqrt2)) / 2 = erfc(-z/sqrt2) / 2 (Abramowitz & Stegun 7.1.2).
 *     Both identities are exact; they only avoid the cancellation of 1 + (-1+e)
 *     for negative z, where the literal forms lose every digit in double.
 *   - rounding to fp16 / bf16 is IEEE round-to-nearest-even with subnormals kept
 *     and overflow to +-inf.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define KTO_F16 0
#define KTO_BF16 1

#define KTO_GELU_ERF 0
#define KTO_GELU_TANH 1
#define KTO_GEGLU 2
#define KTO_NONE 3 /* no activation: H~ = P (two chained linear layers) */
#define KTO_GELU_SIGMOID 4 /* x * sigmoid(1.702 x) */
#define KTO_SILU 5         /* x * sigmoid(x) */

/* ------------------------------------------------------------------------ */
/* fp16 / bf16 codecs, written from the bit formats.                         */
/* fp16: 1 sign, 5 exponent (bias 15), 10 fraction bits.                     */
/* bf16: 1 sign, 8 exponent (bias 127), 7 fraction bits.                     */
/* ------------------------------------------------------------------------ */

double oracle_f16_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return s ? -v : v;
}

double oracle_bf16_to_f64(uint16_t b) {
    int s = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* subnormal: f * 2^-133 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/128) * 2^(e-127) */
    }
    return s ? -v : v;
}

/*
 * Generic RNE encoder for a binary format with `fbits` fraction bits, minimum
 * normal exponent `emin`, exponent bias `bias` and largest finite value `maxf`.
 * The quantum at magnitude a is 2^(max(floor(log2 a), emin) - fbits); a / q is
 * exact in double (power-of-two scaling), nearbyint() in the default rounding
 * mode rounds it to the nearest integer with ties to even, and n * q is the
 * rounded value.  Overflow past maxf gives infinity.
 */
static uint16_t encode_rne(double x, int fbits, int emin, int bias, double maxf,
                           uint16_t inf_bits, uint16_t nan_bits) {
    if (isnan(x)) return nan_bits;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | inf_bits);
    int e2;
    frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1)  => floor(log2 a) = e2 - 1 */
    int E = e2 - 1;
    if (E < emin) E = emin;
    double q = ldexp(1.0, E - fbits);
    double n = nearbyint(a / q);
    double r = n * q;
    if (r > maxf) return (uint16_t)(sign | inf_bits);
    if (r < ldexp(1.0, emin)) {
        return (uint16_t)(sign | (uint16_t)n); /* subnormal: fraction field = n */
    }
    int er;
    frexp(r, &er);
    int RE = er - 1; /* r in [2^RE, 2^(RE+1)) */
    uint16_t frac = (uint16_t)(ldexp(r, fbits - RE) - ldexp(1.0, fbits));
    uint16_t expo = (uint16_t)(RE + bias);
    return (uint16_t)(sign | (uint16_t)(expo << fbits) | frac);
}

uint16_t oracle_f64_to_f16(double x) {
    return encode_rne(x, 10, -14, 15, 65504.0, 0x7C00, 0x7E00);
}

uint16_t oracle_f64_to_bf16(double x) {
    /* largest finite bf16: (2 - 2^-7) * 2^127 */
    return encode_rne(x, 7, -126, 127, ldexp(255.0, 120), 0x7F80, 0x7FC0);
}

static double decode(uint16_t v, int dtype) {
    return dtype == KTO_BF16 ? oracle_bf16_to_f64(v) : oracle_f16_to_f64(v);
}

static uint16_t encode(double x, int dtype) {
    return dtype == KTO_BF16 ? oracle_f64_to_bf16(x) : oracle_f64_to_f16(x);
}

void oracle_decode(const uint16_t* in, double* out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = decode(in[i], dtype);
}

void oracle_encode(const double* in, uint16_t* out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = encode(in[i], dtype);
}

/* ------------------------------------------------------------------------ */
/* GELU, both forms, float64.                                                */
/* ------------------------------------------------------------------------ */

/* gelu_erf(z) = z * Phi(z) = 0.5 * z * (1 + erf(z / sqrt 2)) = 0.5 * z * erfc(-z / sqrt 2) */
double oracle_gelu_erf(double z) {
    return 0.5 * z * erfc(-z * 0.70710678118654752440);
}

/* gelu_tanh(z) = 0.5 * z * (1 + tanh(u)),  u = sqrt(2/pi) * (z + 0.044715 z^3)
 *             = z / (1 + exp(-2u))                                             */
double oracle_gelu_tanh(double z) {
    double u = 0.79788456080286535588 * (z + 0.044715 * z * z * z);
    return z / (1.0 + exp(-2.0 * u));
}

/* sigmoid-weighted forms: z * sigmoid(a z) = z / (1 + exp(-a z)) */
double oracle_gelu_sigmoid(double z) { return z / (1.0 + exp(-1.702 * z)); }
double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

void oracle_gelu_vec(const double* z, double* out, int64_t n, int form) {
    for (int64_t i = 0; i < n; ++i) {
        if (form == KTO_GELU_TANH) out[i] = oracle_gelu_tanh(z[i]);
        else if (form == KTO_GELU_SIGMOID) out[i] = oracle_gelu_sigmoid(z[i]);
        else if (form == KTO_SILU) out[i] = oracle_silu(z[i]);
        else out[i] = oracle_gelu_erf(z[i]);
    }
}

/* LayerNorm of one row, float64: mean, biased variance (divide by D), then
 * (x - mean) / sqrt(var + eps) * gamma + beta. */
void oracle_layernorm_row(const double* x, const double* gamma, const double* beta, double eps,
                          double* out, int64_t D) {
    double mean = 0.0;
    for (int64_t k = 0; k < D; ++k) mean += x[k];
    mean /= (double)D;
    double var = 0.0;
    for (int64_t k = 0; k < D; ++k) var += (x[k] - mean) * (x[k] - mean);
    var /= (double)D;
    double inv = 1.0 / sqrt(var + eps);
    for (int64_t k = 0; k < D; ++k) out[k] = (x[k] - mean) * inv * gamma[k] + beta[k];
}

/* ------------------------------------------------------------------------ */
/* Linear layer in float64: C[m,n] = sum_k A[m,k] * B[k,n] (+ bias[n]).      */
/* A is [M][K], B is [K][N], C is [M][N], all row-major.  Each C[m,n] is a   */
/* sum over k = 0, 1, ..., K-1 in that order; the bias is added last.        */
/* ------------------------------------------------------------------------ */

static void linear_row(const double* a_row, const double* B, const double* bias,
                       double* c_row, int64_t K, int64_t N) {
    for (int64_t n = 0; n < N; ++n) c_row[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double a = a_row[k];
        const double* b = B + k * N;
        for (int64_t n = 0; n < N; ++n) c_row[n] += a * b[n];
    }
    if (bias)
        for (int64_t n = 0; n < N; ++n) c_row[n] += bias[n];
}

void oracle_linear(const double* A, const double* B, const double* bias, double* C,
                   int64_t M, int64_t K, int64_t N) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) linear_row(A + m * K, B, bias, C + m * N, K, N);
}

/* ------------------------------------------------------------------------ */
/* The activation step on one row of P (length F_up), producing H~ (length F). */
/* ------------------------------------------------------------------------ */

static void activation_row(const double* p, double* h, int64_t F, int act) {
    if (act == KTO_GEGLU) {
        /* value = first half, gate = second half */
        for (int64_t j = 0; j < F; ++j) h[j] = p[j] * oracle_gelu_erf(p[F + j]);
    } else if (act == KTO_GELU_TANH) {
        for (int64_t j = 0; j < F; ++j) h[j] = oracle_gelu_tanh(p[j]);
    } else if (act == KTO_NONE) {
        for (int64_t j = 0; j < F; ++j) h[j] = p[j];
    } else if (act == KTO_GELU_SIGMOID) {
        for (int64_t j = 0; j < F; ++j) h[j] = oracle_gelu_sigmoid(p[j]);
    } else if (act == KTO_SILU) {
        for (int64_t j = 0; j < F; ++j) h[j] = oracle_silu(p[j]);
    } else {
        for (int64_t j = 0; j < F; ++j) h[j] = oracle_gelu_erf(p[j]);
    }
}

void oracle_activation(const double* P, double* Hx, int64_t M, int64_t F, int act) {
    int64_t Fup = (act == KTO_GEGLU) ? 2 * F : F;
    for (int64_t m = 0; m < M; ++m) activation_row(P + m * Fup, Hx + m * F, F, act);
}

/* ------------------------------------------------------------------------ */
/* The whole MLP, on a chosen subset of rows (rows[] = NULL means all rows).  */
/* Inputs are the 16-bit bit patterns of the I/O dtype.  Outputs, for row i   */
/* of the subset: H_out[i][F] (rounded H bits, may be NULL), Yx_out[i][D]     */
/* (float64, before the final rounding, may be NULL), Y_out[i][D] (rounded,   */
/* may be NULL).  Returns 0, or -1 on a bad argument / allocation failure.    */
/* ------------------------------------------------------------------------ */

int oracle_mlp_rows_ex(int64_t M, int64_t D, int64_t F, int act, int dtype, int bias,
                       const uint16_t* X, const uint16_t* W_up, const uint16_t* W_down,
                       const uint16_t* b_up, const uint16_t* b_down,
                       const uint16_t* R, const uint16_t* ln_gamma, const uint16_t* ln_beta,
                       double ln_eps, int w_layout,
                       const int64_t* rows, int64_t nrows,
                       uint16_t* H_out, double* Yx_out, uint16_t* Y_out) {
    if (M < 1 || D < 1 || F < 1 || nrows < 0) return -1;
    if (act < 0 || act > 5 || (dtype != KTO_F16 && dtype != KTO_BF16)) return -1;
    if ((ln_gamma == NULL) != (ln_beta == NULL) || (w_layout != 0 && w_layout != 1)) return -1;
    if (rows == NULL) nrows = M;
    for (int64_t i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return -1;
    int64_t Fup = (act == KTO_GEGLU) ? 2 * F : F;

    double* wu = (double*)malloc(sizeof(double) * (size_t)(D * Fup));
    double* wd = (double*)malloc(sizeof(double) * (size_t)(F * D));
    double* bu = (double*)malloc(sizeof(double) * (size_t)Fup);
    double* bd = (double*)malloc(sizeof(double) * (size_t)D);
    if (!wu || !wd || !bu || !bd) {
        free(wu); free(wd); free(bu); free(bd);
        return -1;
    }
    if (w_layout == 0) {
        oracle_decode(W_up, wu, D * Fup, dtype);
        oracle_decode(W_down, wd, F * D, dtype);
    } else {
        /* [out][in] storage: W_up is [F_up][D], W_down is [D][F]; transpose exactly */
        for (int64_t j = 0; j < Fup; ++j)
            for (int64_t k = 0; k < D; ++k) wu[k * Fup + j] = decode(W_up[j * D + k], dtype);
        for (int64_t n = 0; n < D; ++n)
            for (int64_t j = 0; j < F; ++j) wd[j * D + n] = decode(W_down[n * F + j], dtype);
    }
    double* lg = NULL;
    double* lb = NULL;
    if (ln_gamma) {
        lg = (double*)malloc(sizeof(double) * (size_t)D);
        lb = (double*)malloc(sizeof(double) * (size_t)D);
        if (!lg || !lb) {
            free(wu); free(wd); free(bu); free(bd); free(lg); free(lb);
            return -1;
        }
        oracle_decode(ln_gamma, lg, D, dtype);
        oracle_decode(ln_beta, lb, D, dtype);
    }
    if (bias) {
        oracle_decode(b_up, bu, Fup, dtype);
        oracle_decode(b_down, bd, D, dtype);
    }
    int failed = 0;

#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)D);
        double* p = (double*)malloc(sizeof(double) * (size_t)Fup);
        double* hx = (double*)malloc(sizeof(double) * (size_t)F);
        double* h = (double*)malloc(sizeof(double) * (size_t)F);
        double* y = (double*)malloc(sizeof(double) * (size_t)D);
        double* xn = (double*)malloc(sizeof(double) * (size_t)D);
        if (!x || !p || !hx || !h || !y || !xn) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < nrows; ++i) {
                int64_t m = rows ? rows[i] : i;
                /* step 1: the row of X, exactly, in float64 */
                oracle_decode(X + m * D, x, D, dtype);
                if (lg) {
                    /* optional prologue: LayerNorm, rounded once to the I/O dtype */
                    oracle_layernorm_row(x, lg, lb, ln_eps, xn, D);
                    for (int64_t k = 0; k < D; ++k) x[k] = decode(encode(xn[k], dtype), dtype);
                }
                /* step 2: up projection (+ b_up) */
                linear_row(x, wu, bias ? bu : NULL, p, D, Fup);
                /* step 3: activation (GEGLU: value * gelu_erf(gate)) */
                activation_row(p, hx, F, act);
                /* step 4: the one rounding of H to the I/O dtype */
                for (int64_t j = 0; j < F; ++j) {
                    uint16_t hb = encode(hx[j], dtype);
                    if (H_out) H_out[i * F + j] = hb;
                    h[j] = decode(hb, dtype);
                }
                /* step 5: down projection (+ b_down) from the rounded H */
                linear_row(h, wd, bias ? bd : NULL, y, F, D);
                /* optional residual, added before the one rounding of Y */
                if (R)
                    for (int64_t n = 0; n < D; ++n) y[n] += decode(R[m * D + n], dtype);
                for (int64_t n = 0; n < D; ++n) {
                    if (Yx_out) Yx_out[i * D + n] = y[n];
                    if (Y_out) Y_out[i * D + n] = encode(y[n], dtype);
                }
            }
        }
        free(x); free(p); free(hx); free(h); free(y); free(xn);
    }
    free(wu); free(wd); free(bu); free(bd); free(lg); free(lb);
    return failed ? -1 : 0;
}

int oracle_mlp_rows(int64_t M, int64_t D, int64_t F, int act, int dtype, int bias,
                    const uint16_t* X, const uint16_t* W_up, const uint16_t* W_down,
                    const uint16_t* b_up, const uint16_t* b_down,
                    const int64_t* rows, int64_t nrows,
                    uint16_t* H_out, double* Yx_out, uint16_t* Y_out) {
    return oracle_mlp_rows_ex(M, D, F, act, dtype, bias, X, W_up, W_down, b_up, b_down, NULL, NULL, NULL,
                              0.0, 0, rows, nrows, H_out, Yx_out, Y_out);
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Fused-epilogue GEMM oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library.  It shares no source, header, table or helper with the
 * CUDA path: every decode, index computation and rounding below is written
 * out here from the definitions.
 *
 * What it computes, one output row at a time, in fp64:
 *
 *   acc(l,m,n) = sum_k a(l,m,k) * b(l,k,n)          a = op(A), b = op(B)
 *   t          = alpha*scale_a*scale_b*acc + beta*c(l,m,n) + bias
 *   t          = max(t, 0)                          if the activation is ReLU
 *   t          = t * Phi(t) = t/2 * (1 + erf(t/sqrt2))   if it is GELU
 *   D(l,m,n)   = round-to-nearest-even(t) in D's type
 *
 * Sources (page title, section):
 *  - "CUTLASS" (knowledge-base page), opening section: the operation is
 *    C = alpha * op(A) * op(B) + beta * C, op in {N, T}, column-major BLAS
 *    convention; D may be the same buffer as C ("Technical Documentation:
 *    NVIDIA/cutlass", "Launching a GEMM kernel in CUDA").
 *  - "CUTLASS" (knowledge-base page), "Epilogues": bias, activation and
 *    scaling are applied to the accumulated tile before it is written.
 *  - "Utilities for SM100", "Background - SM100 epilogue flow": accumulator,
 *    then the optional source C, then the fusion (bias, activation), then the
 *    store of D.
 *  - "Technical Documentation: NVIDIA/cutlass", "Blackwell Narrow Precision
 *    Data Types" table: e4m3 has 4 exponent and 3 mantissa bits, signed.
 *    The encoding details (bias 7, no infinities, S.1111.111 is NaN, largest
 *    finite 448) are the OCP 8-bit float E4M3 definition the table points to.
 *  - Per-tensor dequantisation scales scale_a, scale_b multiply the
 *    accumulator (the block-scaled form D = C + (A x SFA)(B x SFB) of
 *    "Blackwell SM100 GEMMs", "Block Scaled GEMMs", with one scale per
 *    tensor).
 *  - Block scaling (sf_vec > 0), "Technical Documentation: NVIDIA/cutlass",
 *    "Block Scaled GEMMs": acc = sum_k (a(m,k) * SFA(m, k/SV)) *
 *    (b(k,n) * SFB(n, k/SV)), SV = sf_vec elements of K per scale factor.
 *    "Blackwell Narrow Precision Data Types": mx_float8 pairs an 8-bit float
 *    with a ue8m0 scale (8 exponent bits, no sign, no mantissa), SV = 32; the
 *    value of a ue8m0 code e is 2^(e-127) and e = 255 is NaN (the OCP MX
 *    definition the table points to).  "Scale Factor Layouts": each
 *    512-byte basic block holds 128 rows x 4 scale factors, row r's four
 *    factors at byte (r % 32) * 16 + ((r % 128) / 32) * 4 (M0SF0-3, M32SF0-3,
 *    M64SF0-3, M96SF0-3, then M1...), and the blocks follow each other along
 *    K first (K-major), then along M; one such tensor per batch.
 *    nv_float4 pairs e2m1 data (2 exponent bits, 1 mantissa bit, signed)
 *    with a ue4m3 scale (4 exponent bits, 3 mantissa bits, no sign), SV =
 *    16 (same table and "Blackwell Block Scaled Narrow Precision Data
 *    Types").  Reading: e2m1 has bias 1 and no inf or NaN, so its codes are
 *    +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}; ue4m3 is e4m3 without the sign bit
 *    (bias 7, 0x7F NaN).  Two e2m1 elements share a byte, the one of lower
 *    storage index in the low nibble.
 *
 * Every product of two operands (<= 11 significant bits each) is exact in
 * fp64, and the fp64 sum over K carries a relative error of order K * 2^-53,
 * far below any output type's half-ulp, so the single final rounding is the
 * only rounding that matters.
 *
 * Readings where the pages leave a step open:
 *  - bias is added after alpha scaling and is not scaled itself;
 *  - beta == 0 means C is not read at all (a NaN in C does not propagate);
 *  - ReLU(t) = t > 0 ? t : 0 (so NaN maps to 0, like fmaxf);
 *  - GELU is the exact Gaussian-CDF form x * Phi(x) (the pages name no
 *    GELU; the tanh approximation is not used);
 *  - a batch index l adds l * stride_x elements to operand x's base.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element type codes of this oracle's own interface. */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3, OR_UE8M0 = 4, OR_E2M1 = 5, OR_UE4M3 = 6 };

typedef struct {
    int64_t M, N, K, L;
    int32_t op_a, op_b;                          /* 0 = N (as stored), 1 = T */
    int32_t order_a, order_b, order_c, order_d;  /* 0 = column-major, 1 = row-major */
    int64_t lda, ldb, ldc, ldd;                  /* leading dimensions, elements */
    int64_t stride_a, stride_b, stride_c, stride_d, stride_bias; /* batch strides, elements */
    int32_t dtype_a, dtype_b, dtype_c, dtype_d;
    double alpha, beta, scale_a, scale_b;
    int32_t has_bias;      /* bias is fp32 */
    int32_t bias_per_row;  /* 0: bias[n] broadcast down the columns; 1: bias[m] */
    int32_t act;           /* 0 = identity, 1 = ReLU, 2 = GELU */
    int32_t sf_vec;        /* 0: no block scaling; 32: ue8m0 scale per 32 K elements;
                              16: ue4m3 scale per 16 K elements */
} oracle_problem_t;

/* ---------------------------------------------------------------------------
 * Bit-level codecs.  A binary float with `eb` exponent bits and `mb` stored
 * mantissa bits has bias 2^(eb-1)-1; a zero exponent field means subnormal
 * (value = mant * 2^(1-bias-mb)).  IEEE formats reserve the all-ones exponent
 * for inf/NaN; e4m3 uses it for normal numbers except mantissa 111 (NaN);
 * e2m1 has no special values at all.  `ieee`: 1 IEEE, 0 e4m3's rule, -1 none.
 * ------------------------------------------------------------------------- */
static int type_bits(int dt, int* eb, int* mb, int* ieee) {
    switch (dt) {
        case OR_F32:  *eb = 8; *mb = 23; *ieee = 1; return 32;
        case OR_F16:  *eb = 5; *mb = 10; *ieee = 1; return 16;
        case OR_BF16: *eb = 8; *mb = 7;  *ieee = 1; return 16;
        case OR_E4M3: *eb = 4; *mb = 3;  *ieee = 0; return 8;
        case OR_E2M1: *eb = 2; *mb = 1;  *ieee = -1; return 4;
        default: return 0;
    }
}

double oracle_decode(int dt, uint32_t bits) {
    int eb, mb, ieee;
    if (dt == OR_UE8M0) return (bits & 0xFFu) == 0xFFu ? NAN : ldexp(1.0, (int)(bits & 0xFFu) - 127);
    if (dt == OR_UE4M3) return oracle_decode(OR_E4M3, bits & 0x7Fu);     /* no sign bit */
    if (!type_bits(dt, &eb, &mb, &ieee)) return NAN;
    const uint32_t mant = bits & ((1u << mb) - 1u);
    const uint32_t expf = (bits >> mb) & ((1u << eb) - 1u);
    const int neg = (bits >> (mb + eb)) & 1u;
    const int bias = (1 << (eb - 1)) - 1;
    const uint32_t all_ones = (1u << eb) - 1u;
    double v;
    if (expf == all_ones && ieee == 1) {
        v = mant ? NAN : INFINITY;
    } else if (expf == all_ones && ieee == 0 && mant == (1u << mb) - 1u) {
        v = NAN;
    } else if (expf == 0) {
        v = ldexp((double)mant, 1 - bias - mb);
    } else {
        v = ldexp((double)(mant | (1u << mb)), (int)expf - bias - mb);
    }
    return neg ? -v : v;
}

/* Round-to-nearest, ties-to-even, from fp64 into an IEEE type (f32/f16/bf16).
 * Overflow goes to infinity as IEEE 754 prescribes for this rounding mode. */
uint32_t oracle_encode(int dt, double v) {
    int eb, mb, ieee;
    if (!type_bits(dt, &eb, &mb, &ieee) || ieee != 1) return 0xFFFFFFFFu;
    const int bias = (1 << (eb - 1)) - 1;
    const uint32_t sign = signbit(v) ? (1u << (eb + mb)) : 0u;
    const uint32_t inf_bits = sign | (((1u << eb) - 1u) << mb);
    if (isnan(v)) return inf_bits | (1u << (mb - 1));   /* quiet NaN */
    const double a = fabs(v);
    if (isinf(a)) return inf_bits;
    if (a == 0.0) return sign;
    const int emin = 1 - bias;
    const int emax = bias;
    const double max_finite = ldexp(2.0 - ldexp(1.0, -mb), emax);
    int e2;
    frexp(a, &e2);               /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;              /* a in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;      /* subnormal range shares emin's quantum */
    /* a / 2^(E-mb) is exact in fp64 (power-of-two scaling); nearbyint rounds it
     * to an integer with ties to even under the default rounding mode. */
    const double r = nearbyint(ldexp(a, mb - E));
    const double res = ldexp(r, E - mb);
    if (res > max_finite) return inf_bits;
    if (r == 0.0) return sign;
    frexp(res, &e2);
    E = e2 - 1;
    if (E < emin) {
        return sign | (uint32_t)ldexp(res, mb - emin);
    }
    const uint32_t mant = (uint32_t)(ldexp(res, mb - E) - ldexp(1.0, mb));
    return sign | ((uint32_t)(E + bias) << mb) | mant;
}

static uint32_t load_bits(const void* base, int dt, int64_t idx) {
    switch (dt) {
        case OR_F32: { uint32_t x; memcpy(&x, (const char*)base + 4 * idx, 4); return x; }
        case OR_F16:
        case OR_BF16: { uint16_t x; memcpy(&x, (const char*)base + 2 * idx, 2); return x; }
        case OR_E4M3: return ((const uint8_t*)base)[idx];
        case OR_E2M1: {
            const uint8_t byte = ((const uint8_t*)base)[idx / 2];
            return idx % 2 ? (uint32_t)(byte >> 4) : (uint32_t)(byte & 0xFu);
        }
        default: return 0;
    }
}

static void store_bits(void* base, int dt, int64_t idx, uint32_t bits) {
    switch (dt) {
        case OR_F32: memcpy((char*)base + 4 * idx, &bits, 4); break;
        case OR_F16:
        case OR_BF16: { uint16_t x = (uint16_t)bits; memcpy((char*)base + 2 * idx, &x, 2); break; }
        default: break;
    }
}

/* ---------------------------------------------------------------------------
 * Addressing, BLAS convention.  op(A) is M x K: with op N the stored matrix is
 * M x K, with op T it is K x M.  A stored R x S matrix is read at
 * r * ld + s (row-major) or r + s * ld (column-major).
 * ------------------------------------------------------------------------- */
static int64_t stored_index(int order, int64_t r, int64_t s, int64_t ld) {
    return order == 1 ? r * ld + s : r + s * ld;
}

static int64_t a_index(const oracle_problem_t* p, int64_t l, int64_t m, int64_t k) {
    const int64_t off = p->op_a == 0 ? stored_index(p->order_a, m, k, p->lda)
                                     : stored_index(p->order_a, k, m, p->lda);
    return l * p->stride_a + off;
}

static int64_t b_index(const oracle_problem_t* p, int64_t l, int64_t k, int64_t n) {
    const int64_t off = p->op_b == 0 ? stored_index(p->order_b, k, n, p->ldb)
                                     : stored_index(p->order_b, n, k, p->ldb);
    return l * p->stride_b + off;
}

static int64_t cd_index(int order, int64_t ld, int64_t stride, int64_t l, int64_t m, int64_t n) {
    return l * stride + stored_index(order, m, n, ld);
}

static int nthreads_or_default(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_max_threads(void) { return nthreads_or_default(0); }

/* Byte offset of scale factor (row, kf) of batch l in a tensor of `rows`
 * rows and `sfk` factors per row (the basic-block layout above). */
int64_t oracle_sf_index(int64_t l, int64_t row, int64_t kf, int64_t rows, int64_t sfk) {
    const int64_t kblocks = (sfk + 3) / 4, mblocks = (rows + 127) / 128;
    const int64_t block = (row / 128) * kblocks + kf / 4;
    return l * mblocks * kblocks * 512 + block * 512 + (row % 32) * 16 + ((row % 128) / 32) * 4 + kf % 4;
}

static double sf_value(const uint8_t* sf, int64_t l, int64_t row, int64_t k, int64_t rows, const oracle_problem_t* p) {
    const int64_t sfk = (p->K + p->sf_vec - 1) / p->sf_vec;
    const int sf_type = p->sf_vec == 16 ? OR_UE4M3 : OR_UE8M0;      /* nv_float4 : mx types */
    return oracle_decode(sf_type, sf[oracle_sf_index(l, row, k / p->sf_vec, rows, sfk)]);
}

/*
 * b(l, k, n) decoded into a k-major fp64 panel (K x N).  The last panel is
 * kept and reused when the next call names the same storage with the same
 * bytes (an FNV-1a hash of the operand's storage span is part of the key), so
 * repeated calls on one operand decode it once.  Not thread-safe: calls into
 * the oracle are sequential.
 */
static double* g_panel = NULL;
static size_t g_panel_cap = 0;
static struct {
    const void* base;
    const void* sfb;
    int64_t K, N, l, ldb, stride_b;
    int32_t op_b, order_b, dtype_b, sf_vec;
    uint64_t hash, sf_hash;
    int valid;
} g_key;

static uint64_t fnv1a(const uint8_t* p, size_t n) {
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 1099511628211ull;
    }
    return h;
}

static const double* b_panel(const oracle_problem_t* p, const void* B, const uint8_t* SFB, int64_t l) {
    const int64_t K = p->K, N = p->N;
    int eb, mb, ieee;
    const int bits = type_bits(p->dtype_b, &eb, &mb, &ieee);
    /* the storage span this batch of B occupies (whole bytes) */
    const int64_t srows = p->op_b == 0 ? K : N, scols = p->op_b == 0 ? N : K;
    const int64_t outer = p->order_b == 1 ? srows : scols;
    const int64_t inner = p->order_b == 1 ? scols : srows;
    const int64_t span = outer > 0 && inner > 0 ? (outer - 1) * p->ldb + inner : 0;
    const int64_t bit0 = l * p->stride_b * bits;
    const uint8_t* first = (const uint8_t*)B + (size_t)(bit0 / 8);
    const uint64_t h = fnv1a(first, (size_t)((bit0 % 8 + span * bits + 7) / 8));
    uint64_t sh = 0;
    if (p->sf_vec > 0) {
        const int64_t sfk = (K + p->sf_vec - 1) / p->sf_vec;
        const int64_t per = ((N + 127) / 128) * ((sfk + 3) / 4) * 512;
        sh = fnv1a(SFB + l * per, (size_t)per);
    }
    if (g_key.valid && g_key.base == B && g_key.K == K && g_key.N == N && g_key.l == l && g_key.ldb == p->ldb &&
        g_key.stride_b == p->stride_b && g_key.op_b == p->op_b && g_key.order_b == p->order_b &&
        g_key.dtype_b == p->dtype_b && g_key.hash == h && g_key.sf_vec == p->sf_vec &&
        (p->sf_vec == 0 || (g_key.sfb == (const void*)SFB && g_key.sf_hash == sh)))
        return g_panel;
    const size_t need = (size_t)(K > 0 ? K : 1) * (size_t)N;
    if (need > g_panel_cap) {
        free(g_panel);
        g_panel = (double*)malloc(sizeof(double) * need);
        g_panel_cap = g_panel ? need : 0;
        g_key.valid = 0;
        if (!g_panel) return NULL;
    }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) {
            double v = oracle_decode(p->dtype_b, load_bits(B, p->dtype_b, b_index(p, l, k, n)));
            if (p->sf_vec > 0) v *= sf_value(SFB, l, n, k, N, p);      /* b(k,n) * SFB(n, k/SV) */
            g_panel[k * N + n] = v;
        }
    g_key.base = B;
    g_key.sfb = SFB;
    g_key.sf_vec = p->sf_vec;
    g_key.sf_hash = sh;
    g_key.K = K;
    g_key.N = N;
    g_key.l = l;
    g_key.ldb = p->ldb;
    g_key.stride_b = p->stride_b;
    g_key.op_b = p->op_b;
    g_key.order_b = p->order_b;
    g_key.dtype_b = p->dtype_b;
    g_key.hash = h;
    g_key.valid = 1;
    return g_panel;
}

/*
 * Computes the full output rows listed in `rows` (each entry is l*M + m).
 * Row i of the result goes to Dout[i*N .. i*N+N-1], packed in D's type, and,
 * when Tout is not NULL, the fp64 value before rounding to Tout[i*N + n].
 * The full GEMM is the call with every row listed.
 * Returns 0 on success, a negative code on bad arguments or allocation failure.
 */
int oracle_gemm_rows_sf(const oracle_problem_t* p, const void* A, const void* B, const uint8_t* SFA,
                        const uint8_t* SFB, const void* C, const float* bias, int64_t nrows, const int64_t* rows,
                        void* Dout, double* Tout, int nthreads) {
    int eb, mb, ieee;
    if (!p || p->M < 0 || p->N < 0 || p->K < 0 || p->L < 1) return -1;
    if (!type_bits(p->dtype_a, &eb, &mb, &ieee) || !type_bits(p->dtype_b, &eb, &mb, &ieee)) return -2;
    if (!type_bits(p->dtype_d, &eb, &mb, &ieee) || ieee != 1) return -3;
    const int use_c = p->beta != 0.0;
    if (use_c && (!C || !type_bits(p->dtype_c, &eb, &mb, &ieee))) return -4;
    if (p->has_bias && !bias) return -5;
    if (p->sf_vec < 0 || (p->sf_vec > 0 && (!SFA || !SFB))) return -7;
    const int64_t M = p->M, N = p->N, K = p->K;
    const double scale = p->alpha * p->scale_a * p->scale_b;
    const int nt = nthreads_or_default(nthreads);
    if (nrows == 0 || N == 0) return 0;

    int status = 0;
    for (int64_t l = 0; l < p->L; ++l) {
        int64_t in_batch = 0;
        for (int64_t i = 0; i < nrows; ++i) in_batch += (rows[i] / M) == l;
        if (!in_batch) continue;
        const double* Bd = b_panel(p, B, SFB, l);
        if (!Bd) return -6;

#pragma omp parallel num_threads(nt)
        {
            double* acc = (double*)malloc(sizeof(double) * (size_t)N);
            if (!acc) {
#pragma omp atomic write
                status = -6;
            }
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < nrows; ++i) {
                if (!acc || rows[i] / M != l) continue;
                const int64_t m = rows[i] % M;
                for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
                /* i-k-j order: one a(m,k) times the k-th row of b, summed. */
                for (int64_t k = 0; k < K; ++k) {
                    double a = oracle_decode(p->dtype_a, load_bits(A, p->dtype_a, a_index(p, l, m, k)));
                    if (p->sf_vec > 0) a *= sf_value(SFA, l, m, k, M, p);     /* a(m,k) * SFA(m, k/SV) */
                    const double* brow = Bd + k * N;
                    for (int64_t n = 0; n < N; ++n) acc[n] += a * brow[n];
                }
                for (int64_t n = 0; n < N; ++n) {
                    double t = scale * acc[n];
                    if (use_c)
                        t += p->beta * oracle_decode(p->dtype_c,
                                 load_bits(C, p->dtype_c, cd_index(p->order_c, p->ldc, p->stride_c, l, m, n)));
                    if (p->has_bias)
                        t += (double)bias[l * p->stride_bias + (p->bias_per_row ? m : n)];
                    if (p->act == 1) t = t > 0.0 ? t : 0.0;
                    if (p->act == 2) t = 0.5 * t * (1.0 + erf(t * 0.70710678118654752440));
                    if (Tout) Tout[i * N + n] = t;
                    store_bits(Dout, p->dtype_d, i * N + n, oracle_encode(p->dtype_d, t));
                }
            }
            free(acc);
        }
    }
    return status;
}

int oracle_gemm_rows(const oracle_problem_t* p, const void* A, const void* B, const void* C, const float* bias,
                     int64_t nrows, const int64_t* rows, void* Dout, double* Tout, int nthreads) {
    if (p && p->sf_vec != 0) return -7;
    return oracle_gemm_rows_sf(p, A, B, NULL, NULL, C, bias, nrows, rows, Dout, Tout, nthreads);
}

/* Round-to-nearest-even into e4m3 with saturation ("satfinite"): finite
 * values beyond the largest finite magnitude 448 become +-448, NaN becomes
 * the NaN code S.1111.111 (0x7F); e4m3 has no infinities.  Subnormals have
 * quantum 2^-9 (exponent field 0, bias 7, 3 mantissa bits). */
uint32_t oracle_encode_e4m3(double v) {
    if (isnan(v)) return 0x7Fu;
    const uint32_t sign = signbit(v) ? 0x80u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    const int mb = 3, bias = 7, emin = 1 - bias;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;
    if (E < emin) E = emin;
    double r = nearbyint(ldexp(a, mb - E));    /* exact scaling, ties to even */
    double res = ldexp(r, E - mb);
    if (res > 448.0 || isinf(a)) return sign | 0x7Eu;  /* satfinite: 1.1111.110 = 448 */
    if (r == 0.0) return sign;
    frexp(res, &e2);
    E = e2 - 1;
    if (E < emin) return sign | (uint32_t)ldexp(res, mb - emin);          /* subnormal */
    const uint32_t mant = (uint32_t)(ldexp(res, mb - E) - ldexp(1.0, mb));
    return sign | ((uint32_t)(E + bias) << mb) | mant;
}

void oracle_encode_e4m3_array(const double* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_encode_e4m3(v[i]);
}

/* Round-to-nearest-even into e2m1 with saturation: magnitudes from 6 up
 * become 6 (code 7), the sign goes to bit 3.  Bias 1 and one mantissa bit:
 * below 1 the quantum is 0.5 (code 1 = 0.5), then 2^(E-1) for values in
 * [2^E, 2^(E+1)).  NaN has no code; it is given 0 (callers never pass one). */
uint32_t oracle_encode_e2m1(double v) {
    if (isnan(v)) return 0u;
    const uint32_t sign = signbit(v) ? 0x8u : 0u;
    const double a = fabs(v);
    if (a >= 6.0) return sign | 0x7u;
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;
    if (E < 0) E = 0;                          /* subnormal range shares exponent 0's quantum */
    const double r = nearbyint(ldexp(a, 1 - E));    /* exact scaling, ties to even */
    const double res = ldexp(r, E - 1);
    if (res == 0.0) return sign;
    frexp(res, &e2);
    E = e2 - 1;
    if (E < 0) return sign | 0x1u;             /* 0.5 */
    const uint32_t mant = (uint32_t)(ldexp(res, 1 - E) - 2.0);
    return sign | ((uint32_t)(E + 1) << 1) | mant;
}

void oracle_encode_e2m1_array(const double* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_encode_e2m1(v[i]);
}

/* Scatters packed rows (as produced by oracle_gemm_rows for every row, in
 * order) into D's own storage layout: D(l,m,n) at l*stride_d + (m,n) by
 * order_d and ldd.  Lets a test build a full D buffer the way a caller lays
 * it out. */
int oracle_scatter_d(const oracle_problem_t* p, const void* packed, void* Dstore) {
    int eb, mb, ieee;
    if (!type_bits(p->dtype_d, &eb, &mb, &ieee)) return -1;
    for (int64_t l = 0; l < p->L; ++l)
        for (int64_t m = 0; m < p->M; ++m)
            for (int64_t n = 0; n < p->N; ++n)
                store_bits(Dstore, p->dtype_d, cd_index(p->order_d, p->ldd, p->stride_d, l, m, n),
                           load_bits(packed, p->dtype_d, (l * p->M + m) * p->N + n));
    return 0;
}

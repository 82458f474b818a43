/*
 * moe_oracle.c -- plain, slow fp64 CPU oracle of the routed-expert MXFP4 MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * What it computes (sources: the Deltafin pages, "Deltafin 的功能" and "工作原理":
 * 16 routed experts per layer picked by the router, experts kept at their
 * released MXFP4 precision; the layer math is the routed-expert layer named by
 * the project brief: top-16 of E by router logit, softmax over the 16 selected
 * logits, SwiGLU expert FFN, router-weighted combine):
 *
 *   l_e   = sum_h x_h W_r[e,h] (+ skew_e)             exact (fixed-point), see route
 *   S     = the k experts of largest l, ties -> lower index, in descending order
 *   w_j   = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the k selected   (fp64)
 *   g     = W_g x, u = W_u x, h = silu(g) * u,  o = W_d h                   (fp64)
 *   y     = sum_j w_j o_j                                                   (fp64)
 *
 * MXFP4 (OCP Microscaling v1.0): element = E2M1(code) * 2^(scale_byte - 127),
 * one E8M0 scale byte per 32 consecutive elements along K.
 *
 * Parity pins live in tests/test_oracle_*.py.  Functions with no external pin are
 * marked "parity unpinned" below (none at present).
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Threads of the OpenMP loops (rows and tokens are independent; the arithmetic of
 * each result does not depend on the thread count).  Returns the previous value. */
int orc_set_threads(int n) {
    int prev = omp_get_max_threads();
    if (n > 0) omp_set_num_threads(n);
    return prev;
}

/* ------------------------------------------------------------------ SplitMix64
 * Steele, Lea & Flood, "Fast Splittable Pseudorandom Number Generators" (2014),
 * in counter mode: u64(seed, stream, i) is output i of SplitMix64 started at
 * key(seed, stream) = mix(mix(seed + G) ^ mix(stream + 2G)). */
#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output i (0-based) of plain SplitMix64 whose state starts at `state`. */
uint64_t orc_splitmix64_at(uint64_t state, uint64_t i) {
    return sm_mix(state + (i + 1) * SM_GAMMA);
}

uint64_t orc_u64(uint64_t seed, uint64_t stream, uint64_t i) {
    uint64_t key = sm_mix(sm_mix(seed + SM_GAMMA) ^ sm_mix(stream + 2 * SM_GAMMA));
    return sm_mix(key + (i + 1) * SM_GAMMA);
}

/* Expert e of the pool drawn with `seed`, in its logical row-major form:
 *   codes : gate [I][H/2] | up [I][H/2] | down [H][I/2]   (element 2j in the low nibble)
 *   scales: gate [I][H/32] | up [I][H/32] | down [H][I/32]
 * Code byte b is byte (b mod 8) of u64(seed, 2e, b/8): two uniform E2M1 codes.
 * Scale byte j is 118 + (u64(seed, 2e+1, j) >> 32) mod 5: exponents -9..-5. */
void orc_gen_expert(uint64_t seed, int e, int H, int I, uint8_t *codes, uint8_t *scales) {
    size_t ncode = (size_t)3 * H * I / 2, nscale = (size_t)3 * H * I / 32;
    uint64_t key_c = sm_mix(sm_mix(seed + SM_GAMMA) ^ sm_mix((uint64_t)(2 * e) + 2 * SM_GAMMA));
    uint64_t key_s = sm_mix(sm_mix(seed + SM_GAMMA) ^ sm_mix((uint64_t)(2 * e + 1) + 2 * SM_GAMMA));
    for (size_t b = 0; b < ncode; b += 8) {
        uint64_t r = sm_mix(key_c + (uint64_t)(b / 8 + 1) * SM_GAMMA);
        for (size_t q = 0; q < 8 && b + q < ncode; q++) codes[b + q] = (uint8_t)(r >> (8 * q));
    }
    for (size_t j = 0; j < nscale; j++) {
        uint64_t r = sm_mix(key_s + (uint64_t)(j + 1) * SM_GAMMA);
        scales[j] = (uint8_t)(118 + (r >> 32) % 5);
    }
}

/* ------------------------------------------------------------ OCP MX element types */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(unsigned code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* E8M0: 2^(b-127); 0xFF is NaN. */
double orc_e8m0_value(unsigned b) {
    if ((b & 0xFF) == 0xFF) return NAN;
    return ldexp(1.0, (int)(b & 0xFF) - 127);
}

/* E4M3 (OCP "FN" variant): bias 7, no infinities, 0x7F/0xFF NaN, max 448. */
double orc_e4m3_value(unsigned c) {
    unsigned s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, (int)e - 7);
    return s ? -v : v;
}

/* Round v to E4M3: nearest finite value, ties to the even code, |v| beyond the
 * largest finite magnitude saturates to +-448 (the "satfinite" conversion). */
unsigned orc_e4m3_encode(double v) {
    unsigned sign = (v < 0 || (v == 0 && signbit(v))) ? 0x80u : 0u;
    double a = fabs(v);
    unsigned best = 0;
    double bestd = INFINITY;
    for (unsigned c = 0; c < 0x7F; c++) {          /* the 127 finite non-negative codes */
        double d = fabs(orc_e4m3_value(c) - a);
        if (d < bestd || (d == bestd && (c & 1u) == 0u)) { best = c; bestd = d; }
    }
    return sign | best;
}

/* MXFP8 quantisation of n values in blocks of 32 (OCP MX v1.0, section 6.3):
 * shared exponent X = floor(log2(amax)) - 8 (8 = E4M3 emax), clamped to [-127,127];
 * element code = E4M3(v / 2^X) with saturation.  amax == 0 gives X = -127.
 * codes[n], sbytes[ceil(n/32)], deq[n] (nullable) = dequantised values. */
void orc_quant_mxfp8(const double *v, int n, uint8_t *codes, uint8_t *sbytes, double *deq) {
    for (int b0 = 0; b0 < n; b0 += 32) {
        int b1 = b0 + 32 < n ? b0 + 32 : n;
        double amax = 0.0;
        for (int i = b0; i < b1; i++) if (fabs(v[i]) > amax) amax = fabs(v[i]);
        int X = -127;
        if (amax > 0.0) {
            int ex;
            frexp(amax, &ex);                      /* amax = f * 2^ex, f in [0.5, 1) */
            X = (ex - 1) - 8;
            if (X < -127) X = -127;
            if (X > 127) X = 127;
        }
        sbytes[b0 / 32] = (uint8_t)(X + 127);
        for (int i = b0; i < b1; i++) {
            unsigned c = orc_e4m3_encode(ldexp(v[i], -X));
            codes[i] = (uint8_t)c;
            if (deq) deq[i] = ldexp(orc_e4m3_value(c), X);
        }
    }
}

/* Round v to E2M1: nearest of the 8 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to
 * the even code (mantissa bit 0), |v| beyond 6 saturates to +-6; the sign bit is
 * that of v (so small negatives give -0, code 8). */
unsigned orc_e2m1_encode(double v) {
    unsigned sign = (v < 0 || (v == 0 && signbit(v))) ? 8u : 0u;
    double a = fabs(v);
    if (a >= 6.0) return sign | 7u;                 /* saturation (also where |v - m| loses m) */
    unsigned best = 0;
    double bestd = INFINITY;
    for (unsigned c = 0; c < 8; c++) {
        double d = fabs(E2M1_MAG[c] - a);
        if (d < bestd || (d == bestd && (c & 1u) == 0u)) { best = c; bestd = d; }
    }
    return sign | best;
}

/* MXFP4 quantisation of n values in blocks of 32 (OCP MX v1.0): shared exponent
 * X = floor(log2(amax)) - 2 (2 = E2M1 emax), clamped to [-127, 127]; element code =
 * E2M1(v / 2^X) with saturation.  amax == 0 gives X = -127.
 * codes[n] (one code per byte), sbytes[ceil(n/32)], deq[n] (nullable). */
void orc_quant_mxfp4(const double *v, int n, uint8_t *codes, uint8_t *sbytes, double *deq) {
    for (int b0 = 0; b0 < n; b0 += 32) {
        int b1 = b0 + 32 < n ? b0 + 32 : n;
        double amax = 0.0;
        for (int i = b0; i < b1; i++) if (fabs(v[i]) > amax) amax = fabs(v[i]);
        int X = -127;
        if (amax > 0.0) {
            int ex;
            frexp(amax, &ex);
            X = (ex - 1) - 2;
            if (X < -127) X = -127;
            if (X > 127) X = 127;
        }
        sbytes[b0 / 32] = (uint8_t)(X + 127);
        for (int i = b0; i < b1; i++) {
            unsigned c = orc_e2m1_encode(ldexp(v[i], -X));
            codes[i] = (uint8_t)c;
            if (deq) deq[i] = ldexp(orc_e2m1_value(c), X);
        }
    }
}

/* ----------------------------------------------------------------- bf16 helpers */

double orc_bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to bf16, nearest-even, directly (no intermediate fp32). */
uint16_t orc_bf16_round(double v) {
    uint16_t sign = (v < 0 || (v == 0 && signbit(v))) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7FC0;
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);                                  /* a in [2^(ex-1), 2^ex) */
    int e = ex - 1;                                 /* unbiased exponent of a */
    if (e < -126) e = -126;                         /* subnormal range: fixed quantum */
    double q = ldexp(a, 7 - e);                     /* significand in units of the last place */
    double r = nearbyint(q);                        /* current rounding mode: nearest-even */
    uint32_t m = (uint32_t)r;
    int E = e + 127;                                /* biased exponent if normal */
    if (m >= 256) { m >>= 1; E += 1; }              /* rounding carried into the next binade */
    if (m < 128) E = 0;                             /* subnormal (only when e == -126) */
    if (E >= 255) return sign | 0x7F80;             /* overflow to infinity */
    return sign | (uint16_t)((uint32_t)E << 7) | (uint16_t)(m & 0x7F);
}

/* ------------------------------------------------------------------ routing
 * Exact router logits.  A finite bf16 value is (-1)^s * m * 2^(E' - 134) with
 * m = the 8-bit significand (implicit bit included for E > 0) and E' = max(E, 1);
 * a finite fp32 skew is (-1)^s * m * 2^(E' - 150) with a 24-bit m.  Every term
 * is therefore an integer multiple of 2^-268, and the logit is held exactly as a
 * two's-complement integer in units of 2^-268, in base-2^32 limbs. */
#define XL 22                      /* 704 bits: terms reach bit 524, sums of 2^31 terms fit */

typedef struct { int64_t d[XL]; } exact_t;

static void ex_add(exact_t *a, int neg, uint64_t m, int shift) {
    int li = shift / 32, sh = shift % 32;
    /* m < 2^24 and sh < 32: value m << sh < 2^56 split into two 32-bit digits */
    uint64_t v = m << sh;
    int64_t lo = (int64_t)(v & 0xFFFFFFFFu), hi = (int64_t)(v >> 32);
    if (neg) { lo = -lo; hi = -hi; }
    a->d[li] += lo;
    a->d[li + 1] += hi;
}

static void ex_normalise(exact_t *a) {
    for (int i = 0; i < XL - 1; i++) {
        int64_t c = a->d[i] >> 32;                 /* arithmetic shift: floor division */
        a->d[i] -= c * ((int64_t)1 << 32);
        a->d[i + 1] += c;
    }
}

/* -1, 0, +1 for a < b, a == b, a > b (both normalised). */
static int ex_cmp(const exact_t *a, const exact_t *b) {
    if (a->d[XL - 1] != b->d[XL - 1]) return a->d[XL - 1] < b->d[XL - 1] ? -1 : 1;
    for (int i = XL - 2; i >= 0; i--)
        if (a->d[i] != b->d[i]) return a->d[i] < b->d[i] ? -1 : 1;   /* digits in [0, 2^32) */
    return 0;
}

/* The exact value rounded to the nearest double (ties to even). */
static double ex_to_double(const exact_t *a) {
    exact_t t = *a;
    int neg = t.d[XL - 1] < 0;
    if (neg) {                                     /* two's-complement negate, then renormalise */
        for (int i = 0; i < XL; i++) t.d[i] = -t.d[i];
        ex_normalise(&t);
    }
    int top = -1;
    for (int i = XL - 1; i >= 0; i--) if (t.d[i]) { top = i; break; }
    if (top < 0) return neg ? -0.0 : 0.0;
    /* gather 96 bits from the top three digits, then the sticky rest */
    uint64_t d2 = (uint64_t)t.d[top], d1 = top >= 1 ? (uint64_t)t.d[top - 1] : 0,
             d0 = top >= 2 ? (uint64_t)t.d[top - 2] : 0;
    int sticky = 0;
    for (int i = top - 3; i >= 0; i--) if (t.d[i]) sticky = 1;
    int lz = 0;
    while (!((d2 << lz) & 0x80000000ULL)) lz++;    /* d2 has a bit set in [0, 32) */
    /* 64 most significant bits, starting at the leading one */
    __uint128_t w96 = ((__uint128_t)d2 << 64) | ((__uint128_t)d1 << 32) | d0;
    w96 <<= (32 + lz);                             /* leading one now at bit 127 */
    uint64_t hi = (uint64_t)(w96 >> 64);
    if ((uint64_t)w96 != 0) sticky = 1;
    if (sticky) hi |= 1;                           /* below the rounding bit: breaks ties only */
    double r = (double)hi;                         /* one correctly rounded conversion */
    int exp2 = 32 * top + 31 - lz - 63 - 268;      /* weight of hi's bit 0 */
    r = ldexp(r, exp2);
    return neg ? -r : r;
}

/* returns 0, or -1 if a non-finite input was seen */
static int bf16_parts(uint16_t b, int *neg, uint32_t *m, int *Ep) {
    int E = (b >> 7) & 0xFF;
    if (E == 0xFF) return -1;
    *neg = (b >> 15) & 1;
    *m = (b & 0x7F) | (E ? 0x80u : 0u);
    *Ep = E ? E : 1;
    return 0;
}

static int exact_logit(const uint16_t *x, const uint16_t *w, int H, const float *skew_e, exact_t *out) {
    memset(out, 0, sizeof(*out));
    for (int h = 0; h < H; h++) {
        int n1, n2, e1, e2;
        uint32_t m1, m2;
        if (bf16_parts(x[h], &n1, &m1, &e1) || bf16_parts(w[h], &n2, &m2, &e2)) return -1;
        if (m1 == 0 || m2 == 0) continue;
        ex_add(out, n1 ^ n2, (uint64_t)m1 * m2, e1 + e2);     /* unit 2^(e1+e2-268) */
    }
    if (skew_e) {
        uint32_t u;
        memcpy(&u, skew_e, 4);
        int E = (u >> 23) & 0xFF;
        if (E == 0xFF) return -1;
        uint32_t m = (u & 0x7FFFFF) | (E ? 0x800000u : 0u);
        int Ep = E ? E : 1;
        if (m) ex_add(out, (u >> 31) & 1, m, Ep + 118);       /* 2^(Ep-150) = 2^(Ep+118-268) */
    }
    ex_normalise(out);
    return 0;
}

/* Route M tokens: top-k of E by exact logit (ties -> lower index), in descending
 * order, and softmax weights over the k selected logits.
 * x [M][H] bf16, Wr [E][H] bf16, skew [E] fp32 (nullable).
 * idx [M][k], w [M][k] fp64, logits [M][E] fp64 (nullable; the exact value rounded).
 * Returns 0, or -1 on non-finite input, -2 on bad sizes. */
int orc_route(const uint16_t *x, int M, int H, const uint16_t *Wr, int E, const float *skew, int k,
              int32_t *idx, double *w, double *logits) {
    if (M < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return -2;
    int rc = 0;
    /* tokens are independent: each thread routes whole tokens with its own buffers */
    #pragma omp parallel
    {
        exact_t *l = (exact_t *)malloc(sizeof(exact_t) * (size_t)E);
        char *taken = (char *)malloc((size_t)E);
        if (!l || !taken) {
            #pragma omp atomic write
            rc = -2;
        }
        #pragma omp for schedule(dynamic, 1)
        for (int m = 0; m < M; m++) {
            if (!l || !taken) continue;
            const uint16_t *xm = x + (size_t)m * H;
            int bad = 0;
            for (int e = 0; e < E && !bad; e++)
                if (exact_logit(xm, Wr + (size_t)e * H, H, skew ? skew + e : NULL, &l[e])) bad = 1;
            if (bad) {
                #pragma omp atomic write
                rc = -1;
                continue;
            }
            if (logits) for (int e = 0; e < E; e++) logits[(size_t)m * E + e] = ex_to_double(&l[e]);
            memset(taken, 0, (size_t)E);
            for (int j = 0; j < k; j++) {              /* k passes of "largest remaining, lowest index" */
                int best = -1;
                for (int e = 0; e < E; e++) {
                    if (taken[e]) continue;
                    if (best < 0 || ex_cmp(&l[e], &l[best]) > 0) best = e;
                }
                taken[best] = 1;
                idx[(size_t)m * k + j] = best;
            }
            double lmax = ex_to_double(&l[idx[(size_t)m * k]]), z = 0.0;
            for (int j = 0; j < k; j++) z += exp(ex_to_double(&l[idx[(size_t)m * k + j]]) - lmax);
            for (int j = 0; j < k; j++)
                w[(size_t)m * k + j] = exp(ex_to_double(&l[idx[(size_t)m * k + j]]) - lmax) / z;
        }
        free(l);
        free(taken);
    }
    return rc;
}

/* ------------------------------------------------------------------- expert FFN */

/* Dot product of row `row` of an MXFP4 matrix with K columns and the vector v:
 * sum over 32-blocks of 2^(scale-127) * sum_j E2M1(code_j) * v_j. */
static double mx_row_dot(const uint8_t *codes, const uint8_t *scales, size_t row, int K, const double *v) {
    const uint8_t *c = codes + row * (size_t)(K / 2);
    const uint8_t *s = scales + row * (size_t)(K / 32);
    double acc = 0.0;
    for (int b = 0; b < K / 32; b++) {
        double sc = orc_e8m0_value(s[b]), part = 0.0;
        for (int j = 32 * b; j < 32 * b + 32; j++) {
            unsigned code = (j & 1) ? (c[j / 2] >> 4) : (c[j / 2] & 15);
            part += orc_e2m1_value(code) * v[j];
        }
        acc += sc * part;
    }
    return acc;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Apply one expert (logical layout, see orc_gen_expert) to n rows x [n][H]:
 * y [n][H] = W_d (silu(W_g x) * (W_u x)); h [n][I] (nullable) receives h.
 * h_mode 1: h is MXFP8-quantised along I (orc_quant_mxfp8) before W_d;
 * h_mode 2: h is MXFP4-quantised along I (orc_quant_mxfp4) before W_d.
 * Rows are independent; the loop over rows is the outer one for clarity. */
void orc_expert_forward(const uint8_t *codes, const uint8_t *scales, int H, int I,
                        const double *x, int n, double *y, double *h, int h_mode) {
    const uint8_t *cg = codes, *cu = codes + (size_t)I * H / 2, *cd = codes + (size_t)I * H;
    const uint8_t *sg = scales, *su = scales + (size_t)I * H / 32, *sd = scales + (size_t)I * H / 16;
    double *hv = (double *)malloc(sizeof(double) * (size_t)I);
    uint8_t *qc = (uint8_t *)malloc((size_t)I), *qs = (uint8_t *)malloc((size_t)I / 32 + 1);
    for (int r = 0; r < n; r++) {
        const double *xr = x + (size_t)r * H;
        #pragma omp parallel for schedule(static)
        for (int i = 0; i < I; i++) {
            double g = mx_row_dot(cg, sg, (size_t)i, H, xr);
            double u = mx_row_dot(cu, su, (size_t)i, H, xr);
            hv[i] = silu(g) * u;
        }
        if (h_mode == 1) orc_quant_mxfp8(hv, I, qc, qs, hv);
        if (h_mode == 2) orc_quant_mxfp4(hv, I, qc, qs, hv);
        if (h) memcpy(h + (size_t)r * I, hv, sizeof(double) * (size_t)I);
        #pragma omp parallel for schedule(static)
        for (int o = 0; o < H; o++) {
            y[(size_t)r * H + o] = mx_row_dot(cd, sd, (size_t)o, I, hv);
        }
    }
    free(hv);
    free(qc);
    free(qs);
}

/* ------------------------------------------------- MXFP8 rounding ambiguity
 * Test support for the tensor-core prefill path.  There h is computed in fp32, so
 * the oracle knows the GPU's h_i only to within an error radius r_i (orc_h_radius),
 * and an MXFP8 decision that falls inside that radius may go either way: the
 * element may round to either E4M3 neighbour, and a block whose max |h| sits near a
 * power of two may take either shared exponent.  Both sides apply the same OCP
 * rule (orc_quant_mxfp8) to the value they hold. */

/* Shared exponent of a block with max |v| = amax (OCP MX v1.0: floor(log2 amax) - emax,
 * clamped to [-127, 127]; -127 for amax == 0), emax = 8 for E4M3, 2 for E2M1. */
static int mx_block_exp(double amax, int emax) {
    if (!(amax > 0.0)) return -127;
    int ex;
    frexp(amax, &ex);
    int X = (ex - 1) - emax;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    return X;
}

/* v quantised at shared exponent X and dequantised: E4M3 (fmt 8) or E2M1 (fmt 4). */
static double mx_at(double v, int X, int fmt) {
    if (fmt == 4) return ldexp(orc_e2m1_value(orc_e2m1_encode(ldexp(v, -X))), X);
    return ldexp(orc_e4m3_value(orc_e4m3_encode(ldexp(v, -X))), X);
}

/* delta[i] = the largest |alternative - nominal| of the MX value (fmt 8: MXFP8, 4:
 * MXFP4) of v[i] when each element of its 32-block may be anywhere in
 * [v - radius, v + radius]: every shared exponent a block max in its range can give
 * is tried, and at each exponent the quantised value is monotone in the element, so
 * its extremes over the interval are the quantised ends of the interval.  The
 * nominal value is that of orc_quant_mxfp8 / orc_quant_mxfp4. */
void orc_mx_ambiguity(const double *v, const double *radius, int n, int fmt, double *delta) {
    const int emax = fmt == 4 ? 2 : 8;
    for (int b0 = 0; b0 < n; b0 += 32) {
        int b1 = b0 + 32 < n ? b0 + 32 : n;
        double amax = 0.0, alo = 0.0, ahi = 0.0;
        for (int i = b0; i < b1; i++) {
            double a = fabs(v[i]), lo = a - radius[i] > 0.0 ? a - radius[i] : 0.0;
            if (a > amax) amax = a;
            if (lo > alo) alo = lo;
            if (a + radius[i] > ahi) ahi = a + radius[i];
        }
        int X = mx_block_exp(amax, emax), Xlo = mx_block_exp(alo, emax), Xhi = mx_block_exp(ahi, emax);
        for (int i = b0; i < b1; i++) {
            double q = mx_at(v[i], X, fmt), d = 0.0;
            for (int Xa = Xlo; Xa <= Xhi; Xa++) {
                double e1 = fabs(mx_at(v[i] - radius[i], Xa, fmt) - q);
                double e2 = fabs(mx_at(v[i] + radius[i], Xa, fmt) - q);
                if (e1 > d) d = e1;
                if (e2 > d) d = e2;
            }
            delta[i] = d;
        }
    }
}

void orc_mxfp8_ambiguity(const double *v, const double *radius, int n, double *delta) {
    orc_mx_ambiguity(v, radius, n, 8, delta);
}

/* Dot product as mx_row_dot, also returning sum_t (|P_{t-1}| + |S_t|) over the
 * 32-element blocks t in ascending K, with S_t the block's scaled sum and P_t the
 * running sum after it (P_0 = 0). */
static double mx_row_dot_steps(const uint8_t *codes, const uint8_t *scales, size_t row, int K, const double *v,
                               double *step_mag) {
    const uint8_t *c = codes + row * (size_t)(K / 2);
    const uint8_t *s = scales + row * (size_t)(K / 32);
    double acc = 0.0, sp = 0.0;
    for (int b = 0; b < K / 32; b++) {
        double sc = orc_e8m0_value(s[b]), part = 0.0;
        for (int j = 32 * b; j < 32 * b + 32; j++) {
            unsigned code = (j & 1) ? (c[j / 2] >> 4) : (c[j / 2] & 15);
            part += orc_e2m1_value(code) * v[j];
        }
        sp += fabs(acc) + fabs(sc * part);
        acc += sc * part;
    }
    *step_mag = sp;
    return acc;
}

/* h = silu(W_g x) * (W_u x) of one expert for rows x [n][H] (x already MXFP8-exact),
 * and the error radius of the fp32 h the tensor-core path computes, per element.
 * The error model:
 *  (1) each block-scaled MMA step of K = 32 (one E8M0 block of both operands) adds
 *      its block sum S_t, exact, to the fp32 accumulator P_{t-1} with an error of at
 *      most rel * (|P_{t-1}| + |S_t|) (rel = 2^-23, one fp32 ulp of the larger
 *      operand: covers round-to-nearest or truncation of the sum, and truncation of
 *      the smaller operand when it is aligned to the larger), so |g_gpu - g| <=
 *      dg = rel * sum_t (|P_{t-1}| + |S_t|), the steps taken in ascending K, the
 *      order the MMAs run in; likewise du;
 *  (2) silu(g) * u is then evaluated in fp32 with a fast exponential (whose
 *      documented error grows linearly in |g|) and a fast division: relative error
 *      at most (8 + 2|g|) 2^-23;
 *  so, with |silu'| <= 1.1,
 *      r = 1.1 dg (|u| + du) + |silu(g)| du + (8 + 2|g|) 2^-23 |h|.
 * h, radius [n][I]. */
void orc_h_radius(const uint8_t *codes, const uint8_t *scales, int H, int I, const double *x, int n, double rel,
                  double *h, double *radius) {
    const uint8_t *cg = codes, *cu = codes + (size_t)I * H / 2;
    const uint8_t *sg = scales, *su = scales + (size_t)I * H / 32;
    for (int r = 0; r < n; r++) {
        const double *xr = x + (size_t)r * H;
        #pragma omp parallel for schedule(static)
        for (int i = 0; i < I; i++) {
            double Pg, Pu;
            double g = mx_row_dot_steps(cg, sg, (size_t)i, H, xr, &Pg);
            double u = mx_row_dot_steps(cu, su, (size_t)i, H, xr, &Pu);
            /* the fp64 running sums stand in for the exact ones: 1e-9 of margin */
            double dg = rel * Pg * (1.0 + 1e-9), du = rel * Pu * (1.0 + 1e-9);
            double sg_ = silu(g), hv = sg_ * u;
            h[(size_t)r * I + i] = hv;
            radius[(size_t)r * I + i] =
                1.1 * dg * (fabs(u) + du) + fabs(sg_) * du + (8.0 + 2.0 * fabs(g)) * ldexp(1.0, -23) * fabs(hv);
        }
    }
}

/* Per output row o of one expert applied to the rows x [n][H] with MX-quantised h
 * (fmt 8: MXFP8, 4: MXFP4): yamb[o] = sum_i |W_d[o][i]| * delta_i, with delta from
 * orc_mx_ambiguity on the radii of orc_h_radius (step error `rel`): the largest
 * change of o that equally valid decisions on the GPU's h can make. */
void orc_expert_ambiguity(const uint8_t *codes, const uint8_t *scales, int H, int I,
                          const double *x, int n, double rel, int fmt, double *yamb) {
    const uint8_t *cd = codes + (size_t)I * H;
    const uint8_t *sd = scales + (size_t)I * H / 16;
    double *hv = (double *)malloc(sizeof(double) * (size_t)n * I);
    double *rd = (double *)malloc(sizeof(double) * (size_t)n * I);
    double *dl = (double *)malloc(sizeof(double) * (size_t)I);
    orc_h_radius(codes, scales, H, I, x, n, rel, hv, rd);
    for (int r = 0; r < n; r++) {
        orc_mx_ambiguity(hv + (size_t)r * I, rd + (size_t)r * I, I, fmt, dl);
        #pragma omp parallel for schedule(static)
        for (int o = 0; o < H; o++) {
            const uint8_t *c = cd + (size_t)o * (I / 2);
            const uint8_t *sc = sd + (size_t)o * (I / 32);
            double acc = 0.0;
            for (int i = 0; i < I; i++) {
                if (dl[i] == 0.0) continue;
                unsigned code = (i & 1) ? (c[i / 2] >> 4) : (c[i / 2] & 15);
                acc += fabs(orc_e2m1_value(code)) * orc_e8m0_value(sc[i / 32]) * dl[i];
            }
            yamb[(size_t)r * H + o] = acc;
        }
    }
    free(hv);
    free(rd);
    free(dl);
}

/* ------------------------------------------------------------- stacked-layer glue
 * Pre-scale of the MoE input (exact): x_hat = x * 2^-p with p = floor(log2(amax|x|)) - 2,
 * so amax|x_hat| lies in [4, 8).  amax == 0 gives p = 0.  Result rounded to bf16
 * (exact unless it falls below the bf16 normal range). */
int orc_prescale_exponent(const uint16_t *x, int H) {
    double amax = 0.0;
    for (int h = 0; h < H; h++) {
        double a = fabs(orc_bf16_value(x[h]));
        if (a > amax) amax = a;
    }
    if (amax == 0.0) return 0;
    int ex;
    frexp(amax, &ex);
    return (ex - 1) - 2;
}

void orc_prescale(const uint16_t *x, int H, uint16_t *out) {
    int p = orc_prescale_exponent(x, H);
    for (int h = 0; h < H; h++) out[h] = orc_bf16_round(ldexp(orc_bf16_value(x[h]), -p));
}

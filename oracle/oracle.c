/*
 * oracle.c -- plain, slow, obviously-correct CPU definition of the scaled FP8
 * cast.  TEST INFRASTRUCTURE ONLY: it is called by the test-suite, by the
 * smoke check and by the CPU-baseline leg of the benchmark, never by the
 * product path.  It shares no code, header, table or constant with the CUDA
 * library; it uses only integer bit manipulation and exact double arithmetic.
 *
 * Sources (the pages this restates, cited by page title and section):
 *  - "Mixed Precision FP16/BF16/FP8" (mind-map card): bit layouts 1+5+10,
 *    1+8+7, E4M3 max 448, E5M2 max 57344, FP16 max 65504, min normal 2^-14,
 *    min subnormal 2^-24.
 *  - "Practice c06/E3, worked solution": scale = largest power of two that
 *    keeps the window's largest |x| below the format's largest finite value
 *    with a margin; previous scale kept under a hysteresis rule.
 *  - "what actually breaks low precision training" ("What the measurements
 *    said"): MX blocks of 32 share a power of two given by the OCP formula,
 *    so the largest values of a block clip; one extra bit of exponent
 *    headroom removes the clipping.  ("First, catching myself"): signed zero.
 *
 * Readings adopted where the pages are silent:
 *  - sat-RNE: round to the nearest value of the format's grid, extended with
 *    unbounded exponent above the maximum; a tie goes to the even significand.
 *    A result beyond the maximum finite value (or an infinite input)
 *    saturates to sign|max and counts as clipped.  NaN -> sign|0x7F, never
 *    clipped.  Zeros and values rounding to zero keep their sign.
 *  - amax = max |x| over the tensor taken as an unsigned max of the fp32
 *    abs-bits (NaN > Inf > finite); any NaN makes amax the canonical NaN.
 *  - MX: E = floor(log2(block amax)) - emax_elem + headroom, clamped to
 *    [-127, 127]; zero block -> -127; a block holding NaN/Inf -> E8M0 0xFF and
 *    every element byte sign|0x7F.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

/* --------------------------------------------------------------------------
 * Generic minifloat description.  fmt 0 = OCP E4M3 (FN kind: no infinity,
 * only S.1111.111 is NaN), fmt 1 = OCP E5M2 (IEEE kind), fmt 2 = IEEE FP16
 * (IEEE kind; used only to pin the generic codec against a known format).
 * ------------------------------------------------------------------------ */
typedef struct {
    int ebits, mbits, bias;
    int ieee;        /* 1: all-ones exponent is Inf/NaN; 0: FN kind          */
    int emax;        /* unbiased exponent of the largest finite value        */
    uint32_t maxcode;/* code of the largest finite positive value            */
    uint32_t nancode;/* positive quiet NaN code used for NaN results         */
} mf_t;

static mf_t mf_of(int fmt) {
    mf_t f;
    if (fmt == 0) {          /* E4M3: 1+4+3, bias 7, max 1.110b x 2^8 = 448  */
        f.ebits = 4; f.mbits = 3; f.bias = 7; f.ieee = 0; f.emax = 8;
        f.maxcode = 0x7E; f.nancode = 0x7F;
    } else if (fmt == 1) {   /* E5M2: 1+5+2, bias 15, max 1.11b x 2^15       */
        f.ebits = 5; f.mbits = 2; f.bias = 15; f.ieee = 1; f.emax = 15;
        f.maxcode = 0x7B; f.nancode = 0x7F;
    } else {                 /* FP16: 1+5+10, bias 15, max (2-2^-10) 2^15    */
        f.ebits = 5; f.mbits = 10; f.bias = 15; f.ieee = 1; f.emax = 15;
        f.maxcode = 0x7BFF; f.nancode = 0x7E00;
    }
    return f;
}

static int code_bits(const mf_t* f) { return 1 + f->ebits + f->mbits; }

/* Decode a code to a double (exact: every value of these formats is a
 * double).  NaN codes give NaN, infinity codes give +-inf. */
double orc_decode(int fmt, uint32_t code) {
    mf_t f = mf_of(fmt);
    int nb = code_bits(&f);
    uint32_t s = (code >> (nb - 1)) & 1u;
    uint32_t ef = (code >> f.mbits) & ((1u << f.ebits) - 1u);
    uint32_t mfield = code & ((1u << f.mbits) - 1u);
    uint32_t eall = (1u << f.ebits) - 1u;
    double v;
    if (f.ieee && ef == eall) {
        v = (mfield == 0) ? INFINITY : NAN;
    } else if (!f.ieee && ef == eall && mfield == ((1u << f.mbits) - 1u)) {
        v = NAN;
    } else if (ef == 0) {
        v = ldexp((double)mfield, 1 - f.bias - f.mbits);           /* subnormal */
    } else {
        v = ldexp((double)((1u << f.mbits) + mfield), (int)ef - f.bias - f.mbits);
    }
    return s ? -v : v;
}

/* Encode the exact value (-1)^sign * sig * 2^x (sig a non-negative integer)
 * with round-to-nearest-even on the grid extended above the maximum, then
 * saturate.  *clipped is set to 1 when saturation changed the result. */
static uint32_t encode_exact(const mf_t* f, int sign, uint64_t sig, int x, int* clipped) {
    int nb = code_bits(f);
    uint32_t sbit = sign ? (1u << (nb - 1)) : 0u;
    *clipped = 0;
    if (sig == 0) return sbit;                      /* signed zero            */
    int L = 63;                                     /* index of sig's top bit */
    while (((sig >> L) & 1u) == 0) L--;
    int k = L + x;                                  /* floor(log2 |value|)    */
    int emin = 1 - f->bias;                         /* smallest normal exp.   */
    int qe = (k < emin ? emin : k) - f->mbits;      /* grid spacing exponent  */
    /* n = round_half_even(value / 2^qe) */
    int shift = x - qe;
    uint64_t n;
    if (shift >= 0) {
        n = sig << shift;                           /* exact, n < 2^(mbits+1) */
    } else {
        int r = -shift;
        if (r > 64) {
            n = 0;                                  /* value < half a step    */
        } else {
            uint64_t q = (r == 64) ? 0 : (sig >> r);
            uint64_t rem = (r == 64) ? sig : (sig & ((1ull << r) - 1ull));
            uint64_t half = 1ull << (r - 1);
            n = q;
            if (rem > half || (rem == half && (q & 1u))) n = q + 1;
        }
    }
    /* overflow: the rounded magnitude n*2^qe exceeds the largest finite value.
     * If k > emax the magnitude is at least 2^(emax+1) > max; if k == emax it
     * overflows when n is above the largest finite significand. */
    uint32_t maxn = (f->maxcode & ((1u << f->mbits) - 1u)) + (1u << f->mbits);
    if (k > f->emax || (k == f->emax && n > maxn)) {
        *clipped = 1;
        return sbit | f->maxcode;
    }
    if (n == 0) return sbit;                        /* rounded to zero        */
    if (n == (1ull << (f->mbits + 1))) { n >>= 1; qe += 1; }   /* carry      */
    if (n < (1ull << f->mbits)) return sbit | (uint32_t)n;      /* subnormal */
    uint32_t ef = (uint32_t)(qe + f->mbits + f->bias);
    uint32_t mant = (uint32_t)(n - (1ull << f->mbits));
    return sbit | (ef << f->mbits) | mant;
}

/* Encode a double exactly (used to pin the codec: sums and products of
 * format values, FP16 against numpy).  Infinity saturates and clips, NaN maps
 * to sign|NaN code. */
uint32_t orc_encode_double(int fmt, double v, int* clipped) {
    mf_t f = mf_of(fmt);
    uint64_t b;
    memcpy(&b, &v, 8);
    int s = (int)(b >> 63);
    uint32_t ef = (uint32_t)((b >> 52) & 0x7FFu);
    uint64_t mfield = b & ((1ull << 52) - 1ull);
    int nb = code_bits(&f);
    *clipped = 0;
    if (ef == 0x7FF) {
        if (mfield) return (s ? (1u << (nb - 1)) : 0u) | f.nancode;
        *clipped = 1;
        return (s ? (1u << (nb - 1)) : 0u) | f.maxcode;
    }
    if (ef == 0) return encode_exact(&f, s, mfield, -1074, clipped);
    return encode_exact(&f, s, mfield | (1ull << 52), (int)ef - 1075, clipped);
}

/* Cast one fp32 value (given by its bits) multiplied by 2^e. */
static uint32_t cast_f32_bits(const mf_t* f, uint32_t xb, int e, int* clipped) {
    int s = (int)(xb >> 31);
    uint32_t ef = (xb >> 23) & 0xFFu;
    uint32_t mfield = xb & 0x7FFFFFu;
    uint32_t sbit = s ? (1u << (code_bits(f) - 1)) : 0u;
    *clipped = 0;
    if (ef == 0xFF) {
        if (mfield) return sbit | f->nancode;                       /* NaN   */
        *clipped = 1;                                               /* +-Inf */
        return sbit | f->maxcode;
    }
    if (ef == 0) return encode_exact(f, s, mfield, -149 + e, clipped);
    return encode_exact(f, s, mfield | 0x800000u, (int)ef - 150 + e, clipped);
}

uint32_t orc_cast_scalar(int fmt, uint32_t xbits, int e, int* clipped) {
    mf_t f = mf_of(fmt);
    return cast_f32_bits(&f, xbits, e, clipped);
}

/* dtype 0 = fp32 (elements are uint32 bit patterns), 1 = bf16 (uint16 bit
 * patterns; a bf16 is the upper half of the fp32 with the same value). */
static inline uint32_t load_bits(const void* x, int dtype, int64_t i) {
    if (dtype == 0) return ((const uint32_t*)x)[i];
    return ((uint32_t)((const uint16_t*)x)[i]) << 16;
}

static inline uint32_t canon_amax(uint32_t a) {
    return a > 0x7F800000u ? 0x7FC00000u : a;
}

#define ORC_CHUNK 65536

/* amax = max |x| as abs-bits (see header).  Returns fp32 bits. */
uint32_t orc_amax(const void* x, int dtype, int64_t n, int nthreads) {
    int64_t nchunks = (n + ORC_CHUNK - 1) / ORC_CHUNK;
    uint32_t best = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static) reduction(max : best)
    for (int64_t c = 0; c < nchunks; c++) {
        int64_t lo = c * ORC_CHUNK, hi = lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n;
        for (int64_t i = lo; i < hi; i++) {
            uint32_t a = load_bits(x, dtype, i) & 0x7FFFFFFFu;
            if (a > best) best = a;
        }
    }
    return canon_amax(best);
}

/* Per-tensor cast of n elements with scale 2^e.  Writes q[n]; returns the
 * number of clipped elements; *amax_bits receives the tensor's amax. */
int64_t orc_cast(const void* x, int dtype, int64_t n, int fmt, int e,
                 uint8_t* q, uint32_t* amax_bits, int nthreads) {
    mf_t f = mf_of(fmt);
    int64_t nchunks = (n + ORC_CHUNK - 1) / ORC_CHUNK;
    int64_t clipped = 0;
    uint32_t best = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static) reduction(+ : clipped) reduction(max : best)
    for (int64_t c = 0; c < nchunks; c++) {
        int64_t lo = c * ORC_CHUNK, hi = lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n;
        for (int64_t i = lo; i < hi; i++) {
            uint32_t xb = load_bits(x, dtype, i);
            uint32_t a = xb & 0x7FFFFFFFu;
            if (a > best) best = a;
            int cl;
            q[i] = (uint8_t)cast_f32_bits(&f, xb, e, &cl);
            clipped += cl;
        }
    }
    if (amax_bits) *amax_bits = canon_amax(best);
    return clipped;
}

/* Cast only the elements at positions idx[0..m): q[j] and clip[j] (0/1). */
void orc_cast_at(const void* x, int dtype, const int64_t* idx, int64_t m, int fmt,
                 int e, uint8_t* q, uint8_t* clip) {
    mf_t f = mf_of(fmt);
    for (int64_t j = 0; j < m; j++) {
        int cl;
        q[j] = (uint8_t)cast_f32_bits(&f, load_bits(x, dtype, idx[j]), e, &cl);
        clip[j] = (uint8_t)cl;
    }
}

/* Scale exponent rule, written as its definition: the largest integer e in
 * [-126, 126] with 2^e * A <= fmax * 2^-margin, found by trying every e from
 * the top.  A*2^e and fmax*2^-m are exact in double for every fp32 A and
 * every e here.  If none qualifies the bottom of the range is returned.
 * *ok = 0 (and 0 is returned) when A is zero or not finite: the caller then
 * keeps its previous exponent. */
int orc_scale_exp(uint32_t amax_bits, int fmt, int margin, int* ok) {
    mf_t f = mf_of(fmt);
    uint32_t a = amax_bits & 0x7FFFFFFFu;
    if (a == 0 || a >= 0x7F800000u) { *ok = 0; return 0; }
    *ok = 1;
    float af;
    memcpy(&af, &a, 4);
    double fmax = orc_decode(fmt, f.maxcode);
    double limit = ldexp(fmax, -margin);
    for (int e = 126; e >= -126; e--)
        if (ldexp((double)af, e) <= limit) return e;
    return -126;
}

/* MX shared exponent of one block from its amax bits (see header). */
int orc_mx_exp(uint32_t amax_bits, int fmt, int headroom) {
    mf_t f = mf_of(fmt);
    uint32_t a = amax_bits & 0x7FFFFFFFu;
    if (a == 0) return -127;
    float af;
    memcpy(&af, &a, 4);
    int p;
    frexp((double)af, &p);                /* af = m * 2^p, m in [0.5, 1)     */
    int E = (p - 1) - f.emax + headroom;   /* floor(log2 af) = p - 1          */
    if (E < -127) E = -127;
    if (E > 127) E = 127;
    return E;
}

/* MX cast of a row-major [rows, cols] tensor, 32-element blocks along the
 * last dimension.  q: [rows, cols]; e8m0: [rows, cols/32].  Returns the
 * clipped count. */
int64_t orc_mx_cast(const void* x, int dtype, int64_t rows, int64_t cols, int fmt,
                    int headroom, uint8_t* q, uint8_t* e8m0, int nthreads) {
    mf_t f = mf_of(fmt);
    int64_t nblocks = rows * (cols / 32);
    int64_t clipped = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static, 2048) reduction(+ : clipped)
    for (int64_t b = 0; b < nblocks; b++) {
        int64_t base = b * 32;
        uint32_t amax = 0;
        for (int j = 0; j < 32; j++) {
            uint32_t a = load_bits(x, dtype, base + j) & 0x7FFFFFFFu;
            if (a > amax) amax = a;
        }
        if (amax >= 0x7F800000u) {                    /* NaN or Inf in block */
            e8m0[b] = 0xFF;
            for (int j = 0; j < 32; j++)
                q[base + j] = (uint8_t)(((load_bits(x, dtype, base + j) >> 31) << 7) | 0x7Fu);
            continue;
        }
        int E = orc_mx_exp(amax, fmt, headroom);
        e8m0[b] = (uint8_t)(E + 127);
        for (int j = 0; j < 32; j++) {
            int cl;
            q[base + j] = (uint8_t)cast_f32_bits(&f, load_bits(x, dtype, base + j), -E, &cl);
            clipped += cl;
        }
    }
    return clipped;
}

static inline double bits_to_double(uint32_t b) {
    float v;
    memcpy(&v, &b, 4);
    return (double)v;
}

/* Error statistics of a per-tensor cast: deq = decode(q) * 2^-e; over the
 * elements whose input is finite, out[0] = mean((deq-x)^2), out[1] =
 * mean(deq-x), out[2] = number of such elements.  Partial sums are kept per
 * fixed chunk and added in chunk order. */
void orc_stats(const void* x, int dtype, int64_t n, const uint8_t* q, int fmt, int e,
               double* out, int nthreads) {
    int64_t nchunks = (n + ORC_CHUNK - 1) / ORC_CHUNK;
    double sq = 0, sm = 0;
    int64_t cnt = 0;
    double scale_inv = ldexp(1.0, -e);
    if (nthreads < 1) nthreads = 1;
    for (int64_t c0 = 0; c0 < nchunks; c0 += 4096) {
        int64_t c1 = c0 + 4096 < nchunks ? c0 + 4096 : nchunks;
        double psq[4096], psm[4096];
        int64_t pc[4096];
#pragma omp parallel for num_threads(nthreads) schedule(static)
        for (int64_t c = c0; c < c1; c++) {
            int64_t lo = c * ORC_CHUNK, hi = lo + ORC_CHUNK < n ? lo + ORC_CHUNK : n;
            double a2 = 0, a1 = 0;
            int64_t k = 0;
            for (int64_t i = lo; i < hi; i++) {
                uint32_t xb = load_bits(x, dtype, i);
                if ((xb & 0x7FFFFFFFu) >= 0x7F800000u) continue;
                double d = orc_decode(fmt, q[i]) * scale_inv - bits_to_double(xb);
                a2 += d * d;
                a1 += d;
                k++;
            }
            psq[c - c0] = a2; psm[c - c0] = a1; pc[c - c0] = k;
        }
        for (int64_t c = c0; c < c1; c++) { sq += psq[c - c0]; sm += psm[c - c0]; cnt += pc[c - c0]; }
    }
    out[0] = cnt ? sq / (double)cnt : 0.0;
    out[1] = cnt ? sm / (double)cnt : 0.0;
    out[2] = (double)cnt;
}

/* Error statistics of an MX cast: deq = decode(q) * 2^E per block; blocks
 * whose E8M0 byte is the NaN code 0xFF are skipped. */
void orc_mx_stats(const void* x, int dtype, int64_t rows, int64_t cols, const uint8_t* q,
                  const uint8_t* e8m0, int fmt, double* out, int nthreads) {
    int64_t nblocks = rows * (cols / 32);
    int64_t per = ORC_CHUNK / 32;
    int64_t nchunks = (nblocks + per - 1) / per;
    double sq = 0, sm = 0;
    int64_t cnt = 0;
    if (nthreads < 1) nthreads = 1;
    for (int64_t c0 = 0; c0 < nchunks; c0 += 4096) {
        int64_t c1 = c0 + 4096 < nchunks ? c0 + 4096 : nchunks;
        double psq[4096], psm[4096];
        int64_t pc[4096];
#pragma omp parallel for num_threads(nthreads) schedule(static)
        for (int64_t c = c0; c < c1; c++) {
            int64_t lo = c * per, hi = lo + per < nblocks ? lo + per : nblocks;
            double a2 = 0, a1 = 0;
            int64_t k = 0;
            for (int64_t b = lo; b < hi; b++) {
                if (e8m0[b] == 0xFF) continue;
                double s = ldexp(1.0, (int)e8m0[b] - 127);
                for (int j = 0; j < 32; j++) {
                    uint32_t xb = load_bits(x, dtype, b * 32 + j);
                    double d = orc_decode(fmt, q[b * 32 + j]) * s - bits_to_double(xb);
                    a2 += d * d;
                    a1 += d;
                    k++;
                }
            }
            psq[c - c0] = a2; psm[c - c0] = a1; pc[c - c0] = k;
        }
        for (int64_t c = c0; c < c1; c++) { sq += psq[c - c0]; sm += psm[c - c0]; cnt += pc[c - c0]; }
    }
    out[0] = cnt ? sq / (double)cnt : 0.0;
    out[1] = cnt ? sm / (double)cnt : 0.0;
    out[2] = (double)cnt;
}

/* --------------------------------------------------------------------------
 * MX scale-rounding rules and block direction.
 *
 * "what actually breaks low precision training" ("The part I would rather not
 * write"): NVIDIA's MXFP8 pre-training recipe rounds the shared scale up
 * instead of using the specification's floor, and a 2025 study compares
 * floor, ceil and nearest rounding of the scale.  Readings adopted:
 *   rule 0  OCP floor: E = floor(log2 A) - emax_elem
 *   rule 1  ceil: the smallest integer E with A * 2^-E <= fmax (the scaled
 *           block max never exceeds the format maximum)
 *   rule 2  nearest: the integer E nearest to log2(A / fmax) (no ties: the
 *           half-way point would need A / fmax = 2^k * sqrt 2)
 * then E += headroom and E is clamped to [-127, 127]; a zero block gets -127.
 * axis 0: blocks of 32 consecutive elements of a row (e8m0 [rows, cols/32]);
 * axis 1: blocks of 32 consecutive rows of a column (e8m0 [rows/32, cols]).
 * ------------------------------------------------------------------------ */
int orc_mx_exp_rule(uint32_t amax_bits, int fmt, int rule, int headroom) {
    if (rule == 0) return orc_mx_exp(amax_bits, fmt, headroom);
    mf_t f = mf_of(fmt);
    uint32_t a = amax_bits & 0x7FFFFFFFu;
    if (a == 0) return -127;
    float af;
    memcpy(&af, &a, 4);
    double A = (double)af;
    double fmax = orc_decode(fmt, f.maxcode);
    int E0 = -400;                       /* smallest E with A * 2^-E <= fmax */
    for (int e = -200; e <= 200; e++)
        if (ldexp(A, -e) <= fmax) { E0 = e; break; }
    int E = E0;
    if (rule == 2) {
        /* E0 puts the scaled max in (fmax/2, fmax], E0 - 1 in (fmax, 2 fmax];
         * keep E0 when its log distance is the smaller one:
         * fmax / (A 2^-E0) <= (A 2^-(E0-1)) / fmax  <=>  fmax^2 2^(2 E0 - 1) <= A^2
         * (both sides exact in double: 18- and 48-bit significands). */
        if (!(fmax * fmax * ldexp(1.0, 2 * E0 - 1) <= A * A)) E = E0 - 1;
    }
    E += headroom;
    if (E < -127) E = -127;
    if (E > 127) E = 127;
    return E;
}

int64_t orc_mx_cast_ex(const void* x, int dtype, int64_t rows, int64_t cols, int fmt, int rule,
                       int headroom, int axis, uint8_t* q, uint8_t* e8m0, int nthreads) {
    mf_t f = mf_of(fmt);
    int64_t nblocks = rows * cols / 32;
    int64_t clipped = 0;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static, 2048) reduction(+ : clipped)
    for (int64_t b = 0; b < nblocks; b++) {
        /* element j of block b sits at idx(b, j) */
        int64_t r0, c0, step;
        if (axis == 0) { r0 = b / (cols / 32); c0 = (b % (cols / 32)) * 32; step = 1; }
        else { r0 = (b / cols) * 32; c0 = b % cols; step = cols; }
        int64_t base = r0 * cols + c0;
        uint32_t amax = 0;
        for (int j = 0; j < 32; j++) {
            uint32_t a = load_bits(x, dtype, base + j * step) & 0x7FFFFFFFu;
            if (a > amax) amax = a;
        }
        if (amax >= 0x7F800000u) {
            e8m0[b] = 0xFF;
            for (int j = 0; j < 32; j++)
                q[base + j * step] =
                    (uint8_t)(((load_bits(x, dtype, base + j * step) >> 31) << 7) | 0x7Fu);
            continue;
        }
        int E = orc_mx_exp_rule(amax, fmt, rule, headroom);
        e8m0[b] = (uint8_t)(E + 127);
        for (int j = 0; j < 32; j++) {
            int cl;
            q[base + j * step] = (uint8_t)cast_f32_bits(&f, load_bits(x, dtype, base + j * step), -E, &cl);
            clipped += cl;
        }
    }
    return clipped;
}

/* --------------------------------------------------------------------------
 * Counts that drive dynamic loss scaling ("Mixed Precision FP16/BF16/FP8":
 * on Inf/NaN halve the loss scale and skip the step) and the underflow rate
 * ("what actually breaks low precision training", "What the measurements
 * said": clip rates and underflow rates).  Readings: an element is
 * non-finite when the input is NaN or +-Inf; it underflowed when the input is
 * finite and nonzero and its 8-bit result is a zero (+0 or -0).
 * ------------------------------------------------------------------------ */
void orc_count_special(const void* x, int dtype, int64_t n, const uint8_t* q,
                       int64_t* nonfinite, int64_t* underflow) {
    int64_t nf = 0, uf = 0;
    for (int64_t i = 0; i < n; i++) {
        uint32_t a = load_bits(x, dtype, i) & 0x7FFFFFFFu;
        if (a >= 0x7F800000u) nf++;
        else if (a != 0 && (q[i] & 0x7Fu) == 0) uf++;
    }
    *nonfinite = nf;
    *underflow = uf;
}


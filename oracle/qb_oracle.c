/*
 * qb_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar CPU statement of what the block-quantized weight x
 * quantized activation product computes.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load it; the library's product path
 * never does.  It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (the decode engine's documentation pages):
 *   numerics page  -- the decode engine's numerics module page:
 *                     ActScaling::PerBlock, absmax, wide_scale, rne_div,
 *                     quantize_blocks, exact_sum, scaled_to_f32, dot, fdot,
 *                     tree, f32_to_f16, ftz, structs Scale / Segment /
 *                     CodedRow / Unreadable, constants NAN, COEF_BOUND.
 *   lane page       -- its lane module page: block_sums, deliver, lane, and
 *                     the excess-form identity of the unit sums; group and
 *                     deliver32 for ActScaling::Sub32 (block_scale,
 *                     quantize, ACT_BLOCK = 32, GROUP = 256 on the
 *                     numerics page).  The int8 cache's score path:
 *                     cache_row, int8_codes, INV_127, quantize_head and
 *                     int8_score on the numerics page.
 *   colizig OPS page -- FP8: e4m3ToF32, dequantRow, matmulFp8 (E4M3 weights
 *                     with 128x128 block scales; a float path checked there
 *                     against "dequantize then f32 matmul").
 *
 * Readings taken where the pages are silent (each restated where used):
 *   R1  an activation block whose largest magnitude is 0 gets the scale
 *       128*2^0 and all-zero codes (wide_scale is defined for amax > 0 only);
 *   R2  a denormal activation element is read as zero for the codes as well
 *       as for absmax;  a NaN element gets code 0;
 *   R3  an activation block holding an infinity has no scale: it is marked
 *       m = 0 and every row's dot with it is the engine's NaN;
 *   R4  SUM_WINDOW never binds: the two terms of a block are summed exactly
 *       (they fit a 128-bit integer for every finite f16 scale);
 *   R5  rounding to f32 happens on the f32 grid including its subnormal
 *       quantum 2^-149, and a subnormal result is then flushed to a zero of
 *       its sign;
 *   R6  LANES = 8 and the tree is ((l0+l1)+(l2+l3))+((l4+l5)+(l6+l7));
 *   R7  a row with any unreadable block (f16 scale inf or NaN) is NAN.
 *   R13 (Sub32) an all-zero activation block gets the scale 8*2^0 and zero
 *       codes, a block holding an infinity m = 0 (as R1, R3 for PerBlock);
 *   R14 (Sub32) SUM_WINDOW never binds here either: a group's terms are
 *       summed exactly, whatever the spread of their exponents (a 384-bit
 *       integer holds every case), then rounded once as in R5.
 *   R15 (Sub32) a group whose nonzero terms lie 318 or more places above
 *       the least exponent of its terms is NAN (never for block_scale
 *       scales with f16 weight scales; only a caller's out-of-range e).
 *   R17 (int8 cache) the reciprocal under which a cache row's codes are
 *       taken is the f32 quotient 1/s, correctly rounded (the page's recip
 *       seeds Newton steps from a table it does not print).
 *   R19 (FP8) matmulFp8 is read as the page's own check: each weight the f32
 *       product of its decoded byte and its block scale, the dot exact (a
 *       640-bit integer), rounded once to nearest even, subnormals kept; a
 *       GPU result is held to the f32 summation bound
 *       (K + 4) * 2^-24 * sum |x_i * w_i| around it.
 *   R20 (two-word codes) a code crossing in two words is the 16-bit integer
 *       256*hi + lo (hi the signed high byte, lo the unsigned low byte);
 *       its block sums, combine, rounding and fold are PerBlock's.
 *   R18 (int8 cache) a score against a key row whose f16 scale is infinite
 *       or NaN (a row whose amax*INV_127 overflows binary16) is NAN, as an
 *       unreadable weight scale is (R7); a query block without a scale too.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * Contraction must stay off: the f32 rule multiplies and adds separately.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef __int128 i128;
typedef unsigned __int128 u128;

#define OR_F16 1
#define OR_Q8_0 8
#define OR_Q4K 12
#define OR_Q6K 14

/* the engine's one NaN: quiet, no payload, no sign (numerics page, NAN) */
static float engine_nan(void) {
    uint32_t b = 0x7FC00000u;
    float f;
    memcpy(&f, &b, 4);
    return f;
}

static uint32_t f32_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }
static float bits_f32(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }

/* ftz: a denormal flushed to a zero of its sign (numerics page, ftz) */
float or_ftz(float x) {
    if (x != 0.0f && fabsf(x) < 1.17549435e-38f) return copysignf(0.0f, x);
    return x;
}

/* ---------------------------------------------------------------------
 * Scale: a stored f16 scale is sig*2^exp exactly (numerics page, struct
 * Scale; Unreadable for an infinite or NaN scale).  Returns -1 if unreadable.
 * ------------------------------------------------------------------- */
int or_f16_scale(uint16_t h, int64_t *sig, int *ex) {
    int E = (h >> 10) & 31, f = h & 1023;
    if (E == 31) return -1;
    if (E == 0) { *sig = f; *ex = -24; }          /* subnormal: f * 2^-24 */
    else { *sig = 1024 + f; *ex = E - 25; }       /* (1024+f) * 2^(E-25) */
    if (h & 0x8000) *sig = -*sig;
    return 0;
}

/* ---------------------------------------------------------------------
 * absmax: the largest magnitude, a denormal read as zero, folded from +0,
 * a NaN passed over (numerics page, absmax).  Infinity is kept.
 * ------------------------------------------------------------------- */
float or_absmax(const float *x, int n) {
    float a = 0.0f;
    for (int i = 0; i < n; i++) {
        float v = fabsf(x[i]);
        if (isnan(v)) continue;
        if (v < 1.17549435e-38f) v = 0.0f;
        if (v > a) a = v;
    }
    return a;
}

/* a finite normal f32 as X * 2^E with X a signed integer (|X| < 2^24) */
static void f32_split(float x, int64_t *X, int *E) {
    uint32_t b = f32_bits(x);
    int e8 = (b >> 23) & 0xFF;
    int64_t m = (int64_t)((b & 0x7FFFFF) | 0x800000);
    *X = (b >> 31) ? -m : m;
    *E = e8 - 150;
}

/* ---------------------------------------------------------------------
 * wide_scale: the least m*2^e, m in 128..255, with 127*m*2^e >= amax, for a
 * finite positive amax (numerics page, wide_scale; WIDE_BITS = 8).
 * Stated as a search: for every exponent e near amax's, the least m that
 * satisfies the bound is ceil(amax / (127*2^e)); keep the candidates with m
 * in range and return the smallest value.
 * ------------------------------------------------------------------- */
void or_wide_scale(float amax, int *m_out, int *e_out) {
    int64_t M; int E;
    f32_split(amax, &M, &E);                       /* amax = M * 2^E, M > 0 */
    int best_m = 0, best_e = 0;
    for (int j = -40; j <= 40; j++) {              /* e = E + j */
        /* m = ceil(M * 2^E / (127 * 2^(E+j))) = ceil(M / (127 * 2^j)) */
        u128 num = (u128)M, den = 127;
        if (j >= 0) den <<= j; else num <<= -j;
        u128 mm = (num + den - 1) / den;
        if (mm < 128 || mm > 255) continue;
        int e = E + j;
        if (best_m == 0) { best_m = (int)mm; best_e = e; continue; }
        /* compare mm*2^e with best_m*2^best_e exactly */
        int lo = e < best_e ? e : best_e;
        u128 a = (u128)mm << (e - lo), b = (u128)best_m << (best_e - lo);
        if (a < b) { best_m = (int)mm; best_e = e; }
    }
    *m_out = best_m;
    *e_out = best_e;
}

/* round-to-nearest-even division of a non-negative num by a positive den */
static u128 rne_udiv(u128 num, u128 den) {
    u128 q = num / den, r = num - q * den;
    if (2 * r > den || (2 * r == den && (q & 1))) q += 1;
    return q;
}

/* ---------------------------------------------------------------------
 * rne_div: the nearest integer to x / (m*2^e), ties to even, exactly
 * (numerics page, rne_div).  A denormal or NaN x gives 0 (readings R2).
 * ------------------------------------------------------------------- */
int or_rne_div(float x, int m, int e) {
    if (isnan(x) || fabsf(x) < 1.17549435e-38f) return 0;
    int64_t X; int Ex;
    f32_split(x, &X, &Ex);
    int neg = X < 0;
    u128 ax = (u128)(neg ? -X : X);
    int sh = Ex - e;                                /* x/s = X * 2^sh / m */
    u128 num, den;
    if (sh >= 0) {
        if (sh > 60) return neg ? -0x7FFFFFFF : 0x7FFFFFFF; /* cannot occur for |x| <= 127*s */
        num = ax << sh; den = (u128)m;
    } else {
        if (-sh > 100) return 0;                    /* |x/s| < 2^-60: nearest integer 0 */
        num = ax; den = (u128)m << (-sh);
    }
    int64_t q = (int64_t)rne_udiv(num, den);
    return (int)(neg ? -q : q);
}

/* ---------------------------------------------------------------------
 * quantize_blocks: x (a whole number of blocks) quantized per weight block of
 * `block` elements under m*2^e, m in 128..255 (numerics page, quantize_blocks,
 * ActScaling::PerBlock).  Also the per-16-element unit sums of the codes, the
 * activation side's S of the lane page.  Codes and scales are laid out
 * [ncols][K] and [ncols][K/block]; m=0 marks a block holding an infinity (R3).
 * ------------------------------------------------------------------- */
void or_quantize_blocks(const float *x, int64_t K, int ncols, int block,
                        int8_t *codes, uint8_t *m_out, int16_t *e_out, int16_t *sums16) {
    int64_t nb = K / block;
    for (int c = 0; c < ncols; c++) {
        for (int64_t b = 0; b < nb; b++) {
            const float *xb = x + (int64_t)c * K + b * block;
            int8_t *cb = codes + (int64_t)c * K + b * block;
            float amax = or_absmax(xb, block);
            int m, e;
            if (isinf(amax)) { m = 0; e = 0; }             /* R3 */
            else if (amax == 0.0f) { m = 128; e = 0; }     /* R1 */
            else or_wide_scale(amax, &m, &e);
            for (int i = 0; i < block; i++) {
                int q = (m == 0) ? 0 : or_rne_div(xb[i], m, e);
                cb[i] = (int8_t)q;
            }
            m_out[(int64_t)c * nb + b] = (uint8_t)m;
            e_out[(int64_t)c * nb + b] = (int16_t)e;
        }
        for (int64_t u = 0; u < K / 16; u++) {
            int s = 0;
            for (int i = 0; i < 16; i++) s += codes[(int64_t)c * K + u * 16 + i];
            sums16[(int64_t)c * (K / 16) + u] = (int16_t)s;
        }
    }
}

/* ---------------------------------------------------------------------
 * scaled_to_f32: v*2^ex rounded once to f32, to nearest with ties to even,
 * a denormal flushed to a zero of its sign (numerics page, scaled_to_f32);
 * past the top infinite (numerics page, ldexp).  Reading R5: the rounding is
 * on the f32 grid (quantum 2^(x-23) for a normal leading place x, 2^-149
 * below 2^-126), the flush after it.  An exact zero gives +0.
 * ------------------------------------------------------------------- */
float or_scaled_to_f32(i128 v, int ex) {
    if (v == 0) return 0.0f;
    int neg = v < 0;
    u128 a = neg ? (u128)(-v) : (u128)v;
    int p = 127;
    while (!((a >> p) & 1)) p--;                    /* leading place of a */
    int x = p + ex;                                 /* value in [2^x, 2^(x+1)) */
    int sub = x < -126;                             /* below the least normal f32 */
    int qe = sub ? -149 : x - 23;                   /* quantum of the f32 grid there */
    int shift = qe - ex;
    u128 r;
    if (shift <= 0) r = a << (-shift);
    else if (shift >= 128) r = 0;                   /* far below half a quantum */
    else r = rne_udiv(a, (u128)1 << shift);
    /* value = r * 2^qe, r <= 2^24 */
    if (sub && r < ((u128)1 << 23)) return neg ? -0.0f : 0.0f;       /* subnormal: flush */
    if (r == 0) return neg ? -0.0f : 0.0f;
    double d = ldexp((double)(uint64_t)r, qe);
    if (d >= 3.4028236692093846e38) return neg ? -INFINITY : INFINITY;  /* >= 2^128 */
    float f = (float)d;                             /* exact: representable */
    return neg ? -f : f;
}

/* ---------------------------------------------------------------------
 * Unpacking a row record into the logical coded row (CodedRow / Segment):
 * codes and their per-segment coefficients.  The byte layout is this
 * library's own (the pages fix none); see the synth module's docstring.
 * ------------------------------------------------------------------- */
static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

int64_t or_record_bytes(int fmt, int64_t K) {
    switch (fmt) {
    case OR_Q8_0: return (K + 2 * (K / 32) + 15) / 16 * 16;
    case OR_Q4K: return 144 * (K / 256);
    case OR_Q6K: return (210 * (K / 256) + 15) / 16 * 16;
    case OR_F16: return 2 * K;
    }
    return -1;
}

/* Q4_K-like: q[K] in 0..15, sc[K/32], mn[K/32] in 0..63, d/dmin bits [K/256] */
void or_unpack_q4k(const uint8_t *rec, int64_t K, uint8_t *q, uint8_t *sc, uint8_t *mn,
                   uint16_t *d, uint16_t *dmin) {
    for (int64_t b = 0; b < K / 256; b++) {
        const uint8_t *blk = rec + 144 * b;
        d[b] = rd16(blk);
        dmin[b] = rd16(blk + 2);
        uint64_t s48 = 0, m48 = 0;
        for (int i = 0; i < 6; i++) {
            s48 |= (uint64_t)blk[4 + i] << (8 * i);
            m48 |= (uint64_t)blk[10 + i] << (8 * i);
        }
        for (int s = 0; s < 8; s++) {
            sc[b * 8 + s] = (uint8_t)((s48 >> (6 * s)) & 63);
            mn[b * 8 + s] = (uint8_t)((m48 >> (6 * s)) & 63);
            for (int j = 0; j < 16; j++) {
                uint8_t byte = blk[16 + 16 * s + j];
                q[b * 256 + 32 * s + j] = byte & 15;
                q[b * 256 + 32 * s + 16 + j] = byte >> 4;
            }
        }
    }
}

/* Q6_K-like: q[K] in 0..63, sc[K/16] int8, d bits [K/256] */
void or_unpack_q6k(const uint8_t *rec, int64_t K, uint8_t *q, int8_t *sc, uint16_t *d) {
    int64_t nsb = K / 256;
    for (int64_t b = 0; b < nsb; b++) {
        const uint8_t *blk = rec + 208 * b;
        d[b] = rd16(rec + 208 * nsb + 2 * b);
        for (int u = 0; u < 16; u++) sc[b * 16 + u] = (int8_t)blk[192 + u];
        for (int c = 0; c < 8; c++) {
            for (int j = 0; j < 16; j++) {
                uint8_t byte = blk[16 * c + j];
                q[b * 256 + 32 * c + j] = byte & 15;
                q[b * 256 + 32 * c + 16 + j] = byte >> 4;
            }
            for (int half = 0; half < 2; half++) {
                for (int i = 0; i < 16; i++) {
                    int k = i / 4, bb = i % 4;
                    uint8_t hbyte = blk[128 + 8 * c + 4 * half + bb];
                    int hbits = (hbyte >> (2 * k)) & 3;
                    q[b * 256 + 32 * c + 16 * half + i] |= (uint8_t)(hbits << 4);
                }
            }
        }
    }
}

/* Q8_0: q[K] int8, d bits [K/32] */
void or_unpack_q8_0(const uint8_t *rec, int64_t K, int8_t *q, uint16_t *d) {
    for (int64_t i = 0; i < K; i++) q[i] = (int8_t)rec[i];
    for (int64_t b = 0; b < K / 32; b++) d[b] = rd16(rec + K + 2 * b);
}

/* one unpacked row: the logical coded row */
typedef struct {
    int fmt;
    int64_t K;
    uint8_t *q;      /* Q4_K / Q6_K codes (unsigned) */
    int8_t *q8;      /* Q8_0 codes */
    uint8_t *sc, *mn;/* Q4_K sub-block scales and offsets, per 32 */
    int8_t *sc6;     /* Q6_K sub-scales, per 16 */
    uint16_t *d, *dm;/* f16 bits of the block scales */
} or_row;

static int row_alloc(or_row *w, int fmt, int64_t K) {
    memset(w, 0, sizeof *w);
    w->fmt = fmt; w->K = K;
    w->q = malloc((size_t)K); w->q8 = malloc((size_t)K);
    w->sc = malloc((size_t)(K / 32 + 1)); w->mn = malloc((size_t)(K / 32 + 1));
    w->sc6 = malloc((size_t)(K / 16 + 1));
    w->d = malloc(2 * (size_t)(K / 32 + 1)); w->dm = malloc(2 * (size_t)(K / 32 + 1));
    return (w->q && w->q8 && w->sc && w->mn && w->sc6 && w->d && w->dm) ? 0 : -1;
}
static void row_free(or_row *w) {
    free(w->q); free(w->q8); free(w->sc); free(w->mn); free(w->sc6); free(w->d); free(w->dm);
}
static int row_unpack(or_row *w, const uint8_t *rec) {
    if (w->fmt == OR_Q8_0) or_unpack_q8_0(rec, w->K, w->q8, w->d);
    else if (w->fmt == OR_Q4K) or_unpack_q4k(rec, w->K, w->q, w->sc, w->mn, w->d, w->dm);
    else if (w->fmt == OR_Q6K) or_unpack_q6k(rec, w->K, w->q, w->sc6, w->d);
    else return -1;
    return 0;
}
static int fmt_block(int fmt) { return fmt == OR_Q8_0 ? 32 : 256; }

/* ---------------------------------------------------------------------
 * block_sums: a block's two exact sums, sum coef*a and sum offs*a, taken
 * element by element (lane page, block_sums; numerics page, struct Segment:
 * the coefficients are the codes times their sub-block scales, the offsets
 * the offset terms).  Q8_0: coef = q.  Q4_K-like: coef = sc*q, offs = mn,
 * second scale -dmin.  Q6_K-like: coef = sc*(q-32), no offsets.
 * ------------------------------------------------------------------- */
typedef struct {
    int64_t C, O;
    uint16_t s1, s2;  /* f16 bits of the first and second scale */
    int kind;         /* 0: one scale; 1: second scale enters as -s2 */
} or_block;

static void block_sums(const or_row *w, int64_t b, const int8_t *a, or_block *ob) {
    ob->C = 0; ob->O = 0; ob->kind = 0; ob->s2 = 0;
    if (w->fmt == OR_Q8_0) {
        for (int i = 0; i < 32; i++) ob->C += (int64_t)w->q8[b * 32 + i] * a[b * 32 + i];
        ob->s1 = w->d[b];
    } else if (w->fmt == OR_Q4K) {
        for (int i = 0; i < 256; i++) {
            int64_t e = b * 256 + i;
            int s = i / 32;
            int64_t coef = (int64_t)w->sc[b * 8 + s] * w->q[e];
            int64_t offs = w->mn[b * 8 + s];
            ob->C += coef * a[e];
            ob->O += offs * a[e];
        }
        ob->s1 = w->d[b]; ob->s2 = w->dm[b]; ob->kind = 1;
    } else {
        for (int i = 0; i < 256; i++) {
            int64_t e = b * 256 + i;
            int u = i / 16;
            int64_t coef = (int64_t)w->sc6[b * 16 + u] * ((int64_t)w->q[e] - 32);
            ob->C += coef * a[e];
        }
        ob->s1 = w->d[b];
    }
}

/* ---------------------------------------------------------------------
 * lane: the block's value -- its scale times the coefficient sum plus its
 * second scale times the offset sum, both times the activation scale m*2^e,
 * summed exactly and rounded once (lane page, lane; numerics page, exact_sum,
 * scaled_to_f32, ActScaling::PerBlock).  NaN for an unreadable block (R3, R7).
 * kind 0: one scale; kind 1: value = s_a*(s1*C - s2*O).
 * ------------------------------------------------------------------- */
float or_lane_value(int64_t C, int64_t O, uint16_t s1, uint16_t s2, int kind, int m, int e) {
    int64_t sig1, sig2 = 0; int ex1, ex2 = 0;
    if (m == 0) return engine_nan();
    if (or_f16_scale(s1, &sig1, &ex1)) return engine_nan();
    if (kind == 1 && or_f16_scale(s2, &sig2, &ex2)) return engine_nan();
    i128 t1 = (i128)sig1 * m * C;                   /* at 2^(ex1+e) */
    if (kind == 0) return or_scaled_to_f32(t1, ex1 + e);
    i128 t2 = -(i128)sig2 * m * O;                  /* at 2^(ex2+e) */
    int lo = ex1 < ex2 ? ex1 : ex2;
    i128 sum = (t1 << (ex1 - lo)) + (t2 << (ex2 - lo));   /* exact (R4): < 2^75 */
    return or_scaled_to_f32(sum, lo + e);
}

/* ---------------------------------------------------------------------
 * Per-block results of every (column, row, block): the two exact sums and the
 * rounded value.  Layouts [ncols][rows][K/block].  Any of C/O/v may be NULL.
 * ------------------------------------------------------------------- */
int or_block_values(int fmt, const uint8_t *W, int64_t rows, int64_t K, const int8_t *codes,
                    const uint8_t *am, const int16_t *ae, int ncols, int64_t *C, int64_t *O, float *v) {
    or_row w;
    int64_t nb = K / fmt_block(fmt), rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = 0; r < rows; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++) {
            for (int64_t b = 0; b < nb; b++) {
                or_block ob;
                block_sums(&w, b, codes + (int64_t)c * K, &ob);
                int64_t idx = ((int64_t)c * rows + r) * nb + b;
                if (C) C[idx] = ob.C;
                if (O) O[idx] = ob.O;
                if (v) v[idx] = or_lane_value(ob.C, ob.O, ob.s1, ob.s2, ob.kind,
                                              am[(int64_t)c * nb + b], ae[(int64_t)c * nb + b]);
            }
        }
    }
    row_free(&w);
    return 0;
}

/* ---------------------------------------------------------------------
 * dot: the f32 the engine produces for row . act under PerBlock -- each
 * block's value rounded once, the rounded pieces added in order from +0 in
 * f32 with ftz (numerics page, dot and the f32 rules).  Rows [r0, r1) of the
 * matrix; out[c*rows + r].  A NaN row is the engine's NaN.
 * ------------------------------------------------------------------- */
int or_gemv_rows(int fmt, const uint8_t *W, int64_t rows, int64_t r0, int64_t r1, int64_t K,
                 const int8_t *codes, const uint8_t *am, const int16_t *ae, int ncols, float *out) {
    or_row w;
    int64_t nb = K / fmt_block(fmt), rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = r0; r < r1; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++) {
            float acc = 0.0f;
            for (int64_t b = 0; b < nb; b++) {
                or_block ob;
                block_sums(&w, b, codes + (int64_t)c * K, &ob);
                float v = or_lane_value(ob.C, ob.O, ob.s1, ob.s2, ob.kind,
                                        am[(int64_t)c * nb + b], ae[(int64_t)c * nb + b]);
                acc = or_ftz(acc + v);
            }
            if (isnan(acc)) acc = engine_nan();
            out[(int64_t)c * rows + r] = acc;
        }
    }
    row_free(&w);
    return 0;
}

int or_gemv(int fmt, const uint8_t *W, int64_t rows, int64_t K, const int8_t *codes,
            const uint8_t *am, const int16_t *ae, int ncols, float *out) {
    return or_gemv_rows(fmt, W, rows, 0, rows, K, codes, am, ae, ncols, out);
}

/* ---------------------------------------------------------------------
 * The lane's own delivery, for cross-checking block_sums: per 16-element unit
 * the array hands P' = sum q*a', the weight image Q = sum q, the activation
 * side S' = sum a', with a' = a + 128 (one-word excess form) and q the
 * decoder's unsigned code; the unit's signed sums follow from the identity
 *   sum (q - z)*a = P' - 128*Q - z*S' + 128*16*z,   sum a = S' - 128*16,
 * and the block sums are C = sum_u c_u * sum(q-z)*a, O = sum_u n_u * sum a
 * (lane page, opening description; deliver / block_sums).  For Q8_0 the
 * unsigned code is q+128 with z = 128 and c_u = 1; for Q4_K z = 0, c_u = sc,
 * n_u = mn; for Q6_K z = 32, c_u = sc, no offsets.
 * ------------------------------------------------------------------- */
int or_block_sums_excess(int fmt, const uint8_t *W, int64_t rows, int64_t K, const int8_t *codes,
                         int ncols, int64_t *C, int64_t *O) {
    or_row w;
    int blk = fmt_block(fmt);
    int64_t nb = K / blk, rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = 0; r < rows; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++) {
            const int8_t *a = codes + (int64_t)c * K;
            for (int64_t b = 0; b < nb; b++) {
                int64_t Cs = 0, Os = 0;
                for (int u = 0; u < blk / 16; u++) {
                    int64_t P1 = 0, Q = 0, S1 = 0, z, cu, nu;
                    for (int i = 0; i < 16; i++) {
                        int64_t e = b * blk + 16 * u + i;
                        int64_t ap = (int64_t)a[e] + 128;
                        int64_t qu = (fmt == OR_Q8_0) ? (int64_t)w.q8[e] + 128 : (int64_t)w.q[e];
                        P1 += qu * ap; Q += qu; S1 += ap;
                    }
                    if (fmt == OR_Q8_0) { z = 128; cu = 1; nu = 0; }
                    else if (fmt == OR_Q4K) { z = 0; cu = w.sc[b * 8 + u / 2]; nu = w.mn[b * 8 + u / 2]; }
                    else { z = 32; cu = w.sc6[b * 16 + u]; nu = 0; }
                    Cs += cu * (P1 - 128 * Q - z * S1 + 128 * 16 * z);
                    Os += nu * (S1 - 128 * 16);
                }
                int64_t idx = ((int64_t)c * rows + r) * nb + b;
                C[idx] = Cs;
                O[idx] = Os;
            }
        }
    }
    row_free(&w);
    return 0;
}

/* ---------------------------------------------------------------------
 * Two-word activation codes (lane page, opening description and WordSums;
 * numerics page, Words): a code that crosses in two words is a 16-bit integer
 * a = 256*hi + lo, hi its signed high byte and lo its unsigned low byte.  The
 * block's sums against such codes are the same definitions as block_sums --
 * sum coef*a and sum offs*a, element by element -- now over 16-bit codes; the
 * lane combines them with the block's scales and the activation scale
 * exactly and rounds once (or_lane_value: the terms stay below 2^56, shifted
 * by at most 29 places, inside its 128-bit sum), and dot adds the rounded
 * values in block order.
 * ------------------------------------------------------------------- */
static void block_sums_w2(const or_row *w, int64_t b, const int16_t *a, or_block *ob) {
    ob->C = 0; ob->O = 0; ob->kind = 0; ob->s2 = 0;
    if (w->fmt == OR_Q8_0) {
        for (int i = 0; i < 32; i++) ob->C += (int64_t)w->q8[b * 32 + i] * a[b * 32 + i];
        ob->s1 = w->d[b];
    } else if (w->fmt == OR_Q4K) {
        for (int i = 0; i < 256; i++) {
            int64_t e = b * 256 + i;
            int s = i / 32;
            ob->C += (int64_t)w->sc[b * 8 + s] * w->q[e] * a[e];
            ob->O += (int64_t)w->mn[b * 8 + s] * a[e];
        }
        ob->s1 = w->d[b]; ob->s2 = w->dm[b]; ob->kind = 1;
    } else {
        for (int i = 0; i < 256; i++) {
            int64_t e = b * 256 + i;
            ob->C += (int64_t)w->sc6[b * 16 + i / 16] * ((int64_t)w->q[e] - 32) * a[e];
        }
        ob->s1 = w->d[b];
    }
}

/* Per (column, row, block) sums and rounded values for two-word codes; layouts as or_block_values. */
int or_block_values_w2(int fmt, const uint8_t *W, int64_t rows, int64_t K, const int16_t *codes,
                       const uint8_t *am, const int16_t *ae, int ncols, int64_t *C, int64_t *O, float *v) {
    or_row w;
    int64_t nb = K / fmt_block(fmt), rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = 0; r < rows; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++)
            for (int64_t b = 0; b < nb; b++) {
                or_block ob;
                block_sums_w2(&w, b, codes + (int64_t)c * K, &ob);
                int64_t idx = ((int64_t)c * rows + r) * nb + b;
                if (C) C[idx] = ob.C;
                if (O) O[idx] = ob.O;
                if (v) v[idx] = or_lane_value(ob.C, ob.O, ob.s1, ob.s2, ob.kind,
                                              am[(int64_t)c * nb + b], ae[(int64_t)c * nb + b]);
            }
    }
    row_free(&w);
    return 0;
}

/* dot for two-word codes: rows [r0, r1), out[c*rows + r], the rounded block values added in order from +0. */
int or_gemv_w2_rows(int fmt, const uint8_t *W, int64_t rows, int64_t r0, int64_t r1, int64_t K,
                    const int16_t *codes, const uint8_t *am, const int16_t *ae, int ncols, float *out) {
    or_row w;
    int64_t nb = K / fmt_block(fmt), rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = r0; r < r1; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++) {
            float acc = 0.0f;
            for (int64_t b = 0; b < nb; b++) {
                or_block ob;
                block_sums_w2(&w, b, codes + (int64_t)c * K, &ob);
                acc = or_ftz(acc + or_lane_value(ob.C, ob.O, ob.s1, ob.s2, ob.kind,
                                                 am[(int64_t)c * nb + b], ae[(int64_t)c * nb + b]));
            }
            if (isnan(acc)) acc = engine_nan();
            out[(int64_t)c * rows + r] = acc;
        }
    }
    row_free(&w);
    return 0;
}

/* The lane's two-word delivery (lane page, opening description): per
 * 16-element unit and per word, P' = sum q*a', Q = sum q, S' = sum a', where
 * the high word crosses in excess form (a' = hi + 128) and the low byte as
 * itself (a' = lo); the unit's signed sums are the excess word's
 *   P' - 128*Q - z*S' + 128*16*z  and  S' - 128*16
 * weighted by 256, plus the low byte's  P' - z*S'  and  S'.  Block sums as in
 * or_block_sums_excess. */
int or_block_sums_excess_w2(int fmt, const uint8_t *W, int64_t rows, int64_t K, const int16_t *codes,
                            int ncols, int64_t *C, int64_t *O) {
    or_row w;
    int blk = fmt_block(fmt);
    int64_t nb = K / blk, rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = 0; r < rows; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++) {
            const int16_t *a = codes + (int64_t)c * K;
            for (int64_t b = 0; b < nb; b++) {
                int64_t Cs = 0, Os = 0;
                for (int u = 0; u < blk / 16; u++) {
                    int64_t Ph = 0, Pl = 0, Q = 0, Sh = 0, Sl = 0, z, cu, nu;
                    for (int i = 0; i < 16; i++) {
                        int64_t e = b * blk + 16 * u + i;
                        int64_t code = a[e];
                        int64_t lo = code & 255, hi = (code - lo) / 256;   /* code = 256*hi + lo, lo in 0..255 */
                        int64_t ah = hi + 128;                             /* the high word in excess form */
                        int64_t qu = (fmt == OR_Q8_0) ? (int64_t)w.q8[e] + 128 : (int64_t)w.q[e];
                        Ph += qu * ah; Pl += qu * lo; Q += qu; Sh += ah; Sl += lo;
                    }
                    if (fmt == OR_Q8_0) { z = 128; cu = 1; nu = 0; }
                    else if (fmt == OR_Q4K) { z = 0; cu = w.sc[b * 8 + u / 2]; nu = w.mn[b * 8 + u / 2]; }
                    else { z = 32; cu = w.sc6[b * 16 + u]; nu = 0; }
                    const int64_t dot = 256 * (Ph - 128 * Q - z * Sh + 128 * 16 * z) + (Pl - z * Sl);
                    const int64_t sum = 256 * (Sh - 128 * 16) + Sl;
                    Cs += cu * dot;
                    Os += nu * sum;
                }
                int64_t idx = ((int64_t)c * rows + r) * nb + b;
                C[idx] = Cs;
                O[idx] = Os;
            }
        }
    }
    row_free(&w);
    return 0;
}

/* ---------------------------------------------------------------------
 * Unreadable blocks: count the blocks whose f16 scale is inf or NaN
 * (numerics page, struct Unreadable; reads).
 * ------------------------------------------------------------------- */
int64_t or_count_unreadable(int fmt, const uint8_t *W, int64_t rows, int64_t K) {
    or_row w;
    int64_t rec = or_record_bytes(fmt, K), n = 0, nb = K / fmt_block(fmt);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = 0; r < rows; r++) {
        row_unpack(&w, W + r * rec);
        for (int64_t b = 0; b < nb; b++) {
            int64_t s; int e;
            int bad = or_f16_scale(w.d[b], &s, &e) != 0;
            if (fmt == OR_Q4K) bad |= or_f16_scale(w.dm[b], &s, &e) != 0;
            n += bad;
        }
    }
    row_free(&w);
    return n;
}

/* ---------------------------------------------------------------------
 * f32_to_f16: x rounded to binary16, to nearest with ties to even,
 * subnormals kept, past the top infinite (numerics page, f32_to_f16).
 * Stated on the integers: |x| = X * 2^E exactly, rounded to a multiple of the
 * binary16 quantum at its place (2^(x-10) for x >= -14, 2^-24 below).
 * NaN gives the quiet NaN 0x7E00.
 * ------------------------------------------------------------------- */
uint16_t or_f32_to_f16(float x) {
    uint32_t b = f32_bits(x);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000);
    if (isnan(x)) return 0x7E00;
    if (isinf(x)) return sign | 0x7C00;
    int e8 = (b >> 23) & 0xFF;
    uint64_t X = b & 0x7FFFFF;
    int E;
    if (e8 == 0) E = -149;                 /* f32 subnormal: X * 2^-149 */
    else { X |= 0x800000; E = e8 - 150; }
    if (X == 0) return sign;
    int p = 63;
    while (!((X >> p) & 1)) p--;
    int xl = p + E;                        /* leading place */
    int sub = xl < -14;                    /* below the least normal binary16 */
    int qe = sub ? -24 : xl - 10;          /* binary16 quantum there */
    int shift = qe - E;
    uint64_t r;
    if (shift <= 0) r = X << (-shift);
    else if (shift >= 64) r = 0;
    else {
        uint64_t q = X >> shift, rem = X & ((1ull << shift) - 1), half = 1ull << (shift - 1);
        r = q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0);
    }
    /* value = r * 2^qe; encode */
    if (r == 0) return sign;
    if (sub) {
        if (r < 1024) return sign | (uint16_t)r;            /* subnormal */
        return sign | (uint16_t)(1 << 10);                  /* rounded up to 2^-14 */
    }
    if (r == 2048) { r = 1024; qe += 1; }                   /* carry into the next binade */
    int ebias = qe + 10 + 15;                               /* leading place + bias */
    if (ebias >= 31) return sign | 0x7C00;
    return sign | (uint16_t)(ebias << 10) | (uint16_t)(r - 1024);
}

/* binary16 widened to f32, exactly */
float or_f16_to_f32(uint16_t h) {
    int E = (h >> 10) & 31, f = h & 1023;
    float s = (h & 0x8000) ? -1.0f : 1.0f;
    if (E == 31) return f ? engine_nan() : s * INFINITY;
    if (E == 0) return s * (float)ldexp((double)f, -24);
    return s * (float)ldexp((double)(1024 + f), E - 25);
}

/* ---------------------------------------------------------------------
 * F16 weights: fdot -- sum a_i*b_i in LANES lanes (element i in lane i mod
 * LANES, in index order, from +0), then the balanced pairwise tree (numerics
 * page, fdot, tree, and the f32 rules; reading R6).  The activation is first
 * rounded to f16 by f32_to_f16 (the caller passes x16).  out[c*rows + r].
 * ------------------------------------------------------------------- */
int or_gemv_f16(const uint16_t *W, int64_t rows, int64_t K, const uint16_t *x16, int ncols, float *out) {
    for (int c = 0; c < ncols; c++) {
        const uint16_t *xc = x16 + (int64_t)c * K;
        for (int64_t r = 0; r < rows; r++) {
            const uint16_t *w = W + r * K;
            float l[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            for (int64_t i = 0; i < K; i++) {
                float p = or_ftz(or_f16_to_f32(w[i]) * or_f16_to_f32(xc[i]));
                l[i % 8] = or_ftz(l[i % 8] + p);
            }
            float t01 = or_ftz(l[0] + l[1]), t23 = or_ftz(l[2] + l[3]);
            float t45 = or_ftz(l[4] + l[5]), t67 = or_ftz(l[6] + l[7]);
            float acc = or_ftz(or_ftz(t01 + t23) + or_ftz(t45 + t67));
            if (isnan(acc)) acc = engine_nan();
            out[(int64_t)c * rows + r] = acc;
        }
    }
    return 0;
}

/* f32 -> f16 for a whole activation, [n] */
void or_quantize_f16(const float *x, int64_t n, uint16_t *x16) {
    for (int64_t i = 0; i < n; i++) x16[i] = or_f32_to_f16(x[i]);
}

/* scaled_to_f32 over 64-bit inputs, for tests: v * 2^ex; v given as hi:lo */
float or_scaled_to_f32_2x64(int64_t hi, uint64_t lo, int ex) {
    i128 v = ((i128)hi << 64) | (i128)lo;
    return or_scaled_to_f32(v, ex);
}

/* the f32 bits of a float, for ctypes callers */
uint32_t or_bits(float f) { return f32_bits(f); }
float or_from_bits(uint32_t b) { return bits_f32(b); }


/* =====================================================================
 * ActScaling::Sub32 (numerics page: block_scale, quantize, ACT_BLOCK,
 * GROUP, exact_sum, dot; lane page: group, deliver32).
 * ===================================================================== */

/* ---------------------------------------------------------------------
 * block_scale: the least m*2^e, m in 8..15, with 127*m*2^e >= amax, for a
 * finite positive amax (numerics page, block_scale).  The same search as
 * wide_scale with a 4-bit significand.
 * ------------------------------------------------------------------- */
void or_block_scale(float amax, int *m_out, int *e_out) {
    int64_t M; int E;
    f32_split(amax, &M, &E);
    int best_m = 0, best_e = 0;
    for (int j = -40; j <= 40; j++) {
        u128 num = (u128)M, den = 127;
        if (j >= 0) den <<= j; else num <<= -j;
        u128 mm = (num + den - 1) / den;
        if (mm < 8 || mm > 15) continue;
        int e = E + j;
        if (best_m == 0) { best_m = (int)mm; best_e = e; continue; }
        int lo = e < best_e ? e : best_e;
        u128 a = (u128)mm << (e - lo), b = (u128)best_m << (best_e - lo);
        if (a < b) { best_m = (int)mm; best_e = e; }
    }
    *m_out = best_m;
    *e_out = best_e;
}

/* ---------------------------------------------------------------------
 * quantize: x (a whole number of groups) quantized per ACT_BLOCK = 32
 * elements under block_scale (numerics page, quantize, ActScaling::Sub32),
 * codes by rne_div; readings R2, R13.  Scales [ncols][K/32]; unit sums as
 * for quantize_blocks.
 * ------------------------------------------------------------------- */
void or_quantize_sub32(const float *x, int64_t K, int ncols, int8_t *codes, uint8_t *m_out, int16_t *e_out,
                       int16_t *sums16) {
    int64_t nb = K / 32;
    for (int c = 0; c < ncols; c++) {
        for (int64_t b = 0; b < nb; b++) {
            const float *xb = x + (int64_t)c * K + b * 32;
            int8_t *cb = codes + (int64_t)c * K + b * 32;
            float amax = or_absmax(xb, 32);
            int m, e;
            if (isinf(amax)) { m = 0; e = 0; }             /* R13 */
            else if (amax == 0.0f) { m = 8; e = 0; }       /* R13 */
            else or_block_scale(amax, &m, &e);
            for (int i = 0; i < 32; i++) cb[i] = (int8_t)((m == 0) ? 0 : or_rne_div(xb[i], m, e));
            m_out[(int64_t)c * nb + b] = (uint8_t)m;
            e_out[(int64_t)c * nb + b] = (int16_t)e;
        }
        for (int64_t u = 0; u < K / 16; u++) {
            int sum = 0;
            for (int i = 0; i < 16; i++) sum += codes[(int64_t)c * K + u * 16 + i];
            sums16[(int64_t)c * (K / 16) + u] = (int16_t)sum;
        }
    }
}

/* ---------------------------------------------------------------------
 * exact_sum of sig_k * 2^E_k (|sig_k| < 2^63) rounded once to f32 (numerics
 * page, exact_sum, scaled_to_f32; readings R5, R14): the terms are added
 * exactly in a 384-bit two's-complement integer aligned at the least
 * exponent, then rounded to nearest even on the f32 grid (2^-149 quantum
 * below 2^-126), a subnormal result flushed to a zero of its sign, past the
 * top infinite.  No terms, or an exact zero, is +0.
 * ------------------------------------------------------------------- */
#define OR_WL 12  /* 32-bit limbs: 384 bits */
typedef struct { uint32_t w[OR_WL]; } or_wide;

static void wide_add_shifted(or_wide *acc, int64_t sig, int shift) {
    /* acc += sig * 2^shift, two's complement, shift >= 0, shift + 64 < 384 */
    uint32_t t[OR_WL];
    uint64_t mag = sig < 0 ? (uint64_t)0 - (uint64_t)sig : (uint64_t)sig;
    memset(t, 0, sizeof t);
    int limb = shift / 32, bit = shift % 32;
    /* place mag << bit across limbs */
    u128 v = (u128)mag << bit;
    for (int i = 0; i < 4 && limb + i < OR_WL; i++) t[limb + i] = (uint32_t)(v >> (32 * i));
    if (sig < 0) {  /* negate t */
        uint64_t carry = 1;
        for (int i = 0; i < OR_WL; i++) {
            uint64_t x = (uint64_t)(uint32_t)~t[i] + carry;
            t[i] = (uint32_t)x;
            carry = x >> 32;
        }
    }
    uint64_t carry = 0;
    for (int i = 0; i < OR_WL; i++) {
        uint64_t x = (uint64_t)acc->w[i] + t[i] + carry;
        acc->w[i] = (uint32_t)x;
        carry = x >> 32;
    }
}

float or_exact_sum_f32(const int64_t *sig, const int *E, int n) {
    if (n == 0) return 0.0f;
    int lo = E[0];
    for (int k = 1; k < n; k++) if (E[k] < lo) lo = E[k];
    or_wide acc;
    memset(&acc, 0, sizeof acc);
    for (int k = 0; k < n; k++) {
        if (sig[k] == 0) continue;
        if (E[k] - lo + 64 >= 32 * OR_WL - 2) return engine_nan();  /* cannot occur for f16 x block_scale terms */
        wide_add_shifted(&acc, sig[k], E[k] - lo);
    }
    int neg = (acc.w[OR_WL - 1] >> 31) & 1;
    if (neg) {  /* magnitude */
        uint64_t carry = 1;
        for (int i = 0; i < OR_WL; i++) {
            uint64_t x = (uint64_t)(uint32_t)~acc.w[i] + carry;
            acc.w[i] = (uint32_t)x;
            carry = x >> 32;
        }
    }
    int p = -1;                                      /* leading place of the magnitude */
    for (int i = OR_WL - 1; i >= 0 && p < 0; i--)
        if (acc.w[i]) for (int b = 31; b >= 0; b--) if ((acc.w[i] >> b) & 1) { p = 32 * i + b; break; }
    if (p < 0) return 0.0f;
    int x = p + lo;
    int sub = x < -126;
    int qe = sub ? -149 : x - 23;
    int shift = qe - lo;                             /* places below the quantum */
    uint64_t r;
    if (shift <= 0) {
        r = 0;                                       /* exact: the magnitude < 2^25 in quanta */
        for (int i = OR_WL - 1; i >= 0; i--) r = (r << 32) | acc.w[i];  /* p <= 24 here */
        r <<= -shift;
    } else {
        /* r = floor(mag / 2^shift), rem against half */
        r = 0;
        for (int bpos = p; bpos >= shift; bpos--) r = (r << 1) | ((acc.w[bpos / 32] >> (bpos % 32)) & 1);
        int half = (acc.w[(shift - 1) / 32] >> ((shift - 1) % 32)) & 1;
        int below = 0;
        for (int bpos = shift - 2; bpos >= 0 && !below; bpos--) below = (acc.w[bpos / 32] >> (bpos % 32)) & 1;
        if (half && (below || (r & 1))) r += 1;
    }
    if (sub && r < ((uint64_t)1 << 23)) return neg ? -0.0f : 0.0f;
    if (r == 0) return neg ? -0.0f : 0.0f;
    double d = ldexp((double)r, qe);
    if (d >= 3.4028236692093846e38) return neg ? -INFINITY : INFINITY;
    float f = (float)d;
    return neg ? -f : f;
}

/* ---------------------------------------------------------------------
 * group (lane page): group g (GROUP = 256 elements) of a row -- every 32-
 * element sub-block's two exact sums times its weight block's scales and its
 * own activation scale, the terms summed exactly and rounded once (numerics
 * page, dot under ActScaling::Sub32).  Q8_0: the sub-block is a weight
 * block, term d_s*m_s*2^e_s*C_s.  Q4_K-like: terms d*m_s*C_s and
 * -dmin*m_s*O_s at the sub-block's activation exponent.  Q6_K-like: the two
 * 16-element weight sub-blocks of the activation block make one C_s.  NaN for
 * an unreadable weight scale or an activation block without a scale.
 * ------------------------------------------------------------------- */
static float group_value(const or_row *w, int64_t g, const int8_t *a, const uint8_t *am, const int16_t *ae) {
    int64_t sig[16]; int E[16]; int n = 0;
    for (int s = 0; s < 8; s++) {
        int64_t sb = g * 8 + s;                       /* 32-element activation block */
        int m = am[sb], e = ae[sb];
        if (m == 0) return engine_nan();
        int64_t C = 0, O = 0, sg; int ex;
        uint16_t d1, d2 = 0; int kind = 0;
        if (w->fmt == OR_Q8_0) {
            for (int i = 0; i < 32; i++) C += (int64_t)w->q8[sb * 32 + i] * a[sb * 32 + i];
            d1 = w->d[sb];
        } else if (w->fmt == OR_Q4K) {
            for (int i = 0; i < 32; i++) {
                int64_t el = sb * 32 + i;
                C += (int64_t)w->sc[sb] * w->q[el] * a[el];
                O += (int64_t)w->mn[sb] * a[el];
            }
            d1 = w->d[g]; d2 = w->dm[g]; kind = 1;
        } else {
            for (int i = 0; i < 32; i++) {
                int64_t el = sb * 32 + i;
                C += (int64_t)w->sc6[el / 16] * ((int64_t)w->q[el] - 32) * a[el];
            }
            d1 = w->d[g];
        }
        if (or_f16_scale(d1, &sg, &ex)) return engine_nan();
        sig[n] = sg * m * C; E[n] = ex + e; n++;
        if (kind == 1) {
            if (or_f16_scale(d2, &sg, &ex)) return engine_nan();
            sig[n] = -sg * m * O; E[n] = ex + e; n++;
        }
    }
    return or_exact_sum_f32(sig, E, n);
}

/* ---------------------------------------------------------------------
 * dot under Sub32: the groups' values added in order from +0 in f32 with ftz
 * (numerics page, dot).  K a whole number of groups; rows [r0, r1);
 * out[c*rows + r]; activation scales [ncols][K/32].
 * ------------------------------------------------------------------- */
int or_gemv_sub32_rows(int fmt, const uint8_t *W, int64_t rows, int64_t r0, int64_t r1, int64_t K,
                       const int8_t *codes, const uint8_t *am, const int16_t *ae, int ncols, float *out) {
    or_row w;
    if (K % 256) return -1;
    int64_t ng = K / 256, rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = r0; r < r1; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++) {
            float acc = 0.0f;
            for (int64_t g = 0; g < ng; g++)
                acc = or_ftz(acc + group_value(&w, g, codes + (int64_t)c * K, am + (int64_t)c * (K / 32),
                                               ae + (int64_t)c * (K / 32)));
            if (isnan(acc)) acc = engine_nan();
            out[(int64_t)c * rows + r] = acc;
        }
    }
    row_free(&w);
    return 0;
}

/* the group values themselves: v[c][r][g] */
int or_group_values(int fmt, const uint8_t *W, int64_t rows, int64_t K, const int8_t *codes, const uint8_t *am,
                    const int16_t *ae, int ncols, float *v) {
    or_row w;
    if (K % 256) return -1;
    int64_t ng = K / 256, rec = or_record_bytes(fmt, K);
    if (row_alloc(&w, fmt, K)) { row_free(&w); return -1; }
    for (int64_t r = 0; r < rows; r++) {
        row_unpack(&w, W + r * rec);
        for (int c = 0; c < ncols; c++)
            for (int64_t g = 0; g < ng; g++)
                v[((int64_t)c * rows + r) * ng + g] =
                    group_value(&w, g, codes + (int64_t)c * K, am + (int64_t)c * (K / 32), ae + (int64_t)c * (K / 32));
    }
    row_free(&w);
    return 0;
}


/* =====================================================================
 * The int8 cache's score path (numerics page: cache_row, int8_codes,
 * INV_127, quantize_head, int8_score).
 * ===================================================================== */

/* INV_127 (numerics page): 1/127 as an f32, to nearest (0x3C010204). */
#define OR_INV_127 (1.0f / 127.0f)

/* ---------------------------------------------------------------------
 * int8_codes for one element (numerics page, int8_codes): x*inv as an f32
 * product (operands and result flushed), to the nearest integer with ties to
 * even, kept within +-127; a NaN product gives 0; an infinite inv (the
 * reciprocal of a scale that rounded to zero) gives 0.
 * ------------------------------------------------------------------- */
int or_int8_code(float x, float inv) {
    if (isinf(inv)) return 0;
    float p = or_ftz(or_ftz(x) * inv);
    if (isnan(p)) return 0;
    if (p >= 127.0f) return 127;
    if (p <= -127.0f) return -127;
    return (int)rintf(p);                /* default rounding: to nearest, ties to even */
}

/* ---------------------------------------------------------------------
 * cache_row (numerics page): n rows of d elements, each stored as int8 codes
 * under one f16 scale.  amax = absmax(row); the scale is
 * f32_to_f16(amax * INV_127) (an f32 product, flushed); the codes are
 * int8_codes of the row under the reciprocal of that scale (reading R17);
 * a scale that rounds to zero gives an infinite reciprocal and all-zero
 * codes.  codes [n][d], scales (binary16 bits) [n].
 * ------------------------------------------------------------------- */
void or_cache_rows(const float *x, int64_t n, int d, int8_t *codes, uint16_t *scales) {
    for (int64_t r = 0; r < n; r++) {
        const float *xr = x + r * d;
        float amax = or_absmax(xr, d);
        uint16_t h = or_f32_to_f16(or_ftz(amax * OR_INV_127));
        float s = or_f16_to_f32(h);
        float inv = 1.0f / s;
        for (int i = 0; i < d; i++) codes[r * d + i] = (int8_t)or_int8_code(xr[i], inv);
        scales[r] = h;
    }
}

/* ---------------------------------------------------------------------
 * quantize_head (numerics page): nh query heads of d elements as the array
 * reads them.  scaling 1 (ActScaling::Sub32): each head padded with zeros to
 * a whole number of groups, dp = 256*ceil(d/256) elements, quantized per 32
 * (quantize); codes [nh][dp], scales [nh][dp/32].  scaling 0
 * (ActScaling::PerBlock): the whole head one block (quantize_blocks with
 * block = d, wide_scale); codes [nh][d], scales [nh][1].
 * ------------------------------------------------------------------- */
int or_quantize_heads(int scaling, const float *q, int nh, int d, int8_t *codes, uint8_t *m, int16_t *e) {
    if (d <= 0 || d % 16) return -1;
    if (scaling == 1) {
        int dp = (d + 255) / 256 * 256;
        float *buf = (float *)calloc((size_t)dp, sizeof(float));
        int16_t *s16 = (int16_t *)malloc((size_t)dp / 16 * sizeof(int16_t));
        if (!buf || !s16) { free(buf); free(s16); return -1; }
        for (int h = 0; h < nh; h++) {
            memcpy(buf, q + (int64_t)h * d, (size_t)d * sizeof(float));
            or_quantize_sub32(buf, dp, 1, codes + (int64_t)h * dp, m + (int64_t)h * (dp / 32),
                              e + (int64_t)h * (dp / 32), s16);
        }
        free(buf);
        free(s16);
        return 0;
    }
    int16_t *s16 = (int16_t *)malloc((size_t)d / 16 * sizeof(int16_t));
    if (!s16) return -1;
    for (int h = 0; h < nh; h++)
        or_quantize_blocks(q + (int64_t)h * d, d, 1, d, codes + (int64_t)h * d, m + h, e + h, s16);
    free(s16);
    return 0;
}

/* ---------------------------------------------------------------------
 * int8_score (numerics page): a query head (nb blocks of blk codes with
 * scales m*2^e; codes past d are padding) against a cached key row (d int8
 * codes, f16 scale ks): per block, D_b = sum of q_i*k_i; the term
 * sig(ks) * m_b * D_b at exponent exp(ks) + e_b; the terms summed exactly
 * and rounded once (exact_sum, reading R5).  NaN for a query block without a
 * scale or an unreadable key scale (R18).
 * ------------------------------------------------------------------- */
float or_int8_score(const int8_t *qc, const uint8_t *m, const int16_t *e, int blk, int nb, int d, const int8_t *kc,
                    uint16_t ks) {
    int64_t sg;
    int ex;
    if (or_f16_scale(ks, &sg, &ex)) return engine_nan();
    int64_t *sig = (int64_t *)malloc((size_t)nb * sizeof(int64_t));
    int *E = (int *)malloc((size_t)nb * sizeof(int));
    if (!sig || !E) { free(sig); free(E); return engine_nan(); }
    float r;
    int bad = 0;
    for (int b = 0; b < nb; b++) {
        if (m[b] == 0) { bad = 1; break; }
        int64_t D = 0;
        for (int i = b * blk; i < (b + 1) * blk && i < d; i++) D += (int64_t)qc[i] * kc[i];
        sig[b] = sg * m[b] * D;
        E[b] = ex + e[b];
    }
    r = bad ? engine_nan() : or_exact_sum_f32(sig, E, nb);
    free(sig);
    free(E);
    return r;
}

/* ---------------------------------------------------------------------
 * The scores of nh query heads against L cached key rows of nkv key heads
 * (query head h reads key head h / (nh / nkv)): out[h*L + p] = the f32
 * product of int8_score and `scale` (flushed), NaN as the engine's.  Query
 * as or_quantize_heads writes it; key codes [nkv][lcap][d], key scales
 * [nkv][lcap] (positions 0..L-1 of each head used).
 * ------------------------------------------------------------------- */
int or_kv_scores(int scaling, const int8_t *qc, const uint8_t *qm, const int16_t *qe, int nh, int d,
                 const int8_t *kc, const uint16_t *ks, int64_t L, int64_t lcap, int nkv, float scale, float *out) {
    if (nkv <= 0 || nh % nkv || d <= 0 || d % 16 || L > lcap) return -1;
    int dp = scaling == 1 ? (d + 255) / 256 * 256 : d;
    int blk = scaling == 1 ? 32 : d, nb = dp / blk;
    for (int h = 0; h < nh; h++) {
        int kvh = h / (nh / nkv);
        for (int64_t p = 0; p < L; p++) {
            int64_t row = (int64_t)kvh * lcap + p;
            float v = or_int8_score(qc + (int64_t)h * dp, qm + (int64_t)h * nb, qe + (int64_t)h * nb, blk, nb, d,
                                    kc + row * d, ks[row]);
            v = or_ftz(v * scale);
            if (isnan(v)) v = engine_nan();
            out[(int64_t)h * L + p] = v;
        }
    }
    return 0;
}


/* =====================================================================
 * FP8 E4M3 weights with 128x128 block scales (colizig OPS page, FP8:
 * e4m3ToF32, dequantRow, matmulFp8).
 * ===================================================================== */

/* ---------------------------------------------------------------------
 * e4m3ToF32: an OCP E4M3 byte [s:1][e:4][m:3], exponent bias 7, as a number:
 * e = 0 -> (m/8) * 2^-6 (subnormal; m = 0 is a zero of the sign), otherwise
 * (1 + m/8) * 2^(e-7); e = 15 with m = 7 is NaN (the format has no
 * infinity).  Written from the format's definition with ldexp.
 * ------------------------------------------------------------------- */
float or_e4m3_to_f32(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return engine_nan();
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return (float)(s ? -v : v);
}

/* ---------------------------------------------------------------------
 * The exact dot of n f32 pairs, rounded once: every product x_i * w_i is an
 * integer times a power of two (24-bit by 24-bit significands), added exactly
 * into a two's-complement integer of 640 bits whose bit j weighs 2^(j - 298)
 * (products of finite f32 values lie between 2^-298 and 2^256, and 2^31 terms
 * add 31 more places); the sum is then rounded to nearest even on the f32
 * grid, subnormals kept (ordinary f32 arithmetic: the FP8 path has no flush
 * rule), past the top infinite.  A NaN operand, an infinity times zero, or
 * infinities of both signs give NaN; otherwise an infinite product gives that
 * infinity.  An exact zero is +0.
 * ------------------------------------------------------------------- */
#define OR_DL 20   /* 32-bit limbs: 640 bits */
#define OR_DOFF 298

static void dot_add(uint32_t *acc, uint64_t mag, int neg, int pos) {
    /* acc += (neg ? -1 : 1) * mag * 2^pos, 0 <= pos, pos + 64 < 640 */
    uint32_t t[OR_DL];
    memset(t, 0, sizeof t);
    int limb = pos / 32, bit = pos % 32;
    u128 v = (u128)mag << bit;
    for (int i = 0; i < 4 && limb + i < OR_DL; i++) t[limb + i] = (uint32_t)(v >> (32 * i));
    if (neg) {
        uint64_t carry = 1;
        for (int i = 0; i < OR_DL; i++) {
            uint64_t y = (uint64_t)(uint32_t)~t[i] + carry;
            t[i] = (uint32_t)y;
            carry = y >> 32;
        }
    }
    uint64_t carry = 0;
    for (int i = 0; i < OR_DL; i++) {
        uint64_t y = (uint64_t)acc[i] + t[i] + carry;
        acc[i] = (uint32_t)y;
        carry = y >> 32;
    }
}

/* an f32 as sig * 2^e with sig < 2^24 (zero: sig 0) */
static void f32_parts(float f, uint64_t *sig, int *e, int *neg) {
    uint32_t b;
    memcpy(&b, &f, 4);
    *neg = (int)(b >> 31);
    int E = (int)((b >> 23) & 0xFF);
    uint32_t m = b & 0x7FFFFF;
    *sig = E ? (m | 0x800000u) : m;
    *e = (E ? E : 1) - 150;
}

float or_exact_dot_f32(const float *x, const float *w, int64_t n) {
    uint32_t acc[OR_DL];
    memset(acc, 0, sizeof acc);
    int pinf = 0, ninf = 0;
    for (int64_t i = 0; i < n; i++) {
        const float a = x[i], b = w[i];
        if (isnan(a) || isnan(b)) return engine_nan();
        if (isinf(a) || isinf(b)) {
            if (a == 0.0f || b == 0.0f) return engine_nan();   /* infinity times zero */
            if ((a < 0) != (b < 0)) ninf = 1; else pinf = 1;
            continue;
        }
        uint64_t sa, sb;
        int ea, eb, na, nb;
        f32_parts(a, &sa, &ea, &na);
        f32_parts(b, &sb, &eb, &nb);
        if (sa == 0 || sb == 0) continue;
        dot_add(acc, sa * sb, na != nb, ea + eb + OR_DOFF);
    }
    if (pinf && ninf) return engine_nan();
    if (pinf) return INFINITY;
    if (ninf) return -INFINITY;
    int neg = (int)((acc[OR_DL - 1] >> 31) & 1);
    if (neg) {
        uint64_t carry = 1;
        for (int i = 0; i < OR_DL; i++) {
            uint64_t y = (uint64_t)(uint32_t)~acc[i] + carry;
            acc[i] = (uint32_t)y;
            carry = y >> 32;
        }
    }
    int p = -1;  /* leading place of the magnitude */
    for (int i = OR_DL - 1; i >= 0 && p < 0; i--)
        if (acc[i]) for (int k = 31; k >= 0; k--) if ((acc[i] >> k) & 1) { p = 32 * i + k; break; }
    if (p < 0) return 0.0f;
    int x2 = p - OR_DOFF;                       /* leading exponent */
    int qe = x2 < -126 ? -149 : x2 - 23;        /* the f32 quantum there */
    int q = qe + OR_DOFF;                       /* its bit position */
    /* mantissa = acc >> q (at most 25 bits), then nearest even on the rest */
    uint64_t mant = 0;
    for (int k = p; k >= q; k--) mant = (mant << 1) | ((acc[k / 32] >> (k % 32)) & 1);
    int half = q >= 1 ? (int)((acc[(q - 1) / 32] >> ((q - 1) % 32)) & 1) : 0;
    int sticky = 0;
    for (int k = q - 2; k >= 0 && !sticky; k--) sticky = (acc[k / 32] >> (k % 32)) & 1;
    if (half && (sticky || (mant & 1))) mant++;
    if (mant == (1ull << 24)) { mant >>= 1; qe++; }
    float r;
    if (mant < (1ull << 23)) {                  /* subnormal (qe = -149) */
        uint32_t bits = (uint32_t)mant;
        memcpy(&r, &bits, 4);
    } else {
        int e2 = qe + 23;                       /* exponent of the leading bit */
        if (e2 > 127) return neg ? -INFINITY : INFINITY;
        uint32_t bits = ((uint32_t)(e2 + 127) << 23) | ((uint32_t)mant & 0x7FFFFFu);
        memcpy(&r, &bits, 4);
    }
    return neg ? -r : r;
}

/* ---------------------------------------------------------------------
 * matmulFp8 read as "dequantize then f32 matmul" (the page's own check): the
 * weight W[r][i] is the f32 product of its decoded byte and its 128x128 block
 * scale (dequantRow folds the scale), rounded to nearest; the row's dot with
 * each activation column x[c][:] is then taken exactly and rounded once to
 * f32 (or_exact_dot_f32).  Scales [ceil(rows/128)][ceil(K/128)].  Also the
 * sum of |x_i * w_i| in double (absdot), the scale against which a GPU's f32
 * summation error is bounded.  A NaN result is the engine's NaN.
 * ------------------------------------------------------------------- */
int or_gemv_fp8(const uint8_t *W, const float *scales, int64_t rows, int64_t K, const float *x, int ncols,
                float *out, double *absdot) {
    int64_t kb = (K + 127) / 128;
    float *w = (float *)malloc((size_t)K * sizeof(float));
    if (!w) return -1;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t i = 0; i < K; i++) {
            float s = scales[(r / 128) * kb + i / 128];
            w[i] = or_e4m3_to_f32(W[r * K + i]) * s;   /* one f32 product, to nearest */
        }
        for (int c = 0; c < ncols; c++) {
            const float *xc = x + (int64_t)c * K;
            float v = or_exact_dot_f32(xc, w, K);
            out[(int64_t)c * rows + r] = isnan(v) ? engine_nan() : v;
            if (absdot) {
                double ab = 0.0;
                for (int64_t i = 0; i < K; i++) ab += fabs((double)xc[i] * (double)w[i]);
                absdot[(int64_t)c * rows + r] = ab;
            }
        }
    }
    free(w);
    return 0;
}

/*
 * CPU oracle of the routed MoE prefill layer.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * CPU-baseline leg of the benchmark load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls
 * it.  It is written to be read against the pages, not to be fast: plain
 * loops, fp64 arithmetic, no blocking, no reordering of any sum.  Build with
 * -ffp-contract=off so that every a*b+c rounds twice, as written.
 *
 * Sources (page title, then section):
 *  [P1] "Round 4 Track C: Prefill MoE Plan (mm_clear + mm_hist + mm_scan +
 *       mm_place) & Epilogue / Gather Audit" -- section 1 items 1, 2 and 4
 *       (histogram, padded scan with -1 tail rows, stable place, row gather)
 *       and section 3 (the plan buffers compared bit for bit).
 *  [P3] "Batched resident MoE experts on Apple Silicon: a flat parallel
 *       expert pass" -- section 1 (an immutable (token, expert, weight) job
 *       list; per job gate/up projection -> gated activation -> weighted down
 *       projection) and section 3 (the same per-token top-k summation order).
 *  [P4] "Add --moe-mode sweep-prefill" -- Mechanism (experts walked in
 *       ascending id over contiguous slices).
 *  [P1] again, section 2: the benchmarks run the experts from quantized
 *       weight packs (8-, 4- and 2-bit block formats).  The quantized form
 *       here is 8-bit floating point E4M3 (the OCP 8-bit floating point
 *       format: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *       infinities, S.1111.111 = NaN, largest finite 448) with one fp32
 *       scale per expert and output feature; and 4-bit MXFP4 (the OCP
 *       Microscaling format: E2M1 elements -- 1 sign, 2 exponent bits with
 *       bias 1, 1 mantissa bit, magnitudes 0 .. 6 -- in blocks of 32 along
 *       the reduction axis sharing a power-of-two scale 2^(S-127), S an
 *       unsigned 8-bit exponent).
 *
 * Readings taken where the pages leave a step open:
 *  - flat entry i = t*k + j (token-major); ties inside an expert keep
 *    increasing i;
 *  - id -1 marks a skipped slot: no row, pos = -1, no contribution;
 *  - an empty expert gets zero rows and zero tiles;
 *  - pad rows carry srt_tok = -1 and srt_w = +0.0f; gathered pad rows are
 *    all-zero bits;
 *  - gated activation is SwiGLU: h = silu(g) * u with silu(z) = z/(1+e^-z),
 *    g from the gate weight, u from the up weight;
 *  - the routing weight scales each job's down projection; the token's
 *    output sums its slots j = 0..k-1 in order starting from zero.
 *
 * Every function here is pinned by the CPU tests (brute force on tiny
 * inputs, closed forms, library cross-checks and invariants).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_ID (-2)
#define ORC_ERR_CAP (-3)
#define ORC_ERR_MEM (-4)

/* ---- widening of 16-bit inputs (exact) --------------------------------- */

static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float v;
    memcpy(&v, &u, sizeof v);
    return (double)v;
}

static double f16_value(uint16_t h)
{
    int sign = h >> 15, ex = (h >> 10) & 0x1f, man = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);               /* subnormal: man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(man | 0x400), ex - 25); /* (1024+man) * 2^(ex-25) */
    return sign ? -v : v;
}

static double value16(uint16_t b, int is_f16)
{
    return is_f16 ? f16_value(b) : bf16_value(b);
}

/* fp64 -> fp32 (C conversion, nearest) -> bf16 (nearest, ties to even). */
static double to_bf16(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) != 0x7f800000u)
        u += 0x7fffu + ((u >> 16) & 1u);
    u &= 0xffff0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- E4M3 weights [P1 sec. 2; the OCP E4M3 definition] ----------------- */

/* Value of an E4M3 code: exponent field 0 is subnormal (m/8 * 2^-6), the
 * rest normal ((1 + m/8) * 2^(e-7)); S.1111.111 is NaN. */
static double e4m3_value(uint8_t c)
{
    int sign = c >> 7, ex = (c >> 3) & 15, man = c & 7;
    double v;
    if (ex == 15 && man == 7)
        return NAN;
    if (ex == 0)
        v = ldexp((double)man, -9);
    else
        v = ldexp((double)(8 + man), ex - 10);
    return sign ? -v : v;
}

/* Nearest E4M3 code to v, ties to the even code (the one whose mantissa
 * field is even), magnitudes past 448 saturated to 448; the sign is kept
 * (a negative value that rounds to zero gives -0).  Written as a search
 * over the 127 non-negative finite magnitudes, which are in increasing
 * order of their codes. */
static uint8_t e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    int c, best = 0;
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    for (c = 1; c <= 0x7e; c++) {
        double lo = e4m3_value((uint8_t)(c - 1)), hi = e4m3_value((uint8_t)c);
        if (a > hi)
            continue;
        /* lo <= a <= hi */
        if (a - lo < hi - a)
            best = c - 1;
        else if (a - lo > hi - a)
            best = c;
        else
            best = ((c - 1) & 1) == 0 ? c - 1 : c;
        break;
    }
    return (uint8_t)(sign | best);
}

/*
 * Quantize bf16 weights W [E][K][M] (M the output feature, contiguous) to
 * E4M3 codes q [E][K][M] with one fp32 scale per (expert, output feature):
 *   amax = max over k of |W[e][k][m]|
 *   scale[e][m] = amax / 448 (fp32 division), or 1 when that is 0
 *   q[e][k][m] = e4m3_encode(W[e][k][m] / scale[e][m]) (fp32 division)
 * so the dequantized weight is e4m3_value(q) * scale.  W must be finite.
 */
void oracle_quantize_e4m3(const uint16_t *W, int E, int K, int M, uint8_t *q, float *scale)
{
    long e, k, m;
    for (e = 0; e < E; e++) {
        for (m = 0; m < M; m++) {
            float amax = 0.0f, s;
            for (k = 0; k < K; k++) {
                float a = (float)fabs(bf16_value(W[(e * K + k) * M + m]));
                if (a > amax)
                    amax = a;
            }
            s = amax / 448.0f;
            if (s == 0.0f)
                s = 1.0f;
            scale[e * M + m] = s;
            for (k = 0; k < K; k++) {
                long i = (e * K + k) * M + m;
                q[i] = e4m3_encode((float)bf16_value(W[i]) / s);
            }
        }
    }
}

/* ---- MXFP4 weights [P1 sec. 2; the OCP Microscaling (MX) MXFP4 format] ---- */

/* Value of an E2M1 (4-bit) code: 1 sign bit, 2 exponent bits (bias 1), 1
 * mantissa bit; exponent field 0 is subnormal (m/2), the rest normal
 * ((1 + m/2) * 2^(e-1)).  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no
 * infinities, no NaN. */
static double e2m1_value(uint8_t c)
{
    int sign = (c >> 3) & 1, ex = (c >> 1) & 3, man = c & 1;
    double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sign ? -v : v;
}

/* Nearest E2M1 code to v, ties to the even code (the one whose mantissa
 * bit is 0), magnitudes past 6 saturated to 6; the sign is kept (a
 * negative value that rounds to zero gives -0).  A search over the eight
 * non-negative magnitudes, which increase with their codes. */
static uint8_t e2m1_encode(double v)
{
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    int c, best = 0;
    if (a >= 6.0)
        return (uint8_t)(sign | 0x7);
    for (c = 1; c <= 7; c++) {
        double lo = e2m1_value((uint8_t)(c - 1)), hi = e2m1_value((uint8_t)c);
        if (a > hi)
            continue;
        /* lo <= a <= hi */
        if (a - lo < hi - a)
            best = c - 1;
        else if (a - lo > hi - a)
            best = c;
        else /* a tie: the code whose mantissa bit is 0 */
            best = (c & 1) ? c - 1 : c;
        break;
    }
    return (uint8_t)(sign | best);
}

#define MX_BLOCK 32
#define E2M1_EMAX 2 /* exponent of the largest E2M1 normal: 6 = 1.5 * 2^2 */

/*
 * Quantize bf16 weights W [E][K][M] (M the output feature, contiguous) to
 * MXFP4 along the reduction axis K: for each expert e, output feature m and
 * block b of 32 consecutive k (K a multiple of 32, M even):
 *   amax = max |W| over the block
 *   x = floor(log2(amax)) - 2, clamped to [-127, 127]; x = -127 when amax = 0
 *   scales[e][b][m] = x + 127 (an 8-bit power-of-two exponent, E8M0)
 *   code = e2m1_encode(W / 2^x) (exact division by a power of two)
 * so the dequantized weight is e2m1_value(code) * 2^x.  Codes are packed two
 * per byte along M: byte codes[e][k][m/2] holds feature m (even) in its low
 * four bits and feature m + 1 in its high four bits.  W must be finite.
 */
void oracle_quantize_mxfp4(const uint16_t *W, int E, int K, int M, uint8_t *codes,
                           uint8_t *scales)
{
    long e, b, k, m;
    for (e = 0; e < E; e++) {
        for (b = 0; b < K / MX_BLOCK; b++) {
            for (m = 0; m < M; m++) {
                double amax = 0.0;
                int x = -127, fe;
                for (k = b * MX_BLOCK; k < (b + 1) * MX_BLOCK; k++) {
                    double a = fabs(bf16_value(W[(e * K + k) * M + m]));
                    if (a > amax)
                        amax = a;
                }
                if (amax > 0.0) {
                    frexp(amax, &fe); /* amax = f * 2^fe, f in [0.5, 1): floor(log2) = fe - 1 */
                    x = fe - 1 - E2M1_EMAX;
                    if (x < -127)
                        x = -127;
                    if (x > 127)
                        x = 127;
                }
                scales[(e * (K / MX_BLOCK) + b) * M + m] = (uint8_t)(x + 127);
                for (k = b * MX_BLOCK; k < (b + 1) * MX_BLOCK; k++) {
                    uint8_t c = e2m1_encode(ldexp(bf16_value(W[(e * K + k) * M + m]), -x));
                    uint8_t *byte = &codes[(e * K + k) * (M / 2) + m / 2];
                    if ((m & 1) == 0)
                        *byte = (uint8_t)((*byte & 0xf0) | c);
                    else
                        *byte = (uint8_t)((*byte & 0x0f) | (c << 4));
                }
            }
        }
    }
}

/*
 * The dequantized weights e2m1_value(code) * 2^(scale - 127) as bf16 bit
 * patterns W [E][K][M].  Every such value with scale <= 252 is a bf16 value
 * (at most two significant bits, exponent inside bf16's range), so this is
 * exact; returns ORC_ERR_ARG if some value is not (a scale byte above 252).
 */
int oracle_dequantize_mxfp4(const uint8_t *codes, const uint8_t *scales, int E, int K, int M,
                            uint16_t *W)
{
    long e, k, m;
    for (e = 0; e < E; e++)
        for (k = 0; k < K; k++)
            for (m = 0; m < M; m++) {
                uint8_t byte = codes[(e * K + k) * (M / 2) + m / 2];
                uint8_t c = (m & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf);
                int s = scales[(e * (K / MX_BLOCK) + k / MX_BLOCK) * M + m];
                double v = ldexp(e2m1_value(c), s - 127);
                float f = (float)v;
                uint32_t u;
                if (s > 252 || (double)f != v)
                    return ORC_ERR_ARG;
                memcpy(&u, &f, sizeof u);
                if (u & 0xffffu)
                    return ORC_ERR_ARG;
                W[(e * K + k) * M + m] = (uint16_t)(u >> 16);
            }
    return ORC_OK;
}

/*
 * E4M3 activations: one row x[0..d-1] (exact bf16 values) with a power-of-
 * two scale 2^e, e the smallest integer with max |x| <= 448 * 2^e (e = 0
 * for an all-zero row); codes are e4m3_encode(x * 2^-e), exact scaling.
 * Writes the codes (if q) and returns e.
 */
static int quantize_row_e4m3(const double *x, int d, uint8_t *q)
{
    double amax = 0.0;
    int c, e = 0;
    for (c = 0; c < d; c++)
        if (fabs(x[c]) > amax)
            amax = fabs(x[c]);
    if (amax > 0.0) {
        e = ilogb(amax) - 8;             /* amax in [2^(e+8), 2^(e+9)) */
        if (amax > ldexp(448.0, e))
            e++;
    }
    if (q)
        for (c = 0; c < d; c++)
            q[c] = e4m3_encode((float)ldexp(x[c], -e));
    return e;
}

/* The row replaced by its dequantized values value(code) * 2^e. */
static void dequantize_row_e4m3(double *x, int d)
{
    int c, e = quantize_row_e4m3(x, d, NULL);
    for (c = 0; c < d; c++)
        x[c] = ldexp(e4m3_value(e4m3_encode((float)ldexp(x[c], -e))), e);
}

/* Rows of a bf16 matrix x [R][d]: codes [R][d] and exponents e [R]. */
void oracle_quantize_rows_e4m3(const uint16_t *x, long R, int d, uint8_t *q, int32_t *e)
{
    long r;
    int c;
    double *row = (double *)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
    if (!row)
        return;
    for (r = 0; r < R; r++) {
        for (c = 0; c < d; c++)
            row[c] = bf16_value(x[r * (long)d + c]);
        e[r] = quantize_row_e4m3(row, d, q + r * (long)d);
    }
    free(row);
}

/* ---- routing plan [P1 sec. 1 items 1-2, sec. 3; P4 Mechanism] ---------- */

/*
 * The plan is a stable counting sort of the flat (token, slot) entries by
 * expert id.  Its result is what [P1]'s serial rank loop computes ("rank =
 * number of earlier entries of the block with the same expert", added to the
 * block's base), which the page's optimised place reproduces bit for bit.
 *
 *   counts[e]      = number of entries routed to expert e
 *   offsets[e]     = sum over e' < e of counts[e'] rounded up to tm
 *   offsets[E]     = R_pad, the padded row total
 *   pos[i]         = row of flat entry i (-1 for a skipped slot)
 *   srt_tok[row]   = token of the entry in that row, -1 in pad rows
 *   srt_w[row]     = routing weight of that entry (bit copy), +0 in pad rows
 *   tile_expert[n] = expert owning rows [n*tm, (n+1)*tm)
 *
 * Returns R_pad, or ORC_ERR_ID if an id lies outside [-1, E), or
 * ORC_ERR_CAP if R_pad exceeds cap.
 */
long oracle_plan(const int32_t *ids, const float *w, int T, int k, int E, int tm,
                 int32_t *offsets, int32_t *counts, int32_t *srt_tok, float *srt_w,
                 int32_t *pos, int32_t *tile_expert, long cap)
{
    long n = (long)T * (long)k;
    long i, r;
    int e;
    int32_t *cursor;

    if (T < 0 || k < 1 || E < 1 || tm < 1)
        return ORC_ERR_ARG;

    /* 1. per-expert row counts (the histogram) */
    for (e = 0; e < E; e++)
        counts[e] = 0;
    for (i = 0; i < n; i++) {
        int id = ids[i];
        if (id == -1)
            continue;
        if (id < -1 || id >= E)
            return ORC_ERR_ID;
        counts[id]++;
    }

    /* 2. exclusive scan of the tile-padded counts, ascending expert id */
    offsets[0] = 0;
    for (e = 0; e < E; e++) {
        long tiles = ((long)counts[e] + tm - 1) / tm;
        offsets[e + 1] = (int32_t)(offsets[e] + tiles * tm);
    }
    if ((long)offsets[E] > cap)
        return ORC_ERR_CAP;

    /* 3. stable place: walk the entries in increasing i with one cursor per
     *    expert that starts at the expert's first row */
    cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!cursor)
        return ORC_ERR_MEM;
    for (e = 0; e < E; e++)
        cursor[e] = offsets[e];
    for (i = 0; i < n; i++) {
        int id = ids[i];
        if (id == -1) {
            pos[i] = -1;
            continue;
        }
        r = cursor[id]++;
        pos[i] = (int32_t)r;
        srt_tok[r] = (int32_t)(i / k);
        srt_w[r] = w[i];
    }
    free(cursor);

    /* 4. the tail rows of each expert's last tile */
    for (e = 0; e < E; e++) {
        for (r = (long)offsets[e] + counts[e]; r < (long)offsets[e + 1]; r++) {
            srt_tok[r] = -1;
            srt_w[r] = 0.0f;
        }
    }

    /* 5. tile table */
    for (e = 0; e < E; e++) {
        long t;
        for (t = offsets[e] / tm; t < offsets[e + 1] / tm; t++)
            tile_expert[t] = e;
    }
    return (long)offsets[E];
}

/* ---- row gather [P1 sec. 1 item 4] ------------------------------------- */

/* xs[r] = x[srt_tok[r]] for a real row, an all-zero row for a pad row. */
void oracle_gather(const uint16_t *x, int T, int d, const int32_t *srt_tok,
                   long R_pad, uint16_t *xs)
{
    long r;
    for (r = 0; r < R_pad; r++) {
        int t = srt_tok[r];
        if (t >= 0 && t < T)
            memcpy(xs + r * (long)d, x + (long)t * d, sizeof(uint16_t) * (size_t)d);
        else
            memset(xs + r * (long)d, 0, sizeof(uint16_t) * (size_t)d);
    }
}

/* ---- one job of the flat expert pass [P3 sec. 1] ----------------------- */

/*
 * For one routed row x (length d) and expert e:
 *   g[n] = sum_c x[c] * Wg[e][c][n]      (c = 0..d-1 in order)
 *   u[n] = sum_c x[c] * Wu[e][c][n]
 *   h[n] = silu(g[n]) * u[n],  silu(z) = z / (1 + exp(-z))
 *   o[m] = sum_n h[n] * Wd[e][n][m]      (n = 0..f-1 in order)
 * Weights have layouts Wg, Wu [E][d][f] and Wd [E][f][d], either bf16 or
 * E4M3 codes with scales [E][f] (gate, up) and [E][d] (down): a weight
 * matrix is read through wmat_t, whose value is exact in fp64 either way.
 * mirror != 0 rounds h to bf16 before the down projection, as a GPU that
 * stores h in bf16 does (used only for the second, reported reference).
 */
typedef struct {
    const uint16_t *b16; /* bf16 weights, or NULL */
    const uint8_t *q8;   /* E4M3 codes when b16 is NULL */
    const float *scale;  /* [E][cols] with q8 */
    long rows, cols;     /* per expert */
} wmat_t;

/* e4m3_value of every code, filled once (same values, looked up) */
static double e4m3_table[256];
static pthread_once_t e4m3_once = PTHREAD_ONCE_INIT;

static void e4m3_fill(void)
{
    int c;
    for (c = 0; c < 256; c++)
        e4m3_table[c] = e4m3_value((uint8_t)c);
}

/* Weight [e][r][c] of W, as a value. */
static double wval(const wmat_t *W, long e, long r, long c)
{
    long i = (e * W->rows + r) * W->cols + c;
    if (W->b16)
        return bf16_value(W->b16[i]);
    return e4m3_table[W->q8[i]] * (double)W->scale[e * W->cols + c];
}

static void expert_job(const uint16_t *xrow, int x_is_f16, const wmat_t *Wg,
                       const wmat_t *Wu, const wmat_t *Wd, long e, int d, int f,
                       int mirror, int a8, double *xv, double *g, double *u, double *h,
                       double *hq, double *o)
{
    int c, n, m;
    for (c = 0; c < d; c++)
        xv[c] = value16(xrow[c], x_is_f16);
    if (a8) /* gate/up sees the row's E4M3 values (quantize_row_e4m3) */
        dequantize_row_e4m3(xv, d);
    for (n = 0; n < f; n++) {
        g[n] = 0.0;
        u[n] = 0.0;
    }
    for (c = 0; c < d; c++) {
        if (Wg->b16 && Wu->b16) { /* the same sums, with the rows addressed once */
            const uint16_t *wg = Wg->b16 + (e * Wg->rows + c) * (long)f;
            const uint16_t *wu = Wu->b16 + (e * Wu->rows + c) * (long)f;
            for (n = 0; n < f; n++) {
                g[n] += xv[c] * bf16_value(wg[n]);
                u[n] += xv[c] * bf16_value(wu[n]);
            }
            continue;
        }
        for (n = 0; n < f; n++) {
            g[n] += xv[c] * wval(Wg, e, c, n);
            u[n] += xv[c] * wval(Wu, e, c, n);
        }
    }
    for (n = 0; n < f; n++) {
        h[n] = g[n] / (1.0 + exp(-g[n])) * u[n];
        if (mirror)
            h[n] = to_bf16(h[n]);
        /* with E4M3 activations h's codes are decided from h as stored, in
         * bf16 (the same precision on both sides: one bf16 step can move a
         * value across an E4M3 midpoint, a whole E4M3 step) */
        hq[n] = a8 ? to_bf16(h[n]) : h[n];
    }
    if (a8) /* ... and the down projection sees those E4M3 values (h itself is kept) */
        dequantize_row_e4m3(hq, f);
    for (m = 0; m < d; m++)
        o[m] = 0.0;
    for (n = 0; n < f; n++) {
        if (Wd->b16) {
            const uint16_t *wd = Wd->b16 + (e * Wd->rows + n) * (long)d;
            for (m = 0; m < d; m++)
                o[m] += hq[n] * bf16_value(wd[m]);
            continue;
        }
        for (m = 0; m < d; m++)
            o[m] += hq[n] * wval(Wd, e, n, m);
    }
}

/* A job: one routed row, its expert, and where its results go. */
typedef struct {
    const uint16_t *xrow;
    int e;
    double *h; /* [f] or NULL */
    double *o; /* [d] */
} job_t;

typedef struct {
    const job_t *jobs;
    long njobs;
    int tid, nthreads;
    int x_is_f16, d, f, mirror, a8;
    const wmat_t *Wg, *Wu, *Wd;
    int failed;
} pass_t;

static void *pass_worker(void *arg)
{
    pass_t *p = (pass_t *)arg;
    long d = p->d, f = p->f, j;
    double *xv = (double *)malloc(sizeof(double) * (size_t)(d + 4 * f));
    double *g, *u, *hbuf, *hq;
    if (!xv) {
        p->failed = 1;
        return NULL;
    }
    g = xv + d;
    u = g + f;
    hbuf = u + f;
    hq = hbuf + f;
    /* jobs are independent; each thread takes every nthreads-th job, so the
     * arithmetic of a job does not depend on the thread count */
    for (j = p->tid; j < p->njobs; j += p->nthreads) {
        const job_t *jb = &p->jobs[j];
        expert_job(jb->xrow, p->x_is_f16, p->Wg, p->Wu, p->Wd, jb->e, p->d, p->f,
                   p->mirror, p->a8, xv, g, u, jb->h ? jb->h : hbuf, hq, jb->o);
    }
    free(xv);
    return NULL;
}

/* Run the flat parallel pass over a job list on nthreads host threads. */
static int run_pass(const job_t *jobs, long njobs, int x_is_f16, int d, int f,
                    int mirror, int a8, const wmat_t *Wg, const wmat_t *Wu,
                    const wmat_t *Wd, int nthreads)
{
    pthread_t th[256];
    pass_t ps[256];
    int started[256];
    int t, failed = 0;
    pthread_once(&e4m3_once, e4m3_fill);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((long)nthreads > njobs)
        nthreads = njobs > 0 ? (int)njobs : 1;
    for (t = 0; t < nthreads; t++) {
        ps[t].jobs = jobs;
        ps[t].njobs = njobs;
        ps[t].tid = t;
        ps[t].nthreads = nthreads;
        ps[t].x_is_f16 = x_is_f16;
        ps[t].d = d;
        ps[t].f = f;
        ps[t].mirror = mirror;
        ps[t].a8 = a8;
        ps[t].Wg = Wg;
        ps[t].Wu = Wu;
        ps[t].Wd = Wd;
        ps[t].failed = 0;
        started[t] = 0;
    }
    for (t = 1; t < nthreads; t++)
        started[t] = pthread_create(&th[t], NULL, pass_worker, &ps[t]) == 0;
    pass_worker(&ps[0]);
    for (t = 1; t < nthreads; t++) {
        if (started[t])
            pthread_join(th[t], NULL);
        else
            pass_worker(&ps[t]); /* could not start a thread: do its share here */
    }
    for (t = 0; t < nthreads; t++)
        failed |= ps[t].failed;
    return failed ? ORC_ERR_MEM : ORC_OK;
}

/* ---- the layer for a set of tokens [P3 sec. 1, sec. 3] ----------------- */

/*
 * y[ti][m] for the tokens tokens[0..ntok-1] (any subset, any order):
 *   build the job list of every (token, slot j) with ids[t*k+j] != -1,
 *   run each job through its expert (expert_job), then for each token
 *   y = sum over j = 0..k-1 in order of w[t*k+j] * o_(t,j), from 0.0.
 * mirror != 0 gives the bf16 mirror instead: h rounded to bf16 in the job,
 * each weighted slot output rounded to bf16, slots summed in fp32 in order,
 * the sum rounded to bf16.
 * Returns ORC_OK, ORC_ERR_ID for an id outside [-1, E), ORC_ERR_ARG for a
 * token outside [0, T), or ORC_ERR_MEM.
 */
static int layer_tokens(const uint16_t *x, int x_is_f16, const int32_t *ids,
                        const float *w, const wmat_t *Wg, const wmat_t *Wu,
                        const wmat_t *Wd, int T, int d, int E, int k, int f,
                        const int32_t *tokens, int ntok, int mirror, int a8, int nthreads,
                        double *y)
{
    long ti, j, nj = 0, m;
    job_t *jobs = NULL;
    double *obuf;
    long *slot_job;
    int rc;

    for (ti = 0; ti < ntok; ti++) {
        int t = tokens[ti];
        if (t < 0 || t >= T)
            return ORC_ERR_ARG;
        for (j = 0; j < k; j++) {
            int e = ids[(long)t * k + j];
            if (e == -1)
                continue;
            if (e < -1 || e >= E)
                return ORC_ERR_ID;
            nj++;
        }
    }
    jobs = (job_t *)calloc((size_t)(nj > 0 ? nj : 1), sizeof(job_t));
    obuf = (double *)malloc(sizeof(double) * (size_t)(nj > 0 ? nj : 1) * (size_t)d);
    slot_job = (long *)malloc(sizeof(long) * (size_t)(ntok > 0 ? ntok : 1) * (size_t)k);
    if (!jobs || !obuf || !slot_job) {
        free(jobs);
        free(obuf);
        free(slot_job);
        return ORC_ERR_MEM;
    }

    /* the immutable job list */
    nj = 0;
    for (ti = 0; ti < ntok; ti++) {
        int t = tokens[ti];
        for (j = 0; j < k; j++) {
            int e = ids[(long)t * k + j];
            if (e == -1) {
                slot_job[ti * k + j] = -1;
                continue;
            }
            jobs[nj].xrow = x + (long)t * d;
            jobs[nj].e = e;
            jobs[nj].h = NULL;
            jobs[nj].o = obuf + nj * (long)d;
            slot_job[ti * k + j] = nj;
            nj++;
        }
    }

    /* one flat pass over all jobs */
    rc = run_pass(jobs, nj, x_is_f16, d, f, mirror, a8, Wg, Wu, Wd, nthreads);

    /* per-token combine in slot order */
    if (rc == ORC_OK) {
        for (ti = 0; ti < ntok; ti++) {
            int t = tokens[ti];
            double *yt = y + ti * (long)d;
            if (!mirror) {
                for (m = 0; m < d; m++)
                    yt[m] = 0.0;
                for (j = 0; j < k; j++) {
                    long jb = slot_job[ti * k + j];
                    double wt;
                    if (jb < 0)
                        continue;
                    wt = (double)w[(long)t * k + j];
                    for (m = 0; m < d; m++)
                        yt[m] += wt * jobs[jb].o[m];
                }
            } else {
                for (m = 0; m < d; m++) {
                    float acc = 0.0f;
                    for (j = 0; j < k; j++) {
                        long jb = slot_job[ti * k + j];
                        if (jb < 0)
                            continue;
                        acc += (float)to_bf16((double)w[(long)t * k + j] * jobs[jb].o[m]);
                    }
                    yt[m] = to_bf16((double)acc);
                }
            }
        }
    }
    free(jobs);
    free(obuf);
    free(slot_job);
    return rc;
}

static wmat_t bf16_mat(const uint16_t *W, long rows, long cols)
{
    wmat_t m = {W, NULL, NULL, rows, cols};
    return m;
}

static wmat_t e4m3_mat(const uint8_t *q, const float *scale, long rows, long cols)
{
    wmat_t m = {NULL, q, scale, rows, cols};
    return m;
}

int oracle_layer_tokens(const uint16_t *x, int x_is_f16, const int32_t *ids,
                        const float *w, const uint16_t *Wg, const uint16_t *Wu,
                        const uint16_t *Wd, int T, int d, int E, int k, int f,
                        const int32_t *tokens, int ntok, int mirror, int nthreads,
                        double *y)
{
    wmat_t g = bf16_mat(Wg, d, f), u = bf16_mat(Wu, d, f), dn = bf16_mat(Wd, f, d);
    return layer_tokens(x, x_is_f16, ids, w, &g, &u, &dn, T, d, E, k, f, tokens, ntok,
                        mirror, 0, nthreads, y);
}

/* The same layer with E4M3 weights: Wg, Wu codes [E][d][f] with scales
 * [E][f], Wd codes [E][f][d] with scales [E][d].  a8 != 0 also gives both
 * projections E4M3 inputs: gate/up each row's E4M3 values and down the
 * E4M3 values of h rounded to bf16 (how h is stored), each quantized per row
 * by quantize_row_e4m3. */
int oracle_layer_tokens_e4m3(const uint16_t *x, int x_is_f16, const int32_t *ids,
                             const float *w, const uint8_t *Wg, const float *sg,
                             const uint8_t *Wu, const float *su, const uint8_t *Wd,
                             const float *sd, int T, int d, int E, int k, int f,
                             const int32_t *tokens, int ntok, int mirror, int a8,
                             int nthreads, double *y)
{
    wmat_t g = e4m3_mat(Wg, sg, d, f), u = e4m3_mat(Wu, su, d, f), dn = e4m3_mat(Wd, sd, f, d);
    return layer_tokens(x, x_is_f16, ids, w, &g, &u, &dn, T, d, E, k, f, tokens, ntok,
                        mirror, a8, nthreads, y);
}

/* ---- stage-level views used to check one GPU stage at a time ------------ */

/*
 * Expert FFN on given routed rows: for each listed row r of xs (16-bit,
 * [*, d]) with expert row_expert[i] and routing weight row_w[i]:
 *   h_out[i][n] = h of that job and ys_out[i][m] = row_w[i] * o[m].
 * Same arithmetic as oracle_layer_tokens' jobs.
 */
static int expert_rows(const uint16_t *xs, int x_is_f16, int d, int f,
                       const int64_t *rows, int nrows, const int32_t *row_expert,
                       const float *row_w, int E, const wmat_t *Wg,
                       const wmat_t *Wu, const wmat_t *Wd, int mirror, int a8,
                       int nthreads, double *h_out, double *ys_out)
{
    long i, m;
    job_t *jobs = (job_t *)calloc((size_t)(nrows > 0 ? nrows : 1), sizeof(job_t));
    int rc;
    if (!jobs)
        return ORC_ERR_MEM;
    for (i = 0; i < nrows; i++) {
        if (row_expert[i] < 0 || row_expert[i] >= E) {
            free(jobs);
            return ORC_ERR_ID;
        }
        jobs[i].xrow = xs + rows[i] * (long)d;
        jobs[i].e = row_expert[i];
        jobs[i].h = h_out + i * (long)f;
        jobs[i].o = ys_out + i * (long)d;
    }
    rc = run_pass(jobs, nrows, x_is_f16, d, f, mirror, a8, Wg, Wu, Wd, nthreads);
    if (rc == ORC_OK) {
        for (i = 0; i < nrows; i++)
            for (m = 0; m < d; m++)
                ys_out[i * (long)d + m] *= (double)row_w[i];
    }
    free(jobs);
    return rc;
}

int oracle_expert_rows(const uint16_t *xs, int x_is_f16, int d, int f,
                       const int64_t *rows, int nrows, const int32_t *row_expert,
                       const float *row_w, int E, const uint16_t *Wg,
                       const uint16_t *Wu, const uint16_t *Wd, int mirror,
                       int nthreads, double *h_out, double *ys_out)
{
    wmat_t g = bf16_mat(Wg, d, f), u = bf16_mat(Wu, d, f), dn = bf16_mat(Wd, f, d);
    return expert_rows(xs, x_is_f16, d, f, rows, nrows, row_expert, row_w, E, &g, &u, &dn,
                       mirror, 0, nthreads, h_out, ys_out);
}

int oracle_expert_rows_e4m3(const uint16_t *xs, int x_is_f16, int d, int f,
                            const int64_t *rows, int nrows, const int32_t *row_expert,
                            const float *row_w, int E, const uint8_t *Wg, const float *sg,
                            const uint8_t *Wu, const float *su, const uint8_t *Wd,
                            const float *sd, int mirror, int a8, int nthreads, double *h_out,
                            double *ys_out)
{
    wmat_t g = e4m3_mat(Wg, sg, d, f), u = e4m3_mat(Wu, su, d, f), dn = e4m3_mat(Wd, sd, f, d);
    return expert_rows(xs, x_is_f16, d, f, rows, nrows, row_expert, row_w, E, &g, &u, &dn,
                       mirror, a8, nthreads, h_out, ys_out);
}

/*
 * Combine of given weighted rows: y[t][m] = sum over j = 0..k-1 in order of
 * Ys[pos[t*k+j]][m] (bf16 rows, skipped when pos is -1), in fp64 from 0.0.
 */
void oracle_combine(const uint16_t *Ys, const int32_t *pos, int T, int k, int d,
                    double *y)
{
    long t, j, m;
    for (t = 0; t < T; t++) {
        double *yt = y + t * (long)d;
        for (m = 0; m < d; m++)
            yt[m] = 0.0;
        for (j = 0; j < k; j++) {
            long p = pos[t * k + j];
            if (p < 0)
                continue;
            for (m = 0; m < d; m++)
                yt[m] += bf16_value(Ys[p * (long)d + m]);
        }
    }
}

/* bf16 rounding as the oracle does it, exposed so the tests can pin it. */
double oracle_round_bf16(double v) { return to_bf16(v); }
double oracle_value16(uint16_t b, int is_f16) { return value16(b, is_f16); }
double oracle_e4m3_value(uint8_t c) { return e4m3_value(c); }
uint8_t oracle_e4m3_encode(float v) { return e4m3_encode(v); }
double oracle_e2m1_value(uint8_t c) { return e2m1_value(c); }
uint8_t oracle_e2m1_encode(double v) { return e2m1_encode(v); }

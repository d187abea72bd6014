/*
 * moe_oracle.c -- the CPU oracle of the quantized MoE decode layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load it. Plain loops, f64 unless the
 * page fixes a precision, no blocking, no fusion. Build with
 * -ffp-contract=off: the f32 steps of the selection must not be contracted.
 *
 * Pins (tests/test_oracle_*.py, run without a GPU): bf16 / f16 conversions
 * against library conversions; hand-packed Q2_K / Q3_K blocks against closed
 * forms; the integer-dot form against the dequantise-then-dot form by brute
 * force; q8_1 round-trip bounds; router sums against exact rational sums;
 * each step of the score against 60-digit arithmetic; the selection against brute force over
 * all k-subsets and its invariants; SwiGLU against its closed form; the
 * layer against special cases with closed-form outputs.
 */
#include "moe_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- numbers */

/* f32 -> bf16 by round-to-nearest-even: add 0x7FFF plus the lowest kept bit
 * and keep the high half (moe_v41.rs, fn bf16_bytes). */
uint16_t orc_bf16_from_f32(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    uint32_t lsb = (b >> 16) & 1u;
    return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

double orc_bf16_to_f64(uint16_t h)
{
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* IEEE binary16 -> f64 (exact). */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, mant = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)mant, -24);
    else if (e == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), e - 25);
    return sign ? -v : v;
}

/* f32 -> IEEE binary16, round to nearest even, from the definition: drop the
 * low bits of the 24-bit significand, round the remainder half to even. */
uint16_t orc_f16_from_f32(float f)
{
    uint32_t b;
    memcpy(&b, &f, 4);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    uint32_t a = b & 0x7FFFFFFFu;
    if (a >= 0x7F800000u)
        return sign | (a > 0x7F800000u ? 0x7E00 : 0x7C00);
    int e = (int)(a >> 23);
    if (e == 0)
        return sign; /* f32 subnormals are far below half the f16 unit */
    uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
    int E = e - 127 + 15; /* binary16 biased exponent if normal */
    int shift = E >= 1 ? 13 : 14 - E;
    if (shift > 25)
        return sign;
    uint32_t q = mant >> shift;
    uint32_t rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q++;
    if (E >= 1) {
        uint32_t h = ((uint32_t)E << 10) + (q - 1024u);
        if (h >= 0x7C00u)
            return sign | 0x7C00;
        return sign | (uint16_t)h;
    }
    return sign | (uint16_t)q; /* subnormal (q = 1024 is the smallest normal) */
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ------------------------------------------------------------ K-quant blocks */

/* Q2_K super-block, 84 bytes, 256 weights (public GGUF layout; the pages name
 * the format, moe_v41.rs MoeV41LayerWeights, and give no layout):
 *   scales[16]  byte s: low nibble = 4-bit scale, high nibble = 4-bit min of
 *               sub-block s (16 weights)
 *   qs[64]      2-bit quants: weight j sits in byte 32*(j/128) + j%32 at bit
 *               offset 2*((j%128)/32)
 *   d, dmin     f16 super-block factors for the scales and the mins
 * weight j = d * scale(j/16) * q_j - dmin * min(j/16). */
void orc_dequant_q2k(const uint8_t *blk, double w[256])
{
    const uint8_t *scales = blk, *qs = blk + 16;
    double d = orc_f16_to_f64(rd16(blk + 80)), dmin = orc_f16_to_f64(rd16(blk + 82));
    for (int j = 0; j < 256; j++) {
        int half = j / 128, g = (j % 128) / 32, l = j % 32, s = j / 16;
        int q = (qs[32 * half + l] >> (2 * g)) & 3;
        w[j] = d * (double)(scales[s] & 15) * (double)q - dmin * (double)(scales[s] >> 4);
    }
}

/* Q3_K super-block, 110 bytes, 256 weights (public GGUF layout):
 *   hmask[32]   high bit of weight j = bit j/32 of hmask[j%32]
 *   qs[64]      low two bits, placed as in Q2_K
 *   scales[12]  sixteen 6-bit scales: low 4 bits of scale i in byte i (i<8,
 *               low nibble) or byte i-8 (i>=8, high nibble); high 2 bits at
 *               bit 2*(i/4) of byte 8 + i%4; stored with a +32 offset
 *   d           f16 super-block factor
 * q_j = low2 - (high bit ? 0 : 4) in [-4, 3]; weight j = d * (scale(j/16)) * q_j. */
void orc_dequant_q3k(const uint8_t *blk, double w[256])
{
    const uint8_t *hmask = blk, *qs = blk + 32, *sc = blk + 96;
    double d = orc_f16_to_f64(rd16(blk + 108));
    for (int j = 0; j < 256; j++) {
        int half = j / 128, g = (j % 128) / 32, l = j % 32, i = j / 16;
        int low2 = (qs[32 * half + l] >> (2 * g)) & 3;
        int hbit = (hmask[l] >> (j / 32)) & 1;
        int q = low2 - (hbit ? 0 : 4);
        int low4 = i < 8 ? (sc[i] & 15) : (sc[i - 8] >> 4);
        int high2 = (sc[8 + i % 4] >> (2 * (i / 4))) & 3;
        int scale = (low4 | (high2 << 4)) - 32;
        w[j] = d * (double)scale * (double)q;
    }
}

/* q8_1 block: f16 d, f16 s, int8 q[32] (36 bytes) -- the activation format
 * the K-quant GEMVs consume (moe_v41.rs module doc: activation quantised to
 * q8_1). Decisions in f32: amax = max |x|, d = amax / 127 (one f32
 * rounding), q = round-half-away(x / d) with an f32 division, q = 0 when
 * amax = 0; stored d = f16(d), s = f16(d * sum q). */
void orc_quant_q8_1(const float *x, int n, uint8_t *out)
{
    for (int b = 0; b < n / 32; b++) {
        const float *xb = x + 32 * b;
        uint8_t *o = out + 36 * b;
        float amax = 0.0f;
        for (int i = 0; i < 32; i++) {
            float a = fabsf(xb[i]);
            if (a > amax)
                amax = a;
        }
        float d = amax / 127.0f;
        int sum = 0;
        for (int i = 0; i < 32; i++) {
            int q = amax == 0.0f ? 0 : (int)roundf(xb[i] / d);
            o[4 + i] = (uint8_t)(int8_t)q;
            sum += q;
        }
        uint16_t dh = orc_f16_from_f32(d), sh = orc_f16_from_f32(d * (float)sum);
        o[0] = (uint8_t)dh;
        o[1] = (uint8_t)(dh >> 8);
        o[2] = (uint8_t)sh;
        o[3] = (uint8_t)(sh >> 8);
    }
}

/* value i of a q8_1 block = f16(d) * q_i */
void orc_dequant_q8_1(const uint8_t *blk, double v[32])
{
    double d = orc_f16_to_f64(rd16(blk));
    for (int i = 0; i < 32; i++)
        v[i] = d * (double)(int8_t)blk[4 + i];
}

static double clampd(double v, double lo, double hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* Input-making only (the tiny layer's experts are quantised N(0, 0.02)
 * weights): a simple non-iterative Q2_K quantiser. Per 16-weight sub-block,
 * min = -min(0, min x), scale = (max x + min) / 3; d, dmin = the largest scale
 * and min over 15, stored f16; codes rounded against the stored factors. */
void orc_quantize_q2k(const float *x, uint8_t *blk)
{
    double scale[16], mins[16], ms = 0, mm = 0;
    for (int s = 0; s < 16; s++) {
        double mn = 0, mx = -INFINITY;
        for (int i = 0; i < 16; i++) {
            double v = x[16 * s + i];
            if (v < mn)
                mn = v;
            if (v > mx)
                mx = v;
        }
        scale[s] = (mx - mn) / 3.0;
        mins[s] = -mn;
        if (scale[s] > ms)
            ms = scale[s];
        if (mins[s] > mm)
            mm = mins[s];
    }
    memset(blk, 0, 84);
    uint16_t dh = orc_f16_from_f32((float)(ms / 15.0)), mh = orc_f16_from_f32((float)(mm / 15.0));
    double d = orc_f16_to_f64(dh), dmin = orc_f16_to_f64(mh);
    for (int s = 0; s < 16; s++) {
        int sc = d > 0 ? (int)clampd(round(scale[s] / d), 0, 15) : 0;
        int mc = dmin > 0 ? (int)clampd(round(mins[s] / dmin), 0, 15) : 0;
        blk[s] = (uint8_t)(sc | (mc << 4));
        double step = d * sc;
        for (int i = 0; i < 16; i++) {
            int j = 16 * s + i;
            int q = step > 0 ? (int)clampd(round((x[j] + dmin * mc) / step), 0, 3) : 0;
            blk[16 + 32 * (j / 128) + j % 32] |= (uint8_t)(q << (2 * ((j % 128) / 32)));
        }
    }
    blk[80] = (uint8_t)dh;
    blk[81] = (uint8_t)(dh >> 8);
    blk[82] = (uint8_t)mh;
    blk[83] = (uint8_t)(mh >> 8);
}

/* Input-making only: a simple non-iterative Q3_K quantiser. Per sub-block,
 * the element of largest magnitude v maps to -4: scale = -v / 4; d = the
 * largest |scale| / 31 stored f16; 6-bit codes and quants rounded against the
 * stored factors. */
void orc_quantize_q3k(const float *x, uint8_t *blk)
{
    double scale[16], ma = 0;
    for (int s = 0; s < 16; s++) {
        double v = 0;
        for (int i = 0; i < 16; i++)
            if (fabs(x[16 * s + i]) > fabs(v))
                v = x[16 * s + i];
        scale[s] = -v / 4.0;
        if (fabs(scale[s]) > ma)
            ma = fabs(scale[s]);
    }
    memset(blk, 0, 110);
    uint16_t dh = orc_f16_from_f32((float)(ma / 31.0));
    double d = orc_f16_to_f64(dh);
    for (int s = 0; s < 16; s++) {
        int code = d > 0 ? (int)clampd(round(scale[s] / d), -32, 31) : 0;
        int c6 = code + 32;
        if (s < 8)
            blk[96 + s] |= (uint8_t)(c6 & 15);
        else
            blk[96 + s - 8] |= (uint8_t)((c6 & 15) << 4);
        blk[96 + 8 + s % 4] |= (uint8_t)(((c6 >> 4) & 3) << (2 * (s / 4)));
        double step = d * code;
        for (int i = 0; i < 16; i++) {
            int j = 16 * s + i;
            int q = step != 0 ? (int)clampd(round(x[j] / step), -4, 3) : 0;
            int hbit = q >= 0, low2 = q >= 0 ? q : q + 4;
            blk[32 + 32 * (j / 128) + j % 32] |= (uint8_t)(low2 << (2 * ((j % 128) / 32)));
            if (hbit)
                blk[j % 32] |= (uint8_t)(1u << (j / 32));
        }
    }
    blk[108] = (uint8_t)dh;
    blk[109] = (uint8_t)(dh >> 8);
}

/* ------------------------------------------------------------------ router */

/* logits[t, e] = sum_j x[t, j] * W[e, j]: bf16 operands, products exact, the
 * sum in f64, rounded once to f32 (moe_v41.rs module doc: an f32-accumulated
 * GEMM of the bf16 input against the bf16 gate weight). */
void orc_router_logits(const uint16_t *x, const uint16_t *w, int dim, int n, int m,
                       float *logits)
{
    for (int t = 0; t < m; t++)
        for (int e = 0; e < n; e++) {
            double s = 0.0;
            for (int j = 0; j < dim; j++)
                s += orc_bf16_to_f64(x[(size_t)t * dim + j]) * orc_bf16_to_f64(w[(size_t)e * dim + j]);
            logits[(size_t)t * n + e] = (float)s;
        }
}

/* ---------------------------------------------------------------- selection */

/* 1 when the long-double value v lies within 2^-56 (relative) of the
 * midpoint between r = (float)v and its neighbour on v's side: there the
 * long-double evaluation (error far below 2^-60 relative) cannot certify on
 * which side of the midpoint the exact value lies. */
static int near_midpoint(long double v, float r)
{
    if (!isfinite(r) || (long double)r == v)
        return 0;
    float nb = v > (long double)r ? nextafterf(r, INFINITY) : nextafterf(r, -INFINITY);
    long double mid = ((long double)r + (long double)nb) / 2.0L;
    return fabsl(v - mid) <= ldexpl(fabsl(v), -56);
}

/* The f32 rounding (to nearest, ties to even) of an exact value known as the
 * long double v; *near_mid is set when that rounding is not certain. */
static float rn_f32(long double v, int *near_mid)
{
    float r = (float)v;
    if (near_midpoint(v, r))
        *near_mid = 1;
    return r;
}

/* score = sqrt(softplus(logit / temp)) as the page writes it in f32
 * (moe_v41.rs, fn softplus: x for x > 20, else x.exp().ln_1p(); fn
 * route_from_logits: the .sqrt() of that), each f32 operation taken as
 * correctly rounded:
 *   t  = f32(logit / temp)
 *   e  = f32(e^t)                (t <= 20)
 *   sp = f32(ln(1 + e))          (t <= 20), else sp = t
 *   s  = f32(sqrt(sp))
 * e and sp are evaluated in long double and rounded to f32; *near_mid is set
 * when either rounding lies within 2^-56 of a midpoint (then not certain). */
float orc_score(float logit, float temp, int *near_mid)
{
    int nm = 0;
    float t = logit / temp;
    float sp;
    if (t > 20.0f) {
        sp = t;
    } else {
        float e = rn_f32(expl((long double)t), &nm);
        sp = rn_f32(log1pl((long double)e), &nm);
    }
    if (near_mid)
        *near_mid = nm;
    return sqrtf(sp);
}

/* a ranks before b: larger key first, NaN keys after all others, equal keys
 * (and NaN pairs) by ascending expert id -- the order a stable sort of ids
 * 0..n-1 by descending key gives (moe_v41.rs, fn route_from_logits). */
static int ranks_before(float ka, int a, float kb, int b)
{
    int na = isnan(ka), nb = isnan(kb);
    if (na || nb) {
        if (na && nb)
            return a < b;
        return nb;
    }
    if (ka > kb)
        return 1;
    if (ka < kb)
        return 0;
    return a < b;
}

/* The selection of moe_v41.rs fn route_from_logits, per token:
 *   scores s_e = score(logit_e); keys s_e + bias_e (f32 add);
 *   order = ids stably sorted by descending key; picks = its first k;
 *   weights = the picks' unbiased scores; if norm_topk_prob and k > 1 they
 *   are divided by (f32 sum in pick order) + 1e-20; then times route_scale.
 * picks / weights [m*k] in pick order; scores [m*n] optional; flags [m]. */
int orc_route(const orc_cfg *c, const float *logits, const float *bias, int m,
              int32_t *picks, float *weights, float *scores, int32_t *flags)
{
    int n = c->n_routed, k = c->topk;
    float *sc = (float *)malloc(sizeof(float) * n), *key = (float *)malloc(sizeof(float) * n);
    int *order = (int *)malloc(sizeof(int) * n);
    if (!sc || !key || !order) {
        free(sc);
        free(key);
        free(order);
        return -1;
    }
    for (int t = 0; t < m; t++) {
        int fl = 0;
        for (int e = 0; e < n; e++) {
            int nm = 0;
            float l = logits[(size_t)t * n + e];
            sc[e] = orc_score(l, c->gate_temp, &nm);
            key[e] = sc[e] + bias[e];
            if (nm)
                fl |= ORC_FLAG_NEAR_MID;
            if (!isfinite(l) || !isfinite(key[e]))
                fl |= ORC_FLAG_NONFINITE;
            if (scores)
                scores[(size_t)t * n + e] = sc[e];
        }
        /* stable insertion sort of ids by descending key */
        for (int i = 0; i < n; i++) {
            int id = i, j = i;
            while (j > 0 && ranks_before(key[id], id, key[order[j - 1]], order[j - 1])) {
                order[j] = order[j - 1];
                j--;
            }
            order[j] = id;
        }
        float wt[64];
        for (int i = 0; i < k; i++) {
            picks[(size_t)t * k + i] = order[i];
            wt[i] = sc[order[i]];
        }
        if (c->norm_topk_prob && k > 1) {
            float sum = 0.0f;
            for (int i = 0; i < k; i++)
                sum = sum + wt[i];
            sum = sum + 1e-20f;
            for (int i = 0; i < k; i++)
                wt[i] = wt[i] / sum;
        }
        for (int i = 0; i < k; i++)
            weights[(size_t)t * k + i] = wt[i] * c->route_scale;
        if (flags)
            flags[t] = fl;
    }
    free(sc);
    free(key);
    free(order);
    return 0;
}

/* The route header, the plan and the pointer table of m tokens from their
 * picks and weights (pick order), as moe_v41/device_route.rs describes them:
 * module doc and fn header_words (per token: status, picks, weight bits, the
 * slots of the plan), fn route_select_launch (pointer = base + slot *
 * slot_bytes + offset; a slot of -1 is read as slot 0 and sets the miss
 * flag), fn device_route_check (the plan in ascending expert id). The pages
 * give the layout for one token; for m tokens the reading is one header row
 * per token, then the plan tail:
 *   row t, 1 + 3k words: [0] status (flags & ORC_FLAG_NONFINITE, | 1 for a
 *     miss); [1..k] picks; [k+1..2k] weight bits; [2k+1..3k] the slots of
 *     the token's picks in ascending id (-1 written as 0);
 *   tail at po = m (1 + 3k): [po] ne = distinct picked experts;
 *     [po + 1 + p] = first pair of plan expert p (p < ne), [po + 1 + ne] =
 *     m k; [po + 2 + m k + p] = plan expert p (ascending id).
 * Pairs (expert, token) run expert by expert in ascending id, tokens ascending
 * within one; plan_w / plan_rows hold each pair's weight and token; ptrs holds
 * gate at [p], up at [m k + p], down at [2 m k + p] for plan expert p. Words
 * of hdr beyond these are left as they are. Returns ne. */
int orc_plan(int m, int k, int n, const int32_t *picks, const float *weights,
             const int32_t *flags, const int32_t *slot_row, uint64_t base,
             uint64_t slot_bytes, uint64_t gate_off, uint64_t up_off, uint64_t down_off,
             int32_t *hdr, float *plan_w, int32_t *plan_rows, uint64_t *ptrs)
{
    int cap = m * k, po = m * (1 + 3 * k);
    for (int t = 0; t < m; t++) {
        int32_t *row = hdr + (size_t)t * (1 + 3 * k);
        int status = flags ? (flags[t] & ORC_FLAG_NONFINITE) : 0;
        int asc[64];
        for (int i = 0; i < k; i++) {
            row[1 + i] = picks[t * k + i];
            memcpy(&row[1 + k + i], &weights[t * k + i], 4);
            asc[i] = picks[t * k + i];
        }
        for (int i = 1; i < k; i++)
            for (int j = i; j > 0 && asc[j] < asc[j - 1]; j--) {
                int v = asc[j];
                asc[j] = asc[j - 1];
                asc[j - 1] = v;
            }
        for (int i = 0; i < k; i++) {
            int sl = slot_row[asc[i]];
            if (sl < 0)
                status |= 1;
            row[1 + 2 * k + i] = sl < 0 ? 0 : sl;
        }
        row[0] = status;
    }
    int ne = 0, q = 0;
    for (int e = 0; e < n; e++) {
        int first = q;
        for (int t = 0; t < m; t++)
            for (int i = 0; i < k; i++)
                if (picks[t * k + i] == e) {
                    plan_rows[q] = t;
                    plan_w[q] = weights[t * k + i];
                    q++;
                }
        if (q == first)
            continue;
        int sl = slot_row[e] < 0 ? 0 : slot_row[e];
        uint64_t b = base + (uint64_t)sl * slot_bytes;
        ptrs[ne] = b + gate_off;
        ptrs[cap + ne] = b + up_off;
        ptrs[2 * cap + ne] = b + down_off;
        hdr[po + 1 + ne] = first;
        hdr[po + 2 + cap + ne] = e;
        ne++;
    }
    hdr[po] = ne;
    hdr[po + 1 + ne] = q;
    return ne;
}

/* Clamped SwiGLU: silu(min(g, L)) * clamp(u, -L, L), silu(z) = z / (1 + e^-z);
 * L <= 0 means no clamp (moe_v41.rs MoeV41Cfg swiglu_limit; the page names
 * the limit and not the formula). */
double orc_swiglu(double g, double u, double limit)
{
    if (limit > 0) {
        if (g > limit)
            g = limit;
        u = clampd(u, -limit, limit);
    }
    return g / (1.0 + exp(-g)) * u;
}

/* ------------------------------------------------------ row-parallel helper */

typedef struct {
    void (*fn)(void *ctx, int r0, int r1);
    void *ctx;
    int r0, r1;
} orc_job;

static void *orc_job_run(void *p)
{
    orc_job *j = (orc_job *)p;
    j->fn(j->ctx, j->r0, j->r1);
    return NULL;
}

/* runs fn over rows [0, rows) split into `threads` contiguous ranges; each
 * row is computed exactly as in the single-threaded loop */
static void orc_parallel_rows(void (*fn)(void *, int, int), void *ctx, int rows, int threads)
{
    if (threads <= 1 || rows < 2 * threads) {
        fn(ctx, 0, rows);
        return;
    }
    if (threads > 256)
        threads = 256;
    pthread_t th[256];
    orc_job jobs[256];
    int ok[256];
    for (int i = 0; i < threads; i++) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].r0 = (int)((long)rows * i / threads);
        jobs[i].r1 = (int)((long)rows * (i + 1) / threads);
        ok[i] = i > 0 && pthread_create(&th[i], NULL, orc_job_run, &jobs[i]) == 0;
    }
    fn(ctx, jobs[0].r0, jobs[0].r1);
    for (int i = 1; i < threads; i++) {
        if (ok[i])
            pthread_join(th[i], NULL);
        else
            fn(ctx, jobs[i].r0, jobs[i].r1); /* thread creation failed: run inline */
    }
}

/* ------------------------------------------------------------------ experts */

typedef struct {
    const uint8_t *blocks; /* rows of K-quant super-blocks */
    int nb, q3;            /* super-blocks per row, Q3_K (else Q2_K) */
    const double *v;       /* dequantised activation */
    double *out;
} orc_gemv_ctx;

/* out[r] = sum_j dequant(W)[r, j] * v[j] in f64 */
static void orc_gemv_rows(void *p, int r0, int r1)
{
    orc_gemv_ctx *c = (orc_gemv_ctx *)p;
    size_t bb = c->q3 ? 110 : 84;
    double w[256];
    for (int r = r0; r < r1; r++) {
        double s = 0.0;
        for (int b = 0; b < c->nb; b++) {
            const uint8_t *blk = c->blocks + ((size_t)r * c->nb + b) * bb;
            if (c->q3)
                orc_dequant_q3k(blk, w);
            else
                orc_dequant_q2k(blk, w);
            for (int j = 0; j < 256; j++)
                s += w[j] * c->v[256 * b + j];
        }
        c->out[r] = s;
    }
}

static void orc_dequant_q8_row(const uint8_t *q8, int n, double *v)
{
    for (int b = 0; b < n / 32; b++)
        orc_dequant_q8_1(q8 + 36 * b, v + 32 * b);
}

/* One routed expert for one token (moe_v41.rs module doc: three K-quant
 * GEMVs on the raw blocks, gate and up Q2_K, down Q3_K, the activation
 * quantised to q8_1 in between):
 *   g, u = dequant(Q2_K) . dequant(q8_1 x)          (f64, stored f32)
 *   h    = SwiGLU(g, u)                               (f64, stored f32)
 *   h_q8 = q8_1(h)                                    (f32 decisions)
 *   dn   = dequant(Q3_K) . dequant(h_q8)              (f64, stored f32)  */
void orc_expert_token(const orc_cfg *c, const uint8_t *gate, const uint8_t *up,
                      const uint8_t *down, const uint8_t *x_q8, float *g, float *u,
                      float *h, uint8_t *h_q8, float *dn, int threads)
{
    int dim = c->dim, inter = c->inter;
    double *xv = (double *)malloc(sizeof(double) * dim);
    double *gd = (double *)malloc(sizeof(double) * inter), *ud = (double *)malloc(sizeof(double) * inter);
    double *hv = (double *)malloc(sizeof(double) * inter), *dd = (double *)malloc(sizeof(double) * dim);
    float *hf = (float *)malloc(sizeof(float) * inter);
    orc_dequant_q8_row(x_q8, dim, xv);
    orc_gemv_ctx cg = {gate, dim / 256, 0, xv, gd}, cu = {up, dim / 256, 0, xv, ud};
    orc_parallel_rows(orc_gemv_rows, &cg, inter, threads);
    orc_parallel_rows(orc_gemv_rows, &cu, inter, threads);
    for (int r = 0; r < inter; r++) {
        hf[r] = (float)orc_swiglu(gd[r], ud[r], c->swiglu_limit);
        if (g)
            g[r] = (float)gd[r];
        if (u)
            u[r] = (float)ud[r];
        if (h)
            h[r] = hf[r];
    }
    uint8_t *hq = h_q8 ? h_q8 : (uint8_t *)malloc((size_t)36 * inter / 32);
    orc_quant_q8_1(hf, inter, hq);
    orc_dequant_q8_row(hq, inter, hv);
    orc_gemv_ctx cd = {down, inter / 256, 1, hv, dd};
    orc_parallel_rows(orc_gemv_rows, &cd, dim, threads);
    for (int r = 0; r < dim; r++)
        dn[r] = (float)dd[r];
    if (!h_q8)
        free(hq);
    free(xv);
    free(gd);
    free(ud);
    free(hv);
    free(dd);
    free(hf);
}

typedef struct {
    const uint16_t *w; /* bf16 rows */
    int cols;
    const double *v;
    double *out;
} orc_bf16_ctx;

static void orc_bf16_rows(void *p, int r0, int r1)
{
    orc_bf16_ctx *c = (orc_bf16_ctx *)p;
    for (int r = r0; r < r1; r++) {
        double s = 0.0;
        for (int j = 0; j < c->cols; j++)
            s += orc_bf16_to_f64(c->w[(size_t)r * c->cols + j]) * c->v[j];
        c->out[r] = s;
    }
}

/* The bf16 shared expert for one token (moe_v41.rs module doc: resident bf16,
 * on the dense GEMM): gs, us = W1 x, W3 x (f64, stored f32); hs = bf16 of the
 * f32-rounded SwiGLU(gs, us); sd = W2 hs (f64, stored f32). */
void orc_shared_token(const orc_cfg *c, const uint16_t *w1, const uint16_t *w3,
                      const uint16_t *w2, const uint16_t *x, float *gs, float *us,
                      uint16_t *hs, float *sd, int threads)
{
    int dim = c->dim, inter = c->inter;
    double *xv = (double *)malloc(sizeof(double) * dim), *hv = (double *)malloc(sizeof(double) * inter);
    double *gd = (double *)malloc(sizeof(double) * inter), *ud = (double *)malloc(sizeof(double) * inter);
    double *dd = (double *)malloc(sizeof(double) * dim);
    for (int j = 0; j < dim; j++)
        xv[j] = orc_bf16_to_f64(x[j]);
    orc_bf16_ctx c1 = {w1, dim, xv, gd}, c3 = {w3, dim, xv, ud};
    orc_parallel_rows(orc_bf16_rows, &c1, inter, threads);
    orc_parallel_rows(orc_bf16_rows, &c3, inter, threads);
    for (int r = 0; r < inter; r++) {
        uint16_t hb = orc_bf16_from_f32((float)orc_swiglu(gd[r], ud[r], c->swiglu_limit));
        hv[r] = orc_bf16_to_f64(hb);
        if (gs)
            gs[r] = (float)gd[r];
        if (us)
            us[r] = (float)ud[r];
        if (hs)
            hs[r] = hb;
    }
    orc_bf16_ctx c2 = {w2, inter, hv, dd};
    orc_parallel_rows(orc_bf16_rows, &c2, dim, threads);
    for (int r = 0; r < dim; r++)
        sd[r] = (float)dd[r];
    free(xv);
    free(hv);
    free(gd);
    free(ud);
    free(dd);
}

/* -------------------------------------------------------------------- layer */

/* One MoE layer step (sh_kquant: the shared expert's w1, w3 are Q2_K and w2
 * Q3_K blocks, passed through the uint16_t pointers as raw bytes):
 *   logits, picks, weights as above; per token the plan = its picks in
 *   ascending expert id (moe_v41/device_route.rs, fn device_route_check:
 *   plan weights in ascending id);
 *   acc = sum over the plan, in that order, of w * down (f32), then the
 *   shared expert's output is added last (moe_v41.rs, fn shared_side: added
 *   into acc after the routed experts);
 *   residual += acc; x_next = bf16(residual). */
int orc_layer(const orc_cfg *c, int m, const uint16_t *x, const uint16_t *router_w,
              const float *bias, const uint8_t *const *experts, uint64_t gate_off,
              uint64_t up_off, uint64_t down_off, const uint16_t *sh_w1,
              const uint16_t *sh_w3, const uint16_t *sh_w2, int sh_kquant, float *residual,
              uint16_t *x_next, float *logits, int32_t *picks, float *weights,
              int32_t *flags, float *acc, float *sd, int threads)
{
    int n = c->n_routed, k = c->topk, dim = c->dim;
    float *lg = (float *)malloc(sizeof(float) * (size_t)m * n);
    int32_t *pk = (int32_t *)malloc(sizeof(int32_t) * (size_t)m * k);
    float *wt = (float *)malloc(sizeof(float) * (size_t)m * k);
    int32_t *fl = (int32_t *)malloc(sizeof(int32_t) * (size_t)m);
    float *xf = (float *)malloc(sizeof(float) * dim), *dn = (float *)malloc(sizeof(float) * dim);
    float *a = (float *)malloc(sizeof(float) * dim), *s = (float *)malloc(sizeof(float) * dim);
    uint8_t *xq = (uint8_t *)malloc((size_t)36 * dim / 32);
    int rc = 0;
    orc_router_logits(x, router_w, dim, n, m, lg);
    orc_route(c, lg, bias, m, pk, wt, NULL, fl);
    for (int t = 0; t < m && rc == 0; t++) {
        const uint16_t *xt = x + (size_t)t * dim;
        for (int j = 0; j < dim; j++)
            xf[j] = (float)orc_bf16_to_f64(xt[j]);
        orc_quant_q8_1(xf, dim, xq);
        for (int r = 0; r < dim; r++)
            a[r] = 0.0f;
        /* the plan: this token's picks in ascending expert id */
        int plan[64];
        float pw[64];
        for (int i = 0; i < k; i++) {
            plan[i] = pk[(size_t)t * k + i];
            pw[i] = wt[(size_t)t * k + i];
        }
        for (int i = 1; i < k; i++)
            for (int j = i; j > 0 && plan[j] < plan[j - 1]; j--) {
                int ti = plan[j];
                plan[j] = plan[j - 1];
                plan[j - 1] = ti;
                float tw = pw[j];
                pw[j] = pw[j - 1];
                pw[j - 1] = tw;
            }
        for (int i = 0; i < k; i++) {
            const uint8_t *slot = experts[plan[i]];
            if (!slot) {
                rc = -1;
                break;
            }
            orc_expert_token(c, slot + gate_off, slot + up_off, slot + down_off, xq, NULL, NULL,
                             NULL, NULL, dn, threads);
            for (int r = 0; r < dim; r++)
                a[r] = a[r] + pw[i] * dn[r];
        }
        if (rc)
            break;
        if (sh_w1 && sh_w3 && sh_w2 && sh_kquant) {
            /* the shared expert on the routed experts' kernels (moe_v41.rs
             * MoeV41LayerWeights: Q2_K w1, w3 and Q3_K w2; struct MoeV41
             * sh_q8: its own q8_1 of the SwiGLU output): the routed
             * expert's arithmetic, weight 1, added after the routed sum */
            orc_expert_token(c, (const uint8_t *)sh_w1, (const uint8_t *)sh_w3,
                             (const uint8_t *)sh_w2, xq, NULL, NULL, NULL, NULL, s, threads);
            for (int r = 0; r < dim; r++)
                a[r] = a[r] + s[r];
        } else if (sh_w1 && sh_w3 && sh_w2) {
            orc_shared_token(c, sh_w1, sh_w3, sh_w2, xt, NULL, NULL, NULL, s, threads);
            for (int r = 0; r < dim; r++)
                a[r] = a[r] + s[r];
        } else {
            for (int r = 0; r < dim; r++)
                s[r] = 0.0f;
        }
        for (int r = 0; r < dim; r++) {
            float *res = residual + (size_t)t * dim + r;
            *res = *res + a[r];
            x_next[(size_t)t * dim + r] = orc_bf16_from_f32(*res);
            if (acc)
                acc[(size_t)t * dim + r] = a[r];
            if (sd)
                sd[(size_t)t * dim + r] = s[r];
        }
    }
    if (logits)
        memcpy(logits, lg, sizeof(float) * (size_t)m * n);
    if (picks)
        memcpy(picks, pk, sizeof(int32_t) * (size_t)m * k);
    if (weights)
        memcpy(weights, wt, sizeof(float) * (size_t)m * k);
    if (flags)
        memcpy(flags, fl, sizeof(int32_t) * (size_t)m);
    free(lg);
    free(pk);
    free(wt);
    free(fl);
    free(xf);
    free(dn);
    free(a);
    free(s);
    free(xq);
    return rc;
}

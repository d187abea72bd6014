// moe_route.cu -- router logits and the device selection.
//
// One launch does both: every CTA computes the logits of its router rows
// (weights prefetched into shared memory by one bulk copy before the
// programmatic-launch wait, so the fetch overlaps the previous kernel), then
// takes a ticket; the CTA that takes the last ticket runs the selection for
// all tokens and writes the route header, the plan weights and rows and the
// gate/up/down pointer table (page spark_model/layers/moe_v41/device_route.rs,
// module doc and fn route_select_launch). No CTA ever waits on another.
//
// Selection (page spark_model/layers/moe_v41.rs, fn softplus and
// fn route_from_logits): score = the f32 chain sqrt(ln_1p(exp(l / temp))),
// each step correctly rounded, key = score + bias, stable descending order,
// top k, weights renormalised in f32. The score is evaluated in the router
// epilogue, where every CTA takes a few of the rows, in float-float single
// precision with double-precision fallbacks near rounding midpoints (FP64 is
// a slow pipe on GB300). The selecting CTA is latency-bound: it reads everything it needs in
// one round of loads, ranks each token with one warp (k rounds of a warp-wide
// maximum over 64-bit sortable values), and only stores afterwards.
#pragma once
#include "moe_common.cuh"

namespace moe {

struct RouteArgs {
    const uint16_t *x;  // bf16 [m, dim]
    const uint16_t *w;  // bf16 [n, dim]
    float *logits;      // f32 [m, n]
    float *scores;      // f32 [m, n]: exact scores (written by the router when selecting)
    float *keys;        // f32 [m, n]: score + bias
    int dim, n, m, rows_per_cta;
    // selection
    int do_select;
    const float *bias;
    const int32_t *slot_row;
    const char *arena_base;
    unsigned long long slot_bytes, gate_off, up_off, down_off;
    float temp, route_scale;
    int norm, k;
    int32_t *hdr;
    float *plan_w;
    int32_t *plan_rows;
    unsigned long long *ptrs;
    uint32_t *ctrl;  // [MOE_CTRL_TICKET], [MOE_CTRL_STATUS]
    unsigned long long wait_ns;  // bound on each wait
};

// ------------------------------------------------------------------ the score
//
// Page moe_v41.rs, fn softplus and fn route_from_logits: the score is the f32
// chain t.exp().ln_1p().sqrt() (t itself in place of the first two steps for
// t > 20), t = f32(l / temp). Each step is taken as a correctly rounded f32
// operation:
//   e = RN(e^t),  p = RN(ln(1 + e)),  s = RN(sqrt(p)).
// sqrt is the IEEE operation. For e and p, CUDA's expf / log1pf give a
// candidate within two ulp, and the rounding is decided exactly against the
// midpoints m between neighbouring f32 values:
//   e:  e^t >= m
//   p:  ln(1 + e) >= m  <=>  e >= e^m - 1   (both sides increasing)
// Level 1 evaluates e^t and e^m - 1 in float-float single precision (pairs of
// f32, unevaluated sums hi + lo; Dekker's and Knuth's exact sum and product)
// to about 2^-41 relative: FP64 is a slow pipe on GB300. A decision closer
// than 2^-37 relative goes to level 2, CUDA's double-precision exp / log1p
// (error below 2^-51), and one closer than 2^-48 there to level 3, e^x in
// double-double (Taylor series after a reduction by ln 2, about 2^-100),
// decided at 2^-70.

struct ff {
    float hi, lo;
};

__device__ __forceinline__ ff ff_two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

__device__ __forceinline__ ff ff_fast_two_sum(float a, float b)  // |a| >= |b|
{
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ ff ff_two_prod(float a, float b)
{
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ ff ff_add(ff a, ff b)
{
    const ff s = ff_two_sum(a.hi, b.hi);
    return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ ff ff_mul(ff a, ff b)
{
    const ff p = ff_two_prod(a.hi, b.hi);
    return ff_fast_two_sum(p.hi, __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo)));
}

// 1/n!, n = 0 .. 14: the exact rationals rounded to f32 twice (hi, then the
// rest). A table in constant memory (one broadcast load a step) and loops
// that are not unrolled keep this code small: it runs once per launch, so its
// instructions are fetched cold.
__constant__ float2 c_inv_fact[15] = {
    {1.0f, 0.0f},
    {1.0f, 0.0f},
    {0x1.0p-1f, 0.0f},
    {0x1.555556p-3f, -0x1.555556p-28f},
    {0x1.555556p-5f, -0x1.555556p-30f},
    {0x1.111112p-7f, -0x1.dddddep-32f},
    {0x1.6c16c2p-10f, -0x1.27d27ep-35f},
    {0x1.a01a02p-13f, -0x1.7f97fap-39f},
    {0x1.a01a02p-16f, -0x1.7f97fap-42f},
    {0x1.71de3ap-19f, 0x1.55b1ccp-45f},
    {0x1.27e4fcp-22f, -0x1.10ec14p-47f},
    {0x1.ae6456p-26f, 0x1.fd5138p-52f},
    {0x1.1eed8ep-29f, 0x1.ff1b12p-54f},
    {0x1.612462p-33f, -0x1.8af25ep-58f},
    {0x1.93974ap-37f, 0x1.180f94p-62f},
};

__device__ __forceinline__ ff ff_inv_fact(int n)
{
    const float2 c = c_inv_fact[n];
    return {c.x, c.y};
}

// 2^(j / 32), j = 0 .. 31, as float-float pairs (hi = the f32 rounding, lo =
// the f32 rounding of the rest; the pairs are within 2^-49 relative)
__constant__ float2 c_exp2_32[32] = {
    {0x1p+0f, 0x0p+0f},
    {0x1.059b0ep+0f, -0x1.9d4f52p-25f},
    {0x1.0b5586p+0f, 0x1.9f3122p-25f},
    {0x1.11301ep+0f, -0x1.fdb496p-25f},
    {0x1.172b84p+0f, -0x1.c15742p-27f},
    {0x1.1d4874p+0f, -0x1.d2e8cap-25f},
    {0x1.2387a6p+0f, 0x1.ceac48p-25f},
    {0x1.29e9ep+0f, -0x1.5c0424p-25f},
    {0x1.306fep+0f, 0x1.4636e2p-25f},
    {0x1.371a74p+0f, -0x1.18aac6p-25f},
    {0x1.3dea64p+0f, 0x1.824684p-25f},
    {0x1.44e086p+0f, 0x1.8624b4p-30f},
    {0x1.4bfdaep+0f, -0x1.593abcp-25f},
    {0x1.5342b6p+0f, -0x1.2c561p-25f},
    {0x1.5ab07ep+0f, -0x1.5bd5ecp-27f},
    {0x1.6247ecp+0f, -0x1.f8b55p-25f},
    {0x1.6a09e6p+0f, 0x1.9fcef4p-26f},
    {0x1.71f75ep+0f, 0x1.1d8beep-25f},
    {0x1.7a1148p+0f, -0x1.829fdp-25f},
    {0x1.82589ap+0f, -0x1.accc7cp-26f},
    {0x1.8ace54p+0f, 0x1.15506ep-27f},
    {0x1.93737cp+0f, -0x1.e64744p-25f},
    {0x1.9c4918p+0f, 0x1.51f848p-27f},
    {0x1.a5503cp+0f, -0x1.b83b54p-25f},
    {0x1.ae89fap+0f, -0x1.a94b14p-26f},
    {0x1.b7f77p+0f, -0x1.a09438p-25f},
    {0x1.c199bep+0f, -0x1.3d56b2p-27f},
    {0x1.cb720ep+0f, -0x1.8837ccp-27f},
    {0x1.d5818ep+0f, -0x1.822dbcp-27f},
    {0x1.dfc974p+0f, -0x1.908c94p-25f},
    {0x1.ea4afap+0f, 0x1.52486cp-27f},
    {0x1.f50766p+0f, -0x1.246ebp-26f},
};

// 2^q for q in [-126, 127], exactly
__device__ __forceinline__ float pow2i(int q) { return __int_as_float((q + 127) << 23); }

// x 2^n for |n| <= 252, exact when the result is a normal f32 (two exact
// power-of-two steps, so that 2^n itself need not be representable)
__device__ __forceinline__ float scale2(float x, int n)
{
    const int h = n / 2;
    return __fmul_rn(__fmul_rn(x, pow2i(h)), pow2i(n - h));
}

__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }

// Tang's table-driven reduction of x (|x.hi| <= 110): k = round(x 32 / ln2),
// x = k ln2 / 32 + r with ln2 / 32 in three parts (k times the first two
// formed exactly as float-float products), |r| < 0.0109. Returns r; j = k
// mod 32, q = floor(k / 32): e^x = 2^q 2^(j / 32) e^r.
__device__ __forceinline__ ff tang_reduce(ff x, int &j, int &q)
{
    const float P1 = 0x1.62ep-6f, P2 = 0x1.0bfbe8p-20f, P3 = 0x1.cf79acp-45f;
    const float kf = rintf(__fmul_rn(x.hi, 0x1.715476p+5f));
    const int k = (int)kf;
    j = k & 31;
    q = k >> 5;  // arithmetic shift: floor
    ff r = ff_add(x, ff_neg(ff_two_prod(kf, P1)));
    r = ff_add(r, ff_neg(ff_two_prod(kf, P2)));
    return ff_add(r, {-__fmul_rn(kf, P3), 0.0f});
}

// e^x = 2^q P, P in [0.98, 2] as float-float: 2^(j/32) from the table times
// the Taylor series of e^r to r^5 / 5! (remainder below 2^-48)
__device__ ff exp_ff(ff x, int &q)
{
    int j;
    const ff r = tang_reduce(x, j, q);
    ff p = ff_inv_fact(5);
#pragma unroll 1
    for (int n = 4; n >= 0; --n)
        p = ff_add(ff_mul(p, r), ff_inv_fact(n));
    const float2 tj = c_exp2_32[j];
    return ff_mul({tj.x, tj.y}, p);
}

// e^m - 1 for m in [2^-26, 21]: below 1/8 the series m (1 + m/2! + ... +
// m^8/9!) (remainder below 2^-48 relative), else e^m - 1 (e^m - 1 >= 1/8
// loses at most 3.1 bits to the cancellation)
__device__ ff expm1_ff(ff m)
{
    if (m.hi < 0.125f) {
        ff p = ff_inv_fact(9);
#pragma unroll 1
        for (int n = 8; n >= 1; --n)
            p = ff_add(ff_mul(p, m), ff_inv_fact(n));
        return ff_mul(p, m);
    }
    int q;
    const ff P = exp_ff(m, q);
    const float sc = pow2i(q);  // q <= 30
    return ff_add({__fmul_rn(P.hi, sc), __fmul_rn(P.lo, sc)}, {-1.0f, 0.0f});
}

// ---- levels 2 and 3 (rare: a decision within 2^-37 of a midpoint)

struct dd {
    double hi, lo;
};

__device__ __forceinline__ dd dd_two_sum(double a, double b)
{
    const double s = __dadd_rn(a, b);
    const double bb = __dsub_rn(s, a);
    return {s, __dadd_rn(__dsub_rn(a, __dsub_rn(s, bb)), __dsub_rn(b, bb))};
}

__device__ __forceinline__ dd dd_fast_two_sum(double a, double b)  // |a| >= |b|
{
    const double s = __dadd_rn(a, b);
    return {s, __dsub_rn(b, __dsub_rn(s, a))};
}

__device__ __forceinline__ dd dd_add(dd a, dd b)
{
    const dd s = dd_two_sum(a.hi, b.hi);
    const dd t = dd_two_sum(a.lo, b.lo);
    dd u = dd_fast_two_sum(s.hi, __dadd_rn(s.lo, t.hi));
    return dd_fast_two_sum(u.hi, __dadd_rn(u.lo, t.lo));
}

__device__ __forceinline__ dd dd_mul(dd a, dd b)
{
    const double p = __dmul_rn(a.hi, b.hi);
    const double e = __fma_rn(a.hi, b.hi, -p);
    return dd_fast_two_sum(p, __fma_rn(a.hi, b.lo, __fma_rn(a.lo, b.hi, e)));
}

// a / n for a small positive integer n: the remainder of the rounded
// quotient is exact (one fma), and carries the low part
__device__ __forceinline__ dd dd_div_int(dd a, double n)
{
    const double q1 = __ddiv_rn(a.hi, n);
    const double rem = __fma_rn(-q1, n, a.hi);
    return dd_fast_two_sum(q1, __ddiv_rn(__dadd_rn(rem, a.lo), n));
}

// e^x in double-double for |x| <= 110: k = round(x / ln2), r = x - k ln2
// with ln2 = L1 + L2 + L3 (L1 of 32 bits, so k L1 is exact; k L2 an exact
// double-double product), |r| <= 0.35; e^r = 1 + r (1 + r/2 (1 + r/3 (... (1
// + r/24)))), remainder below 2^-120; times 2^k (exact).
__device__ __noinline__ dd exp_dd(double x)
{
    const double L1 = 0x1.62e42fee00000p-1, L2 = 0x1.a39ef35793c76p-33, L3 = 0x1.cc01f97b57a08p-87;
    const double k = rint(__dmul_rn(x, 0x1.71547652b82fep+0));
    dd r = dd_two_sum(x, -__dmul_rn(k, L1));
    const double p2 = __dmul_rn(k, L2);
    r = dd_add(r, {-p2, -__fma_rn(k, L2, -p2)});
    r = dd_add(r, {-__dmul_rn(k, L3), 0.0});
    dd p = {1.0, 0.0};
#pragma unroll 1
    for (int n = 24; n >= 1; --n)
        p = dd_add({1.0, 0.0}, dd_div_int(dd_mul(r, p), (double)n));
    const int ki = (int)k;
    const double s1 = __longlong_as_double((long long)(1023 + ki / 2) << 52);
    const double s2 = __longlong_as_double((long long)(1023 + ki - ki / 2) << 52);
    return {__dmul_rn(__dmul_rn(p.hi, s1), s2), __dmul_rn(__dmul_rn(p.lo, s1), s2)};
}

// The nearest f32 of an exact value V known through `above(m)` = (V > m) for
// a midpoint m, with `sure` cleared when the comparison is too close: the
// candidate c (V's rounding at a precision far above f32) and its two
// neighbours, decided against the two midpoints around c.
template <typename Above>
__device__ __forceinline__ float decide_near(float c, Above above, bool &sure)
{
    const unsigned cb = __float_as_uint(c);
    const float lo = cb > 0u ? __uint_as_float(cb - 1u) : c, hi = __uint_as_float(cb + 1u);
    const double mlo = 0.5 * ((double)lo + (double)c), mhi = 0.5 * ((double)c + (double)hi);  // exact
    bool s1 = true, s2 = true;
    const bool a_hi = above(mhi, s1);
    const bool a_lo = above(mlo, s2);
    sure = s1 && s2 && (lo != c || a_lo);
    return a_hi ? hi : (a_lo ? c : lo);
}

// RN(e^t) for t in [-104, 20] at levels 2 and 3
__device__ __noinline__ float exp_rn_slow(float t)
{
    const double E = exp((double)t);
    bool sure;
    const float c = __double2float_rn(E);
    float r = decide_near(c, [&](double m, bool &ok) {
        ok = fabs(E - m) > 0x1.0p-48 * E;
        return E > m;
    }, sure);
    if (sure)
        return r;
    const dd E3 = exp_dd((double)t);
    return decide_near(c, [&](double m, bool &ok) {
        const dd D = dd_add(E3, {-m, 0.0});
        ok = fabs(D.hi) > 0x1.0p-70 * m;
        return D.hi > 0.0;
    }, sure);
}

// RN(ln(1 + y)) for y in [2^-25, e^20] at levels 2 and 3 (level 3 compares
// y with e^m - 1 for the midpoints m)
__device__ __noinline__ float log1p_rn_slow(float y)
{
    const double L = log1p((double)y);
    bool sure;
    const float c = __double2float_rn(L);
    float r = decide_near(c, [&](double m, bool &ok) {
        ok = fabs(L - m) > 0x1.0p-48 * L;
        return L > m;
    }, sure);
    if (sure)
        return r;
    return decide_near(c, [&](double m, bool &ok) {
        const dd X = dd_add(exp_dd(m), {-1.0, 0.0});
        const dd D = dd_add({(double)y, 0.0}, {-X.hi, -X.lo});
        ok = fabs(D.hi) > 0x1.0p-70 * (double)y;
        return D.hi > 0.0;
    }, sure);
}

// ---- level 1

// RN(e^t) for t in [-104, 20] in float-float: the candidate c = expf(t) and
// its neighbours c_-2 .. c_+2 (f32 steps), the four midpoints between them
// scaled by 2^-q (exact: c 2^-q is near P), compared with P = e^t 2^-q. The
// number n of midpoints below e^t places it: the rounding is c_(n-2) for n
// = 1..3. Returns false when a decision is closer than 2^-37 relative or c
// is off by two steps.
__device__ __forceinline__ bool exp_rn_ff(float t, float &out)
{
    const unsigned cb = max(__float_as_uint(expf(t)), 2u);
    int q;
    const ff P = exp_ff({t, 0.0f}, q);
    const float tol = 0x1.0p-37f * P.hi;
    int n = 0;
    bool sure = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = __uint_as_float(cb + i - 2), b = __uint_as_float(cb + i - 1);
        const ff M = {scale2(b, -q), scale2(__fsub_rn(a, b), -q - 1)};  // (a + b) / 2 2^-q
        const ff D = ff_add(P, ff_neg(M));
        sure = sure && fabsf(D.hi) > tol;
        n += D.hi > 0.0f;
    }
    if (!sure || n == 0 || n == 4)
        return false;
    out = __uint_as_float(cb - 2 + n);
    return true;
}

// RN(ln(1 + y)) for y in [2^-25, e^20] in float-float, on a converged group
// of four lanes (mask gmask, first lane src0, this lane's place v): the
// candidate c = log1pf(y) and its neighbours c_-2 .. c_+2; lane v evaluates
// e^m_v - 1 for the midpoint m_v between c_(v-2) and c_(v-1); the group
// gathers the four and compares each with y. Returns false as exp_rn_ff.
__device__ __forceinline__ bool log1p_rn_ff(float y, int v, unsigned gmask, int src0, float &out)
{
    const unsigned cb = __float_as_uint(log1pf(y));
    const float a = __uint_as_float(cb + v - 2), b = __uint_as_float(cb + v - 1);
    const ff X = expm1_ff({b, __fmul_rn(__fsub_rn(a, b), 0.5f)});  // the exact midpoint
    const float tol = 0x1.0p-37f * y;
    int n = 0;
    bool sure = true;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float xh = __shfl_sync(gmask, X.hi, src0 + i), xl = __shfl_sync(gmask, X.lo, src0 + i);
        const ff D = ff_add({y, 0.0f}, {-xh, -xl});
        sure = sure && fabsf(D.hi) > tol;
        n += D.hi > 0.0f;
    }
    if (!sure || n == 0 || n == 4)
        return false;
    out = __uint_as_float(cb - 2 + n);
    return true;
}

// The routing score of l on a converged group of four lanes that share l
// (v = 0..3, mask gmask, first lane src0); every lane returns it.
// ln(1 + e) rounds to e itself below 2^-25 (ln(1 + e) = e (1 - e/2 + ...)
// lies within e/2 < 2^-26 relative of e, closer than any midpoint).
__device__ __noinline__ float score_chain(float t, int v, unsigned gmask, int src0)
{
    float e = 0.0f;  // e^t < 2^-150 below t = -104: rounds to 0
    if (t >= -104.0f && !exp_rn_ff(t, e))
        e = exp_rn_slow(t);
    float p = e;
    if (e >= 0x1.0p-25f && !log1p_rn_ff(e, v, gmask, src0, p))
        p = log1p_rn_slow(e);
    return __fsqrt_rn(p);
}

__device__ __forceinline__ float score_fast(float l, float temp, int v, unsigned gmask, int src0)
{
    const float t = __fdiv_rn(l, temp);
    if (t > 20.0f)
        return __fsqrt_rn(t);
    if (t != t)
        return t;
    return score_chain(t, v, gmask, src0);
}

// ------------------------------------------------------------------ sortable keys

// One 64-bit value per expert that orders exactly as "ranks before": the key
// mapped to an unsigned integer that grows with it (-0 equal to +0, NaN below
// every number), then the complement of the id so equal keys put the lower id
// first. 0 (a NaN key with id 2^32 - 1) pads empty slots and ranks last.
__device__ __forceinline__ unsigned long long rank_value(float key, int id)
{
    uint32_t u;
    if (isnan(key)) {
        u = 0u;
    } else {
        uint32_t b = key == 0.0f ? 0u : __float_as_uint(key);
        u = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    }
    return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)id);
}

__device__ __forceinline__ int rank_id(unsigned long long v) { return (int)(0xFFFFFFFFu - (uint32_t)v); }

// ------------------------------------------------------------------ selection + plan (whole CTA, 256 threads)

// Shared memory of the selection: a fixed part, then per token its n sortable
// values (u64) and n exact scores (f32).
struct SelectSmem {
    unsigned long long cand[8][MOE_MAX_TOPK];               // per warp: the k best of its share
    unsigned long long fin[MOE_MAX_TOKENS][MOE_MAX_TOPK];   // per token: its k best
    int pick[MOE_MAX_TOKENS][MOE_MAX_TOPK];
    float w[MOE_MAX_TOKENS][MOE_MAX_TOPK];
    int flags[MOE_MAX_TOKENS];
    int first[MOE_MAX_TOKENS * MOE_MAX_TOPK], ent[MOE_MAX_TOKENS * MOE_MAX_TOPK];
};

// the largest of PL (a power of two) values, as a balanced tree
template <int PL>
__device__ __forceinline__ unsigned long long lane_max(const unsigned long long (&v)[PL])
{
    unsigned long long t[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i)
        t[i] = v[i];
#pragma unroll
    for (int w = PL / 2; w >= 1; w /= 2)
#pragma unroll
        for (int i = 0; i < w; ++i)
            t[i] = max(t[i], t[i + w]);
    return t[0];
}

// k rounds of the warp-wide maximum over PL values per lane (distinct; 0
// marks an empty place and ranks last): out[r] = the r-th largest, written
// by lane 0. A round reduces the high words; the low words only when more
// than one lane holds the largest high word (equal keys). The lane holding
// the winner removes it and takes the maximum of the rest.
template <int PL>
__device__ __forceinline__ void warp_topk(unsigned long long (&v)[PL], int k, unsigned long long *out)
{
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    unsigned long long best = lane_max<PL>(v);
    for (int r = 0; r < k; ++r) {
        const unsigned bh = (unsigned)(best >> 32);
        const unsigned hi = __reduce_max_sync(full, bh);
        const unsigned tied = __ballot_sync(full, bh == hi);
        const unsigned lo = (tied & (tied - 1u)) == 0u ? __shfl_sync(full, (unsigned)best, __ffs(tied) - 1)
                                                       : __reduce_max_sync(full, bh == hi ? (unsigned)best : 0u);
        const unsigned long long win = ((unsigned long long)hi << 32) | lo;
        if (lane == 0)
            out[r] = win;
        if (win != 0ull && best == win) {
#pragma unroll
            for (int i = 0; i < PL; ++i)
                v[i] = v[i] == win ? 0ull : v[i];
            best = lane_max<PL>(v);
        }
    }
}

// Calls f with IntC<PL>, PL = per_lane rounded up to a power of two (<= 32)
template <typename F>
__device__ __forceinline__ void with_per_lane(int per_lane, F &&f)
{
    if (per_lane <= 1)
        f(IntC<1>{});
    else if (per_lane <= 2)
        f(IntC<2>{});
    else if (per_lane <= 4)
        f(IntC<4>{});
    else if (per_lane <= 8)
        f(IntC<8>{});
    else if (per_lane <= 16)
        f(IntC<16>{});
    else
        f(IntC<32>{});
}

__host__ __device__ inline size_t sel_v_off() { return align_up(sizeof(SelectSmem), 16); }
__host__ __device__ inline size_t sel_bytes(int m, int n) { return sel_v_off() + (size_t)m * n * (8 + 4); }

template <bool kGlobal>
__device__ __forceinline__ float sel_ld(const float *p)
{
    if constexpr (kGlobal)
        return __ldcg(p);  // written by other CTAs of this kernel: read at L2
    else
        return *p;
}

#define SEL_UNROLL 8

// Selection for all m tokens (256 threads), then the plan: the distinct
// picked experts in ascending id with their (expert, token) pairs, and the
// header. logits, scores, keys: [m, n] in global memory (kGlobal) or shared;
// slot: the slot-table row of every expert, already in shared memory.
template <bool kGlobal>
__device__ void select_and_plan(const RouteArgs &a, const float *logits, const float *scores, const float *keys,
                                const int *slot, uint8_t *smem)
{
    SelectSmem &sm = *reinterpret_cast<SelectSmem *>(smem);
    unsigned long long *val = reinterpret_cast<unsigned long long *>(smem + sel_v_off());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.n, k = a.k, m = a.m, cap = m * k, mn = m * n;
    const FastDiv nd((uint32_t)n), kd((uint32_t)k);  // token of entry i, of pair q: one multiply-high each
    float *sco = reinterpret_cast<float *>(val + (size_t)mn);
    if (tid < MOE_MAX_TOKENS)
        sm.flags[tid] = 0;
    __syncthreads();

    // one round of loads (SEL_UNROLL entries a thread in flight at once)
    for (int b = 0; b < mn; b += 256 * SEL_UNROLL) {
        float kk[SEL_UNROLL], ll[SEL_UNROLL], ss[SEL_UNROLL];
#pragma unroll
        for (int u = 0; u < SEL_UNROLL; ++u) {
            const int i = b + tid + 256 * u;
            kk[u] = i < mn ? sel_ld<kGlobal>(keys + i) : 0.0f;
            ll[u] = i < mn ? sel_ld<kGlobal>(logits + i) : 0.0f;
            ss[u] = i < mn ? sel_ld<kGlobal>(scores + i) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < SEL_UNROLL; ++u) {
            const int i = b + tid + 256 * u;
            if (i < mn) {
                const int t = (int)nd.div((uint32_t)i), e = i - t * n;
                val[i] = rank_value(kk[u], e);
                sco[i] = ss[u];
                if (!isfinite(ll[u]) || !isfinite(kk[u]))
                    atomicOr(&sm.flags[t], MOE_HDR_NONFINITE);
            }
        }
    }
    __syncthreads();

    // Ranking. Each token has a group of gsz warps (8 for one token, down to
    // one warp per token); each warp takes the k best of its share (the
    // experts lane + 32 (wig + gsz i)), then the group's first warp takes the
    // k best of those gsz * k candidates.
    int gsz = 8;
    while (gsz > 1 && gsz * m > 8)
        gsz >>= 1;
    const int group = warp / gsz, wig = warp - group * gsz;
    if (group < m) {
        const int t = group;
        const unsigned long long *vt = val + (size_t)t * n;
        const int stride = 32 * gsz;
        unsigned long long *fin = sm.fin[t];
        unsigned long long *out1 = gsz == 1 ? fin : sm.cand[warp];
        with_per_lane((n + stride - 1) / stride, [&](auto PC) {
            constexpr int PL = decltype(PC)::value;
            unsigned long long v[PL];
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                const int e = wig * 32 + lane + i * stride;
                v[i] = e < n ? vt[e] : 0ull;
            }
            warp_topk<PL>(v, k, out1);
        });
        if (gsz > 1) {
            asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(gsz * 32) : "memory");
            if (wig == 0) {
                const int nc = gsz * k;  // <= 64
                unsigned long long v[2];
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int c = lane + 32 * j, cw = (int)kd.div((uint32_t)c);
                    v[j] = c < nc ? sm.cand[group * gsz + cw][c - cw * k] : 0ull;
                }
                warp_topk<2>(v, k, fin);
            }
        }
        if (wig == 0) {
            // lane 0 holds the picks; a pick outside [0, n) (fewer than k
            // values, impossible for k <= n) would index the tables
            if (lane == 0) {
                for (int r = 0; r < k; ++r) {
                    int id = rank_id(fin[r]);
                    if (id < 0 || id >= n) {
                        if (a.ctrl)
                            atomicOr(a.ctrl + MOE_CTRL_STATUS, (uint32_t)MOE_WS_PLAN);
                        id = 0;
                    }
                    sm.pick[t][r] = id;
                }
            }
            __syncwarp();
            // weights in pick order, each step one f32 rounding
            float sv[MOE_MAX_TOPK];
#pragma unroll
            for (int i = 0; i < MOE_MAX_TOPK; ++i)
                sv[i] = i < k ? sco[(size_t)t * n + sm.pick[t][i]] : 0.0f;
            float sum = 0.0f;
#pragma unroll
            for (int i = 0; i < MOE_MAX_TOPK; ++i)
                if (i < k)
                    sum = __fadd_rn(sum, sv[i]);
            sum = __fadd_rn(sum, 1e-20f);
            if (lane < k) {
                float sc = 0.0f;
#pragma unroll
                for (int i = 0; i < MOE_MAX_TOPK; ++i)
                    sc = lane == i ? sv[i] : sc;
                sm.w[t][lane] = (a.norm && k > 1) ? __fmul_rn(__fdiv_rn(sc, sum), a.route_scale)
                                                  : __fmul_rn(sc, a.route_scale);
            }
        }
    }
    __syncthreads();
    const int po = m * (1 + 3 * k);  // plan tail of the header
    if (warp == 0) {
        // the plan, by one warp: pair q = (token q / k, its pick q % k), two per
        // lane; ranked by (expert, token); the distinct experts in ascending id
        int eq[2], tq[2], rq[2];
        bool fq[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int q = lane + 32 * j;
            tq[j] = (int)kd.div((uint32_t)q);
            eq[j] = q < cap ? sm.pick[tq[j]][q - tq[j] * k] : 0;
            if (q < cap)
                sm.ent[q] = eq[j];
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int q = lane + 32 * j;
            rq[j] = 0;
            fq[j] = false;
            if (q < cap) {
                int earlier = 0;
                for (int q2 = 0, t2 = 0, r2 = 0; q2 < cap; ++q2) {  // pair q2 = token t2, pick r2
                    const int e2 = sm.ent[q2];
                    rq[j] += e2 < eq[j] || (e2 == eq[j] && t2 < tq[j]);
                    earlier += e2 == eq[j] && t2 < tq[j];
                    if (++r2 == k) {
                        r2 = 0;
                        ++t2;
                    }
                }
                fq[j] = earlier == 0;
                sm.first[q] = fq[j];
                a.plan_rows[rq[j]] = tq[j];
                a.plan_w[rq[j]] = sm.w[tq[j]][q - tq[j] * k];
            }
        }
        __syncwarp();
        int ne = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int q = lane + 32 * j;
            ne += __popc(__ballot_sync(0xffffffffu, q < cap && fq[j]));
            if (q < cap && fq[j]) {
                int p = 0;  // distinct experts below this one
                for (int q2 = 0; q2 < cap; ++q2)
                    p += sm.first[q2] && sm.ent[q2] < eq[j];
                const int sl = slot[eq[j]];
                const unsigned long long base =
                    (unsigned long long)a.arena_base + (unsigned long long)(sl < 0 ? 0 : sl) * a.slot_bytes;
                a.ptrs[p] = base + a.gate_off;
                a.ptrs[cap + p] = base + a.up_off;
                a.ptrs[2 * cap + p] = base + a.down_off;
                a.hdr[po + 1 + p] = rq[j];  // the expert's first pair: its pairs start here
                a.hdr[po + 2 + cap + p] = eq[j];
            }
        }
        if (lane == 0) {
            a.hdr[po] = ne;
            a.hdr[po + 1 + ne] = cap;
        }
    } else if (warp == 1 && lane < m) {
        // header rows: status, picks, weight bits, slots of the picks in ascending id
        const int t = lane;
        int32_t *h = a.hdr + (size_t)t * (1 + 3 * k);
        int status = sm.flags[t];
        for (int i = 0; i < k; ++i) {
            const int v = sm.pick[t][i];
            h[1 + i] = v;
            h[1 + k + i] = __float_as_int(sm.w[t][i]);
            int pos = 0;  // the picks of a token are distinct: position in ascending id
            for (int j = 0; j < k; ++j)
                pos += sm.pick[t][j] < v;
            const int sl = slot[v];
            if (sl < 0)
                status |= MOE_HDR_MISS;
            h[1 + 2 * k + pos] = sl < 0 ? 0 : sl;
        }
        h[0] = status;
    }
}

// ------------------------------------------------------------------ kernels

// the router's constants staged before the wait: the slot table (for the
// selection) and the bias of the CTA's rows
__host__ __device__ inline size_t router_pre_bytes(int n, int rows) { return align_up(4 * ((size_t)n + rows), 128); }

// smem: [0,128) barrier + flag; the staged constants; then the CTA's router
// rows, x, logits; the last CTA reuses the rows area for the selection
// KM: the token count the kernel is built for (it holds that case's code
// alone: 1 or 8), or 0 for any m
template <int KM>
__global__ void __launch_bounds__(256) moe_router_kernel(RouteArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int *s_last = reinterpret_cast<int *>(smem + 8);
    int *s_slot = reinterpret_cast<int *>(smem + 128);
    float *s_bias = reinterpret_cast<float *>(s_slot + a.n);
    uint16_t *sw = reinterpret_cast<uint16_t *>(smem + 128 + router_pre_bytes(a.n, a.rows_per_cta));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dim = a.dim, m = a.m;
    const int row0 = blockIdx.x * a.rows_per_cta;
    const int nrows = min(a.rows_per_cta, a.n - row0);
    uint16_t *sx = sw + (size_t)a.rows_per_cta * dim;
    float *red = reinterpret_cast<float *>(sx + (size_t)m * dim);  // logits [rows][m]
    const uint32_t wbytes = (uint32_t)nrows * dim * 2;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0 && nrows > 0) {
        // this CTA's router rows: constant weights, fetched before the wait
        const uint64_t pol = policy_evict_first();
        mbar_arrive_expect_tx(bar, wbytes);
        const char *src = reinterpret_cast<const char *>(a.w + (size_t)row0 * dim);
        char *dst = reinterpret_cast<char *>(sw);
        for (uint32_t off = 0; off < wbytes; off += 32768u)
            bulk_g2s(dst + off, src + off, min(32768u, wbytes - off), bar, pol);
    }
    // the bias and the slot table are layer constants too (kernels that write
    // them, such as the slot-table update, complete before a dependent starts)
    if (a.do_select) {
        for (int e = tid; e < a.n; e += blockDim.x)
            s_slot[e] = __ldg(a.slot_row + e);
        if (tid < nrows)
            s_bias[tid] = __ldg(a.bias + row0 + tid);
    }
    pdl_wait();  // x is produced by the previous kernel
    pdl_launch_dependents();
    {
        const uint4 *gx = reinterpret_cast<const uint4 *>(a.x);
        uint4 *s4 = reinterpret_cast<uint4 *>(sx);
        for (int i = tid; i < m * dim / 8; i += blockDim.x)
            s4[i] = __ldcg(gx + i);
    }
    __syncthreads();
    const bool ok = nrows <= 0 || mbar_wait(bar, 0, a.ctrl + MOE_CTRL_STATUS, a.wait_ns);
    if (__syncthreads_and(ok) == 0)
        return;
    // logits: one warp per row, all tokens at once; lane j takes the 16-byte
    // chunks j + 32 i into four partial sums (i mod 4), added pairwise, then a
    // warp butterfly -- a fixed order per (token, row), whatever m is
    const int nch = dim / 8;
    with_m_k<KM>(m, [&](auto MC) {
        constexpr int M = decltype(MC)::value;
        const uint4 *x4 = reinterpret_cast<const uint4 *>(sx);
        for (int r = warp; r < nrows; r += blockDim.x >> 5) {
            const uint4 *wr = reinterpret_cast<const uint4 *>(sw + (size_t)r * dim);
            float acc[M][4];
#pragma unroll
            for (int t = 0; t < M; ++t)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[t][q] = 0.0f;
            for (int c0 = lane; c0 < nch; c0 += 128) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = c0 + 32 * q;
                    if (c < nch) {
                        const uint4 wv = wr[c];
#pragma unroll
                        for (int t = 0; t < M; ++t)
                            acc[t][q] = fma_bf16x8(wv, x4[(size_t)t * nch + c], acc[t][q]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < M; ++t) {
                float v = (acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]);
#pragma unroll
                for (int o = 16; o; o >>= 1)
                    v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0)
                    red[(size_t)r * m + t] = v;
            }
        }
    });
    __syncthreads();
    // one score a warp first (lane groups of four, lane-major over the
    // warps): the scores take different paths by range, and paths in one
    // warp would run one after another; a group computes one score, the four
    // midpoint tests of its float-float log1p step one a lane
    const int nw = blockDim.x >> 5, grp = lane >> 2, gv = lane & 3;
    {
        const unsigned gmask = 0xFu << (4 * grp);
        const FastDiv md((uint32_t)m);
        for (int i = warp + nw * grp; i < nrows * m; i += nw * 8) {
            const int r = (int)md.div((uint32_t)i), t = i - r * m;
            const float l = red[i];
            const size_t o = (size_t)t * a.n + row0 + r;
            if (gv == 0)
                a.logits[o] = l;
            if (a.do_select) {
                // the exact score of this row, here: a few lanes of every CTA
                // in parallel instead of the selecting CTA
                const float sc = score_fast(l, a.temp, gv, gmask, 4 * grp);
                if (gv == 0) {
                    a.scores[o] = sc;
                    a.keys[o] = __fadd_rn(sc, s_bias[r]);
                }
            }
        }
    }
    if (!a.do_select)
        return;
    // the last CTA to finish its rows runs the selection (no CTA waits)
    __syncthreads();
    if (tid == 0) {
        // acq_rel: releases this CTA's logits/scores/keys (ordered before by
        // the barrier), and the last CTA acquires everyone else's
        unsigned old;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(a.ctrl + MOE_CTRL_TICKET) : "memory");
        *s_last = old == gridDim.x - 1;
    }
    __syncthreads();
    if (!*s_last)
        return;
    // the rows area is no longer needed: it holds the selection
    select_and_plan<true>(a, a.logits, a.scores, a.keys, s_slot, reinterpret_cast<uint8_t *>(sw));
    __syncthreads();
    if (tid == 0) {
        // the plan is written: released to the gate/up kernel's producers,
        // which read it without waiting for this grid to finish (release:
        // this CTA's stores, ordered before by the barrier)
        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(a.ctrl + MOE_CTRL_GATEUP + 5), "r"(1u) : "memory");
        // the ticket, for the next launch (every CTA has taken its own):
        // after the release, which so does not wait for it
        st_relaxed_gpu(a.ctrl + MOE_CTRL_TICKET, 0u);
    }
}

// the selection alone, on caller-provided logits: one CTA of 256 threads
// computes every score and key into shared memory, then selects
__global__ void __launch_bounds__(256) moe_select_kernel(RouteArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const size_t mn = (size_t)a.m * a.n;
    float *sc = reinterpret_cast<float *>(smem + align_up(sel_bytes(a.m, a.n), 128));
    float *ky = sc + mn;
    int *slot = reinterpret_cast<int *>(ky + mn);
    pdl_wait();
    pdl_launch_dependents();
    for (int e = threadIdx.x; e < a.n; e += blockDim.x)
        slot[e] = __ldg(a.slot_row + e);
    {
        // a group of four lanes a score (eight groups a warp)
        const int lane = threadIdx.x & 31, grp = lane >> 2, gv = lane & 3;
        const int ng = (int)(blockDim.x >> 5) * 8;
        {
            const unsigned gmask = 0xFu << (4 * grp);
            for (int i = (int)(threadIdx.x >> 5) * 8 + grp; i < (int)mn; i += ng) {
                const float s = score_fast(a.logits[i], a.temp, gv, gmask, 4 * grp);
                if (gv == 0) {
                    sc[i] = s;
                    ky[i] = __fadd_rn(s, __ldg(a.bias + i % a.n));
                }
            }
        }
    }
    __syncthreads();
    select_and_plan<false>(a, a.logits, sc, ky, slot, smem);
}

#define MOE_SCORES_PER_CTA 64  // eight warps of eight four-lane groups

struct ScoreArgs {
    const float *logits;
    float *scores;
    float temp;
    int count;
};

// the routing score of each of count logits: a group of four lanes each
// (eight groups a warp, MOE_SCORES_PER_CTA a CTA of 256 threads)
__global__ void moe_score_kernel(ScoreArgs a)
{
    pdl_wait();
    const int lane = threadIdx.x & 31, grp = lane >> 2, gv = lane & 3;
    const int i = blockIdx.x * MOE_SCORES_PER_CTA + (int)(threadIdx.x >> 5) * 8 + grp;
    if (i < a.count) {
        const float s = score_fast(a.logits[i], a.temp, gv, 0xFu << (4 * grp), 4 * grp);
        if (gv == 0)
            a.scores[i] = s;
    }
}

}  // namespace moe

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
// fn route_from_logits): score = f32(sqrt(softplus(l / temp))), key = score +
// bias, stable descending order, top k, weights renormalised in f32. The
// score is defined as the correctly rounded f32 of the exact value. FP64 is a
// slow pipe on GB300, so each lane first ranks all its experts with a
// single-precision score (CUDA's expf / log1pf / sqrtf, error a few ulp) and a
// generous error bound, finds the k-th largest lower bound T, and evaluates
// the double-precision score only for the candidates whose upper bound
// reaches T. Every expert outside that set is provably below k candidates,
// so the picks equal the ranking by exact keys.
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
};

// ------------------------------------------------------------------ scores

// The score as defined: the f32 rounding of sqrt(softplus(t)), t = f32(l / temp),
// softplus(x) = x for x > 20. Evaluated in f64 (CUDA's exp, log1p, sqrt) and
// rounded once: the f64 chain's error is far below half an f32 ulp, so the
// rounding equals the exact one except within ~2^-50 of an f32 midpoint.
__device__ __forceinline__ float score_exact(float l, float temp)
{
    const float t = __fdiv_rn(l, temp);
    const double sp = t > 20.0f ? (double)t : log1p(exp((double)t));
    return __double2float_rn(sqrt(sp));
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

#define SEL_PER_WARP MOE_MAX_ROUTED  // values per warp in the first ranking stage

struct SelectSmem {
    int pick[MOE_MAX_TOKENS][MOE_MAX_TOPK];
    float sc[MOE_MAX_TOKENS][MOE_MAX_TOPK];
    float w[MOE_MAX_TOKENS][MOE_MAX_TOPK];
    int flags[MOE_MAX_TOKENS];
    int wflag[8];
    unsigned long long v[8][SEL_PER_WARP];               // per warp: its experts' values
    unsigned long long cand[8][MOE_MAX_TOPK];            // per warp: its k best
    int first[MOE_MAX_TOKENS * MOE_MAX_TOPK], rank[MOE_MAX_TOKENS * MOE_MAX_TOPK],
        ent[MOE_MAX_TOKENS * MOE_MAX_TOPK];
};

__device__ __forceinline__ void group_sync(int group, int gsz)
{
    if (gsz == 1)
        __syncwarp();
    else
        asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(gsz * 32) : "memory");
}

// The picks of token t by a group of gsz warps from exact scores and keys.
// Ranking by counting (no long shuffle chains): every value's rank is the
// number of values ranking before it; stage 1 inside each warp over its
// experts, stage 2 over the group's k best of each warp.
__device__ void select_token_group(const RouteArgs &a, const float *logits, const float *scores,
                                   const float *keys, int t, int group, int gsz, SelectSmem &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wig = warp - group * gsz;
    const int n = a.n, k = a.k, stride = gsz * 32;
    const size_t row = (size_t)t * n;
    const int per_lane = (n + stride - 1) / stride;  // <= SEL_PER_WARP / 32
    bool nonfinite = false;
    for (int i = 0; i < per_lane; ++i) {
        const int e = wig * 32 + lane + i * stride;
        unsigned long long v = 0ull;
        if (e < n) {
            const float key = keys[row + e];
            nonfinite |= !isfinite(logits[row + e]) || !isfinite(key);
            v = rank_value(key, e);
        }
        sm.v[warp][lane + 32 * i] = v;
    }
    if (lane < MOE_MAX_TOPK)
        sm.cand[warp][lane] = 0ull;
    const unsigned nf = __ballot_sync(0xffffffffu, nonfinite);
    if (lane == 0)
        sm.wflag[warp] = nf ? MOE_HDR_NONFINITE : 0;
    __syncwarp();
    const int nv = 32 * per_lane;
    for (int i = 0; i < per_lane; ++i) {
        const unsigned long long mv = sm.v[warp][lane + 32 * i];
        if (mv != 0ull) {
            int r = 0;
            for (int j = 0; j < nv; ++j)
                r += sm.v[warp][j] > mv;
            if (r < k)
                sm.cand[warp][r] = mv;
        }
    }
    group_sync(group, gsz);
    if (wig == 0) {
        // stage 2: the group's gsz * k candidates (<= 64), two per lane
        const int nc = gsz * k;
        for (int c = lane; c < nc; c += 32) {
            const unsigned long long v = sm.cand[group * gsz + c / k][c % k];
            if (v == 0ull)
                continue;
            int r = 0;
            for (int j = 0; j < nc; ++j)
                r += sm.cand[group * gsz + j / k][j % k] > v;
            if (r < k) {
                const int id = rank_id(v);
                sm.pick[t][r] = id;
                sm.sc[t][r] = scores[row + id];
            }
        }
        __syncwarp();
        if (lane == 0) {
            int fl = 0;
            for (int w = 0; w < gsz; ++w)
                fl |= sm.wflag[group * gsz + w];
            sm.flags[t] = fl;
            // weights in pick order, each step one f32 rounding
            if (a.norm && k > 1) {
                float sum = 0.0f;
                for (int i = 0; i < k; ++i)
                    sum = __fadd_rn(sum, sm.sc[t][i]);
                sum = __fadd_rn(sum, 1e-20f);
                for (int i = 0; i < k; ++i)
                    sm.w[t][i] = __fmul_rn(__fdiv_rn(sm.sc[t][i], sum), a.route_scale);
            } else {
                for (int i = 0; i < k; ++i)
                    sm.w[t][i] = __fmul_rn(sm.sc[t][i], a.route_scale);
            }
        }
    }
}

// Selection for all m tokens, then the plan: the distinct picked experts in
// ascending id with their (expert, token) pairs, pair-major, and the header.
__device__ void select_and_plan(const RouteArgs &a, const float *logits, const float *scores, const float *keys,
                                SelectSmem &sm)
{
    const int tid = threadIdx.x, warp = tid >> 5;
    const int n = a.n, k = a.k, m = a.m, cap = m * k;
    // warps in groups: all 8 on one token for m = 1, down to one warp per token
    int gsz = 8;
    while (gsz > 1 && gsz * m > 8)
        gsz >>= 1;
    const int group = warp / gsz;
    if (group < m)
        select_token_group(a, logits, scores, keys, group, group, gsz, sm);
    __syncthreads();
    // pairs: entry q = (token q / k, its pick q % k); rank by (expert, token)
    if (tid < cap) {
        int e = sm.pick[tid / k][tid % k];
        if (e < 0 || e >= n) {  // defensive: a pick outside [0, n) would index the tables
            if (a.ctrl)
                atomicOr(a.ctrl + MOE_CTRL_STATUS, (uint32_t)MOE_WS_PLAN);
            e = 0;
            sm.pick[tid / k][tid % k] = 0;
        }
        sm.ent[tid] = e;
    }
    __syncthreads();
    if (tid < cap) {
        const int e = sm.ent[tid], t = tid / k;
        int rank = 0, earlier = 0;
        for (int q = 0; q < cap; ++q) {
            const int e2 = sm.ent[q], t2 = q / k;
            rank += e2 < e || (e2 == e && t2 < t);
            earlier += e2 == e && t2 < t;
        }
        sm.rank[tid] = rank;
        sm.first[tid] = earlier == 0;
        a.plan_rows[rank] = t;
        a.plan_w[rank] = sm.w[t][tid % k];
    }
    __syncthreads();
    const int po = m * (1 + 3 * k);  // plan tail of the header
    if (tid < cap && sm.first[tid]) {
        const int e = sm.ent[tid];
        int p = 0;
        for (int q = 0; q < cap; ++q)
            p += sm.first[q] && sm.ent[q] < e;
        const int slot = __ldg(a.slot_row + e);
        const unsigned long long base =
            (unsigned long long)a.arena_base + (unsigned long long)(slot < 0 ? 0 : slot) * a.slot_bytes;
        a.ptrs[p] = base + a.gate_off;
        a.ptrs[cap + p] = base + a.up_off;
        a.ptrs[2 * cap + p] = base + a.down_off;
        a.hdr[po + 1 + p] = sm.rank[tid];
        a.hdr[po + 2 + cap + p] = e;
    }
    if (tid == 0) {
        int ne = 0;
        for (int q = 0; q < cap; ++q)
            ne += sm.first[q];
        a.hdr[po] = ne;
        a.hdr[po + 1 + ne] = cap;
    }
    // header rows: status, picks, weight bits, slots of the picks in ascending id
    if (tid >= 32 && tid < 32 + m) {
        const int t = tid - 32;
        int32_t *h = a.hdr + (size_t)t * (1 + 3 * k);
        int sorted[MOE_MAX_TOPK];
        int status = sm.flags[t];
        for (int i = 0; i < k; ++i) {
            h[1 + i] = sm.pick[t][i];
            h[1 + k + i] = __float_as_int(sm.w[t][i]);
            const int v = sm.pick[t][i];
            int j = i;
            while (j > 0 && sorted[j - 1] > v) {
                sorted[j] = sorted[j - 1];
                --j;
            }
            sorted[j] = v;
        }
        for (int i = 0; i < k; ++i) {
            const int slot = __ldg(a.slot_row + sorted[i]);
            if (slot < 0)
                status |= MOE_HDR_MISS;
            h[1 + 2 * k + i] = slot < 0 ? 0 : slot;
        }
        h[0] = status;
    }
}

// ------------------------------------------------------------------ kernels

// smem: [0,128) barrier + flag; then the CTA's router rows, x, warp partials;
// the last CTA reuses the rows area for the selection
__global__ void __launch_bounds__(256) moe_router_kernel(RouteArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    int *s_last = reinterpret_cast<int *>(smem + 8);
    uint16_t *sw = reinterpret_cast<uint16_t *>(smem + 128);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dim = a.dim, m = a.m;
    const int row0 = blockIdx.x * a.rows_per_cta;
    const int nrows = min(a.rows_per_cta, a.n - row0);
    uint16_t *sx = sw + (size_t)a.rows_per_cta * dim;
    float *red = reinterpret_cast<float *>(sx + (size_t)m * dim);  // [8 warps][rows][m]
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
    pdl_wait();  // x is produced by the previous kernel
    pdl_launch_dependents();
    {
        const uint4 *gx = reinterpret_cast<const uint4 *>(a.x);
        uint4 *s4 = reinterpret_cast<uint4 *>(sx);
        for (int i = tid; i < m * dim / 8; i += blockDim.x)
            s4[i] = __ldcg(gx + i);
    }
    __syncthreads();
    const bool ok = nrows <= 0 || mbar_wait(bar, 0, a.ctrl + MOE_CTRL_STATUS);
    if (__syncthreads_and(ok) == 0)
        return;
    // logits: thread-strided 16-byte chunks, warp butterfly, then the 8 warp
    // partials in order -- a fixed order per (token, row), whatever m is
    const int nch = dim / 8;
    for (int r = 0; r < nrows; ++r) {
        const uint4 *wr = reinterpret_cast<const uint4 *>(sw + (size_t)r * dim);
        for (int t = 0; t < m; ++t) {
            const uint4 *xr = reinterpret_cast<const uint4 *>(sx + (size_t)t * dim);
            float acc = 0.0f;
            for (int c = tid; c < nch; c += blockDim.x) {
                const uint4 wv = wr[c], xv = xr[c];
                acc = fmaf(bf16_lo(wv.x), bf16_lo(xv.x), acc);
                acc = fmaf(bf16_hi(wv.x), bf16_hi(xv.x), acc);
                acc = fmaf(bf16_lo(wv.y), bf16_lo(xv.y), acc);
                acc = fmaf(bf16_hi(wv.y), bf16_hi(xv.y), acc);
                acc = fmaf(bf16_lo(wv.z), bf16_lo(xv.z), acc);
                acc = fmaf(bf16_hi(wv.z), bf16_hi(xv.z), acc);
                acc = fmaf(bf16_lo(wv.w), bf16_lo(xv.w), acc);
                acc = fmaf(bf16_hi(wv.w), bf16_hi(xv.w), acc);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1)
                acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0)
                red[((size_t)warp * a.rows_per_cta + r) * m + t] = acc;
        }
    }
    __syncthreads();
    const int nw = blockDim.x >> 5;
    for (int i = tid; i < nrows * m; i += blockDim.x) {
        const int r = i / m, t = i % m;
        float l = 0.0f;
        for (int w = 0; w < nw; ++w)
            l += red[((size_t)w * a.rows_per_cta + r) * m + t];
        const size_t o = (size_t)t * a.n + row0 + r;
        a.logits[o] = l;
        if (a.do_select) {
            // the exact score of this row, here: the f64 chain runs on a few
            // threads of every CTA in parallel instead of in the selecting CTA
            const float sc = score_exact(l, a.temp);
            a.scores[o] = sc;
            a.keys[o] = __fadd_rn(sc, __ldg(a.bias + row0 + r));
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
    SelectSmem *sel = reinterpret_cast<SelectSmem *>(sw);  // the weights are no longer needed
    select_and_plan(a, a.logits, a.scores, a.keys, *sel);
    if (tid == 0)
        atomicExch(a.ctrl + MOE_CTRL_TICKET, 0u);
}

// the selection alone, on caller-provided logits: one CTA of 256 threads
// computes every score and key into shared memory, then selects
__global__ void __launch_bounds__(256) moe_select_kernel(RouteArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    SelectSmem &sel = *reinterpret_cast<SelectSmem *>(smem);
    float *sc = reinterpret_cast<float *>(smem + align_up(sizeof(SelectSmem), 128));
    float *ky = sc + (size_t)a.m * a.n;
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i < a.m * a.n; i += blockDim.x) {
        const float s = score_exact(a.logits[i], a.temp);
        sc[i] = s;
        ky[i] = __fadd_rn(s, __ldg(a.bias + i % a.n));
    }
    __syncthreads();
    select_and_plan(a, a.logits, sc, ky, sel);
}

}  // namespace moe

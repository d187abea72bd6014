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

__device__ __forceinline__ float score_approx(float t)
{
    float sp = t > 20.0f ? t : log1pf(expf(t));
    return sqrtf(sp);
}

__device__ __forceinline__ float score_exact(float t)
{
    double sp = t > 20.0f ? (double)t : log1p(exp((double)t));
    return __double2float_rn(sqrt(sp));
}

// |score_approx - score_exact| plus the key rounding, with a wide margin
// (the single-precision chain is within ~3 ulp; this allows 32 ulp relative
// on the score, 4 ulp on the key, and an absolute floor for subnormal exp).
__device__ __forceinline__ float key_bound(float s, float key)
{
    return s * 0x1p-18f + fabsf(key) * 0x1p-21f + 0x1p-60f;
}

// a ranks before b: larger key first; NaN keys after all numbers; equal keys
// (and two NaNs) by ascending id
__device__ __forceinline__ bool ranks_before(float ka, int ia, float kb, int ib)
{
    bool na = isnan(ka), nb = isnan(kb);
    if (na || nb)
        return (na && nb) ? ia < ib : nb;
    return ka > kb || (ka == kb && ia < ib);
}

// ------------------------------------------------------------------ warp-level top-k merges

// Per-lane best-first lists of (key, id, score), MOE_MAX_TOPK long; the
// sentinel (NaN key, largest id) ranks after everything.
struct CandList {
    float k[MOE_MAX_TOPK], s[MOE_MAX_TOPK];
    int i[MOE_MAX_TOPK];
    __device__ __forceinline__ void clear()
    {
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK; ++j) {
            k[j] = __int_as_float(0x7fffffff);
            i[j] = 0x7fffffff;
            s[j] = 0.0f;
        }
    }
    __device__ __forceinline__ void insert(float key, int id, float sc)
    {
        if (!ranks_before(key, id, k[MOE_MAX_TOPK - 1], i[MOE_MAX_TOPK - 1]))
            return;
        k[MOE_MAX_TOPK - 1] = key;
        i[MOE_MAX_TOPK - 1] = id;
        s[MOE_MAX_TOPK - 1] = sc;
#pragma unroll
        for (int j = MOE_MAX_TOPK - 1; j > 0; --j) {
            if (ranks_before(k[j], i[j], k[j - 1], i[j - 1])) {
                float tk = k[j], ts = s[j];
                int ti = i[j];
                k[j] = k[j - 1];
                i[j] = i[j - 1];
                s[j] = s[j - 1];
                k[j - 1] = tk;
                i[j - 1] = ti;
                s[j - 1] = ts;
            }
        }
    }
    __device__ __forceinline__ void pop()
    {
#pragma unroll
        for (int j = 0; j < MOE_MAX_TOPK - 1; ++j) {
            k[j] = k[j + 1];
            i[j] = i[j + 1];
            s[j] = s[j + 1];
        }
        k[MOE_MAX_TOPK - 1] = __int_as_float(0x7fffffff);
        i[MOE_MAX_TOPK - 1] = 0x7fffffff;
        s[MOE_MAX_TOPK - 1] = 0.0f;
    }
};

// k rounds of a warp-wide best-of-heads: writes the warp's best k (key, id,
// score) to out (lane 0) in rank order. All lanes must call.
__device__ __forceinline__ void warp_merge(CandList &L, int kk, float *ok, int *oi, float *os)
{
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    for (int r = 0; r < kk; ++r) {
        float bk = L.k[0], bs = L.s[0];
        int bi = L.i[0];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float xk = __shfl_xor_sync(full, bk, o), xs = __shfl_xor_sync(full, bs, o);
            const int xi = __shfl_xor_sync(full, bi, o);
            if (ranks_before(xk, xi, bk, bi)) {
                bk = xk;
                bi = xi;
                bs = xs;
            }
        }
        if (L.i[0] == bi && bi != 0x7fffffff)
            L.pop();  // the lane that held the winner (ids are unique)
        if (lane == 0) {
            ok[r] = bk;
            oi[r] = bi;
            os[r] = bs;
        }
    }
}

// per-lane lists of lower bounds (values only): the warp's k largest
__device__ __forceinline__ void warp_topk_values(float (&lo)[MOE_MAX_TOPK], int kk, float *out)
{
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    for (int r = 0; r < kk; ++r) {
        float v = lo[0], mx = v;
#pragma unroll
        for (int o = 16; o; o >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(full, mx, o));
        const unsigned who = __ballot_sync(full, v == mx);
        if (lane == __ffs(who) - 1) {
#pragma unroll
            for (int j = 0; j < MOE_MAX_TOPK - 1; ++j)
                lo[j] = lo[j + 1];
            lo[MOE_MAX_TOPK - 1] = -INFINITY;
        }
        if (lane == 0)
            out[r] = mx;
    }
}

__device__ __forceinline__ void lo_insert(float (&lo)[MOE_MAX_TOPK], float v)
{
    if (!(v > lo[MOE_MAX_TOPK - 1]))
        return;
    lo[MOE_MAX_TOPK - 1] = v;
#pragma unroll
    for (int j = MOE_MAX_TOPK - 1; j > 0; --j) {
        if (lo[j] > lo[j - 1]) {
            float t = lo[j];
            lo[j] = lo[j - 1];
            lo[j - 1] = t;
        }
    }
}

struct TokenPick {
    int id[MOE_MAX_TOPK];
    float s[MOE_MAX_TOPK];
    int flags;
};

// ------------------------------------------------------------------ selection + plan (whole CTA, 256 threads)

struct SelectSmem {
    TokenPick tok[MOE_MAX_TOKENS];
    float w[MOE_MAX_TOKENS][MOE_MAX_TOPK];
    float wlo[8][MOE_MAX_TOPK];                       // per warp: its k largest lower bounds
    float wk[8][MOE_MAX_TOPK], ws[8][MOE_MAX_TOPK];   // per warp: its k best exact candidates
    int wi[8][MOE_MAX_TOPK];
    int wflag[8];
    int warp_sum[2][8];
    int ne;
    int cnt[MOE_MAX_ROUTED];   // tokens that picked expert e
    int pidx[MOE_MAX_ROUTED];  // plan index of e (exclusive prefix of cnt > 0)
    int poff[MOE_MAX_ROUTED];  // first pair of e (exclusive prefix of cnt)
};

__device__ __forceinline__ void group_sync(int group, int gsz)
{
    if (gsz == 1)
        __syncwarp();
    else
        asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(gsz * 32) : "memory");
}

// The picks of one token by a group of gsz warps (experts split across them).
// Pass 1: single-precision keys with error bounds give T, the k-th largest
// lower bound; pass 2: exact keys (f64 scores) for the experts whose upper
// bound reaches T, merged best-first. Writes sm.tok[t] and sm.w[t].
__device__ void select_token_group(const RouteArgs &a, const float *logits, int t, int group, int gsz,
                                   SelectSmem &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wig = warp - group * gsz;
    const int n = a.n, k = a.k, stride = gsz * 32;
    const float *lg = logits + (size_t)t * n;
    float lo[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j)
        lo[j] = -INFINITY;
    bool nonfinite = false;
    for (int e = wig * 32 + lane; e < n; e += stride) {
        const float l = __ldcg(lg + e);
        const float tt = __fdiv_rn(l, a.temp);
        const float sa = score_approx(tt);
        const float ka = __fadd_rn(sa, __ldg(a.bias + e));
        nonfinite |= !isfinite(l) || !isfinite(ka);
        lo_insert(lo, isnan(ka) ? -INFINITY : (isinf(ka) ? ka : ka - key_bound(sa, ka)));
    }
    warp_topk_values(lo, k, sm.wlo[warp]);
    const unsigned nf = __ballot_sync(0xffffffffu, nonfinite);
    if (lane == 0)
        sm.wflag[warp] = nf ? MOE_HDR_NONFINITE : 0;
    group_sync(group, gsz);
    // T: the k-th largest of the group's gsz * k values (every warp of the group)
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j)
        lo[j] = -INFINITY;
    for (int j = lane; j < gsz * k; j += 32)
        lo_insert(lo, sm.wlo[group * gsz + j / k][j % k]);
    float tops[MOE_MAX_TOPK];
    warp_topk_values(lo, k, tops);
    const float T = __shfl_sync(0xffffffffu, tops[k - 1], 0);
    // pass 2
    CandList L;
    L.clear();
    for (int e = wig * 32 + lane; e < n; e += stride) {
        const float l = __ldcg(lg + e);
        const float tt = __fdiv_rn(l, a.temp);
        const float sa = score_approx(tt);
        const float b = __ldg(a.bias + e);
        const float ka = __fadd_rn(sa, b);
        const float hi = isnan(ka) ? -INFINITY : (isinf(ka) ? ka : ka + key_bound(sa, ka));
        if (hi >= T) {
            const float sx = score_exact(tt);
            L.insert(__fadd_rn(sx, b), e, sx);
        }
    }
    warp_merge(L, k, sm.wk[warp], sm.wi[warp], sm.ws[warp]);
    group_sync(group, gsz);
    if (wig == 0) {
        L.clear();
        for (int j = lane; j < gsz * k; j += 32) {
            const int w = group * gsz + j / k, r = j % k;
            L.insert(sm.wk[w][r], sm.wi[w][r], sm.ws[w][r]);
        }
        TokenPick &p = sm.tok[t];
        float kk_[MOE_MAX_TOPK];
        warp_merge(L, k, kk_, p.id, p.s);
        if (lane == 0) {
            int fl = 0;
            for (int w = 0; w < gsz; ++w)
                fl |= sm.wflag[group * gsz + w];
            p.flags = fl;
            // weights in pick order, each step one f32 rounding
            if (a.norm && k > 1) {
                float sum = 0.0f;
                for (int i = 0; i < k; ++i)
                    sum = __fadd_rn(sum, p.s[i]);
                sum = __fadd_rn(sum, 1e-20f);
                for (int i = 0; i < k; ++i)
                    sm.w[t][i] = __fmul_rn(__fdiv_rn(p.s[i], sum), a.route_scale);
            } else {
                for (int i = 0; i < k; ++i)
                    sm.w[t][i] = __fmul_rn(p.s[i], a.route_scale);
            }
        }
    }
}

__device__ void select_and_plan(const RouteArgs &a, const float *logits, SelectSmem &sm)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.n, k = a.k, m = a.m, cap = m * k;
    // warps in groups: all 8 on one token for m = 1, down to one warp per token
    int gsz = 8;
    while (gsz > 1 && gsz * m > 8)
        gsz >>= 1;
    const int group = warp / gsz;
    if (group < m)
        select_token_group(a, logits, group, group, gsz, sm);
    for (int e = tid; e < n; e += blockDim.x)
        sm.cnt[e] = 0;
    __syncthreads();
    // defensive: a pick outside [0, n) would index the tables below
    if (tid < cap) {
        int &id = sm.tok[tid / k].id[tid % k];
        if (id < 0 || id >= n) {
            if (a.ctrl)
                atomicOr(a.ctrl + MOE_CTRL_STATUS, (uint32_t)MOE_WS_PLAN);
            id = 0;
        }
    }
    __syncthreads();
    if (tid < cap)
        atomicAdd(&sm.cnt[sm.tok[tid / k].id[tid % k]], 1);
    __syncthreads();
    // exclusive prefix sums of (cnt > 0) and cnt over e; 4 experts per thread
    int e0 = tid * 4, f[4], c[4], fs = 0, cs = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int e = e0 + i;
        c[i] = e < n ? sm.cnt[e] : 0;
        f[i] = c[i] > 0;
        fs += f[i];
        cs += c[i];
    }
    int fi = fs, ci = cs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int fv = __shfl_up_sync(0xffffffffu, fi, o), cv = __shfl_up_sync(0xffffffffu, ci, o);
        if (lane >= o) {
            fi += fv;
            ci += cv;
        }
    }
    if (lane == 31) {
        sm.warp_sum[0][warp] = fi;
        sm.warp_sum[1][warp] = ci;
    }
    __syncthreads();
    int fb = 0, cb = 0;
    for (int w = 0; w < warp; ++w) {
        fb += sm.warp_sum[0][w];
        cb += sm.warp_sum[1][w];
    }
    if (tid == blockDim.x - 1)
        sm.ne = fb + fi;
    fi = fb + fi - fs;  // exclusive
    ci = cb + ci - cs;
    const int po = m * (1 + 3 * k);  // plan tail of the header
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int e = e0 + i;
        if (e < n) {
            sm.pidx[e] = fi;
            sm.poff[e] = ci;
            if (f[i]) {
                int slot = __ldg(a.slot_row + e);
                unsigned long long s = slot < 0 ? 0ull : (unsigned long long)slot;
                unsigned long long base = (unsigned long long)a.arena_base + s * a.slot_bytes;
                a.ptrs[fi] = base + a.gate_off;
                a.ptrs[cap + fi] = base + a.up_off;
                a.ptrs[2 * cap + fi] = base + a.down_off;
                a.hdr[po + 1 + fi] = ci;
                a.hdr[po + 2 + cap + fi] = e;
            }
        }
        fi += f[i];
        ci += c[i];
    }
    __syncthreads();
    if (tid == 0) {
        a.hdr[po] = sm.ne;
        a.hdr[po + 1 + sm.ne] = cap;
    }
    // pairs: token t's pick e goes to poff[e] + (number of earlier tokens that picked e)
    if (tid < cap) {
        int t = tid / k, i = tid % k, e = sm.tok[t].id[i], rank = 0;
        for (int t2 = 0; t2 < t; ++t2)
            for (int i2 = 0; i2 < k; ++i2)
                rank += sm.tok[t2].id[i2] == e;
        int pair = sm.poff[e] + rank;
        a.plan_rows[pair] = t;
        a.plan_w[pair] = sm.w[t][i];
    }
    // header rows: status, picks, weight bits, slots of the picks in ascending id
    if (tid < m) {
        const TokenPick &p = sm.tok[tid];
        int32_t *h = a.hdr + (size_t)tid * (1 + 3 * k);
        int sorted[MOE_MAX_TOPK];
        int status = p.flags;
        for (int i = 0; i < k; ++i) {
            h[1 + i] = p.id[i];
            h[1 + k + i] = __float_as_int(sm.w[tid][i]);
            int v = p.id[i], j = i;
            while (j > 0 && sorted[j - 1] > v) {
                sorted[j] = sorted[j - 1];
                --j;
            }
            sorted[j] = v;
        }
        for (int i = 0; i < k; ++i) {
            int slot = __ldg(a.slot_row + sorted[i]);
            if (slot < 0)
                status |= MOE_HDR_MISS;
            h[1 + 2 * k + i] = slot < 0 ? 0 : slot;
        }
        h[0] = status;
    }
}

// ------------------------------------------------------------------ kernels

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
        uint64_t pol = policy_evict_first();
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
    bool ok = nrows <= 0 || mbar_wait(bar, 0, a.ctrl + MOE_CTRL_STATUS);
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
                uint4 wv = wr[c], xv = xr[c];
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
        int r = i / m, t = i % m;
        float s = 0.0f;
        for (int w = 0; w < nw; ++w)
            s += red[((size_t)w * a.rows_per_cta + r) * m + t];
        a.logits[(size_t)t * a.n + row0 + r] = s;
    }
    if (!a.do_select)
        return;
    // the last CTA to finish its logits runs the selection
    __threadfence();
    __syncthreads();
    if (tid == 0)
        *s_last = atomicAdd(a.ctrl + MOE_CTRL_TICKET, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!*s_last)
        return;
    __threadfence();
    SelectSmem *sel = reinterpret_cast<SelectSmem *>(sw);  // the weights are no longer needed
    select_and_plan(a, a.logits, *sel);
    if (tid == 0)
        atomicExch(a.ctrl + MOE_CTRL_TICKET, 0u);
}

// the selection alone, on caller-provided logits: one CTA of 256 threads
__global__ void __launch_bounds__(256) moe_select_kernel(RouteArgs a)
{
    __shared__ SelectSmem sel;
    pdl_wait();
    pdl_launch_dependents();
    select_and_plan(a, a.logits, sel);
}

}  // namespace moe

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
// score is the correctly rounded f32 of the exact value, evaluated in double
// precision in the router epilogue, where every CTA takes a few of the rows
// (FP64 is a slow pipe on GB300; spread over the CTAs its latency is paid
// once). The selecting CTA is latency-bound: it reads everything it needs in
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

// k rounds of the warp-wide maximum over PL values per lane (distinct; 0
// marks an empty place and ranks last): out[r] = the r-th largest, written
// by lane 0. The lane holding the winner removes it and rescans its values.
template <int PL>
__device__ __forceinline__ void warp_topk(unsigned long long (&v)[PL], int k, unsigned long long *out)
{
    const int lane = threadIdx.x & 31;
    unsigned long long best = 0ull;
#pragma unroll
    for (int i = 0; i < PL; ++i)
        best = max(best, v[i]);
    for (int r = 0; r < k; ++r) {
        const unsigned hi = __reduce_max_sync(0xffffffffu, (unsigned)(best >> 32));
        const unsigned lo = __reduce_max_sync(0xffffffffu, (unsigned)(best >> 32) == hi ? (unsigned)best : 0u);
        const unsigned long long win = ((unsigned long long)hi << 32) | lo;
        if (lane == 0)
            out[r] = win;
        if (win != 0ull && best == win) {
            best = 0ull;
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                v[i] = v[i] == win ? 0ull : v[i];
                best = max(best, v[i]);
            }
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
                const int t = i / n, e = i - t * n;
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
                    const int c = lane + 32 * j;
                    v[j] = c < nc ? sm.cand[group * gsz + c / k][c % k] : 0ull;
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
            eq[j] = q < cap ? sm.pick[q / k][q % k] : 0;
            tq[j] = q / k;
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
                for (int q2 = 0; q2 < cap; ++q2) {
                    const int e2 = sm.ent[q2], t2 = q2 / k;
                    rq[j] += e2 < eq[j] || (e2 == eq[j] && t2 < tq[j]);
                    earlier += e2 == eq[j] && t2 < tq[j];
                }
                fq[j] = earlier == 0;
                sm.first[q] = fq[j];
                a.plan_rows[rq[j]] = tq[j];
                a.plan_w[rq[j]] = sm.w[tq[j]][q % k];
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
    const bool ok = nrows <= 0 || mbar_wait(bar, 0, a.ctrl + MOE_CTRL_STATUS);
    if (__syncthreads_and(ok) == 0)
        return;
    // logits: one warp per row, all tokens at once; lane j takes the 16-byte
    // chunks j + 32 i into four partial sums (i mod 4), added pairwise, then a
    // warp butterfly -- a fixed order per (token, row), whatever m is
    const int nch = dim / 8;
    with_m(m, [&](auto MC) {
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
    for (int i = tid; i < nrows * m; i += blockDim.x) {
        const int r = i / m, t = i % m;
        const float l = red[i];
        const size_t o = (size_t)t * a.n + row0 + r;
        a.logits[o] = l;
        if (a.do_select) {
            // the exact score of this row, here: the f64 chain runs on a few
            // threads of every CTA in parallel instead of in the selecting CTA
            const float sc = score_exact(l, a.temp);
            a.scores[o] = sc;
            a.keys[o] = __fadd_rn(sc, s_bias[r]);
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
        atomicExch(a.ctrl + MOE_CTRL_TICKET, 0u);
        // a hint for the gate/up kernel's producer: the plan is written, so
        // its dependency wait is about to end (its own wait still orders it)
        *reinterpret_cast<volatile uint32_t *>(a.ctrl + MOE_CTRL_GATEUP + 5) = 1u;
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
    for (int i = threadIdx.x; i < (int)mn; i += blockDim.x) {
        const float s = score_exact(a.logits[i], a.temp);
        sc[i] = s;
        ky[i] = __fadd_rn(s, __ldg(a.bias + i % a.n));
    }
    __syncthreads();
    select_and_plan<false>(a, a.logits, sc, ky, slot, smem);
}

}  // namespace moe

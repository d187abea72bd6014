// moe_prefill.cuh -- the batched (prefill) arm of the MoE layer on tensor cores.
//
// Page spark_model/layers/moe_v41.rs, struct Kernels (gather, scatter_add,
// sum_rows, quant_d2s6 / quant_d4, mmq_q2k_*, mmq_q3k_*, gemm) and struct
// MoeV41 (a_rows: an expert group's gathered rows; a_q8: their q8_1
// activations): for many tokens the routed experts run as GEMMs over each
// expert's group of tokens, the shared expert and the router as dense GEMMs.
// The layer's arithmetic is the decode step's; only its grouping changes.
//
// Every contraction runs on tcgen05.mma (kind::f16, f32 accumulator in TMEM,
// 128 x N tiles, K in steps of 64) in one kernel template, moe_tc_gemm:
//   AK = 0  A (weights) bf16 by TMA          -- router, shared W1 / W3 / W2
//   AK = 1  A dequantised from Q2_K blocks  -- routed gate, up
//   AK = 2  A dequantised from Q3_K blocks  -- routed down
// For AK > 0 a producer warp streams the raw blocks of 128 weight rows with
// 3-D TMA loads (u32 elements over [slot][row][bytes] of the expert arena)
// and four worker warps turn them into fp16 operand tiles in the 128-byte
// swizzled layout (each weight d * sc * q - dmin * m or d * sc * q in f32,
// then rounded to fp16); B is the group's activation rows, fp16, by TMA.
// gate and up (AK = 1) split both operands into fp16 pairs hi + lo (22
// significant bits: the dequantised q8_1 activation, 18 bits, exactly; the
// weight to 2^-23) and accumulate hi.hi + hi.lo + lo.hi, so g and u are as
// exact as f32 sums allow -- h is quantised to q8_1 again, and g, u a few
// 2^-12 off would move some of its roundings. down (AK = 2) takes single
// fp16 parts (about 2^-12 relative per operand): its output is only summed.
// The tensor cores' f32 accumulation is coarser than a sequential f32 sum
// (about 2e-5 relative over K = 4096), so K is split over up to four
// accumulators in TMEM (4 x 128 columns) whose results the epilogue adds in
// f32, in order; over K = 4096 that keeps the router logits within 1e-5.
// One warp issues the MMAs; the four worker warps are the epilogue (TMEM ->
// registers -> global).
#pragma once
#include "moe_tc.cuh"
#include "moe_route.cuh"

namespace moe {

#define TC_M 128        // rows of a tile (weights)
#define TC_NT 128       // columns (tokens) of a tile, at most
#define TC_KC 64        // K per stage (one 128-byte swizzle atom of 16-bit elements)
#define TC_THREADS 192  // warps 0-3 workers / epilogue, 4 producer, 5 MMA
#define TC_BROWS 16     // rows of a B TMA box
#define TC_TMEM_COLS 512  // TMEM columns a CTA holds: up to 4 accumulators of TC_NT columns

// a column task of the routed GEMMs: the expert's slot, its first pair and
// the number of its pairs in this tile
struct TcTask {
    int slot, c0, ncols, pad;
};

struct TcArgs {
    int M, N, K;            // AK = 0: D[M x N] over K; AK > 0: M = rows of the matrix, K its row length
    float *out;             // out[col * ldo + row]
    int ldo;
    const float *colw;      // AK = 2: each column's (pair's) routing weight; else NULL
    const TcTask *tasks;    // AK > 0
    const int *ntasks;      // AK > 0: count of tasks (device)
    int raw_row;            // AK > 0: bytes of one row's blocks in a raw stage (rk / 256 blocks)
    int S, SR;              // operand stages, raw stages
    uint32_t raw_bytes;     // AK > 0: bytes of one raw stage (128 rows x raw_row)
    int rk;                 // AK > 0: K per raw stage
    int ksplit;             // K split over this many accumulators (1, 2 or 4), added in f32 at the end
    uint32_t *status;
    unsigned long long wait_ns;
};

// operands of a stage: hi and lo tiles for the split GEMM (gate, up)
__host__ __device__ constexpr int tc_parts(int AK) { return AK == 1 ? 2 : 1; }

__host__ __device__ inline size_t tc_smem_bytes(int parts, int S, int SR, uint32_t raw_bytes)
{
    // 1024 alignment slack, A and B stages (16 KB a part each), raw stages, barriers + TMEM address
    return 1024 + (size_t)S * 2 * parts * 16384 + (size_t)SR * raw_bytes + 256;
}

// f32 pair -> fp16 pairs hi (the rounding) and lo (the rounding of the rest)
__device__ __forceinline__ void split_half2(float a, float b, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(a, b);
    const float2 back = __half22float2(h);
    const __half2 l = __floats2half2_rn(__fsub_rn(a, back.x), __fsub_rn(b, back.y));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// Q2_K: 64 weights (quarter kq of the super-block at blk) of one row -> 32
// words of fp16 pairs (hi) and of the pairs' remainders (lo), element order.
// w = d sc q - dmin m (one f32 rounding).
__device__ __forceinline__ void dq_q2k_quarter(const uint8_t *blk, int kq, uint32_t (&o)[32], uint32_t (&ol)[32])
{
    const uint32_t *bw = reinterpret_cast<const uint32_t *>(blk);  // 4-byte aligned (84-byte blocks)
    const uint32_t scw = bw[kq];                                   // scales of sub-blocks 4 kq .. 4 kq + 3
    const uint32_t dd = bw[20];
    const float d = f16_bits_to_f32(dd), dmin = f16_bits_to_f32(dd >> 16);
    float ds[4], dm[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const uint32_t sc = (scw >> (8 * u)) & 0xFFu;
        ds[u] = d * (float)(sc & 15u);
        dm[u] = dmin * (float)(sc >> 4);
    }
    const int half = kq >> 1, g0 = 2 * (kq & 1);
    uint32_t W[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        W[i] = bw[4 + 8 * half + i];
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            const uint32_t qq = (W[wi] >> (2 * (g0 + gi))) & 0x03030303u;
            const int u = 2 * gi + (wi >> 2);
            float f[4];
#pragma unroll
            for (int b = 0; b < 4; ++b)  // 2^23 + q exactly, then q
                f[b] = __uint_as_float(__byte_perm(qq, 0x4B000000u, b | 0x7440)) - 8388608.0f;
            split_half2(fmaf(f[0], ds[u], -dm[u]), fmaf(f[1], ds[u], -dm[u]), o[16 * gi + 2 * wi],
                        ol[16 * gi + 2 * wi]);
            split_half2(fmaf(f[2], ds[u], -dm[u]), fmaf(f[3], ds[u], -dm[u]), o[16 * gi + 2 * wi + 1],
                        ol[16 * gi + 2 * wi + 1]);
        }
    }
}

// Q3_K: 64 weights (quarter kq) of one row from a 110-byte block at a 2-byte
// aligned address. w = d * (scale - 32) * q (exact in f32), q = low2 | hbit
// << 2 minus 4.
__device__ __forceinline__ void dq_q3k_quarter(const uint8_t *blk, int kq, uint32_t (&o)[32])
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(blk);
    const uint32_t *W = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(a & 3) * 8u;
    auto word = [&](int i) { return __funnelshift_r(W[i], W[i + 1], sh); };
    uint32_t hm[8], qv[8];
    const int half = kq >> 1, g0 = 2 * (kq & 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        hm[i] = word(i);
        qv[i] = word(8 + 8 * half + i);
    }
    const uint32_t s0 = word(24), s1 = word(25), s2 = word(26);
    const float d = f16_bits_to_f32(word(27));
    const uint32_t scb[3] = {s0, s1, s2};
    auto sbyte = [&](int i) { return (scb[i >> 2] >> (8 * (i & 3))) & 0xFFu; };
    float ds[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = 4 * kq + u;  // sub-block
        const uint32_t lo4 = i < 8 ? (sbyte(i) & 15u) : (sbyte(i - 8) >> 4);
        const uint32_t hi2 = (sbyte(8 + (i & 3)) >> (2 * (i >> 2))) & 3u;
        ds[u] = d * (float)((int)(lo4 | (hi2 << 4)) - 32);
    }
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        const int g = g0 + gi, hsh = 4 * half + g;  // weight j: bit j / 32 of hmask[j % 32]
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
            const uint32_t v = ((qv[wi] >> (2 * g)) & 0x03030303u) | (((hm[wi] >> hsh) & 0x01010101u) << 2);
            const int u = 2 * gi + (wi >> 2);
            float f[4];
#pragma unroll
            for (int b = 0; b < 4; ++b)  // 2^23 + v exactly, then v - 4
                f[b] = __uint_as_float(__byte_perm(v, 0x4B000000u, b | 0x7440)) - 8388612.0f;
            const __half2 h01 = __floats2half2_rn(f[0] * ds[u], f[1] * ds[u]);
            const __half2 h23 = __floats2half2_rn(f[2] * ds[u], f[3] * ds[u]);
            o[16 * gi + 2 * wi] = *reinterpret_cast<const uint32_t *>(&h01);
            o[16 * gi + 2 * wi + 1] = *reinterpret_cast<const uint32_t *>(&h23);
        }
    }
}

// bounded mbarrier wait that gives up for good after the first timeout of
// this thread (`dead`), so that a broken pipeline still ends
__device__ __forceinline__ void tc_wait(uint64_t *bar, uint32_t parity, const TcArgs &a, bool &dead)
{
    if (!dead && !mbar_wait(bar, parity, a.status, a.wait_ns))
        dead = true;
}

template <int AK>
__global__ void __launch_bounds__(TC_THREADS, 1)
    moe_tc_gemm(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                const __grid_constant__ CUtensorMap bmap_lo, TcArgs a)
{
    constexpr int PARTS = tc_parts(AK);
    constexpr uint32_t STG = PARTS * 16384u;  // bytes of a stage's A (or B) tiles: hi, then lo
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int S = a.S, SR = a.SR;
    uint8_t *sa = smem;                    // S x STG
    uint8_t *sb = smem + (size_t)S * STG;  // S x STG
    uint8_t *sraw = sb + (size_t)S * STG;  // SR x raw_bytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(sraw + (size_t)SR * a.raw_bytes);
    uint64_t *full_a = bars, *full_b = bars + S, *empty = bars + 2 * S, *raw_full = bars + 3 * S;
    uint64_t *raw_empty = raw_full + SR, *done = raw_empty + SR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the tile: rows m0 .. m0 + 127 of the weights, columns c0 .. c0 + ncols - 1
    int m0 = blockIdx.y * TC_M, c0, ncols, slot = 0;
    if constexpr (AK == 0) {
        c0 = blockIdx.x * TC_NT;
        ncols = min(TC_NT, a.N - c0);
    } else {
        if ((int)blockIdx.x >= __ldg(a.ntasks))
            return;
        const TcTask t = a.tasks[blockIdx.x];
        slot = t.slot;
        c0 = t.c0;
        ncols = t.ncols;
    }
    const int nb16 = (ncols + TC_BROWS - 1) / TC_BROWS;  // B boxes a stage
    const int n_mma = nb16 * TC_BROWS;                   // MMA N (a multiple of 16)
    const uint32_t idesc = mma_idesc(TC_M, n_mma, AK == 0);
    const int KC = a.K / TC_KC;
    const int per_raw = AK == 0 ? 1 : a.rk / TC_KC;     // operand stages a raw stage feeds

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_a[s], AK == 0 ? 1 : 128);
            mbar_init(&full_b[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int r = 0; r < SR; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], 128);
        }
        mbar_init(done, 1);
        fence_barrier_init();
    }
    if (warp == 0)
        tmem_alloc(tmem_slot, TC_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool dead = false;

    if (warp == 4) {
        // ---------------- producer: B boxes (and A, or the raw blocks)
        if (lane == 0) {
            tma_prefetch_map(&amap);
            tma_prefetch_map(&bmap);
            if constexpr (PARTS == 2)
                tma_prefetch_map(&bmap_lo);
            for (int kc = 0; kc < KC; ++kc) {
                if constexpr (AK > 0) {
                    if (kc % per_raw == 0) {
                        const int rc = kc / per_raw, r = rc % SR;
                        if (rc >= SR)
                            tc_wait(&raw_empty[r], (uint32_t)((rc / SR - 1) & 1), a, dead);
                        mbar_arrive_expect_tx(&raw_full[r], a.raw_bytes);
                        tma_load_3d(sraw + (size_t)r * a.raw_bytes, &amap, rc * (a.raw_row / 4), m0, slot,
                                    &raw_full[r]);
                    }
                }
                const int s = kc % S;
                if (kc >= S)
                    tc_wait(&empty[s], (uint32_t)((kc / S - 1) & 1), a, dead);
                if constexpr (AK == 0) {
                    mbar_arrive_expect_tx(&full_a[s], 16384u);
                    tma_load_2d(sa + (size_t)s * STG, &amap, kc * TC_KC, m0, &full_a[s]);
                }
                mbar_arrive_expect_tx(&full_b[s], (uint32_t)PARTS * nb16 * TC_BROWS * 128u);
                for (int i = 0; i < nb16; ++i) {
                    tma_load_2d(sb + (size_t)s * STG + i * TC_BROWS * 128, &bmap, kc * TC_KC, c0 + i * TC_BROWS,
                                &full_b[s]);
                    if constexpr (PARTS == 2)
                        tma_load_2d(sb + (size_t)s * STG + 16384 + i * TC_BROWS * 128, &bmap_lo, kc * TC_KC,
                                    c0 + i * TC_BROWS, &full_b[s]);
                }
            }
        }
    } else if (warp == 5) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const int kper = KC / a.ksplit;  // K-chunks an accumulator takes
            for (int kc = 0; kc < KC; ++kc) {
                const int s = kc % S;
                const uint32_t ph = (uint32_t)((kc / S) & 1);
                const uint32_t acc = tmem + (uint32_t)(kc / kper) * TC_NT;
                const bool first = kc % kper == 0;
                tc_wait(&full_a[s], ph, a, dead);
                tc_wait(&full_b[s], ph, a, dead);
                tc_fence_after();
                const uint64_t ad = sw128_desc(sa + (size_t)s * STG), bd = sw128_desc(sb + (size_t)s * STG);
#pragma unroll
                for (int k = 0; k < TC_KC / 16; ++k) {  // K = 16 a step: 32 bytes further in the swizzle atom
                    mma_f16(acc, ad + 2 * k, bd + 2 * k, idesc, !first || k > 0);
                    if constexpr (PARTS == 2) {  // + hi . lo + lo . hi (lo tiles 16 KB after the hi tiles)
                        mma_f16(acc, ad + 2 * k, bd + (16384 >> 4) + 2 * k, idesc, true);
                        mma_f16(acc, ad + (16384 >> 4) + 2 * k, bd + 2 * k, idesc, true);
                    }
                }
                mma_commit(&empty[s]);
            }
            mma_commit(done);
        }
    } else {
        // ---------------- workers (AK > 0): raw blocks -> fp16 operand tiles
        if constexpr (AK > 0) {
            const int r = threadIdx.x;  // the tile row this thread builds
            const int bbytes = AK == 1 ? MOE_Q2K_BYTES : MOE_Q3K_BYTES;
            for (int kc = 0; kc < KC; ++kc) {
                const int rc = kc / per_raw, ri = rc % SR, q = kc % per_raw;
                if (q == 0)
                    tc_wait(&raw_full[ri], (uint32_t)((rc / SR) & 1), a, dead);
                const int s = kc % S;
                if (kc >= S)
                    tc_wait(&empty[s], (uint32_t)((kc / S - 1) & 1), a, dead);
                const uint8_t *blk = sraw + (size_t)ri * a.raw_bytes + (size_t)r * a.raw_row + (q >> 2) * bbytes;
                uint32_t o[32];
                uint8_t *tile = sa + (size_t)s * STG;
                if constexpr (AK == 1) {
                    uint32_t ol[32];
                    dq_q2k_quarter(blk, q & 3, o, ol);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4 *>(tile + 16384 + sw128_offset(r, 8 * c)) =
                            make_uint4(ol[4 * c], ol[4 * c + 1], ol[4 * c + 2], ol[4 * c + 3]);
                } else {
                    dq_q3k_quarter(blk, q & 3, o);
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 8 * c)) =
                        make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                fence_proxy_async_smem();  // generic-proxy writes before the MMA reads them
                mbar_arrive(&full_a[s]);
                if (q == per_raw - 1)
                    mbar_arrive(&raw_empty[ri]);
            }
        }
        // ---------------- epilogue: row m0 + threadIdx.x, columns 32 at a time
        tc_wait(done, 0, a, dead);
        tc_fence_after();
        const int row = m0 + (int)threadIdx.x;
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        for (int cb = 0; cb < ncols; cb += 32) {
            float v[32];
            tmem_ld32(lane_addr + (uint32_t)cb, v);
            for (int j = 1; j < a.ksplit; ++j) {
                float w[32];
                tmem_ld32(lane_addr + (uint32_t)(j * TC_NT + cb), w);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = __fadd_rn(v[i], w[i]);
            }
            if (row < a.M) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int col = cb + j;
                    if (col < ncols) {
                        float x = v[j];
                        if constexpr (AK == 2)
                            x = __fmul_rn(__ldg(a.colw + c0 + col), x);
                        a.out[(size_t)(c0 + col) * a.ldo + row] = x;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tmem, TC_TMEM_COLS);
}

// ------------------------------------------------------------------ the batched selection

// Per token: key = score + bias over the n experts, the k best (stable:
// ties to the lower id), weights from the unbiased scores (renormalised in
// f32 in pick order when norm and k > 1, times route_scale) -- the rule of
// fn route_from_logits, as in the decode selection. One warp per token.
struct PTopArgs {
    const float *logits, *scores, *bias;
    int32_t *picks, *flags;
    float *weights;
    int m, n, k, norm;
    float route_scale;
};

__global__ void __launch_bounds__(256) moe_prefill_topk_kernel(PTopArgs a)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= a.m)
        return;
    const int t = warp;
    const float *sc = a.scores + (size_t)t * a.n;
    const float *lg = a.logits + (size_t)t * a.n;
    __shared__ unsigned long long win[8][MOE_MAX_TOPK];
    unsigned long long *out = win[threadIdx.x >> 5];
    bool nonfinite = false;
    with_per_lane((a.n + 31) / 32, [&](auto PC) {
        constexpr int PL = decltype(PC)::value;
        unsigned long long v[PL];
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            const int e = lane + 32 * i;
            if (e < a.n) {
                const float key = __fadd_rn(sc[e], __ldg(a.bias + e));
                nonfinite = nonfinite || !isfinite(key) || !isfinite(lg[e]);
                v[i] = rank_value(key, e);
            } else {
                v[i] = 0ull;
            }
        }
        warp_topk<PL>(v, a.k, out);
    });
    nonfinite = __any_sync(0xffffffffu, nonfinite);
    __syncwarp();
    if (lane == 0) {
        float s[MOE_MAX_TOPK];
        int id[MOE_MAX_TOPK];
        float sum = 0.0f;
        for (int i = 0; i < a.k; ++i) {
            id[i] = min(max(rank_id(out[i]), 0), a.n - 1);
            s[i] = sc[id[i]];
            sum = __fadd_rn(sum, s[i]);
        }
        sum = __fadd_rn(sum, 1e-20f);
        for (int i = 0; i < a.k; ++i) {
            a.picks[(size_t)t * a.k + i] = id[i];
            a.weights[(size_t)t * a.k + i] = (a.norm && a.k > 1) ? __fmul_rn(__fdiv_rn(s[i], sum), a.route_scale)
                                                                 : __fmul_rn(s[i], a.route_scale);
        }
        a.flags[t] = nonfinite ? MOE_HDR_NONFINITE : 0;
    }
}

// ------------------------------------------------------------------ grouping by expert

// One CTA of 1024 threads. The pairs (token, pick) grouped by expert in
// ascending id, tokens ascending within an expert (deterministic): count,
// exclusive scan, then per expert a warp walks the tokens in order and
// places its pairs with ballots. Also the column tasks of the routed GEMMs
// (ceil(count / TC_NT) per expert) and each pick's pair index.
struct PPlanArgs {
    const int32_t *picks;
    const float *weights;
    const int32_t *slot_row;
    int m, n, k;
    int32_t *cnt, *off;      // [n], [n + 1]
    int32_t *pair_tok;       // [P]
    float *pair_w;           // [P]
    int32_t *pick_pair;      // [P]: pair index of pick (t, i)
    TcTask *tasks;           // column tasks
    int32_t *ntasks;
    uint32_t *status;
};

__global__ void __launch_bounds__(1024) moe_prefill_plan_kernel(PPlanArgs a)
{
    __shared__ int s_cnt[MOE_MAX_ROUTED], s_off[MOE_MAX_ROUTED + 1], s_toff[MOE_MAX_ROUTED + 1];
    const int tid = threadIdx.x, P = a.m * a.k;
    for (int e = tid; e < a.n; e += blockDim.x)
        s_cnt[e] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = a.picks[p];
        if (e >= 0 && e < a.n)
            atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0, tacc = 0;
        for (int e = 0; e < a.n; ++e) {
            s_off[e] = acc;
            s_toff[e] = tacc;
            acc += s_cnt[e];
            tacc += (s_cnt[e] + TC_NT - 1) / TC_NT;
        }
        s_off[a.n] = acc;
        s_toff[a.n] = tacc;
        *a.ntasks = tacc;
    }
    __syncthreads();
    for (int e = tid; e <= a.n; e += blockDim.x) {
        a.off[e] = s_off[e];
        if (e < a.n) {
            a.cnt[e] = s_cnt[e];
            const int sl = a.slot_row[e];
            if (s_cnt[e] > 0 && sl < 0)
                atomicOr(a.status, (uint32_t)MOE_WS_PLAN);  // a picked expert is not resident
            for (int j = 0; j * TC_NT < s_cnt[e]; ++j)
                a.tasks[s_toff[e] + j] = TcTask{sl < 0 ? 0 : sl, s_off[e] + j * TC_NT, min(TC_NT, s_cnt[e] - j * TC_NT), 0};
        }
    }
    // per expert, a warp places its pairs in token order
    const int warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    for (int e = warp; e < a.n; e += nw) {
        if (s_cnt[e] == 0)
            continue;
        int base = s_off[e];
        for (int t0 = 0; t0 < a.m; t0 += 32) {
            const int t = t0 + lane;
            int which = -1;
            if (t < a.m)
                for (int i = 0; i < a.k; ++i)
                    if (a.picks[(size_t)t * a.k + i] == e)
                        which = i;
            const unsigned bal = __ballot_sync(0xffffffffu, which >= 0);
            if (which >= 0) {
                const int q = base + __popc(bal & ((1u << lane) - 1u));
                a.pair_tok[q] = t;
                a.pair_w[q] = a.weights[(size_t)t * a.k + which];
                a.pick_pair[(size_t)t * a.k + which] = q;
            }
            base += __popc(bal);
        }
    }
}

// ------------------------------------------------------------------ activations

// x_hat = the dequantised q8_1 of each token's x (f16(d) * q, exact in f32)
// as fp16 hi + lo (exactly: 18 significant bits), then gathered into pair
// order: Xg[p] = x_hat[pair_tok[p]]. One warp per 32-block.
__global__ void moe_prefill_xhat_kernel(const uint16_t *x, int nblk, __half *xhat, __half *xhat_lo)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= nblk)
        return;
    const float v = bf16_to_f32(x[(size_t)warp * 32 + lane]);
    const Q8Block b = q8_quant_warp(v);
    const float xh = __fmul_rn(b.d8, (float)b.q);
    const __half hi = __float2half_rn(xh);
    xhat[(size_t)warp * 32 + lane] = hi;
    xhat_lo[(size_t)warp * 32 + lane] = __float2half_rn(__fsub_rn(xh, __half2float(hi)));
}

__global__ void moe_prefill_gather_kernel(const uint4 *src, const int32_t *pair_tok, int P, int row16, uint4 *dst)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)P * row16)
        return;
    const int p = (int)(i / row16), c = (int)(i % row16);
    dst[i] = src[(size_t)pair_tok[p] * row16 + c];
}

// h = SwiGLU(g, u) per pair, its q8_1 (f32 decisions, f16 scale), and the
// dequantised fp16 h_hat for the down GEMM. One warp per 32-block.
__global__ void moe_prefill_swiglu_kernel(const float *g, const float *u, int nblk, float limit, __half *hhat)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= nblk)
        return;
    const size_t i = (size_t)warp * 32 + lane;
    const Q8Block b = q8_quant_warp(swiglu_f32(g[i], u[i], limit));
    hhat[i] = __float2half_rn(__fmul_rn(b.d8, (float)b.q));
}

// the bf16 shared expert's hs = bf16(SwiGLU(gs, us))
__global__ void moe_prefill_shared_swiglu_kernel(const float *gs, const float *us, size_t count, float limit,
                                                 uint16_t *hs)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count)
        hs[i] = f32_to_bf16(swiglu_f32(gs[i], us[i], limit));
}

// acc[t] = its pairs' weighted down rows in ascending expert id, then sd;
// residual += acc; x_next = bf16(residual)
__global__ void moe_prefill_finish_kernel(const float *dw, const int32_t *picks, const int32_t *pick_pair, int k,
                                          const float *sd, float *acc, float *residual, uint16_t *x_next, int m,
                                          int dim)
{
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)m * dim)
        return;
    const int t = (int)(i / dim), r = (int)(i % dim);
    int e[MOE_MAX_TOPK], q[MOE_MAX_TOPK];
    for (int j = 0; j < k; ++j) {
        e[j] = __ldg(picks + (size_t)t * k + j);
        q[j] = min(max(__ldg(pick_pair + (size_t)t * k + j), 0), m * k - 1);
    }
    for (int j = 1; j < k; ++j)  // ascending expert id (the picks of a token are distinct)
        for (int l = j; l > 0 && e[l] < e[l - 1]; --l) {
            const int te = e[l], tq = q[l];
            e[l] = e[l - 1];
            q[l] = q[l - 1];
            e[l - 1] = te;
            q[l - 1] = tq;
        }
    float s = 0.0f;
    for (int j = 0; j < k; ++j)
        s = __fadd_rn(s, dw[(size_t)q[j] * dim + r]);
    if (sd)
        s = __fadd_rn(s, sd[i]);
    acc[i] = s;
    const float res = __fadd_rn(residual[i], s);
    residual[i] = res;
    x_next[i] = f32_to_bf16(res);
}

}  // namespace moe

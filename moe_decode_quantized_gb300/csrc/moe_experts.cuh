// moe_experts.cu -- the expert GEMVs of one decode step.
//
// Page spark_model/layers/moe_v41.rs (module doc; struct Kernels
// mmvq_q2k_experts, swiglu_q8, mmvq_q3k_experts, accumulate, finish; fn
// shared_side): every routed expert runs three K-quant GEMVs on its raw
// blocks (gate and up Q2_K, down Q3_K) against a q8_1 activation, with a
// clamped SwiGLU in between; the bf16 shared expert runs beside them and is
// added after the routed experts.
//
// Two persistent kernels, one CTA per SM, each a warp-specialised pipeline:
// one producer lane streams whole tasks (contiguous runs of rows) from HBM
// into a ring of shared-memory stages with 1-D bulk copies (TMA engine,
// L2 evict-first), eight consumer warps decode the 2/3-bit quants from shared
// memory with dp4a integer dots and reduce rows with warp shuffles.
//
//   gate/up kernel: tasks = rows of shared W1 / W3 (issued before the
//     programmatic-launch wait: they depend only on x, so they overlap the
//     router and the selection), then 64-super-block row runs of every plan
//     expert's gate and up matrices. Writes g, u (per plan pair) and gs, us.
//   down kernel: tasks = 32-super-block row runs of every plan expert's down
//     matrix and rows of shared W2, all prefetched before the wait (they need
//     only the pointer table); after the wait each CTA builds the q8_1 of
//     SwiGLU(g, u) for the pairs it needs and bf16(SwiGLU(gs, us)). A row
//     group is finished by the warp that completes its last task (a ticket
//     counter per group, no waiting): acc = plan-order sum of w * down, then
//     the shared row, residual += acc, x_next = bf16(residual).
#pragma once
#include "moe_common.cuh"

namespace moe {

struct Task {
    int kind;   // 0 end, 1 routed, 2 shared
    int mat;    // gate/up kernel: 0 gate or W1, 1 up or W3
    int p;      // plan expert
    int row;    // first row (routed) or the row (shared)
    int pair0, npair;
    int tok[MOE_MAX_TOKENS];
};

// ------------------------------------------------------------------ q8_1 (one 32-block per warp)

struct Q8Block {
    int q;      // this lane's quant
    float d;    // f32 scale (the decision scale)
    float d8;   // the f16-rounded scale the dots use
    int s16;    // sum of the quants of this lane's 16-value half
};

// per 32 values: d = amax / 127, q = round-half-away(v / d), q = 0 when amax = 0
__device__ __forceinline__ Q8Block q8_quant_warp(float v)
{
    const unsigned full = 0xffffffffu;
    float amax = fabsf(v);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(full, amax, o));
    Q8Block b;
    b.d = __fdiv_rn(amax, 127.0f);
    b.q = amax == 0.0f ? 0 : (int)roundf(__fdiv_rn(v, b.d));
    b.d8 = __half2float(__float2half_rn(b.d));
    int s = b.q;
#pragma unroll
    for (int o = 8; o; o >>= 1)
        s += __shfl_xor_sync(full, s, o);
    b.s16 = s;
    return b;
}

// Activation row in shared memory: segment sg (256 values) = 272 bytes of
// int8 quants + a 28-float record: [0..7] d8 of its 32-blocks, [8..23] per
// 16-value sub-block either d8 * sum(q) (float, Q2_K min term) or sum(q)
// (int bits, Q3_K offset term).
__host__ __device__ inline size_t act_row_bytes(int cols)
{
    return (size_t)(cols / MOE_QK) * (MOE_SEG_Q_BYTES + 4 * MOE_SEG_REC_FLOATS);
}

__device__ __forceinline__ void q8_store_smem(uint8_t *row, int nseg, int blk, const Q8Block &b,
                                              bool min_term)
{
    const int lane = threadIdx.x & 31;
    int sg = blk >> 3, bi = blk & 7;
    row[sg * MOE_SEG_Q_BYTES + bi * 32 + lane] = (uint8_t)(int8_t)b.q;
    float *rec = reinterpret_cast<float *>(row + nseg * MOE_SEG_Q_BYTES) + sg * MOE_SEG_REC_FLOATS;
    if (lane == 0)
        rec[bi] = b.d8;
    if ((lane & 15) == 0)
        rec[8 + 2 * bi + (lane >> 4)] =
            min_term ? __fmul_rn(b.d8, (float)b.s16) : __int_as_float(b.s16);
}

// ------------------------------------------------------------------ super-block dots

__device__ __forceinline__ uint32_t byte_of(const uint32_t *w, int i) { return (w[i >> 2] >> (8 * (i & 3))) & 0xFFu; }

// Q2_K super-block (84 bytes, 4-byte aligned in shared memory) against a
// q8_1 segment: d * sum_b d8_b (sc_2b dot_2b + sc_2b+1 dot_2b+1)
//               - dmin * sum_s min_s * d8 * sum(q8 of s)
__device__ __forceinline__ float q2k_dot(const uint32_t *blk, const int4 *xq, const float4 *rec)
{
    uint32_t sc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        sc[i] = blk[i];
    const uint32_t dd = blk[20];
    float mn = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 f = rec[2 + i];
        mn = fmaf((float)(byte_of(sc, 4 * i + 0) >> 4), f.x, mn);
        mn = fmaf((float)(byte_of(sc, 4 * i + 1) >> 4), f.y, mn);
        mn = fmaf((float)(byte_of(sc, 4 * i + 2) >> 4), f.z, mn);
        mn = fmaf((float)(byte_of(sc, 4 * i + 3) >> 4), f.w, mn);
    }
    const float4 da = rec[0], db = rec[1];
    const float d8[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
    float main = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t q[8];
#pragma unroll
        for (int w = 0; w < 8; ++w)
            q[w] = blk[4 + 8 * h + w];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int4 xa = xq[8 * h + 2 * g], xb = xq[8 * h + 2 * g + 1];
            const int sh = 2 * g;
            int s0 = __dp4a((int)((q[0] >> sh) & 0x03030303u), xa.x, 0);
            s0 = __dp4a((int)((q[1] >> sh) & 0x03030303u), xa.y, s0);
            s0 = __dp4a((int)((q[2] >> sh) & 0x03030303u), xa.z, s0);
            s0 = __dp4a((int)((q[3] >> sh) & 0x03030303u), xa.w, s0);
            int s1 = __dp4a((int)((q[4] >> sh) & 0x03030303u), xb.x, 0);
            s1 = __dp4a((int)((q[5] >> sh) & 0x03030303u), xb.y, s1);
            s1 = __dp4a((int)((q[6] >> sh) & 0x03030303u), xb.z, s1);
            s1 = __dp4a((int)((q[7] >> sh) & 0x03030303u), xb.w, s1);
            const int sub = 8 * h + 2 * g;
            const int isum = (int)(byte_of(sc, sub) & 15u) * s0 + (int)(byte_of(sc, sub + 1) & 15u) * s1;
            main = fmaf(d8[4 * h + g], (float)isum, main);
        }
    }
    return f16_bits_to_f32(dd) * main - f16_bits_to_f32(dd >> 16) * mn;
}

// Q3_K super-block (110 bytes, 2-byte aligned in shared memory) against a
// q8_1 segment: d * sum_b d8_b (sc_2b (dot_2b - 4 sum_2b) + sc_2b+1 (...)),
// the quants taken as q + 4 in [0, 7] for dp4a and the offset removed.
__device__ __forceinline__ float q3k_dot(const uint8_t *blk, const int4 *xq, const float4 *rec)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(blk);
    const uint32_t *W = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(a & 3) * 8u;  // 0 or 16
    uint32_t f[28];
#pragma unroll
    for (int i = 0; i < 28; ++i)
        f[i] = W[i];
#pragma unroll
    for (int i = 0; i < 27; ++i)
        f[i] = __funnelshift_r(f[i], f[i + 1], sh);
    const float d = f16_bits_to_f32(f[27] >> sh);
    // sixteen 6-bit scales from bytes 96..107 (field words 24..26)
    const uint32_t *scw = f + 24;
    int scale[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t low4 = i < 8 ? (byte_of(scw, i) & 15u) : (byte_of(scw, i - 8) >> 4);
        uint32_t high2 = (byte_of(scw, 8 + (i & 3)) >> (2 * (i >> 2))) & 3u;
        scale[i] = (int)(low4 | (high2 << 4)) - 32;
    }
    const float4 da = rec[0], db = rec[1];
    const float d8[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
    int sq[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 r = rec[2 + i];
        sq[4 * i + 0] = __float_as_int(r.x);
        sq[4 * i + 1] = __float_as_int(r.y);
        sq[4 * i + 2] = __float_as_int(r.z);
        sq[4 * i + 3] = __float_as_int(r.w);
    }
    float acc = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int4 xa = xq[8 * h + 2 * g], xb = xq[8 * h + 2 * g + 1];
            const int qsh = 2 * g, hsh = 4 * h + g;
            int v[8];
#pragma unroll
            for (int w = 0; w < 8; ++w)
                v[w] = (int)(((f[8 + 8 * h + w] >> qsh) & 0x03030303u) |
                             (((f[w] >> hsh) & 0x01010101u) << 2));
            int s0 = __dp4a(v[0], xa.x, 0);
            s0 = __dp4a(v[1], xa.y, s0);
            s0 = __dp4a(v[2], xa.z, s0);
            s0 = __dp4a(v[3], xa.w, s0);
            int s1 = __dp4a(v[4], xb.x, 0);
            s1 = __dp4a(v[5], xb.y, s1);
            s1 = __dp4a(v[6], xb.z, s1);
            s1 = __dp4a(v[7], xb.w, s1);
            const int sub = 8 * h + 2 * g;
            const int isum = scale[sub] * (s0 - 4 * sq[sub]) + scale[sub + 1] * (s1 - 4 * sq[sub + 1]);
            acc = fmaf(d8[4 * h + g], (float)isum, acc);
        }
    }
    return d * acc;
}

// ------------------------------------------------------------------ pipeline helpers

struct Ring {
    uint64_t *full, *empty;
    Task *desc;
    uint8_t *stage;
    uint32_t stage_bytes;
    int S;
    __device__ uint8_t *at(int slot) const { return stage + (size_t)slot * stage_bytes; }
};

// producer side: publishes task i into its slot once the slot is free
__device__ __forceinline__ bool ring_issue(const Ring &r, int i, const Task &t, const void *src,
                                           uint32_t bytes, uint64_t pol, uint32_t *status)
{
    const int slot = i % r.S;
    const uint32_t round = (uint32_t)(i / r.S);
    if (round > 0 && !mbar_wait(&r.empty[slot], (round - 1) & 1u, status))
        return false;
    r.desc[slot] = t;
    mbar_arrive_expect_tx(&r.full[slot], bytes);
    if (bytes)
        bulk_g2s(r.at(slot), src, bytes, &r.full[slot], pol);
    return true;
}

__device__ __forceinline__ void ring_init(const Ring &r)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < r.S; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], 1);
        }
        fence_barrier_init();
    }
}

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"r"(MOE_CONSUMER_WARPS * 32) : "memory");
}

__device__ __forceinline__ Ring ring_carve(uint8_t *smem, int S, uint32_t stage_bytes, size_t stage_off)
{
    Ring r;
    r.S = S;
    r.full = reinterpret_cast<uint64_t *>(smem);
    r.empty = r.full + S;
    r.desc = reinterpret_cast<Task *>(smem + align_up(16 * (size_t)S, 64));
    r.stage = smem + stage_off;
    r.stage_bytes = stage_bytes;
    return r;
}

// bytes before the stages: barriers, descriptors
__host__ __device__ inline size_t ring_head_bytes(int S)
{
    return align_up(align_up(16 * (size_t)S, 64) + sizeof(Task) * (size_t)S, 128);
}

// ------------------------------------------------------------------ gate / up kernel

struct GArgs {
    const uint16_t *x;                 // bf16 [m, dim]
    const uint16_t *w1, *w3;           // shared expert bf16 [inter, dim] (NULL: none)
    const int32_t *hdr;                // route header (plan tail at plan_off)
    const unsigned long long *ptrs;    // [3][cap]
    const int32_t *plan_rows;          // [cap]
    float *g, *u;                      // [cap, inter]
    float *gs, *us;                    // [m, inter]
    uint32_t *status;
    int dim, inter, m, k, cap, plan_off, S;
    uint32_t stage_bytes;
};

__host__ __device__ inline size_t g_act_off(int S) { return ring_head_bytes(S); }
__host__ __device__ inline size_t g_xs_off(int S, int m, int dim) { return g_act_off(S) + align_up((size_t)m * act_row_bytes(dim), 128); }
__host__ __device__ inline size_t g_stage_off(int S, int m, int dim, bool shared)
{
    return g_xs_off(S, m, dim) + (shared ? align_up((size_t)m * dim * 2, 128) : 0);
}
__host__ __device__ inline size_t g_smem_bytes(int S, int m, int dim, bool shared, uint32_t stage_bytes)
{
    return g_stage_off(S, m, dim, shared) + (size_t)S * stage_bytes + 16;
}

__global__ void __launch_bounds__(MOE_THREADS, 1) moe_gateup_kernel(GArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const bool shared = a.w1 != nullptr;
    const Ring ring = ring_carve(smem, a.S, a.stage_bytes, g_stage_off(a.S, a.m, a.dim, shared));
    uint8_t *act = smem + g_act_off(a.S);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + g_xs_off(a.S, a.m, a.dim));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dim = a.dim, inter = a.inter, nb = dim / MOE_QK;
    const size_t arow = act_row_bytes(dim);
    ring_init(ring);
    __syncthreads();

    if (warp == MOE_CONSUMER_WARPS) {
        // ---------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int i = 0;
            bool ok = true;
            if (shared) {
                const int nsh = 2 * inter;
                const int lo = (int)((long long)blockIdx.x * nsh / gridDim.x);
                const int hi = (int)((long long)(blockIdx.x + 1) * nsh / gridDim.x);
                for (int s = lo; s < hi && ok; ++s) {
                    Task t{};
                    t.kind = 2;
                    t.mat = s / inter;
                    t.row = s % inter;
                    const uint16_t *src = (t.mat ? a.w3 : a.w1) + (size_t)t.row * dim;
                    ok = ring_issue(ring, i++, t, src, (uint32_t)dim * 2u, pol, a.status);
                }
            }
            pdl_wait();  // the selection has written the plan and the pointer table
            pdl_launch_dependents();
            const int ne = min(max(__ldcg(a.hdr + a.plan_off), 0), a.cap);
            const int rt = gate_rows_per_task(dim);
            const int tpm = inter / rt;  // tasks per matrix
            const long long total = (long long)ne * 2 * tpm;
            const int lo = (int)(blockIdx.x * total / gridDim.x);
            const int hi = (int)((blockIdx.x + 1) * total / gridDim.x);
            const size_t rowb = (size_t)nb * MOE_Q2K_BYTES;
            for (int tix = lo; tix < hi && ok; ++tix) {
                Task t{};
                t.kind = 1;
                t.p = tix / (2 * tpm);
                const int rem = tix % (2 * tpm);
                t.mat = rem / tpm;
                t.row = (rem % tpm) * rt;
                t.pair0 = __ldcg(a.hdr + a.plan_off + 1 + t.p);
                t.npair = __ldcg(a.hdr + a.plan_off + 2 + t.p) - t.pair0;
                if (t.npair < 1 || t.npair > a.m || t.pair0 < 0 || t.pair0 + t.npair > a.cap) {
                    atomicOr(a.status, (uint32_t)MOE_WS_PLAN);
                    continue;
                }
                bool toks_ok = true;
                for (int j = 0; j < t.npair; ++j) {
                    t.tok[j] = __ldcg(a.plan_rows + t.pair0 + j);
                    toks_ok &= t.tok[j] >= 0 && t.tok[j] < a.m;
                }
                if (!toks_ok) {
                    atomicOr(a.status, (uint32_t)MOE_WS_PLAN);
                    continue;
                }
                const char *src = reinterpret_cast<const char *>(__ldcg(a.ptrs + (size_t)t.mat * a.cap + t.p)) +
                                  (size_t)t.row * rowb;
                ok = ring_issue(ring, i++, t, src, (uint32_t)(rt * rowb), pol, a.status);
            }
            for (int w = 0; w < MOE_CONSUMER_WARPS && ok; ++w) {
                Task t{};
                t.kind = 0;
                ok = ring_issue(ring, i++, t, nullptr, 0, pol, a.status);
            }
        }
        return;
    }

    // ---------------- consumers: the activation first (x is ready: the
    // previous kernel in the stream let this one start only after its own wait)
    const int nblk = a.m * dim / 32;
    for (int b = warp; b < nblk; b += MOE_CONSUMER_WARPS) {
        const int t = b / (dim / 32), bi = b % (dim / 32);
        const float v = bf16_to_f32(__ldcg(a.x + (size_t)t * dim + bi * 32 + lane));
        q8_store_smem(act + t * arow, nb, bi, q8_quant_warp(v), true);
    }
    if (shared) {
        const uint4 *gx = reinterpret_cast<const uint4 *>(a.x);
        uint4 *s4 = reinterpret_cast<uint4 *>(xs);
        for (int i = threadIdx.x; i < a.m * dim / 8; i += MOE_CONSUMER_WARPS * 32)
            s4[i] = __ldcg(gx + i);
    }
    consumers_sync();

    // every thread triggers the dependent launch only after the selection is
    // complete (the first routed task is issued after the producer's wait)
    bool triggered = false;
    for (int j = warp;; j += MOE_CONSUMER_WARPS) {
        const int slot = j % ring.S;
        if (!mbar_wait(&ring.full[slot], (uint32_t)(j / ring.S) & 1u, a.status))
            break;
        const Task t = ring.desc[slot];
        if (t.kind == 0)
            break;
        const uint8_t *st = ring.at(slot);
        if (t.kind == 1 && !triggered) {
            pdl_wait();
            pdl_launch_dependents();
            triggered = true;
        }
        if (t.kind == 1) {
            // 64 super-blocks: lane covers super-blocks lane and lane + 32;
            // one token at a time (tokens of this plan expert), rows reduced
            // over the nb lanes that share them
            const uint32_t *bp0 = reinterpret_cast<const uint32_t *>(st + (size_t)lane * MOE_Q2K_BYTES);
            const uint32_t *bp1 = reinterpret_cast<const uint32_t *>(st + (size_t)(lane + 32) * MOE_Q2K_BYTES);
            const int blk0 = lane % nb, blk1 = (lane + 32) % nb;
            float *out = t.mat ? a.u : a.g;
#pragma unroll 1
            for (int tt = 0; tt < t.npair; ++tt) {
                const uint8_t *xr = act + ring.desc[slot].tok[tt] * arow;
                const float4 *rec = reinterpret_cast<const float4 *>(xr + nb * MOE_SEG_Q_BYTES);
                float v0 = q2k_dot(bp0, reinterpret_cast<const int4 *>(xr + blk0 * MOE_SEG_Q_BYTES),
                                   rec + blk0 * (MOE_SEG_REC_FLOATS / 4));
                float v1 = q2k_dot(bp1, reinterpret_cast<const int4 *>(xr + blk1 * MOE_SEG_Q_BYTES),
                                   rec + blk1 * (MOE_SEG_REC_FLOATS / 4));
                for (int o = nb >> 1; o > 0; o >>= 1) {
                    v0 += __shfl_xor_sync(0xffffffffu, v0, o);
                    v1 += __shfl_xor_sync(0xffffffffu, v1, o);
                }
                if (blk0 == 0) {
                    float *orow = out + (size_t)(t.pair0 + tt) * inter + t.row;
                    orow[lane / nb] = v0;
                    orow[(lane + 32) / nb] = v1;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);
        } else {
            // one bf16 row of W1 or W3 against every token's bf16 x
            float acc[MOE_MAX_TOKENS];
#pragma unroll
            for (int tt = 0; tt < MOE_MAX_TOKENS; ++tt)
                acc[tt] = 0.0f;
            const uint4 *wr = reinterpret_cast<const uint4 *>(st);
            for (int c = lane; c < dim / 8; c += 32) {
                const uint4 wv = wr[c];
#pragma unroll
                for (int tt = 0; tt < MOE_MAX_TOKENS; ++tt) {
                    if (tt < a.m) {
                        const uint4 xv = reinterpret_cast<const uint4 *>(xs + (size_t)tt * dim)[c];
                        float s = acc[tt];
                        s = fmaf(bf16_lo(wv.x), bf16_lo(xv.x), s);
                        s = fmaf(bf16_hi(wv.x), bf16_hi(xv.x), s);
                        s = fmaf(bf16_lo(wv.y), bf16_lo(xv.y), s);
                        s = fmaf(bf16_hi(wv.y), bf16_hi(xv.y), s);
                        s = fmaf(bf16_lo(wv.z), bf16_lo(xv.z), s);
                        s = fmaf(bf16_hi(wv.z), bf16_hi(xv.z), s);
                        s = fmaf(bf16_lo(wv.w), bf16_lo(xv.w), s);
                        s = fmaf(bf16_hi(wv.w), bf16_hi(xv.w), s);
                        acc[tt] = s;
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);
            float *out = t.mat ? a.us : a.gs;
#pragma unroll
            for (int tt = 0; tt < MOE_MAX_TOKENS; ++tt) {
                if (tt < a.m) {
                    float v = acc[tt];
#pragma unroll
                    for (int o = 16; o; o >>= 1)
                        v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0)
                        out[(size_t)tt * inter + t.row] = v;
                }
            }
        }
    }
    if (!triggered) {
        pdl_wait();
        pdl_launch_dependents();
    }
}

// ------------------------------------------------------------------ down kernel

struct DArgs {
    const int32_t *hdr;
    const unsigned long long *ptrs;
    const int32_t *plan_rows;
    const float *plan_w;
    const float *g, *u;           // [cap, inter]
    const float *gs, *us;         // [m, inter]
    const uint16_t *w2;           // shared bf16 [dim, inter] (NULL: none)
    float *down;                  // [cap, dim]
    float *sd;                    // [m, dim]
    float *acc;                   // [m, dim]
    float *residual;              // [m, dim] or NULL
    uint16_t *x_next;             // [m, dim] or NULL
    uint32_t *rgcnt, *status;
    float limit;
    int dim, inter, m, k, cap, plan_off, S, pair_cap;
    uint32_t stage_bytes;
};

__host__ __device__ inline size_t d_small_off(int S) { return ring_head_bytes(S); }
__host__ __device__ inline size_t d_act_off(int S) { return d_small_off(S) + 512; }
__host__ __device__ inline size_t d_hs_off(int S, int pair_cap, int inter)
{
    return d_act_off(S) + align_up((size_t)pair_cap * act_row_bytes(inter), 128);
}
__host__ __device__ inline size_t d_stage_off(int S, int pair_cap, int m, int inter, bool shared)
{
    return d_hs_off(S, pair_cap, inter) + (shared ? align_up((size_t)m * inter * 2, 128) : 0);
}
__host__ __device__ inline size_t d_smem_bytes(int S, int pair_cap, int m, int inter, bool shared,
                                              uint32_t stage_bytes)
{
    return d_stage_off(S, pair_cap, m, inter, shared) + (size_t)S * stage_bytes + 16;
}

// the range of tasks of this CTA and the plan pairs its routed tasks touch
struct DRange {
    int ne, tpr, Tr, lo, hi, pair_lo, pair_hi;
};

__device__ __forceinline__ DRange d_range(const DArgs &a, bool shared)
{
    DRange r;
    r.ne = min(max(__ldcg(a.hdr + a.plan_off), 0), a.cap);
    r.tpr = a.dim / down_rows_per_task(a.inter);
    r.Tr = r.ne * r.tpr;
    const long long T = (long long)r.Tr + (shared ? a.dim : 0);
    r.lo = (int)(blockIdx.x * T / gridDim.x);
    r.hi = (int)((blockIdx.x + 1) * T / gridDim.x);
    r.pair_lo = r.pair_hi = 0;
    if (r.lo < r.Tr && r.lo < r.hi) {
        const int p_lo = r.lo / r.tpr, p_hi = (min(r.hi, r.Tr) - 1) / r.tpr;
        r.pair_lo = min(max(__ldcg(a.hdr + a.plan_off + 1 + p_lo), 0), a.cap);
        r.pair_hi = min(max(__ldcg(a.hdr + a.plan_off + 2 + p_hi), r.pair_lo), a.cap);
    }
    return r;
}

// acc, residual and x_next of row group rg, by one warp
__device__ void finish_row_group(const DArgs &a, int rg, int rd, bool shared, const int *s_rows,
                                 const float *s_w)
{
    const int lane = threadIdx.x & 31, npairs = a.m * a.k;
    for (int it = lane; it < a.m * rd; it += 32) {
        const int t = it / rd, r = rg * rd + it % rd;
        float acc = 0.0f;
        for (int q = 0; q < npairs; ++q)
            if (s_rows[q] == t)
                acc = __fadd_rn(acc, __fmul_rn(s_w[q], __ldcg(a.down + (size_t)q * a.dim + r)));
        if (shared)
            acc = __fadd_rn(acc, __ldcg(a.sd + (size_t)t * a.dim + r));
        a.acc[(size_t)t * a.dim + r] = acc;
        if (a.residual) {
            const float res = __fadd_rn(a.residual[(size_t)t * a.dim + r], acc);
            a.residual[(size_t)t * a.dim + r] = res;
            if (a.x_next)
                a.x_next[(size_t)t * a.dim + r] = f32_to_bf16(res);
        }
    }
}

__global__ void __launch_bounds__(MOE_THREADS, 1) moe_down_kernel(DArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const bool shared = a.w2 != nullptr;
    const Ring ring = ring_carve(smem, a.S, a.stage_bytes, d_stage_off(a.S, a.pair_cap, a.m, a.inter, shared));
    int *s_rows = reinterpret_cast<int *>(smem + d_small_off(a.S));
    float *s_w = reinterpret_cast<float *>(s_rows + 64);
    uint8_t *act = smem + d_act_off(a.S);
    uint16_t *hs = reinterpret_cast<uint16_t *>(smem + d_hs_off(a.S, a.pair_cap, a.inter));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dim = a.dim, inter = a.inter, nb = inter / MOE_QK;
    const int rd = down_rows_per_task(inter);
    const size_t arow = act_row_bytes(inter);
    ring_init(ring);
    __syncthreads();
    const DRange R = d_range(a, shared);

    if (warp == MOE_CONSUMER_WARPS) {
        // ---------------- producer: everything it loads depends only on the
        // pointer table, so the whole range is issued before the wait
        if (lane == 0) {
            pdl_launch_dependents();
            const uint64_t pol = policy_evict_first();
            int i = 0;
            bool ok = true;
            const bool fits = R.pair_hi - R.pair_lo <= a.pair_cap;
            if (!fits)
                atomicOr(a.status, (uint32_t)MOE_WS_PLAN);
            const size_t rowb = (size_t)nb * MOE_Q3K_BYTES;
            for (int tix = R.lo; tix < (fits ? R.hi : R.lo) && ok; ++tix) {
                Task t{};
                const void *src;
                uint32_t bytes;
                if (tix < R.Tr) {
                    t.kind = 1;
                    t.p = tix / R.tpr;
                    t.row = (tix % R.tpr) * rd;
                    t.pair0 = __ldcg(a.hdr + a.plan_off + 1 + t.p);
                    t.npair = __ldcg(a.hdr + a.plan_off + 2 + t.p) - t.pair0;
                    if (t.npair < 1 || t.npair > a.m || t.pair0 < R.pair_lo || t.pair0 + t.npair > R.pair_hi) {
                        atomicOr(a.status, (uint32_t)MOE_WS_PLAN);
                        t.npair = 0;  // issued (the row group's ticket still counts it), computes nothing
                    }
                    src = reinterpret_cast<const char *>(__ldcg(a.ptrs + 2 * (size_t)a.cap + t.p)) + (size_t)t.row * rowb;
                    bytes = (uint32_t)(rd * rowb);
                } else {
                    t.kind = 2;
                    t.row = tix - R.Tr;
                    src = a.w2 + (size_t)t.row * inter;
                    bytes = (uint32_t)inter * 2u;
                }
                ok = ring_issue(ring, i++, t, src, bytes, pol, a.status);
            }
            for (int w = 0; w < MOE_CONSUMER_WARPS && ok; ++w) {
                Task t{};
                t.kind = 0;
                ok = ring_issue(ring, i++, t, nullptr, 0, pol, a.status);
            }
        }
        return;
    }

    // ---------------- consumers: wait for g, u, gs, us; build the activations
    pdl_launch_dependents();
    pdl_wait();
    const int npairs = a.m * a.k;
    for (int q = threadIdx.x; q < npairs; q += MOE_CONSUMER_WARPS * 32) {
        s_rows[q] = __ldcg(a.plan_rows + q);
        s_w[q] = __ldcg(a.plan_w + q);
    }
    const int np = min(R.pair_hi - R.pair_lo, a.pair_cap);
    const int nblk = np * inter / 32;
    for (int b = warp; b < nblk; b += MOE_CONSUMER_WARPS) {
        const int pr = b / (inter / 32), bi = b % (inter / 32);
        const size_t o = (size_t)(R.pair_lo + pr) * inter + bi * 32 + lane;
        const float h = swiglu_f32(__ldcg(a.g + o), __ldcg(a.u + o), a.limit);
        q8_store_smem(act + pr * arow, nb, bi, q8_quant_warp(h), false);
    }
    const bool my_shared = shared && R.hi > R.Tr;
    if (my_shared) {
        for (int i = threadIdx.x; i < a.m * inter; i += MOE_CONSUMER_WARPS * 32)
            hs[i] = f32_to_bf16(swiglu_f32(__ldcg(a.gs + i), __ldcg(a.us + i), a.limit));
    }
    consumers_sync();

    const unsigned expected = (unsigned)R.ne + (shared ? (unsigned)rd : 0u);
    for (int j = warp;; j += MOE_CONSUMER_WARPS) {
        const int slot = j % ring.S;
        if (!mbar_wait(&ring.full[slot], (uint32_t)(j / ring.S) & 1u, a.status))
            break;
        const Task t = ring.desc[slot];
        if (t.kind == 0)
            break;
        const uint8_t *st = ring.at(slot);
        int rg;
        if (t.kind == 1) {
            // 32 super-blocks: lane = (row lane / nb, block lane % nb); one
            // token (plan pair) at a time
            const int blk = lane % nb;
            const uint8_t *bp = st + (size_t)lane * MOE_Q3K_BYTES;
#pragma unroll 1
            for (int tt = 0; tt < t.npair; ++tt) {
                const uint8_t *xr = act + (t.pair0 + tt - R.pair_lo) * arow;
                float v = q3k_dot(bp, reinterpret_cast<const int4 *>(xr + blk * MOE_SEG_Q_BYTES),
                                  reinterpret_cast<const float4 *>(xr + nb * MOE_SEG_Q_BYTES) +
                                      blk * (MOE_SEG_REC_FLOATS / 4));
                for (int o = nb >> 1; o > 0; o >>= 1)
                    v += __shfl_xor_sync(0xffffffffu, v, o);
                if (blk == 0)
                    a.down[(size_t)(t.pair0 + tt) * dim + t.row + lane / nb] = v;
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);
            rg = t.row / rd;
        } else {
            float acc[MOE_MAX_TOKENS];
#pragma unroll
            for (int tt = 0; tt < MOE_MAX_TOKENS; ++tt)
                acc[tt] = 0.0f;
            const uint4 *wr = reinterpret_cast<const uint4 *>(st);
            for (int c = lane; c < inter / 8; c += 32) {
                const uint4 wv = wr[c];
#pragma unroll
                for (int tt = 0; tt < MOE_MAX_TOKENS; ++tt) {
                    if (tt < a.m) {
                        const uint4 xv = reinterpret_cast<const uint4 *>(hs + (size_t)tt * inter)[c];
                        float s = acc[tt];
                        s = fmaf(bf16_lo(wv.x), bf16_lo(xv.x), s);
                        s = fmaf(bf16_hi(wv.x), bf16_hi(xv.x), s);
                        s = fmaf(bf16_lo(wv.y), bf16_lo(xv.y), s);
                        s = fmaf(bf16_hi(wv.y), bf16_hi(xv.y), s);
                        s = fmaf(bf16_lo(wv.z), bf16_lo(xv.z), s);
                        s = fmaf(bf16_hi(wv.z), bf16_hi(xv.z), s);
                        s = fmaf(bf16_lo(wv.w), bf16_lo(xv.w), s);
                        s = fmaf(bf16_hi(wv.w), bf16_hi(xv.w), s);
                        acc[tt] = s;
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);
#pragma unroll
            for (int tt = 0; tt < MOE_MAX_TOKENS; ++tt) {
                if (tt < a.m) {
                    float v = acc[tt];
#pragma unroll
                    for (int o = 16; o; o >>= 1)
                        v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == 0)
                        a.sd[(size_t)tt * dim + t.row] = v;
                }
            }
            rg = t.row / rd;
        }
        // row-group ticket: the warp that brings the count to `expected` finishes it
        __threadfence();
        __syncwarp();
        unsigned last = 0;
        if (lane == 0)
            last = atomicAdd(a.rgcnt + rg, 1u) == expected - 1u;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            finish_row_group(a, rg, rd, shared, s_rows, s_w);
            if (lane == 0)
                atomicExch(a.rgcnt + rg, 0u);
        }
    }
}

// ------------------------------------------------------------------ standalone q8_1 / swiglu

// bytes 0..3 of a q8_1 block: f16(d) | f16(d * sum q) << 16, assembled as one
// 32-bit word (the block is 4-byte aligned: 36-byte stride)
__device__ __forceinline__ uint32_t q8_header_word(float d, int sum)
{
    const uint32_t dh = (uint32_t)__half_as_ushort(__float2half_rn(d));
    const uint32_t sh = (uint32_t)__half_as_ushort(__float2half_rn(__fmul_rn(d, (float)sum)));
    return dh | (sh << 16);
}

// m rows of bf16 -> q8_1 blocks (36 bytes): one warp per block
__global__ void moe_quantize_q8_1_kernel(const uint16_t *x, int nblk, uint8_t *out)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    if (warp >= nblk)
        return;
    const float v = bf16_to_f32(x[(size_t)warp * 32 + lane]);
    const Q8Block b = q8_quant_warp(v);
    int sum = b.s16 + __shfl_xor_sync(0xffffffffu, b.s16, 16);
    uint8_t *o = out + (size_t)warp * MOE_Q8_BYTES;
    o[4 + lane] = (uint8_t)(int8_t)b.q;
    if (lane == 0)
        *reinterpret_cast<uint32_t *>(o) = q8_header_word(b.d, sum);
}

__global__ void moe_swiglu_q8_kernel(const float *g, const float *u, int nblk, float limit, float *h,
                                     uint8_t *out)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    if (warp >= nblk)
        return;
    const size_t i = (size_t)warp * 32 + lane;
    const float v = swiglu_f32(g[i], u[i], limit);
    if (h)
        h[i] = v;
    const Q8Block b = q8_quant_warp(v);
    int sum = b.s16 + __shfl_xor_sync(0xffffffffu, b.s16, 16);
    uint8_t *o = out + (size_t)warp * MOE_Q8_BYTES;
    o[4 + lane] = (uint8_t)(int8_t)b.q;
    if (lane == 0)
        *reinterpret_cast<uint32_t *>(o) = q8_header_word(b.d, sum);
}

}  // namespace moe

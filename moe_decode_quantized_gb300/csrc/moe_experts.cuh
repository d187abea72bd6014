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
// one producer warp (eight issuing lanes) streams whole tasks from HBM into a
// ring of shared-memory stages with 1-D bulk copies (TMA engine, L2
// evict-first), fifteen consumer warps take tasks as they land, decode the
// 2/3-bit quants from shared memory with dp4a integer dots and reduce rows
// with warp shuffles. Tasks are taken from grid-wide counters in chunks.
//
//   gate/up kernel: first the whole shared expert, which depends only on x
//     and so runs before the programmatic-launch wait, beside the router and
//     the selection: W1 row i and W3 row i as two tasks of one CTA (one row
//     a stage; the consumers write gs and us and meet in a shared-memory
//     cell, the second also writes hs = bf16(SwiGLU)), then W2 against hs
//     (once every row is done, grid-wide) into sd. Then, after the wait, the
//     plan experts' gate and up rows, rt rows of each in one task; the
//     consumer writes g, u and h = SwiGLU(g, u) per plan pair. Once the
//     selection has raised its plan-ready hint the routed rows go before the
//     rest of W2.
//   down kernel: tasks = 64-super-block row runs of plan experts' down
//     matrices, all prefetched before the wait (they need only the pointer
//     table); after the wait each CTA builds q8_1(h) for the pairs it needs.
//     With few plan pairs a CTA owns whole row groups of the output (every
//     plan expert's rows of them) and finishes them itself; otherwise its
//     tasks are an expert-major range and a row group is finished by the
//     CTA whose ticket completes it. Finishing: acc = plan-order sum of
//     w * down, then sd, residual += acc, x_next = bf16(residual).
#pragma once
#include "moe_common.cuh"

namespace moe {

struct __align__(16) Task {
    int kind;   // 0 end, 1 routed; gate/up kernel, shared expert: bf16 2 W1 or W3 row, 3 W2 rows;
                // K-quant 4 W1 and W3 rows, 5 W2 rows
    int p;      // plan expert (routed); 0 W1, 1 W3 (shared row)
    int row;    // first row (routed) or the row (shared)
    int pair0, npair;
    int seq;    // the task's index in this CTA's stream (written last by the producer)
    int pad[2];
};

// ------------------------------------------------------------------ q8_1 (one 32-block per warp)

struct Q8Block {
    int q;      // this lane's quant
    float d;    // f32 scale (the decision scale)
    float d8;   // the f16-rounded scale the dots use
    int s16;    // sum of the quants of this lane's 16-value half
};

// round-half-away(fl(v / d)), the q8_1 quant of v, for |v| <= amax and
// d = fl(amax / 127) > 0, given r = fl(1 / d). z = fl(v r) is within
// |v / d| (3 2^-24 + 2^-48) < 381 2^-24 < 2^-15 of fl(v / d) (three relative
// roundings of at most 2^-24 each; |v / d| < 127.0001), so when z is at least
// 2^-15 from every half-integer the two round to the same integer. Nearer
// one (and when r or z is not finite), the quotient itself decides.
__device__ __forceinline__ int q8_code(float v, float d, float r)
{
    const float z = __fmul_rn(v, r);
    const float a = fabsf(z);
    const float f = __fsub_rn(a, floorf(a));  // exact for a < 2^23
    if (!(fabsf(__fsub_rn(f, 0.5f)) >= 0x1.0p-15f))
        return (int)roundf(__fdiv_rn(v, d));
    return (int)roundf(z);
}

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
    b.q = amax == 0.0f ? 0 : q8_code(v, b.d, __frcp_rn(b.d));
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

// One q8_1 block by a group of 4 lanes, 8 values each (the same arithmetic
// as q8_quant_warp: the maximum is exact, each quant the rounding of one IEEE
// quotient (q8_code), the sums integers), so that a warp quantises 8 blocks
// at once. sub: the
// lane's place in its group (lanes 4g .. 4g + 3); v: its values
// 8 sub .. 8 sub + 7 of the block. Stored like q8_store_smem. All 32 lanes
// of the warp call it together (callers loop over 4 x blocks lanes, a
// multiple of 32 since dim and inter are multiples of 256).
__device__ __forceinline__ void q8_block_quad(const float (&v)[8], int sub, uint8_t *row, int nseg, int blk,
                                              bool min_term)
{
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        amax = fmaxf(amax, fabsf(v[j]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    const float r = __frcp_rn(d);
    uint32_t w[2];
    int sum = 0;
#pragma unroll
    for (int j4 = 0; j4 < 2; ++j4) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int q = amax == 0.0f ? 0 : q8_code(v[4 * j4 + b], d, r);
            sum += q;
            word |= (uint32_t)(q & 0xFF) << (8 * b);
        }
        w[j4] = word;
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);  // the half: lanes 0-1 or 2-3 of the group
    const int sg = blk >> 3, bi = blk & 7;
    *reinterpret_cast<uint2 *>(row + sg * MOE_SEG_Q_BYTES + bi * 32 + 8 * sub) = make_uint2(w[0], w[1]);
    const float d8 = __half2float(__float2half_rn(d));
    float *rec = reinterpret_cast<float *>(row + nseg * MOE_SEG_Q_BYTES) + sg * MOE_SEG_REC_FLOATS;
    if (sub == 0)
        rec[bi] = d8;
    if ((sub & 1) == 0)
        rec[8 + 2 * bi + (sub >> 1)] = min_term ? __fmul_rn(d8, (float)sum) : __int_as_float(sum);
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
// The 2-bit fields of a byte are masked in place (value 4^g q) and the 4^g
// is shifted out of the integer sum afterwards (exact: the sum is a multiple
// of 4^g), which saves a shift per weight word; fields 0-2 stay below 128
// (signed bytes), field 3 reaches 0xC0 and its products take the bytes as
// unsigned.
// sum of the four products of unsigned bytes of a and signed bytes of b, plus c
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

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
            // field g masked in place (4^g times the quant); the top field's
            // bytes reach 0xC0, so its products take the bytes as unsigned
            const uint32_t msk = 0x03030303u << (2 * g);
            auto dot = [&](uint32_t a, int b, int c) {
                return g == 3 ? dp4a_us(a, b, c) : __dp4a((int)a, b, c);
            };
            int s0 = dot(q[0] & msk, xa.x, 0);
            s0 = dot(q[1] & msk, xa.y, s0);
            s0 = dot(q[2] & msk, xa.z, s0);
            s0 = dot(q[3] & msk, xa.w, s0);
            int s1 = dot(q[4] & msk, xb.x, 0);
            s1 = dot(q[5] & msk, xb.y, s1);
            s1 = dot(q[6] & msk, xb.z, s1);
            s1 = dot(q[7] & msk, xb.w, s1);
            const int sub = 8 * h + 2 * g;
            const int isum = ((int)(byte_of(sc, sub) & 15u) * s0 + (int)(byte_of(sc, sub + 1) & 15u) * s1) >> (2 * g);
            main = fmaf(d8[4 * h + g], (float)isum, main);
        }
    }
    return f16_bits_to_f32(dd) * main - f16_bits_to_f32(dd >> 16) * mn;
}

// PER Q3_K super-blocks of one lane sharing the same activation columns
// (the activation's quants and scale records loaded once). Q3_K: 32 bytes
// of high bits (bit 4h + g of byte b: value 128h + 32g + b), 64 bytes of
// 2-bit lows (field g of byte 32h + b), 12 bytes of 6-bit scales, f16 d;
// the value is low + 4 high - 4. Per 16-value sub-block the integer sum
//   t = sum low x + 4 sum high x - 4 sum x
// takes two dp4a a weight word: the low field masked in place (4^g low) and
// the high bit masked in place (2^(4h + g) high), both shifted out of the
// sums afterwards (exact: each sum is a multiple of its power of two); the
// top field and the top high bit give unsigned bytes.
template <int PER>
__device__ __forceinline__ void q3k_dot_multi(const uint8_t *st, int lane, const int4 *xq, const float4 *rec,
                                              float (&out)[PER])
{
    const uint32_t *W[PER];
    uint32_t sh[PER], hm[PER][8], S[PER][4];
    float d[PER], acc[PER];
#pragma unroll
    for (int q = 0; q < PER; ++q) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(st + (size_t)(lane + 32 * q) * MOE_Q3K_BYTES);
        W[q] = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
        sh[q] = (uint32_t)(a & 3) * 8u;
        uint32_t w[9];
#pragma unroll
        for (int i = 0; i < 9; ++i)
            w[i] = W[q][i];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            hm[q][i] = __funnelshift_r(w[i], w[i + 1], sh[q]);
        const uint32_t w24 = W[q][24], w25 = W[q][25], w26 = W[q][26], w27 = W[q][27];
        const uint32_t s0 = __funnelshift_r(w24, w25, sh[q]), s1 = __funnelshift_r(w25, w26, sh[q]),
                       s2 = __funnelshift_r(w26, w27, sh[q]);
        // the 16 scales as bytes (0 .. 63): the low nibbles of bytes 0-7 are
        // scales 0-7, their high nibbles scales 8-15; byte 8 + j holds the
        // top two bits of scales j, j + 4, j + 8, j + 12
        S[q][0] = (s0 & 0x0F0F0F0Fu) | ((s2 << 4) & 0x30303030u);
        S[q][1] = (s1 & 0x0F0F0F0Fu) | ((s2 << 2) & 0x30303030u);
        S[q][2] = ((s0 >> 4) & 0x0F0F0F0Fu) | (s2 & 0x30303030u);
        S[q][3] = ((s1 >> 4) & 0x0F0F0F0Fu) | ((s2 >> 2) & 0x30303030u);
        d[q] = f16_bits_to_f32(w27 >> sh[q]);
        acc[q] = 0.0f;
    }
    const float4 da = rec[0], db = rec[1];
    const float d8[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float4 sqa = rec[2 + 2 * h], sqb = rec[3 + 2 * h];  // sums of sub-blocks 8h .. 8h+7
        const int sq[8] = {__float_as_int(sqa.x), __float_as_int(sqa.y), __float_as_int(sqa.z),
                           __float_as_int(sqa.w), __float_as_int(sqb.x), __float_as_int(sqb.y),
                           __float_as_int(sqb.z), __float_as_int(sqb.w)};
        uint32_t qv[PER][8];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            uint32_t w[9];
#pragma unroll
            for (int i = 0; i < 9; ++i)
                w[i] = W[q][8 + 8 * h + i];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                qv[q][i] = __funnelshift_r(w[i], w[i + 1], sh[q]);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int4 xa = xq[8 * h + 2 * g], xb = xq[8 * h + 2 * g + 1];
            const int hsh = 4 * h + g;
            const uint32_t lm = 0x03030303u << (2 * g), hmk = 0x01010101u << hsh;
            const int i0 = 8 * h + 2 * g, i1 = i0 + 1;
            const int xv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
            for (int q = 0; q < PER; ++q) {
                int sl[2], shh[2];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    int a0 = 0, a1 = 0;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint32_t lo = qv[q][4 * b + w] & lm, hi = hm[q][4 * b + w] & hmk;
                        a0 = g == 3 ? dp4a_us(lo, xv[4 * b + w], a0) : __dp4a((int)lo, xv[4 * b + w], a0);
                        a1 = hsh == 7 ? dp4a_us(hi, xv[4 * b + w], a1) : __dp4a((int)hi, xv[4 * b + w], a1);
                    }
                    sl[b] = a0 >> (2 * g);
                    shh[b] = a1 >> hsh;
                }
                const int t0 = sl[0] + 4 * shh[0] - 4 * sq[2 * g], t1 = sl[1] + 4 * shh[1] - 4 * sq[2 * g + 1];
                const int sc0 = (int)__byte_perm(S[q][i0 >> 2], 0u, 0x4440u + (unsigned)(i0 & 3)) - 32;
                const int sc1 = (int)__byte_perm(S[q][i1 >> 2], 0u, 0x4440u + (unsigned)(i1 & 3)) - 32;
                const int isum = sc0 * t0 + sc1 * t1;
                acc[q] = fmaf(d8[4 * h + g], (float)isum, acc[q]);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < PER; ++q)
        out[q] = d[q] * acc[q];
}

// ------------------------------------------------------------------ pipeline helpers

// The plan of the call, cached in shared memory by the producer warp (one
// round of parallel global loads instead of dependent loads per task).
struct PlanCache {
    int ne;
    int next;      // consumers' dynamic task counter
    int hs_ready;  // gate/up: the shared expert's SwiGLU output is in shared memory
    int pad;
    int pair_start[MOE_MAX_TOKENS * MOE_MAX_TOPK + 1];
    int rows[MOE_MAX_TOKENS * MOE_MAX_TOPK];
    unsigned long long ptr[2][MOE_MAX_TOKENS * MOE_MAX_TOPK];
};

struct Ring {
    uint64_t *full, *empty;
    Task *desc;
    PlanCache *pc;
    uint8_t *stage;
    uint32_t stage_bytes;
    int S;                       // at least 2
    uint32_t Sm;                 // ceil(2^32 / S): task i's round i / S = umulhi(i, Sm) (FastDiv)
    unsigned long long wait_ns;  // bound on each wait
    __device__ uint8_t *at(int slot) const { return stage + (size_t)slot * stage_bytes; }
};

// producer side: publishes task i into its slot once the slot is free; the
// stage receives src (bytes) and, after it, src2 (bytes2)
__device__ __forceinline__ bool ring_issue(const Ring &r, int i, const Task &t, const void *src,
                                           uint32_t bytes, uint64_t pol, uint32_t *status,
                                           const void *src2 = nullptr, uint32_t bytes2 = 0)
{
    const uint32_t round = __umulhi((uint32_t)i, r.Sm);
    const int slot = i - (int)round * r.S;
    if (round > 0 && !mbar_wait(&r.empty[slot], (round - 1) & 1u, status, r.wait_ns))
        return false;
    Task tt = t;
    tt.seq = i;
    r.desc[slot] = tt;
    mbar_arrive_expect_tx(&r.full[slot], bytes + bytes2);
    if (bytes)
        bulk_g2s(r.at(slot), src, bytes, &r.full[slot], pol);
    if (bytes2)
        bulk_g2s(r.at(slot) + bytes, src2, bytes2, &r.full[slot], pol);
    return true;
}

__device__ __forceinline__ void ring_init(const Ring &r)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < r.S; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], 1);
            r.desc[s].seq = -1;
        }
        r.pc->next = 0;
        r.pc->hs_ready = 0;
        fence_barrier_init();
    }
}

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"r"(MOE_CONSUMER_WARPS * 32) : "memory");
}

__host__ __device__ inline size_t ring_desc_off(int S) { return align_up(16 * (size_t)S, 64); }
__host__ __device__ inline size_t ring_pc_off(int S) { return align_up(ring_desc_off(S) + sizeof(Task) * (size_t)S, 16); }

// bytes before the stages: barriers, descriptors, plan cache
__host__ __device__ inline size_t ring_head_bytes(int S)
{
    return align_up(ring_pc_off(S) + sizeof(PlanCache), 128);
}

__device__ __forceinline__ Ring ring_carve(uint8_t *smem, int S, uint32_t stage_bytes, size_t stage_off,
                                           unsigned long long wait_ns)
{
    Ring r;
    r.S = S;
    r.Sm = FastDiv((uint32_t)S).m;
    r.wait_ns = wait_ns;
    r.full = reinterpret_cast<uint64_t *>(smem);
    r.empty = r.full + S;
    r.desc = reinterpret_cast<Task *>(smem + ring_desc_off(S));
    r.pc = reinterpret_cast<PlanCache *>(smem + ring_pc_off(S));
    r.stage = smem + stage_off;
    r.stage_bytes = stage_bytes;
    return r;
}

// consumer side: the next task index (dynamic, any warp takes the next task)
__device__ __forceinline__ int ring_grab(const Ring &r)
{
    int j = 0;
    if ((threadIdx.x & 31) == 0)
        j = atomicAdd(&r.pc->next, 1);
    return __shfl_sync(0xffffffffu, j, 0);
}

// Consumer side: waits until slot j % S holds task j. The producer stamps a
// descriptor only after the slot's previous task was consumed, so once the
// stamp reads j the barrier's current phase is task j's and the parity wait
// is unambiguous (a parity wait cannot tell a phase two ahead from the one
// just completed). Bounded like every wait; false after r.wait_ns.
__device__ __forceinline__ bool ring_acquire(const Ring &r, int j, uint32_t *status)
{
    const uint32_t round = __umulhi((uint32_t)j, r.Sm);
    const int slot = j - (int)round * r.S;
    volatile const int *seq = &r.desc[slot].seq;
    if (*seq != j) {
        const uint64_t t0 = globaltimer();
        while (*seq != j) {
            __nanosleep(16);
            if (globaltimer() - t0 > r.wait_ns) {
                atomicOr(status, (uint32_t)MOE_WS_TIMEOUT);
                return false;
            }
        }
    }
    return mbar_wait(&r.full[slot], round & 1u, status, r.wait_ns);
}

// the producer warp caches the plan (all 32 lanes load in parallel, one
// round of independent loads); `which` selects the pointer rows to keep
// (gate/up: 0 and 1, down: 2)
__device__ __forceinline__ void cache_plan(const Ring &r, const int32_t *hdr, int plan_off, const int32_t *plan_rows,
                                           const unsigned long long *ptrs, int cap, int which0, int nwhich)
{
    const int lane = threadIdx.x & 31;
    PlanCache &pc = *r.pc;
    int ps[3], rw[2];
    unsigned long long pt[2][2];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int i = lane + 32 * j;
        ps[j] = i <= cap ? __ldcg(hdr + plan_off + 1 + i) : 0;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        rw[j] = i < cap ? __ldcg(plan_rows + i) : 0;
#pragma unroll
        for (int w = 0; w < 2; ++w)
            pt[j][w] = (i < cap && w < nwhich) ? __ldcg(ptrs + (size_t)(which0 + w) * cap + i) : 0ull;
    }
    const int ne = min(max(__ldcg(hdr + plan_off), 0), cap);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int i = lane + 32 * j;
        if (i <= cap)
            pc.pair_start[i] = min(max(ps[j], 0), cap);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = lane + 32 * j;
        if (i < cap) {
            pc.rows[i] = min(max(rw[j], 0), MOE_MAX_TOKENS - 1);
#pragma unroll
            for (int w = 0; w < 2; ++w)
                if (w < nwhich)
                    pc.ptr[w][i] = pt[j][w];
        }
    }
    if (lane == 0)
        pc.ne = ne;
    __syncwarp();
}

// ------------------------------------------------------------------ gate / up kernel

struct GArgs {
    const uint16_t *x;                 // bf16 [m, dim]
    const void *w1, *w3;               // shared expert [inter, dim], bf16 or Q2_K (NULL: none)
    const void *w2;                    // shared expert [dim, inter], bf16 or Q3_K
    int sk;                            // shared expert: 0 none, 1 bf16, 2 Q2_K / Q3_K
    const int32_t *hdr;                // route header (plan tail at plan_off)
    const unsigned long long *ptrs;    // [3][cap]
    const int32_t *plan_rows;          // [cap]
    float *g, *u, *h;                  // [cap, inter]: h = SwiGLU(g, u)
    float *gs, *us;                    // [m, inter]
    uint16_t *hs;                      // [m, inter] bf16(SwiGLU(gs, us)) (bf16 shared expert)
    float *hsf;                        // [m, inter] SwiGLU(gs, us) (K-quant shared expert)
    float *sd;                         // [m, dim] W2 hs
    uint32_t *status;
    // [0] shared row-task counter, [1] routed-task counter, [2] unused,
    // [3] W2 task counter, [4] shared rows done (hs[i] written), [5] the
    // selection's plan-ready hint; all 0 at the start (the down kernel after
    // this one resets them)
    uint32_t *gctr;
    float limit;
    unsigned long long wait_ns;  // bound on each wait
    int plan_hint;  // the plan comes from the selection in this stream (its hint at gctr[5])
    int stage_x;    // bf16 x and hs staged in shared memory (few tokens); else read from L2
    int dim, inter, m, k, cap, plan_off, S, w2r;
    uint32_t stage_bytes;
};

__host__ __device__ inline size_t g_act_off(int S) { return ring_head_bytes(S); }
__host__ __device__ inline size_t g_xs_off(int S, int m, int dim) { return g_act_off(S) + align_up((size_t)m * act_row_bytes(dim), 128); }
// stage: bf16 x and hs are staged in shared memory (few tokens); else the
// consumers read them from L2 and the ring keeps the room
__host__ __device__ constexpr bool g_stage_x(int m) { return m <= 2; }
__host__ __device__ inline size_t g_hs_off(int S, int m, int dim, bool stage)
{
    return g_xs_off(S, m, dim) + (stage ? align_up((size_t)m * dim * 2, 128) : 0);
}
// Shared rows: the W1 and W3 tasks of a row go to one CTA (chunks of
// MOE_G_CHUNK tasks start at multiples of it) and meet in one of these cells,
// picked by the CTA's pair sequence number: an arrival count (odd after the
// first) and both halves' values
struct PairCell {
    int cnt;
    float v[2][MOE_MAX_TOKENS];
};
#define MOE_PAIR_CELLS 32  // more than the pairs one ring holds
static_assert(MOE_G_CHUNK % 2 == 0, "a chunk holds whole shared-row pairs");
// sk: the shared expert's kind (0 none, 1 bf16, 2 K-quant). The hs area holds
// bf16 hs (staged, bf16) or q8_1(hs) in the activation layout (K-quant).
__host__ __device__ inline size_t g_pair_bytes(int sk)
{
    return sk == 1 ? align_up(sizeof(PairCell) * MOE_PAIR_CELLS, 128) : 0;
}
__host__ __device__ inline size_t g_hs_bytes(int m, int inter, int sk, bool stage)
{
    if (sk == 2)
        return align_up((size_t)m * act_row_bytes(inter), 128);
    return sk == 1 && stage ? align_up((size_t)m * inter * 2, 128) : 0;
}
__host__ __device__ inline size_t g_pair_off(int S, int m, int dim, int inter, int sk, bool stage)
{
    return g_hs_off(S, m, dim, stage) + g_hs_bytes(m, inter, sk, stage);
}
__host__ __device__ inline size_t g_stage_off(int S, int m, int dim, int inter, int sk, bool stage)
{
    return g_pair_off(S, m, dim, inter, sk, stage) + g_pair_bytes(sk);
}
__host__ __device__ inline size_t g_smem_bytes(int S, int m, int dim, int inter, int sk, bool stage,
                                               uint32_t stage_bytes)
{
    return g_stage_off(S, m, dim, inter, sk, stage) + (size_t)S * stage_bytes + 16;
}

// q8_1(hs) of a K-quant shared expert into shared memory (the producer warp,
// once hs is complete grid-wide): m * inter / 8 lane items, a multiple of 32,
// so the whole warp calls q8_block_quad together. Out of line: inlined into
// the producer, this loop made the bf16 layer step 0.3 us slower, although
// that step never runs it.
__device__ __noinline__ void q8_hs_build(const float *hsf, uint8_t *hact, int m, int inter, int lane)
{
    const int nbi = inter / MOE_QK, bpr = inter / 32;
    const size_t arow = act_row_bytes(inter);
    for (int i = lane; i < m * inter / 8; i += 32) {
        const int b = i >> 2, sub = i & 3, t = b / bpr, bi = b - t * bpr;
        const float4 *h4 = reinterpret_cast<const float4 *>(hsf + (size_t)t * inter + bi * 32 + 8 * sub);
        const float4 p = __ldcg(h4), q = __ldcg(h4 + 1);
        const float v[8] = {p.x, p.y, p.z, p.w, q.x, q.y, q.z, q.w};
        q8_block_quad(v, sub, hact + t * arow, nbi, bi, false);
    }
}

// The producer warp: waits (bounded) until every hs row of the shared
// expert is done grid-wide, copies hs into shared memory (bf16) or builds
// q8_1(hs) there (K-quant: four lanes a block, as the activation of the
// Q3_K W2 rows), and raises the CTA's flag (2 instead of 1 after a timeout,
// so that no consumer waits forever).
__device__ bool g_load_hs(const GArgs &a, const Ring &ring, uint16_t *hs_s, int lane)
{
    const uint32_t target = (uint32_t)a.inter;
    bool ok = true;
    if (ld_acquire_gpu(a.gctr + 4) < target) {
        const uint64_t t0 = globaltimer();
        while (ld_acquire_gpu(a.gctr + 4) < target) {
            __nanosleep(16);
            if (globaltimer() - t0 > a.wait_ns) {
                atomicOr(a.status, (uint32_t)MOE_WS_TIMEOUT);
                ok = false;
                break;
            }
        }
    }
    // every lane polled itself: its loads below come after its own acquire
    // (unstaged, the consumers read hs from L2 once the flag is up)
    if (a.sk == 2)
        q8_hs_build(a.hsf, reinterpret_cast<uint8_t *>(hs_s), a.m, a.inter, lane);
    const int n16 = a.stage_x && a.sk == 1 ? a.m * a.inter / 8 : 0;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.hs);
    uint4 *dst = reinterpret_cast<uint4 *>(hs_s);
    for (int i0 = lane; i0 < n16; i0 += 32 * 8) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = i0 + 32 * j < n16 ? __ldcg(src + i0 + 32 * j) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (i0 + 32 * j < n16)
                dst[i0 + 32 * j] = v[j];
    }
    ok = __all_sync(0xffffffffu, ok);
    __syncwarp();
    if (lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile int *>(&ring.pc->hs_ready) = ok ? 1 : 2;
    }
    return ok;
}

// KM: the token count the kernel is built for (it holds that case's code
// alone: 1 or 8), or 0 for any m
template <int KM>
__global__ void __launch_bounds__(MOE_THREADS, 1) moe_gateup_kernel(GArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const bool shared = a.sk != 0, kq = a.sk == 2;
    const bool stage = a.stage_x != 0;
    const Ring ring = ring_carve(smem, a.S, a.stage_bytes, g_stage_off(a.S, a.m, a.dim, a.inter, a.sk, stage), a.wait_ns);
    uint8_t *act = smem + g_act_off(a.S);
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + g_xs_off(a.S, a.m, a.dim));  // staged only
    uint16_t *hs_s = reinterpret_cast<uint16_t *>(smem + g_hs_off(a.S, a.m, a.dim, stage));  // staged (bf16) or q8_1 (K-quant)
    PairCell *cells = reinterpret_cast<PairCell *>(smem + g_pair_off(a.S, a.m, a.dim, a.inter, a.sk, stage));
    // 16-byte chunk i of bf16 x / of hs: shared memory when staged, else L2
    // (kStage: the staging of the token count g_stage_x, known where M is)
    const uint4 *x4s = reinterpret_cast<const uint4 *>(xs), *x4g = reinterpret_cast<const uint4 *>(a.x);
    const uint4 *h4s = reinterpret_cast<const uint4 *>(hs_s), *h4g = reinterpret_cast<const uint4 *>(a.hs);
    const uint8_t *hact = reinterpret_cast<const uint8_t *>(hs_s);  // K-quant: q8_1(hs) rows
    const int nbi = a.inter / MOE_QK;  // super-blocks of a W2 (K-quant) row
    auto ldx = [&](size_t i) { return stage ? x4s[i] : __ldcg(x4g + i); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dim = a.dim, inter = a.inter, nb = dim / MOE_QK;
    const size_t arow = act_row_bytes(dim);
    if (a.sk == 1 && threadIdx.x < MOE_PAIR_CELLS)
        cells[threadIdx.x].cnt = 0;
    ring_init(ring);
    __syncthreads();

    if (warp == MOE_CONSUMER_WARPS) {
        // ---------------- producer warp. Tasks are taken in chunks of
        // MOE_G_CHUNK from grid-wide counters (a CTA that starts late -- its
        // SM still busy with the previous kernel -- simply takes fewer);
        // MOE_PRODUCER_LANES lanes issue a chunk's tasks in parallel.
        const uint64_t pol = policy_evict_first();
        const int P = min(MOE_PRODUCER_LANES, ring.S);
        const bool issuer = lane < P;
        int base = 0;  // index of the next task in this CTA's ring
        bool ok = true;
        int w2_pending = -1;  // W2 left for after the routed work: a chunk taken, or -2 (none taken)
        bool have_hs = false;
        // W2 tasks: w2r bf16 rows, or (K-quant) the Q3_K rows of 64 super-blocks
        const int w2rows = kq ? down_rows_per_task(inter) : a.w2r;
        const uint32_t w2bytes = kq ? (uint32_t)(w2rows * nbi * MOE_Q3K_BYTES) : (uint32_t)a.w2r * inter * 2u;
        auto issue_w2 = [&](int c0, int c1) {
            for (int b = c0; b < c1 && ok; b += P) {
                const int j = b + lane;
                bool mine = true;
                if (issuer && j < c1) {
                    Task t{};
                    t.kind = kq ? 5 : 3;
                    t.row = j * w2rows;
                    mine = ring_issue(ring, base + (j - c0), t, static_cast<const char *>(a.w2) + (size_t)j * w2bytes,
                                      w2bytes, pol, a.status);
                }
                ok = __all_sync(0xffffffffu, mine);
            }
            base += c1 - c0;
        };
        if (shared) {
            // The shared expert depends only on x: all of it runs before the
            // wait. (1) Rows. bf16: task 2i is W1 row i, task 2i + 1 is W3 row
            // i (one row a stage, so the stages fit the routed tasks); of the
            // two consumers of row i the one that finishes second writes
            // hs[i] = bf16(SwiGLU). pair0 carries the CTA's pair sequence
            // number (its meeting cell). K-quant: task i is rows rt i .. of
            // W1 and the same rows of W3 (Q2_K, as a routed task), whose
            // consumer writes gs, us and hs = SwiGLU for every token.
            const int rt = gate_rows_per_task(dim);
            const uint32_t kbytes = (uint32_t)(rt * nb * MOE_Q2K_BYTES);
            const int nsh = kq ? inter / rt : 2 * inter;
            int pseq = 0;
            unsigned nxt = 0;
            if (lane == 0)
                nxt = atomicAdd(a.gctr + 0, (unsigned)MOE_G_CHUNK);
            for (;;) {
                const int c0 = (int)__shfl_sync(0xffffffffu, nxt, 0);
                if (c0 >= nsh || !ok)
                    break;
                if (lane == 0)
                    nxt = atomicAdd(a.gctr + 0, (unsigned)MOE_G_CHUNK);  // the next chunk, in flight meanwhile
                const int c1 = min(c0 + MOE_G_CHUNK, nsh);
                for (int b = c0; b < c1 && ok; b += P) {
                    const int j = b + lane;
                    bool mine = true;
                    if (issuer && j < c1 && kq) {
                        Task t{};
                        t.kind = 4;
                        t.row = j * rt;
                        mine = ring_issue(ring, base + (j - c0), t, static_cast<const char *>(a.w1) + (size_t)j * kbytes,
                                          kbytes, pol, a.status,
                                          static_cast<const char *>(a.w3) + (size_t)j * kbytes, kbytes);
                    } else if (issuer && j < c1) {
                        Task t{};
                        t.kind = 2;
                        t.row = j >> 1;
                        t.p = j & 1;  // 0: W1 (gate), 1: W3 (up)
                        t.pair0 = pseq + ((j - c0) >> 1);
                        mine = ring_issue(ring, base + (j - c0), t,
                                          static_cast<const uint16_t *>(t.p ? a.w3 : a.w1) + (size_t)t.row * dim,
                                          (uint32_t)dim * 2u, pol, a.status);
                    }
                    ok = __all_sync(0xffffffffu, mine);
                }
                base += c1 - c0;
                pseq += (c1 - c0) >> 1;
            }
            // (2) W2 against hs. This warp polls (bounded) two words: every
            // hs row done grid-wide -> it loads hs into shared memory (bf16)
            // or builds q8_1(hs) there (K-quant) and issues W2; the
            // selection's plan-ready hint ->
            // the routed work goes first and W2 (or its rest) after it. No W2
            // task is issued before hs is in shared memory, so nothing queued
            // ahead of a routed task ever waits.
            const int nw2 = dim / w2rows;
            {
                const uint64_t t0 = globaltimer();
                for (;;) {
                    uint32_t done = 0, hint = 0;
                    if (lane == 0) {
                        done = *reinterpret_cast<volatile uint32_t *>(a.gctr + 4);
                        hint = *reinterpret_cast<volatile uint32_t *>(a.gctr + 5);
                    }
                    done = __shfl_sync(0xffffffffu, done, 0);
                    hint = __shfl_sync(0xffffffffu, hint, 0);
                    if (hint != 0u)
                        break;  // W2 entirely after the routed work
                    if (done >= (uint32_t)inter || globaltimer() - t0 > a.wait_ns) {
                        g_load_hs(a, ring, hs_s, lane);  // acquires; times out itself
                        have_hs = true;
                        break;
                    }
                    __nanosleep(16);
                }
            }
            if (have_hs) {
                uint32_t hint = lane == 0 ? *reinterpret_cast<volatile uint32_t *>(a.gctr + 5) : 0u;
                if (lane == 0)
                    nxt = atomicAdd(a.gctr + 3, (unsigned)MOE_G_CHUNK);
                while (ok) {
                    const int c0 = (int)__shfl_sync(0xffffffffu, nxt, 0);
                    if (c0 >= nw2)
                        break;
                    if (__shfl_sync(0xffffffffu, hint, 0) != 0u) {
                        w2_pending = c0;  // taken: issued after the routed work
                        break;
                    }
                    if (lane == 0) {
                        nxt = atomicAdd(a.gctr + 3, (unsigned)MOE_G_CHUNK);
                        hint = *reinterpret_cast<volatile uint32_t *>(a.gctr + 5);  // read one chunk ahead
                    }
                    issue_w2(c0, min(c0 + MOE_G_CHUNK, nw2));
                }
            } else {
                w2_pending = -2;  // nothing taken yet
            }
        }
        // the first routed chunk's ticket does not depend on the plan: taken
        // before the wait, its round trip overlaps the selection
        unsigned nxt = 0;
        if (lane == 0)
            nxt = atomicAdd(a.gctr + 1, (unsigned)MOE_G_CHUNK);
        if (a.plan_hint) {
            // the selecting CTA publishes the plan with a release store of the
            // hint: acquiring it, the plan can be read before the router grid
            // has finished (bounded poll; the wait below still comes before
            // this CTA lets the next kernel start)
            if (ld_acquire_gpu(a.gctr + 5) == 0u) {
                const uint64_t t0 = globaltimer();
                while (ld_acquire_gpu(a.gctr + 5) == 0u) {
                    __nanosleep(16);
                    if (globaltimer() - t0 > a.wait_ns) {
                        if (lane == 0)
                            atomicOr(a.status, (uint32_t)MOE_WS_TIMEOUT);
                        break;
                    }
                }
            }
            __syncwarp();
        } else {
            pdl_wait();  // the plan and the pointer table come from the caller
        }
        cache_plan(ring, a.hdr, a.plan_off, a.plan_rows, a.ptrs, a.cap, 0, 2);
        const PlanCache &pc = *ring.pc;
        const int rt = gate_rows_per_task(dim);
        const int tpe = inter / rt;  // tasks per expert: rt gate rows and the same up rows each
        const FastDiv tpe_d((uint32_t)tpe);
        const int total = pc.ne * tpe;
        const uint32_t bytes = (uint32_t)(rt * nb * MOE_Q2K_BYTES);  // one matrix's rows
        for (;;) {
            const int c0 = (int)__shfl_sync(0xffffffffu, nxt, 0);
            if (c0 >= total || !ok)
                break;
            if (lane == 0)
                nxt = atomicAdd(a.gctr + 1, (unsigned)MOE_G_CHUNK);
            const int c1 = min(c0 + MOE_G_CHUNK, total);
            for (int b = c0; b < c1 && ok; b += P) {
                const int tix = b + lane;
                bool mine = true;
                if (issuer && tix < c1) {
                    Task t{};
                    t.kind = 1;
                    t.p = (int)tpe_d.div((uint32_t)tix);
                    const int r = tix - t.p * tpe;
                    t.row = r * rt;
                    t.pair0 = pc.pair_start[t.p];
                    t.npair = pc.pair_start[t.p + 1] - t.pair0;
                    uint32_t nbytes = bytes;
                    if (t.npair < 1 || t.npair > a.m) {
                        atomicOr(a.status, (uint32_t)MOE_WS_PLAN);
                        t.npair = 0;  // a no-op task keeps the indices contiguous
                        nbytes = 0;
                    }
                    const size_t off = (size_t)r * bytes;
                    mine = ring_issue(ring, base + (tix - c0), t, reinterpret_cast<const char *>(pc.ptr[0][t.p]) + off,
                                      nbytes, pol, a.status, reinterpret_cast<const char *>(pc.ptr[1][t.p]) + off,
                                      nbytes);
                }
                ok = __all_sync(0xffffffffu, mine);
            }
            base += c1 - c0;
        }
        // the next kernel may start once the router grid has completed (it
        // reads the plan before its own wait)
        pdl_wait();
        pdl_launch_dependents();
        if (w2_pending != -1) {
            // the rest of W2, hs first if it is not in shared memory yet (the
            // routed tasks ahead of it never wait)
            const int nw2 = dim / w2rows;
            if (!have_hs)
                g_load_hs(a, ring, hs_s, lane);
            int c0 = w2_pending;
            if (c0 < 0) {
                unsigned nx = 0;
                if (lane == 0)
                    nx = atomicAdd(a.gctr + 3, (unsigned)MOE_G_CHUNK);
                c0 = (int)__shfl_sync(0xffffffffu, nx, 0);
            }
            while (ok && c0 < nw2) {
                unsigned nx = 0;
                if (lane == 0)
                    nx = atomicAdd(a.gctr + 3, (unsigned)MOE_G_CHUNK);
                issue_w2(c0, min(c0 + MOE_G_CHUNK, nw2));
                c0 = (int)__shfl_sync(0xffffffffu, nx, 0);
            }
        }
        for (int b = 0; b < MOE_CONSUMER_WARPS && ok; b += P) {
            bool mine = true;
            if (issuer && b + lane < MOE_CONSUMER_WARPS) {
                Task t{};
                t.kind = 0;
                mine = ring_issue(ring, base + b + lane, t, nullptr, 0, pol, a.status);
            }
            ok = __all_sync(0xffffffffu, mine);
        }
        return;
    }

    // ---------------- consumers: the activation first (x is ready: the
    // previous kernel in the stream let this one start only after its own
    // wait). x is staged with all loads in flight, then quantised from smem.
    if (stage) {
        const uint4 *gx = reinterpret_cast<const uint4 *>(a.x);
        uint4 *s4 = reinterpret_cast<uint4 *>(xs);
        for (int i = threadIdx.x; i < a.m * dim / 8; i += MOE_CONSUMER_WARPS * 32)
            s4[i] = __ldcg(gx + i);
    }
    consumers_sync();
    const int nblk = a.m * dim / 32;
    const FastDiv bpx((uint32_t)(dim / 32));  // 32-value blocks a token row
    for (int i = threadIdx.x; i < nblk * 4; i += MOE_CONSUMER_WARPS * 32) {  // four lanes a block
        const int b = i >> 2, sub = i & 3;
        const int t = (int)bpx.div((uint32_t)b), bi = b - t * (dim / 32);
        const uint4 w = ldx(((size_t)t * dim + bi * 32 + 8 * sub) / 8);
        const float v[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                            bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
        q8_block_quad(v, sub, act + t * arow, nb, bi, true);
    }
    consumers_sync();

    // (the producer triggers the dependent launch, after its wait on the
    // router grid; consumers read the plan from shared memory only)
    bool hs_seen = false;
    for (;;) {
        const int j = ring_grab(ring);
        const int slot = j - (int)__umulhi((uint32_t)j, ring.Sm) * ring.S;
        if (!ring_acquire(ring, j, a.status))
            break;
        const Task t = ring.desc[slot];
        if (t.kind == 0) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);  // END slots are reused when S < warps
            break;
        }
        const uint8_t *st = ring.at(slot);
        if (t.kind == 1) {
            // rt gate rows then the same rt up rows, MOE_G_TASK_SB super-blocks:
            // lane covers super-blocks lane + 32 q, so q and q + 2 are the gate
            // and up parts of the same row (row (lane + 32 q) / nb, block
            // lane % nb); one token at a time, rows reduced over the nb lanes
            // that share them, then h = SwiGLU(g, u) of the row
            constexpr int PER = MOE_G_TASK_SB / 32;
            const int blk = lane % nb;  // the same for all PER super-blocks of the lane
#pragma unroll 1
            for (int tt = 0; tt < t.npair; ++tt) {
                const uint8_t *xr = act + min(ring.pc->rows[t.pair0 + tt], a.m - 1) * arow;
                const int4 *xq = reinterpret_cast<const int4 *>(xr + blk * MOE_SEG_Q_BYTES);
                const float4 *rec = reinterpret_cast<const float4 *>(xr + nb * MOE_SEG_Q_BYTES) +
                                    blk * (MOE_SEG_REC_FLOATS / 4);
                float v[PER];
#pragma unroll
                for (int q = 0; q < PER; ++q)
                    v[q] = q2k_dot(reinterpret_cast<const uint32_t *>(st + (size_t)(lane + 32 * q) * MOE_Q2K_BYTES),
                                   xq, rec);
                for (int o = nb >> 1; o > 0; o >>= 1) {
#pragma unroll
                    for (int q = 0; q < PER; ++q)
                        v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
                }
                if (blk == 0) {
                    const size_t o = (size_t)(t.pair0 + tt) * inter + t.row;
#pragma unroll
                    for (int q = 0; q < PER / 2; ++q) {
                        const int r = (lane + 32 * q) / nb;
                        a.g[o + r] = v[q];
                        a.u[o + r] = v[q + PER / 2];
                        a.h[o + r] = swiglu_f32(v[q], v[q + PER / 2], a.limit);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);
        } else if (t.kind == 2) {
            // W1 row i (t.p = 0) or W3 row i (t.p = 1) against every token's
            // bf16 x into gs or us; the second of the two finishes hs[i]
            const int i = t.row;
            const bool up = t.p != 0;
            const uint4 *wr = reinterpret_cast<const uint4 *>(st);
            with_m_k<KM>(a.m, [&](auto MC) {
                constexpr int M = decltype(MC)::value;
                float ac[M];
#pragma unroll
                for (int tt = 0; tt < M; ++tt)
                    ac[tt] = 0.0f;
                for (int c = lane; c < dim / 8; c += 32) {
                    const uint4 v = wr[c];
#pragma unroll
                    for (int tt = 0; tt < M; ++tt)
                        ac[tt] = fma_bf16x8(
                            v, g_stage_x(M) ? x4s[(size_t)tt * (dim / 8) + c] : __ldcg(x4g + (size_t)tt * (dim / 8) + c),
                            ac[tt]);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ring.empty[slot]);
#pragma unroll
                for (int tt = 0; tt < M; ++tt) {
#pragma unroll
                    for (int o = 16; o; o >>= 1)
                        ac[tt] += __shfl_xor_sync(0xffffffffu, ac[tt], o);
                }
                if (lane == 0) {
                    float *mine = up ? a.us : a.gs;
                    PairCell &pc2 = cells[t.pair0 % MOE_PAIR_CELLS];
#pragma unroll
                    for (int tt = 0; tt < M; ++tt) {
                        mine[(size_t)tt * inter + i] = ac[tt];
                        pc2.v[up][tt] = ac[tt];
                    }
                    __threadfence_block();  // this half's value before the count
                    if (atomicAdd(&pc2.cnt, 1) & 1) {
                        __threadfence_block();  // the other half's value after the count
                        const volatile float *ov = pc2.v[!up];
#pragma unroll
                        for (int tt = 0; tt < M; ++tt) {
                            const float o = ov[tt];
                            const float gv = up ? o : ac[tt], uv = up ? ac[tt] : o;
                            a.hs[(size_t)tt * inter + i] = f32_to_bf16(swiglu_f32(gv, uv, a.limit));
                        }
                        red_add_release_gpu(a.gctr + 4, 1u);  // after this lane's hs stores
                    }
                }
            });
        } else if (t.kind == 4) {
            // K-quant shared rows t.row .. t.row + rt of W1, then the same rows
            // of W3 (Q2_K, lanes laid out as in a routed task), for every
            // token: gs, us and hs = SwiGLU(gs, us) in f32; then the task's
            // rows are counted done grid-wide (release, after every lane's
            // stores)
            constexpr int PER = MOE_G_TASK_SB / 32;
            const int blk = lane % nb;
#pragma unroll 1
            for (int tt = 0; tt < a.m; ++tt) {
                const uint8_t *xr = act + tt * arow;
                const int4 *xq = reinterpret_cast<const int4 *>(xr + blk * MOE_SEG_Q_BYTES);
                const float4 *rec = reinterpret_cast<const float4 *>(xr + nb * MOE_SEG_Q_BYTES) +
                                    blk * (MOE_SEG_REC_FLOATS / 4);
                float v[PER];
#pragma unroll
                for (int q = 0; q < PER; ++q)
                    v[q] = q2k_dot(reinterpret_cast<const uint32_t *>(st + (size_t)(lane + 32 * q) * MOE_Q2K_BYTES),
                                   xq, rec);
                for (int o = nb >> 1; o > 0; o >>= 1) {
#pragma unroll
                    for (int q = 0; q < PER; ++q)
                        v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
                }
                if (blk == 0) {
                    const size_t o = (size_t)tt * inter + t.row;
#pragma unroll
                    for (int q = 0; q < PER / 2; ++q) {
                        const int r = (lane + 32 * q) / nb;
                        a.gs[o + r] = v[q];
                        a.us[o + r] = v[q + PER / 2];
                        a.hsf[o + r] = swiglu_f32(v[q], v[q + PER / 2], a.limit);
                    }
                }
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ring.empty[slot]);
                red_add_release_gpu(a.gctr + 4, (unsigned)gate_rows_per_task(dim));
            }
        } else {
            // W2 rows against every token's hs: bf16 (staged or from L2), or
            // (K-quant) Q3_K against q8_1(hs), both in shared memory once the
            // producer has them there
            if (!hs_seen) {
                if (lane == 0) {
                    volatile int *f = &ring.pc->hs_ready;
                    if (*f == 0) {
                        const uint64_t t0 = globaltimer();
                        while (*f == 0) {
                            __nanosleep(16);
                            if (globaltimer() - t0 > a.wait_ns) {
                                atomicOr(a.status, (uint32_t)MOE_WS_TIMEOUT);
                                break;
                            }
                        }
                    }
                    __threadfence_block();
                }
                __syncwarp();
                hs_seen = true;
            }
            if (t.kind == 5) {
                // 64 Q3_K super-blocks: rows t.row .. of W2, lanes laid out as
                // in a down task, one token at a time
                constexpr int PER = MOE_D_TASK_SB / 32;
                const int blk = lane % nbi;
                const size_t arow_i = act_row_bytes(inter);
#pragma unroll 1
                for (int tt = 0; tt < a.m; ++tt) {
                    const uint8_t *xr = hact + tt * arow_i;
                    const int4 *xq = reinterpret_cast<const int4 *>(xr + blk * MOE_SEG_Q_BYTES);
                    const float4 *rec = reinterpret_cast<const float4 *>(xr + nbi * MOE_SEG_Q_BYTES) +
                                        blk * (MOE_SEG_REC_FLOATS / 4);
                    float v[PER];
                    q3k_dot_multi<PER>(st, lane, xq, rec, v);
                    for (int o = nbi >> 1; o > 0; o >>= 1) {
#pragma unroll
                        for (int q = 0; q < PER; ++q)
                            v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
                    }
                    if (blk == 0) {
#pragma unroll
                        for (int q = 0; q < PER; ++q)
                            a.sd[(size_t)tt * dim + t.row + (lane + 32 * q) / nbi] = v[q];
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ring.empty[slot]);
                continue;
            }
            with_m_k<KM>(a.m, [&](auto MC) {
                constexpr int M = decltype(MC)::value;
                for (int rr = 0; rr < a.w2r; ++rr) {
                    const uint4 *wr = reinterpret_cast<const uint4 *>(st) + (size_t)rr * (inter / 8);
                    float acc[M];
#pragma unroll
                    for (int tt = 0; tt < M; ++tt)
                        acc[tt] = 0.0f;
                    for (int c = lane; c < inter / 8; c += 32) {
                        const uint4 wv = wr[c];
#pragma unroll
                        for (int tt = 0; tt < M; ++tt)
                            acc[tt] = fma_bf16x8(wv,
                                                 g_stage_x(M) ? h4s[(size_t)tt * (inter / 8) + c]
                                                              : __ldcg(h4g + (size_t)tt * (inter / 8) + c),
                                                 acc[tt]);
                    }
#pragma unroll
                    for (int tt = 0; tt < M; ++tt) {
                        float v = acc[tt];
#pragma unroll
                        for (int o = 16; o; o >>= 1)
                            v += __shfl_xor_sync(0xffffffffu, v, o);
                        if (lane == 0)
                            a.sd[(size_t)tt * dim + t.row + rr] = v;
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ring.empty[slot]);
            });
        }
    }
    // the grid-wide counters are reset by the down kernel launched next, once
    // this grid has completed: no CTA waits on an exit ticket here
}

// ------------------------------------------------------------------ down kernel

struct DArgs {
    const int32_t *hdr;
    const unsigned long long *ptrs;
    const int32_t *plan_rows;
    const float *plan_w;
    const float *h;               // [cap, inter] SwiGLU(g, u) per plan pair
    float *down;                  // [cap, dim]
    const float *sd;              // [m, dim] the shared expert's output (the gate/up kernel's)
    float *acc;                   // [m, dim]
    float *residual;              // [m, dim] or NULL
    uint16_t *x_next;             // [m, dim] or NULL
    uint32_t *rgcnt, *status;
    uint32_t *gctr;  // the gate/up kernel's six counters: reset here once that grid has completed
    float limit;
    unsigned long long wait_ns;  // bound on each wait
    int has_shared;  // add sd to the routed sum
    // own_rows > 0: each CTA owns a range of row groups of the output (at
    // most own_rows rows), takes every plan expert's down rows of them,
    // quantises h of every plan pair (pair_cap = m * k) and finishes its own
    // rows from shared memory, with no row-group tickets. 0: expert-major task
    // ranges, tickets, and the CTA that completes a group finishes it.
    int own_rows;
    int dim, inter, m, k, cap, plan_off, S, pair_cap;
    uint32_t stage_bytes;
};

// small area of the down kernel (ints): plan rows [64], plan weights [64],
// each token's pairs in plan order [8][8], the finished-group count, and the
// list of row groups this CTA finishes [dim / rows-per-group]
#define D_SW 64
#define D_TP 128
#define D_NFIN 192
#define D_FIN 196
__host__ __device__ inline size_t d_small_bytes(int dim, int inter)
{
    return align_up(4 * ((size_t)D_FIN + dim / down_rows_per_task(inter)), 128);
}
__host__ __device__ inline size_t d_small_off(int S) { return ring_head_bytes(S); }
__host__ __device__ inline size_t d_act_off(int S, int dim, int inter) { return d_small_off(S) + d_small_bytes(dim, inter); }
// row ownership: the CTA's down rows of every plan pair, f32 [pair_cap][own_rows]
__host__ __device__ inline size_t d_own_off(int S, int pair_cap, int dim, int inter)
{
    return d_act_off(S, dim, inter) + align_up((size_t)pair_cap * act_row_bytes(inter), 128);
}
__host__ __device__ inline size_t d_stage_off(int S, int pair_cap, int dim, int inter, int own_rows)
{
    return d_own_off(S, pair_cap, dim, inter) + align_up(4 * (size_t)pair_cap * own_rows, 128);
}
__host__ __device__ inline size_t d_smem_bytes(int S, int pair_cap, int dim, int inter, int own_rows,
                                               uint32_t stage_bytes)
{
    return d_stage_off(S, pair_cap, dim, inter, own_rows) + (size_t)S * stage_bytes + 16;
}

// the range of tasks of this CTA and the plan pairs its routed tasks touch;
// with row ownership the tasks are (plan expert, owned row group) expert by
// expert, local indices [0, ne * ng)
struct DRange {
    int ne, tpr, Tr, lo, hi, pair_lo, pair_hi;
    bool own;
    int g_lo, ng;
};

// plan expert and row group of the CTA's task tix
__device__ __forceinline__ void d_task(const DRange &R, int tix, int &p, int &grp)
{
    if (R.own) {
        p = tix / R.ng;
        grp = R.g_lo + tix % R.ng;
    } else {
        p = tix / R.tpr;
        grp = tix % R.tpr;
    }
}

// ps: the plan's pair starts as cached by cache_plan (clamped, ne at
// ps_ne), or NULL to read them from the header. OWN: the kernel's path, 1 row
// ownership, 0 tickets (the host launches the instance that matches own_rows)
template <int OWN>
__device__ __forceinline__ DRange d_range(const DArgs &a, const int *ps = nullptr, int ps_ne = 0)
{
    auto start = [&](int i) {  // pair start of plan expert i (i <= ne)
        return ps ? ps[i] : min(max(__ldcg(a.hdr + a.plan_off + 1 + i), 0), a.cap);
    };
    DRange r;
    r.ne = ps ? ps_ne : min(max(__ldcg(a.hdr + a.plan_off), 0), a.cap);
    r.tpr = a.dim / down_rows_per_task(a.inter);
    r.Tr = r.ne * r.tpr;
    r.own = OWN == 1;
    r.g_lo = r.ng = 0;
    if (r.own) {
        r.g_lo = (int)((long long)blockIdx.x * r.tpr / gridDim.x);
        r.ng = (int)((long long)(blockIdx.x + 1) * r.tpr / gridDim.x) - r.g_lo;
        r.lo = 0;
        r.hi = r.ne * r.ng;
        r.pair_lo = 0;
        r.pair_hi = r.hi > 0 ? start(r.ne) : 0;
        return r;
    }
    r.lo = (int)((long long)blockIdx.x * r.Tr / gridDim.x);
    r.hi = (int)((long long)(blockIdx.x + 1) * r.Tr / gridDim.x);
    r.pair_lo = r.pair_hi = 0;
    if (r.lo < r.hi) {
        const int p_lo = r.lo / r.tpr, p_hi = (r.hi - 1) / r.tpr;
        r.pair_lo = start(p_lo);
        r.pair_hi = min(max(start(p_hi + 1), r.pair_lo), a.cap);
    }
    return r;
}

// acc, residual and x_next of row r for token t: the token's pairs in plan
// order (ascending expert id), then the shared row. The down values of pair
// q are dsrc[q * dstride + dcol]: the global down rows (kGlobal, written by
// other CTAs) or the CTA's own rows in shared memory.
template <bool kGlobal>
__device__ __forceinline__ void finish_row(const DArgs &a, int t, int r, bool shared, const int *s_tp,
                                           const float *s_w, const float *dsrc, size_t dstride, int dcol,
                                           bool pre = false, float sd_pre = 0.0f, float res_pre = 0.0f)
{
    const int k = a.k;
    float d[MOE_MAX_TOPK];
#pragma unroll
    for (int i = 0; i < MOE_MAX_TOPK; ++i) {
        const float *src = dsrc + (size_t)s_tp[t * MOE_MAX_TOPK + i] * dstride + dcol;
        d[i] = i < k ? (kGlobal ? __ldcg(src) : *src) : 0.0f;
    }
    // sd and residual: loaded here, or earlier by the caller (pre)
    const float sdv = pre ? sd_pre : shared ? __ldcg(a.sd + (size_t)t * a.dim + r) : 0.0f;
    const float res0 = pre ? res_pre : a.residual ? a.residual[(size_t)t * a.dim + r] : 0.0f;
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < MOE_MAX_TOPK; ++i)
        if (i < k)
            acc = __fadd_rn(acc, __fmul_rn(s_w[s_tp[t * MOE_MAX_TOPK + i]], d[i]));
    if (shared)
        acc = __fadd_rn(acc, sdv);
    a.acc[(size_t)t * a.dim + r] = acc;
    if (a.residual) {
        const float res = __fadd_rn(res0, acc);
        a.residual[(size_t)t * a.dim + r] = res;
        if (a.x_next)
            a.x_next[(size_t)t * a.dim + r] = f32_to_bf16(res);
    }
}

// OWN: 1 for row ownership (own_rows > 0), 0 for row-group tickets; each
// instance holds its own path's code alone
template <int OWN>
__global__ void __launch_bounds__(MOE_THREADS, 1) moe_down_kernel(DArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const bool shared = a.has_shared != 0;
    const Ring ring = ring_carve(smem, a.S, a.stage_bytes, d_stage_off(a.S, a.pair_cap, a.dim, a.inter, a.own_rows), a.wait_ns);
    float *s_own = reinterpret_cast<float *>(smem + d_own_off(a.S, a.pair_cap, a.dim, a.inter));
    int *s_rows = reinterpret_cast<int *>(smem + d_small_off(a.S));
    float *s_w = reinterpret_cast<float *>(s_rows + D_SW);
    int *s_tp = s_rows + D_TP;
    uint8_t *act = smem + d_act_off(a.S, a.dim, a.inter);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dim = a.dim, inter = a.inter, nb = inter / MOE_QK;
    const int rd = down_rows_per_task(inter);
    const size_t arow = act_row_bytes(inter);
    ring_init(ring);
    __syncthreads();

    if (warp == MOE_CONSUMER_WARPS) {
        // ---------------- producer warp: everything it loads depends only on
        // the pointer table, so the whole range is issued before the wait,
        // after one round of loads (the plan, its range from the cached
        // copy); MOE_PRODUCER_LANES lanes issue consecutive tasks in parallel
        pdl_launch_dependents();
        cache_plan(ring, a.hdr, a.plan_off, a.plan_rows, a.ptrs, a.cap, 2, 1);
        const PlanCache &pc = *ring.pc;
        const DRange R = d_range<OWN>(a, pc.pair_start, pc.ne);
        const uint64_t pol = policy_evict_first();
        const int P = min(MOE_PRODUCER_LANES, ring.S);
        const bool issuer = lane < P;
        bool ok = true;
        const bool fits = R.pair_hi - R.pair_lo <= a.pair_cap;
        if (!fits && lane == 0)
            atomicOr(a.status, (uint32_t)MOE_WS_PLAN);
        const uint32_t rbytes = (uint32_t)(rd * nb * MOE_Q3K_BYTES);
        for (int b = R.lo; b < R.hi && ok; b += P) {
            const int tix = b + lane;
            bool mine = true;
            if (issuer && tix < R.hi) {
                Task t{};
                t.kind = 1;
                int r;
                d_task(R, tix, t.p, r);
                t.row = r * rd;
                t.pair0 = pc.pair_start[t.p];
                t.npair = pc.pair_start[t.p + 1] - t.pair0;
                uint32_t bytes = rbytes;
                const void *src = reinterpret_cast<const char *>(pc.ptr[0][t.p]) + (size_t)r * rbytes;
                if (!fits || t.npair < 1 || t.npair > a.m || t.pair0 < R.pair_lo || t.pair0 + t.npair > R.pair_hi) {
                    if (fits)
                        atomicOr(a.status, (uint32_t)MOE_WS_PLAN);
                    t.npair = 0;  // a no-op task: still counted by its row group
                    bytes = 0;
                }
                mine = ring_issue(ring, tix - R.lo, t, src, bytes, pol, a.status);
            }
            ok = __all_sync(0xffffffffu, mine);
        }
        const int base = R.hi - R.lo;
        for (int b = 0; b < MOE_CONSUMER_WARPS && ok; b += P) {
            bool mine = true;
            if (issuer && b + lane < MOE_CONSUMER_WARPS) {
                Task t{};
                t.kind = 0;
                mine = ring_issue(ring, base + b + lane, t, nullptr, 0, pol, a.status);
            }
            ok = __all_sync(0xffffffffu, mine);
        }
        return;
    }
    const DRange R = d_range<OWN>(a);

    // ---------------- consumers: wait for h; build the activations
    pdl_launch_dependents();
    pdl_wait();
    // the gate/up grid has completed (this wait, or the stream's order): its
    // six counters are free for the next launch, which the kernel boundaries
    // order after these stores (one a thread, in the last CTA)
    if (blockIdx.x == gridDim.x - 1 && threadIdx.x < 6)
        st_relaxed_gpu(a.gctr + threadIdx.x, 0u);
    const int npairs = a.m * a.k;
    for (int q = threadIdx.x; q < npairs; q += MOE_CONSUMER_WARPS * 32) {
        s_rows[q] = __ldcg(a.plan_rows + q);
        s_w[q] = __ldcg(a.plan_w + q);
    }
    // q8_1(h) of the plan pairs this CTA's tasks touch, four lanes a block:
    // nq lane items, a multiple of 32, so each warp is wholly in or out of a
    // round; up to DQ rounds a thread with all their loads in flight
    constexpr int DQ = 4, CTH = MOE_CONSUMER_WARPS * 32;
    const int np = min(R.pair_hi - R.pair_lo, a.pair_cap);
    const int nq = np * inter / 32 * 4;
    const FastDiv bpr((uint32_t)(inter / 32));  // 32-value blocks a pair row
    for (int i0 = 0; i0 < nq; i0 += CTH * DQ) {
        float4 hv[DQ][2];
#pragma unroll
        for (int u = 0; u < DQ; ++u) {
            const int i = i0 + (int)threadIdx.x + CTH * u, b = i >> 2, sub = i & 3;
            const int pr = (int)bpr.div((uint32_t)b), bi = b - pr * (inter / 32);
            const float4 *h4 =
                reinterpret_cast<const float4 *>(a.h + (size_t)(R.pair_lo + pr) * inter + bi * 32 + 8 * sub);
            const bool in = i < nq;
            hv[u][0] = in ? __ldcg(h4) : make_float4(0.f, 0.f, 0.f, 0.f);
            hv[u][1] = in ? __ldcg(h4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < DQ; ++u) {
            const int i = i0 + (int)threadIdx.x + CTH * u, b = i >> 2, sub = i & 3;
            const int pr = (int)bpr.div((uint32_t)b), bi = b - pr * (inter / 32);
            if (i >= nq)
                continue;
            const float v[8] = {hv[u][0].x, hv[u][0].y, hv[u][0].z, hv[u][0].w,
                                hv[u][1].x, hv[u][1].y, hv[u][1].z, hv[u][1].w};
            q8_block_quad(v, sub, act + pr * arow, nb, bi, false);
        }
    }
    consumers_sync();
    // each token's pairs in plan order (pairs are grouped by ascending expert)
    if (threadIdx.x < a.m) {
        int c = 0;
        for (int q = 0; q < npairs && c < MOE_MAX_TOPK; ++q)
            if (s_rows[q] == (int)threadIdx.x)
                s_tp[threadIdx.x * MOE_MAX_TOPK + c++] = q;
        for (; c < MOE_MAX_TOPK; ++c)
            s_tp[threadIdx.x * MOE_MAX_TOPK + c] = 0;
    }
    consumers_sync();

    // row ownership: the first round of finished rows (row it = thread) has
    // its sd and residual loaded now, in flight while the tasks compute
    float sd_pre = 0.0f, res_pre = 0.0f;
    const int own_nr = R.ng * rd;
    if (R.own && (int)threadIdx.x < a.m * own_nr) {
        const int tk = (int)threadIdx.x / own_nr, r = R.g_lo * rd + (int)threadIdx.x % own_nr;
        sd_pre = shared ? __ldcg(a.sd + (size_t)tk * dim + r) : 0.0f;
        res_pre = a.residual ? a.residual[(size_t)tk * dim + r] : 0.0f;
    }
    const unsigned expected = (unsigned)R.ne;
    for (;;) {
        const int j = ring_grab(ring);
        const int slot = j - (int)__umulhi((uint32_t)j, ring.Sm) * ring.S;
        if (!ring_acquire(ring, j, a.status))
            break;
        const Task t = ring.desc[slot];
        if (t.kind == 0) {
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);  // END slots are reused when S < warps
            break;
        }
        const uint8_t *st = ring.at(slot);
        if (t.kind == 1) {
            // MOE_D_TASK_SB super-blocks: lane covers super-blocks lane + 32 q
            // (row (lane + 32 q) / nb, block lane % nb); one token (plan pair)
            // at a time
            constexpr int PER = MOE_D_TASK_SB / 32;
            const int blk = lane % nb;
#pragma unroll 1
            for (int tt = 0; tt < t.npair; ++tt) {
                const uint8_t *xr = act + (t.pair0 + tt - R.pair_lo) * arow;
                const int4 *xq = reinterpret_cast<const int4 *>(xr + blk * MOE_SEG_Q_BYTES);
                const float4 *rec = reinterpret_cast<const float4 *>(xr + nb * MOE_SEG_Q_BYTES) +
                                    blk * (MOE_SEG_REC_FLOATS / 4);
                float v[PER];
                q3k_dot_multi<PER>(st, lane, xq, rec, v);
                for (int o = nb >> 1; o > 0; o >>= 1) {
#pragma unroll
                    for (int q = 0; q < PER; ++q)
                        v[q] += __shfl_xor_sync(0xffffffffu, v[q], o);
                }
                if (blk == 0) {
                    float *orow = a.down + (size_t)(t.pair0 + tt) * dim + t.row;
#pragma unroll
                    for (int q = 0; q < PER; ++q)
                        orow[(lane + 32 * q) / nb] = v[q];
                    if (R.own) {
                        float *srow = s_own + (size_t)(t.pair0 + tt) * a.own_rows + (t.row - R.g_lo * rd);
#pragma unroll
                        for (int q = 0; q < PER; ++q)
                            srow[(lane + 32 * q) / nb] = v[q];
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ring.empty[slot]);
        }
    }

    if (R.own) {
        // the CTA's own rows of every token, from its down rows in shared memory
        consumers_sync();
        const int nr = own_nr, r0 = R.g_lo * rd;
        for (int it = threadIdx.x; it < a.m * nr; it += CTH) {
            const int tk = it / nr, rl = it - tk * nr;
            finish_row<false>(a, tk, r0 + rl, shared, s_tp, s_w, s_own, (size_t)a.own_rows, rl,
                              it == (int)threadIdx.x, sd_pre, res_pre);
        }
        return;
    }

    // Row-group tickets, once per CTA: after all of this CTA's tasks, for
    // every row group it touched one acq_rel atomic adding its count of tasks
    // there (release: the CTA's down rows, ordered before it by the barrier;
    // acquire: the other CTAs' rows of a group it completes). The CTA whose
    // addition completes a group finishes it.
    int *s_fin = s_rows + D_FIN;
    int *s_nfin = s_rows + D_NFIN;
    if (threadIdx.x == 0)
        *s_nfin = 0;
    consumers_sync();
    const int ngroups = dim / rd;
    const FastDiv tprd((uint32_t)R.tpr);
    auto count_in = [&](int g) {
        // experts p with lo <= p * tpr + g < hi
        const int a0 = R.lo - g, a1 = R.hi - g;
        const int c0 = a0 <= 0 ? 0 : (int)tprd.div((uint32_t)(a0 + R.tpr - 1));
        const int c1 = a1 <= 0 ? 0 : (int)tprd.div((uint32_t)(a1 + R.tpr - 1));
        return max(0, c1 - c0);
    };
    for (int g0 = threadIdx.x; g0 < ngroups; g0 += 2 * CTH) {
        int cnt[2];
        unsigned old[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {  // both atomics in flight together
            const int g = g0 + j * CTH;
            cnt[j] = g < ngroups ? count_in(g) : 0;
            old[j] = cnt[j] > 0 ? atom_add_acq_rel_gpu(a.rgcnt + g, (unsigned)cnt[j]) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (cnt[j] > 0 && old[j] + (unsigned)cnt[j] == expected)
                s_fin[atomicAdd(s_nfin, 1)] = g0 + j * CTH;  // at most ngroups entries
    }
    consumers_sync();
    // the rows of every group this CTA completed, spread over all consumer
    // threads so that their loads are in flight together
    const int nfin = min(*s_nfin, ngroups), per = a.m * rd;
    for (int it = threadIdx.x; it < nfin * per; it += CTH) {
        const int f = it / per, rem = it - f * per;
        const int r = s_fin[f] * rd + rem % rd;
        finish_row<true>(a, rem / rd, r, shared, s_tp, s_w, a.down, (size_t)a.dim, r);
    }
    for (int f = threadIdx.x; f < nfin; f += CTH)
        atomicExch(a.rgcnt + s_fin[f], 0u);
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

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
// and eight worker warps turn them into fp16 A operands held in tensor
// memory (each thread a row -- its TMEM lane -- written with tcgen05.st; each
// weight d * sc * q - dmin * m or d * sc * q in f32, then rounded to fp16),
// which the MMAs read from TMEM: the large operand never passes through
// shared memory, whose bandwidth would otherwise bound the kernel (fp16 tiles
// written once and read by every MMA). B is the group's activation rows,
// fp16, by TMA.
// gate and up (AK = 1) split both operands into fp16 pairs hi + lo (22
// significant bits: the dequantised q8_1 activation, 18 bits, exactly; the
// weight to 2^-23) and accumulate hi.hi + hi.lo + lo.hi, so g and u are as
// exact as f32 sums allow -- h is quantised to q8_1 again, and g, u a few
// 2^-12 off would move some of its roundings. Up to 64 columns, hi.hi and
// hi.lo are one MMA over the B stage's hi and lo rows side by side: an
// M = 128 MMA takes as long for 16 columns as for 128. down (AK = 2) takes single
// fp16 parts (about 2^-12 relative per operand): its output is only summed.
// The tensor cores' f32 accumulation is coarser than a sequential f32 sum
// (about 2e-5 relative over K = 4096), so the K-chunks are dealt round-robin
// over up to four accumulators in TMEM (4 x 128 columns), each taking its
// chunks in order, whose results the epilogue adds in f32, in order; over
// K = 4096 that keeps the router logits within 1e-5.
// Two warps issue the MMAs (alternate K-chunks); the eight worker warps (two a scheduler: the
// dequantisation is a chain of dependent integer and float steps) are also
// the epilogue (TMEM -> registers -> global).
#pragma once
#include "moe_tc.cuh"
#include "moe_route.cuh"

namespace moe {

#define TC_M 128        // rows of a tile (weights)
#define TC_NT 128       // columns (tokens) of a tile, at most
#define TC_KC 64        // K per stage (one 128-byte swizzle atom of 16-bit elements)
#define TC_WORKERS 8    // worker warps: two threads a tile row (one 32-weight group each)
#define TC_THREADS ((TC_WORKERS + 4) * 32)  // warps 0-7 workers / epilogue, 8 and 9 producers, 10 and 11 MMA
#define TC_BROWS 16     // rows of a B TMA box
#define TC_TMEM_COLS 512  // TMEM columns a CTA holds: up to 4 accumulators of TC_NT columns (dense),
                          // or 2 accumulators and the A stages from column 256 (K-quant)
#define TC_TA0 256        // first TMEM column of the K-quant A stages
#define TC_SB_MAX 8       // stages of the B ring, at most (and of the completion ring: S <= TC_SB_MAX)

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
    int nt;                 // AK = 0: columns of a tile (a multiple of 16, <= TC_NT)
    uint32_t b_buf;         // bytes of the B ring (a multiple of 2048)
    uint32_t *status;
    unsigned long long wait_ns;
};

// operands of a stage: hi and lo tiles for the split GEMM (gate, up)
__host__ __device__ constexpr int tc_parts(int AK) { return AK == 1 ? 2 : 1; }

// AK = 0 keeps its A stages in shared memory, the K-quant kernels in TMEM
__host__ __device__ inline size_t tc_smem_bytes(int AK, int S, int SR, uint32_t raw_bytes, uint32_t b_buf)
{
    // 1024 alignment slack, A stages (16 KB), raw stages, the B ring, barriers + TMEM address
    return 1024 + (AK == 0 ? (size_t)S * 16384 : 0) + (size_t)SR * raw_bytes + b_buf + 512;
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

// super-blocks of a row in one raw stage: Q2_K 4 (K = 1024 a stage), Q3_K 8 (K = 2048)
__host__ __device__ constexpr int tc_raw_blocks(int AK) { return AK == 1 ? 4 : 8; }
__host__ __device__ constexpr int tc_block_bytes(int AK) { return AK == 1 ? MOE_Q2K_BYTES : MOE_Q3K_BYTES; }
__host__ __device__ constexpr int tc_block_words(int AK) { return AK == 1 ? 21 : 28; }

// The words of super-block b of a raw-stage row (16-byte aligned; its
// stride, 336 or 880 bytes, an odd number of 16-byte units, so the eight
// rows of a quarter warp fall in distinct bank groups) by 16-byte loads:
// word i = bytes 4 i .. 4 i + 3 of the block, bytes past its end read as 0.
// O, the block's byte offset, is a constant, so the byte alignment (blocks
// of 84 or 110 bytes) costs shifts between registers only.
template <int O, int BB, int NW>
__device__ __forceinline__ void tc_block_words_at(const uint8_t *row, uint32_t (&E)[NW])
{
    constexpr int off = O & 15, nch = (off + BB + 15) / 16, w0 = off >> 2, sh = (off & 3) * 8;
    uint32_t C[4 * nch];
    const uint4 *p = reinterpret_cast<const uint4 *>(row + (O & ~15));
#pragma unroll
    for (int c = 0; c < nch; ++c) {
        const uint4 v = p[c];
        C[4 * c] = v.x;
        C[4 * c + 1] = v.y;
        C[4 * c + 2] = v.z;
        C[4 * c + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const int w = w0 + i;
        const uint32_t lo = w < 4 * nch ? C[w] : 0u, hi = w + 1 < 4 * nch ? C[w + 1] : 0u;
        E[i] = sh ? __funnelshift_r(lo, hi, sh) : lo;
    }
}

template <int AK>
__device__ __forceinline__ void tc_load_block(const uint8_t *row, int b, uint32_t (&E)[tc_block_words(AK)])
{
    constexpr int BB = tc_block_bytes(AK), NW = tc_block_words(AK);
    switch (b) {
    case 0: tc_block_words_at<0 * BB, BB, NW>(row, E); break;
    case 1: tc_block_words_at<1 * BB, BB, NW>(row, E); break;
    case 2: tc_block_words_at<2 * BB, BB, NW>(row, E); break;
    case 3: tc_block_words_at<3 * BB, BB, NW>(row, E); break;
    default:
        if constexpr (tc_raw_blocks(AK) == 8) {
            switch (b) {
            case 4: tc_block_words_at<4 * BB, BB, NW>(row, E); break;
            case 5: tc_block_words_at<5 * BB, BB, NW>(row, E); break;
            case 6: tc_block_words_at<6 * BB, BB, NW>(row, E); break;
            default: tc_block_words_at<7 * BB, BB, NW>(row, E); break;
            }
        }
    }
}

// Q2_K: the 32 weights of group gi (0, 1) of quarter KQ of a super-block
// (its 21 words bw: scales 0-3, quants 4-19, d and dmin 20) -- elements
// 32 gi .. 32 gi + 31 of the quarter -- to 16 words of fp16 pairs (hi) and of
// the pairs' remainders (lo), element order.
// w = d sc q - dmin m (one f32 rounding). A weight takes one of four values a
// sub-block (q = 0..3): their hi and lo halves form two 8-byte tables, and a
// byte permute with a selector made from two quants (one multiply-add) fetches
// a pair of weights.
template <int KQ>
__device__ __forceinline__ void dq_q2k_group(const uint32_t (&bw)[21], int gi, uint32_t (&o)[16], uint32_t (&ol)[16])
{
    const uint32_t scw = bw[KQ] >> (16 * gi);  // scales of sub-blocks 4 KQ + 2 gi, + 1
    const uint32_t dd = bw[20];
    const float d = f16_bits_to_f32(dd), dmin = f16_bits_to_f32(dd >> 16);
    uint32_t th[2][2], tl[2][2];  // [sub-block][q >> 1]: halves of q = 0, 1 and q = 2, 3
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const uint32_t sc = (scw >> (8 * u)) & 0xFFu;
        const float ds = d * (float)(sc & 15u), dm = dmin * (float)(sc >> 4);
        split_half2(-dm, fmaf(1.0f, ds, -dm), th[u][0], tl[u][0]);
        split_half2(fmaf(2.0f, ds, -dm), fmaf(3.0f, ds, -dm), th[u][1], tl[u][1]);
    }
    constexpr int half = KQ >> 1;
    const int sh = 2 * (2 * (KQ & 1) + gi);
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
        const uint32_t qq = (bw[4 + 8 * half + wi] >> sh) & 0x03030303u;  // four quants, one a byte
        const int u = wi >> 2;
        // selector of halfwords q_a, q_b: nibbles 2 q_a, 2 q_a + 1, 2 q_b, 2 q_b + 1
        const uint32_t s01 = (qq & 0x0303u) * 0x22u + 0x1010u, s23 = (qq >> 16) * 0x22u + 0x1010u;
        o[2 * wi] = __byte_perm(th[u][0], th[u][1], s01);
        o[2 * wi + 1] = __byte_perm(th[u][0], th[u][1], s23);
        ol[2 * wi] = __byte_perm(tl[u][0], tl[u][1], s01);
        ol[2 * wi + 1] = __byte_perm(tl[u][0], tl[u][1], s23);
    }
}

// Q3_K: the 32 weights of group gi of quarter KQ of one row's super-block
// (its 28 words w: hmask 0-7, quants 8-23, scales 24-26, d the low half of
// 27). w = d * (scale - 32) * q (exact in f32), q = low2 | hbit << 2 minus 4.
template <int KQ>
__device__ __forceinline__ void dq_q3k_group(const uint32_t (&w)[28], int gi, uint32_t (&o)[16])
{
    constexpr int half = KQ >> 1, g0 = 2 * (KQ & 1);
    const float d = f16_bits_to_f32(w[27]);
    float ds[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        // sub-block 4 KQ + j: low four bits in byte j of scale word KQ (KQ < 2,
        // low nibbles) or KQ - 2 (high nibbles), high two in byte j of word 2
        const int j = 2 * gi + u;
        const uint32_t lo4 = KQ < 2 ? (w[24 + KQ] >> (8 * j)) & 15u : (w[24 + (KQ & 1)] >> (8 * j + 4)) & 15u;
        const uint32_t hi2 = (w[26] >> (8 * j + 2 * KQ)) & 3u;
        ds[u] = d * (float)((int)(lo4 | (hi2 << 4)) - 32);
    }
    const int g = g0 + gi, hsh = 4 * half + g;  // weight j: bit j / 32 of hmask[j % 32]
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
        const uint32_t v = ((w[8 + 8 * half + wi] >> (2 * g)) & 0x03030303u) | (((w[wi] >> hsh) & 0x01010101u) << 2);
        const int u = wi >> 2;
        // 2^23 + v exactly, then v - 4 and its product with ds, two lanes an
        // instruction (packed f32, each lane rounded to nearest as alone)
        const float2 m4 = make_float2(-8388612.0f, -8388612.0f), d2 = make_float2(ds[u], ds[u]);
        const float2 f01 = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(v, 0x4B000000u, 0x7440)),
                                                             __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7441))),
                                                 m4),
                                      d2);
        const float2 f23 = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(v, 0x4B000000u, 0x7442)),
                                                             __uint_as_float(__byte_perm(v, 0x4B000000u, 0x7443))),
                                                 m4),
                                      d2);
        const __half2 h01 = __float22half2_rn(f01);
        const __half2 h23 = __float22half2_rn(f23);
        o[2 * wi] = *reinterpret_cast<const uint32_t *>(&h01);
        o[2 * wi + 1] = *reinterpret_cast<const uint32_t *>(&h23);
    }
}

// bounded mbarrier wait that gives up for good after the first timeout of
// this thread (`dead`), so that a broken pipeline still ends
__device__ __forceinline__ void tc_wait(uint64_t *bar, uint32_t parity, const TcArgs &a, bool &dead)
{
    if (!dead && !mbar_wait(bar, parity, a.status, a.wait_ns))
        dead = true;
}

// Position i in a ring of n barriers: barrier i % n, phase parity (i / n) & 1,
// stepped by one (the loops of one thread stay free of divisions by the
// run-time ring sizes, which cost a chain of dependent instructions each)
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n)
    {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// one quarter of a super-block (K-chunk kc): once chunk kc - S (position
// `done_pos` of the completion ring of D barriers) has freed A stage `st`,
// this thread's 32 weights into it in TMEM, then the warp's arrival on its
// full barrier
template <int AK, int KQ>
__device__ __forceinline__ void tc_quarter(const uint32_t (&E)[tc_block_words(AK)], int kc, int S, int gi,
                                           uint32_t ta0, uint32_t tac, uint64_t *full_a, uint64_t *mdone, int D,
                                           RingPos &st, RingPos &done_pos, const TcArgs &a, bool &dead)
{
    const int s = st.slot;
    if (kc >= S) {
        tc_wait(&mdone[done_pos.slot], done_pos.phase, a, dead);
        done_pos.next(D);
    }
    st.next(S);
    const uint32_t ta = ta0 + (uint32_t)s * tac;
    uint32_t o[16];
    if constexpr (AK == 1) {
        uint32_t ol[16];
        dq_q2k_group<KQ>(E, gi, o, ol);
        tmem_st16(ta, o);
        tmem_st16(ta + 32, ol);
    } else {
        dq_q3k_group<KQ>(E, gi, o);
        tmem_st16(ta, o);
    }
    tmem_st_wait();
    tc_fence_before();  // the stores before the arrival the MMA thread acquires
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(&full_a[s]);
}

template <int AK>
__global__ void __launch_bounds__(TC_THREADS, 1)
    moe_tc_gemm(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                const __grid_constant__ CUtensorMap bmap_lo, TcArgs a)
{
    constexpr int PARTS = tc_parts(AK);
    constexpr uint32_t TAC = 32 * PARTS;  // TMEM columns of a K-quant A stage: 64 fp16 a row, hi then lo
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int S = a.S, SR = a.SR;
    uint8_t *sa = smem;                                           // AK = 0: S x 16 KB
    uint8_t *sraw = sa + (AK == 0 ? (size_t)S * 16384 : 0);      // SR x raw_bytes
    uint8_t *sb = sraw + (size_t)SR * a.raw_bytes;  // the B ring, b_buf bytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(sb + a.b_buf);
    uint64_t *full_a = bars, *mdone = bars + S, *full_b = mdone + TC_SB_MAX;
    uint64_t *raw_full = full_b + TC_SB_MAX, *raw_empty = raw_full + SR, *done = raw_empty + SR;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the tile: rows m0 .. m0 + 127 of the weights, columns c0 .. c0 + ncols - 1
    int m0 = blockIdx.y * TC_M, c0, ncols, slot = 0;
    if constexpr (AK == 0) {
        c0 = blockIdx.x * a.nt;
        ncols = min(a.nt, a.N - c0);
    } else {
        if ((int)blockIdx.x >= __ldg(a.ntasks))
            return;
        const TcTask t = a.tasks[blockIdx.x];
        slot = t.slot;
        c0 = t.c0;
        ncols = t.ncols;
    }
    const int nb16 = (ncols + TC_BROWS - 1) / TC_BROWS;  // B boxes a stage and part
    const int n_mma = nb16 * TC_BROWS;                   // MMA N (a multiple of 16)
    const uint32_t idesc = mma_idesc(TC_M, n_mma, AK == 0);
    // split GEMM over at most 64 columns: the B stage holds the hi rows and
    // then the lo rows, so one MMA of 2 n_mma columns computes hi.hi and hi.lo
    // side by side in the accumulator (an M = 128 MMA costs the same up to
    // N = 128); the epilogue adds the two halves
    const bool cat = PARTS == 2 && 2 * n_mma <= TC_NT;
    const uint32_t idesc2 = mma_idesc(TC_M, 2 * n_mma, false);
    const int KC = a.K / TC_KC;
    const int per_raw = AK == 0 ? 1 : a.rk / TC_KC;     // A stages a raw stage feeds
    // the B ring holds as many stages as the tile's columns allow: narrow
    // groups keep many loads in flight
    const uint32_t bpart = (uint32_t)nb16 * TC_BROWS * 128u, bstage = PARTS * bpart;
    const int SB = max(1, min(TC_SB_MAX, (int)(a.b_buf / bstage)));
    // One barrier ring tells both the A side (S stages) and the B side (SB
    // stages) which chunks' MMAs are done: a waiter for chunk j has already
    // seen chunk j - D done (it waited for it, or for a later one, before
    // filling the stage now being refilled) and no MMA of chunk j + D can run
    // before the waiter's own next stage, so parity j / D is unambiguous.
    // Even, so that chunks j and j + D are issued by the same MMA thread and
    // their commits reach barrier j % D in order (S, SB <= TC_SB_MAX, even).
    const int D = (max(S, SB) + 1) & ~1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s)
            mbar_init(&full_a[s], AK == 0 ? 1 : TC_WORKERS);  // one arrival a worker warp
        for (int j = 0; j < D; ++j)
            mbar_init(&mdone[j], 1);
        for (int s = 0; s < SB; ++s)
            mbar_init(&full_b[s], 1);
        for (int r = 0; r < SR; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], TC_WORKERS);
        }
        mbar_init(done, 2);  // one commit from each MMA thread
        fence_barrier_init();
    }
    if (warp == 0)
        tmem_alloc(tmem_slot, TC_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool dead = false;

    if (warp == TC_WORKERS) {
        // ---------------- producers: this warp the A side (A tiles, or the
        // raw blocks), the next the B ring, each on its own barriers
        if (lane == 0) {
            tma_prefetch_map(&amap);
            RingPos pf, pw;  // the stage being filled; the one being waited for
            if constexpr (AK > 0) {
                for (int rc = 0; rc < KC / per_raw; ++rc) {  // raw stages
                    if (rc >= SR) {
                        tc_wait(&raw_empty[pw.slot], pw.phase, a, dead);
                        pw.next(SR);
                    }
                    mbar_arrive_expect_tx(&raw_full[pf.slot], a.raw_bytes);
                    tma_load_3d(sraw + (size_t)pf.slot * a.raw_bytes, &amap, rc * (a.raw_row / 4), m0, slot,
                                &raw_full[pf.slot]);
                    pf.next(SR);
                }
            } else {
                for (int kc = 0; kc < KC; ++kc) {
                    if (kc >= S) {  // chunk kc - S done
                        tc_wait(&mdone[pw.slot], pw.phase, a, dead);
                        pw.next(D);
                    }
                    mbar_arrive_expect_tx(&full_a[pf.slot], 16384u);
                    tma_load_2d(sa + (size_t)pf.slot * 16384, &amap, kc * TC_KC, m0, &full_a[pf.slot]);
                    pf.next(S);
                }
            }
        }
    } else if (warp == TC_WORKERS + 1) {
        if (lane == 0) {
            tma_prefetch_map(&bmap);
            if constexpr (PARTS == 2)
                tma_prefetch_map(&bmap_lo);
            RingPos pf, pw;
            for (int kc = 0; kc < KC; ++kc) {
                if (kc >= SB) {  // chunk kc - SB done
                    tc_wait(&mdone[pw.slot], pw.phase, a, dead);
                    pw.next(D);
                }
                const int s = pf.slot;
                pf.next(SB);
                uint8_t *dst = sb + (size_t)s * bstage;
                mbar_arrive_expect_tx(&full_b[s], bstage);
                for (int i = 0; i < nb16; ++i) {
                    tma_load_2d(dst + i * TC_BROWS * 128, &bmap, kc * TC_KC, c0 + i * TC_BROWS, &full_b[s]);
                    if constexpr (PARTS == 2)
                        tma_load_2d(dst + bpart + i * TC_BROWS * 128, &bmap_lo, kc * TC_KC, c0 + i * TC_BROWS,
                                    &full_b[s]);
                }
            }
        }
    } else if (warp == TC_WORKERS + 2 || warp == TC_WORKERS + 3) {
        // ---------------- MMA issuers: two threads (one a warp), thread h the
        // K-chunks h, h + 2, ..., so that one's waits and commits overlap the
        // other's MMAs (an MMA costs about the same for any N <= 128, and
        // the issuing thread's per-chunk waits, commit and stepping would
        // otherwise leave the tensor pipe idle); chunk kc accumulates into
        // accumulator kc % ksplit, so each accumulator takes its chunks in
        // order from one thread (ksplit 1: thread 0 alone)
        if (lane == 0) {
            const int h = warp - (TC_WORKERS + 2), step = a.ksplit > 1 ? 2 : 1;
            RingPos pa, pb, pd;  // A stage, B stage, completion barrier of chunk kc
            if (h == 1) {
                pa.next(S);
                pb.next(SB);
                pd.next(D);
            }
            for (int kc = h; kc < KC && (h == 0 || step == 2); kc += step) {
                const int s = pa.slot, t = pb.slot;
                tc_wait(&full_a[s], pa.phase, a, dead);
                tc_wait(&full_b[t], pb.phase, a, dead);
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(kc & (a.ksplit - 1)) * TC_NT;
                const bool first = kc < a.ksplit;
                const uint64_t bd = sw128_desc(sb + (size_t)t * bstage);
                if constexpr (AK == 0) {
                    const uint64_t ad = sw128_desc(sa + (size_t)s * 16384);
#pragma unroll
                    for (int k = 0; k < TC_KC / 16; ++k)  // K = 16 a step: 32 bytes further in the swizzle atom
                        mma_f16(acc, ad + 2 * k, bd + 2 * k, idesc, !first || k > 0);
                } else {
                    const uint32_t ta = tmem + TC_TA0 + (uint32_t)s * TAC;  // A in TMEM: 8 columns a K = 16 step
                    if (cat) {
#pragma unroll
                        for (int k = 0; k < TC_KC / 16; ++k) {
                            // hi . [hi | lo] over 2 n_mma columns, then + lo . hi
                            mma_f16_ts(acc, ta + 8 * k, bd + 2 * k, idesc2, !first || k > 0);
                            mma_f16_ts(acc, ta + 32 + 8 * k, bd + 2 * k, idesc, true);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < TC_KC / 16; ++k) {
                            mma_f16_ts(acc, ta + 8 * k, bd + 2 * k, idesc, !first || k > 0);
                            if constexpr (PARTS == 2) {  // + hi . lo + lo . hi (lo parts after the hi parts)
                                mma_f16_ts(acc, ta + 8 * k, bd + (bpart >> 4) + 2 * k, idesc, true);
                                mma_f16_ts(acc, ta + 32 + 8 * k, bd + 2 * k, idesc, true);
                            }
                        }
                    }
                }
                mma_commit(&mdone[pd.slot]);  // frees A stage s and B stage t
                for (int i = 0; i < step; ++i) {
                    pa.next(S);
                    pb.next(SB);
                    pd.next(D);
                }
            }
            mma_commit(done);
        }
    } else {
        // ---------------- workers (AK > 0): raw blocks -> fp16 operand tiles
        if constexpr (AK > 0) {
            const int r = threadIdx.x & (TC_M - 1), gi = threadIdx.x >> 7;  // tile row, 32-weight group
            constexpr int NB = tc_raw_blocks(AK);
            // this thread's row of a stage: TMEM lane r, columns 16 gi .. (hi), + 32 (lo)
            const uint32_t ta0 = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + TC_TA0 + 16u * (uint32_t)gi;
            RingPos pr, ps, pw;  // raw stage; A stage; completion barrier of chunk kc - S
            int b = 0;           // super-block within the raw stage
            for (int kb = 0; kb < KC / 4; ++kb) {  // super-blocks along K, four K-chunks each
                if (b == 0)
                    tc_wait(&raw_full[pr.slot], pr.phase, a, dead);
                uint32_t E[tc_block_words(AK)];
                tc_load_block<AK>(sraw + (size_t)pr.slot * a.raw_bytes + (size_t)r * a.raw_row, b, E);
                if (b == NB - 1) {  // the raw stage is all in registers: release it
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&raw_empty[pr.slot]);
                }
                tc_quarter<AK, 0>(E, 4 * kb, S, gi, ta0, TAC, full_a, mdone, D, ps, pw, a, dead);
                tc_quarter<AK, 1>(E, 4 * kb + 1, S, gi, ta0, TAC, full_a, mdone, D, ps, pw, a, dead);
                tc_quarter<AK, 2>(E, 4 * kb + 2, S, gi, ta0, TAC, full_a, mdone, D, ps, pw, a, dead);
                tc_quarter<AK, 3>(E, 4 * kb + 3, S, gi, ta0, TAC, full_a, mdone, D, ps, pw, a, dead);
                if (++b == NB) {
                    b = 0;
                    pr.next(SR);
                }
            }
        }
        // ---------------- epilogue: row m0 + 32 (warp % 4) + lane (the TMEM lane
        // quadrant of the warp), column blocks of 32 shared by warps w, w + 4
        tc_wait(done, 0, a, dead);
        tc_fence_after();
        const int row = m0 + 32 * (warp & 3) + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        for (int cb = 32 * (warp >> 2); cb < ncols; cb += 32 * (TC_WORKERS / 4)) {
            float v[32];
            tmem_ld32(lane_addr + (uint32_t)cb, v);
            if (cat) {  // + the hi . lo half
                float w[32];
                tmem_ld32(lane_addr + (uint32_t)(n_mma + cb), w);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = __fadd_rn(v[i], w[i]);
            }
            for (int j = 1; j < a.ksplit; ++j) {
                float w[32];
                tmem_ld32(lane_addr + (uint32_t)(j * TC_NT + cb), w);
                if (cat) {
                    float w2[32];
                    tmem_ld32(lane_addr + (uint32_t)(j * TC_NT + n_mma + cb), w2);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        w[i] = __fadd_rn(w[i], w2[i]);
                }
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
// ascending id, tokens ascending within an expert (deterministic): each
// warp counts its contiguous range of picks per expert, an exclusive scan
// gives the expert offsets and each warp's first place in every group, and
// each warp places its picks in order (match_any ranks). Also the column
// tasks of the routed GEMMs (ceil(count / TC_NT) per expert) and each pick's
// pair index.
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

#define PLAN_SMEM_PICKS 5120  // m * k up to this: the pair tables are built in shared memory (16-bit)
#define PLAN_WARPS 32         // warps of the plan kernel (1024 threads)

// dynamic shared memory of the plan kernel: per warp and expert a count (then
// a base), and for m * k <= PLAN_SMEM_PICKS the picks and both pair tables
__host__ __device__ inline size_t plan_smem_bytes(int n, int P)
{
    return (size_t)PLAN_WARPS * n * 4 + (P <= PLAN_SMEM_PICKS ? 3 * align_up((size_t)P * 2, 16) : 0);
}

__global__ void __launch_bounds__(1024) moe_prefill_plan_kernel(PPlanArgs a)
{
    __shared__ int s_cnt[MOE_MAX_ROUTED], s_off[MOE_MAX_ROUTED + 1], s_toff[MOE_MAX_ROUTED + 1];
    __shared__ int s_wsum[2][32];
    extern __shared__ __align__(16) uint8_t plan_dyn[];
    const int tid = threadIdx.x, P = a.m * a.k, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const bool staged = P <= PLAN_SMEM_PICKS;
    int *s_wc = reinterpret_cast<int *>(plan_dyn);  // [PLAN_WARPS][n]
    uint16_t *s_pick = reinterpret_cast<uint16_t *>(plan_dyn + (size_t)PLAN_WARPS * a.n * 4);
    uint16_t *s_qp = s_pick + align_up((size_t)P * 2, 16) / 2;  // pair q -> its pick t k + i
    uint16_t *s_pp = s_qp + align_up((size_t)P * 2, 16) / 2;    // pick -> its pair
    auto pick_at = [&](int p) {  // expert of pick p, -1 if out of range
        const int e = staged ? (s_pick[p] == 0xFFFFu ? -1 : (int)s_pick[p]) : __ldg(a.picks + p);
        return e >= 0 && e < a.n ? e : -1;
    };
    for (int e = tid; e < a.n; e += blockDim.x)
        s_cnt[e] = 0;
    for (int i = tid; i < PLAN_WARPS * a.n; i += blockDim.x)
        s_wc[i] = 0;
    __syncthreads();
    // each warp owns the contiguous picks [R warp, R warp + R): its counts per
    // expert, and the totals
    const int R = ((P + PLAN_WARPS - 1) / PLAN_WARPS + 31) / 32 * 32;
    const int p_lo = min(P, R * warp), p_hi = min(P, R * warp + R);
    for (int p = p_lo + lane; p < p_hi; p += 32) {
        int e = __ldg(a.picks + p);
        if (e < 0 || e >= a.n)
            e = -1;
        if (staged)
            s_pick[p] = e < 0 ? (uint16_t)0xFFFFu : (uint16_t)e;  // n <= 1024
        if (e >= 0) {
            atomicAdd(&s_wc[warp * a.n + e], 1);
            atomicAdd(&s_cnt[e], 1);
        }
    }
    __syncthreads();
    // offsets: an exclusive scan over the experts of their pair counts and of
    // their column-task counts (thread e holds expert e; n <= 1024 threads)
    {
        const int c = tid < a.n ? s_cnt[tid] : 0, tc = (c + TC_NT - 1) / TC_NT;
        int ic = c, it = tc;  // inclusive scans within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int uc = __shfl_up_sync(0xffffffffu, ic, o), ut = __shfl_up_sync(0xffffffffu, it, o);
            if (lane >= o) {
                ic += uc;
                it += ut;
            }
        }
        if (lane == 31) {
            s_wsum[0][warp] = ic;
            s_wsum[1][warp] = it;
        }
        __syncthreads();
        if (warp == 0) {  // scan of the warp totals
            int wc = lane < nw ? s_wsum[0][lane] : 0, wt = lane < nw ? s_wsum[1][lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int uc = __shfl_up_sync(0xffffffffu, wc, o), ut = __shfl_up_sync(0xffffffffu, wt, o);
                if (lane >= o) {
                    wc += uc;
                    wt += ut;
                }
            }
            s_wsum[0][lane] = wc;  // inclusive totals of warps 0 .. lane
            s_wsum[1][lane] = wt;
        }
        __syncthreads();
        const int bc = warp > 0 ? s_wsum[0][warp - 1] : 0, bt = warp > 0 ? s_wsum[1][warp - 1] : 0;
        if (tid < a.n) {
            const int off = bc + ic - c;
            s_off[tid] = off;
            s_toff[tid] = bt + it - tc;
            // each warp's first place in the expert's group: its offset plus
            // the counts of the warps before it (whose picks come first)
            int run = off;
            for (int w = 0; w < PLAN_WARPS; ++w) {
                const int cw = s_wc[w * a.n + tid];
                s_wc[w * a.n + tid] = run;
                run += cw;
            }
        }
        if (tid == a.n - 1) {
            s_off[a.n] = bc + ic;
            s_toff[a.n] = bt + it;
            *a.ntasks = bt + it;
        }
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
    // placement: each warp its picks in order, 32 at a time; lanes with the
    // same expert (one match) take consecutive places after the warp's next
    // place in that group. Picks are token-major, a token picks an expert at
    // most once, so each group is in ascending token order.
    for (int p0 = p_lo; p0 < p_hi; p0 += 32) {
        const int p = p0 + lane;
        const int e = p < p_hi ? pick_at(p) : -1;
        const unsigned grp = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(grp & ((1u << lane) - 1u));
        const int base = e >= 0 ? s_wc[warp * a.n + e] : 0;
        __syncwarp();
        if (e >= 0) {
            const int q = base + rank;
            if (rank == 0)
                s_wc[warp * a.n + e] = base + __popc(grp);
            if (staged) {
                s_qp[q] = (uint16_t)p;
                s_pp[p] = (uint16_t)q;
            } else {
                a.pair_tok[q] = p / a.k;
                a.pair_w[q] = a.weights[p];
                a.pick_pair[p] = q;
            }
        }
        __syncwarp();
    }
    if (!staged)
        return;
    // the pair tables from shared memory, in coalesced passes
    __syncthreads();
    const int np = s_off[a.n];
    const FastDiv kd((uint32_t)a.k);
    for (int q = tid; q < np; q += blockDim.x) {
        const int pk = s_qp[q];
        a.pair_tok[q] = (int)kd.div((uint32_t)pk);
        a.pair_w[q] = a.weights[pk];
    }
    for (int p = tid; p < P; p += blockDim.x)
        if (s_pick[p] != 0xFFFFu)
            a.pick_pair[p] = s_pp[p];
}

// ------------------------------------------------------------------ activations

// q8_1 of x (f16(d) * q, exact in f32) as fp16 hi + lo (exactly: 18
// significant bits), written straight into pair order: CTA p takes its
// token's row, eight values a lane, four lanes a 32-block (a group's lanes
// run the same iterations); x is 16-byte aligned
__global__ void moe_prefill_xhat_gather_kernel(const uint16_t *x, const int32_t *pair_tok, int P, int dim, __half *xg,
                                               __half *xg_lo)
{
    const int p = blockIdx.x;
    if (p >= P)
        return;
    const uint16_t *xr = x + (size_t)pair_tok[p] * dim;
    const unsigned gmask = 0xFu << (threadIdx.x & 28);
    for (int it = threadIdx.x; it < dim / 8; it += blockDim.x) {
        const uint4 w = *reinterpret_cast<const uint4 *>(xr + (size_t)it * 8);
        const float v[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                            bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            amax = fmaxf(amax, fabsf(v[j]));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
        const float d = __fdiv_rn(amax, 127.0f), id = __frcp_rn(d), d8 = __half2float(__float2half_rn(d));
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float xh[2];
            __half h[2], l[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int q = amax == 0.0f ? 0 : q8_code(v[2 * j + c], d, id);
                xh[c] = __fmul_rn(d8, (float)q);
                h[c] = __float2half_rn(xh[c]);
                l[c] = __float2half_rn(__fsub_rn(xh[c], __half2float(h[c])));
            }
            const __half2 hh = __halves2half2(h[0], h[1]), ll = __halves2half2(l[0], l[1]);
            hi[j] = *reinterpret_cast<const uint32_t *>(&hh);
            lo[j] = *reinterpret_cast<const uint32_t *>(&ll);
        }
        const size_t o = (size_t)p * dim + (size_t)it * 8;
        *reinterpret_cast<uint4 *>(xg + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(xg_lo + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// h = SwiGLU(g, u) per pair, its q8_1 (f32 decisions, f16 scale), and the
// dequantised fp16 h_hat for the down GEMM. One warp per 32-block.
__global__ void moe_prefill_swiglu_kernel(const float *g, const float *u, int nblk, float limit, __half *hhat)
{
    // four lanes a 32-block, eight consecutive values a lane (the block's
    // four lanes are all in range or all out, so the group's shuffles are safe)
    const size_t it = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (it >= (size_t)nblk * 4)
        return;
    const unsigned gmask = 0xFu << (threadIdx.x & 28);
    const size_t e0 = it * 8;
    const float4 g0 = *reinterpret_cast<const float4 *>(g + e0), g1 = *reinterpret_cast<const float4 *>(g + e0 + 4);
    const float4 u0 = *reinterpret_cast<const float4 *>(u + e0), u1 = *reinterpret_cast<const float4 *>(u + e0 + 4);
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float h[8], amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        h[j] = swiglu_f32(gv[j], uv[j], limit);
        amax = fmaxf(amax, fabsf(h[j]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
    // q8_1 of the block as q8_quant_warp takes it: d = amax / 127, the codes,
    // d8 = f16(d); the dequantised values d8 * q as fp16
    const float d = __fdiv_rn(amax, 127.0f), id = __frcp_rn(d), d8 = __half2float(__float2half_rn(d));
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int q0 = amax == 0.0f ? 0 : q8_code(h[2 * j], d, id);
        const int q1 = amax == 0.0f ? 0 : q8_code(h[2 * j + 1], d, id);
        const __half2 hh = __halves2half2(__float2half_rn(__fmul_rn(d8, (float)q0)),
                                          __float2half_rn(__fmul_rn(d8, (float)q1)));
        o[j] = *reinterpret_cast<const uint32_t *>(&hh);
    }
    *reinterpret_cast<uint4 *>(hhat + e0) = make_uint4(o[0], o[1], o[2], o[3]);
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
template <int V>
__global__ void moe_prefill_finish_kernel(const float *dw, const int32_t *picks, const int32_t *pick_pair, int k,
                                          const float *sd, float *acc, float *residual, uint16_t *x_next, int m,
                                          int dim)
{
    // V consecutive elements of one token a thread (V = 4: 16-byte accesses)
    const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * V;
    if (i >= (size_t)m * dim)
        return;
    const int t = (int)(i / dim), r = (int)(i - (size_t)t * dim);
    // the token's pairs in ascending expert id (its picks are distinct): a
    // compare-swap network over MOE_MAX_TOPK slots, absent picks last
    int e[MOE_MAX_TOPK], q[MOE_MAX_TOPK];
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        e[j] = j < k ? __ldg(picks + (size_t)t * k + j) : INT_MAX;
        q[j] = j < k ? min(max(__ldg(pick_pair + (size_t)t * k + j), 0), m * k - 1) : 0;
    }
#pragma unroll
    for (int j = 1; j < MOE_MAX_TOPK; ++j)
#pragma unroll
        for (int l = j; l > 0; --l)
            if (e[l] < e[l - 1]) {
                const int te = e[l], tq = q[l];
                e[l] = e[l - 1];
                q[l] = q[l - 1];
                e[l - 1] = te;
                q[l - 1] = tq;
            }
    float s[V];
#pragma unroll
    for (int c = 0; c < V; ++c)
        s[c] = 0.0f;
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
        if (j < k) {
            const float *row = dw + (size_t)q[j] * dim + r;
            float v[V];
            if constexpr (V == 4) {
                const float4 w = *reinterpret_cast<const float4 *>(row);
                v[0] = w.x, v[1] = w.y, v[2] = w.z, v[3] = w.w;
            } else {
                v[0] = row[0];
            }
#pragma unroll
            for (int c = 0; c < V; ++c)
                s[c] = __fadd_rn(s[c], v[c]);
        }
    }
#pragma unroll
    for (int c = 0; c < V; ++c) {
        if (sd)
            s[c] = __fadd_rn(s[c], sd[i + c]);
        acc[i + c] = s[c];
        const float res = __fadd_rn(residual[i + c], s[c]);
        residual[i + c] = res;
        x_next[i + c] = f32_to_bf16(res);
    }
}

}  // namespace moe

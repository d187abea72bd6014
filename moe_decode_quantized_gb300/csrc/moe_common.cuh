// moe_common.cuh -- device helpers and the workspace layout of libmoe.so.
//
// sm_103a only. Inline PTX for the Blackwell data movers the kernels use:
// mbarrier-tracked 1-D bulk copies (cp.async.bulk, the TMA engine's untiled
// form) into shared memory, L2 eviction-priority hints, and programmatic
// dependent launch (griddepcontrol) so a kernel's independent prologue runs
// while its predecessor drains. Every wait on an mbarrier is bounded: after
// the kernel's wait_ns of wall time (MOE_WAIT_NS unless the host set another
// bound) the waiting thread records MOE_WS_TIMEOUT in the workspace status
// word and the kernel unwinds instead of hanging.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/moe.h"

#define MOE_QK 256            // weights per K-quant super-block
#define MOE_Q2K_BYTES 84      // Q2_K super-block
#define MOE_Q3K_BYTES 110     // Q3_K super-block
#define MOE_Q8_BYTES 36       // q8_1 block of 32
#define MOE_WAIT_NS 2000000000ull  // default bound on any single wait: 2 s

// one Q2_K task = 128 super-blocks of one matrix (10752 B); one Q3_K task =
// 64 super-blocks (7040 B). Both sizes are multiples of 16 so the bulk copies
// of whole tasks stay 16-byte aligned for every supported shape.
#define MOE_G_TASK_SB 128
#define MOE_D_TASK_SB 64
#define MOE_PRODUCER_LANES 8
#define MOE_G_CHUNK 4  // gate/up tasks taken per grab from the grid-wide counters
// activation layout in shared memory: per 256-value segment, 256 int8 quants
// padded to 272 bytes, and a 28-float scale record (8 block scales d8, then
// 16 per-sub-block values), so lanes on different segments hit different banks
#define MOE_SEG_Q_BYTES 272
#define MOE_SEG_REC_FLOATS 28

#define MOE_CONSUMER_WARPS 15
#define MOE_THREADS ((MOE_CONSUMER_WARPS + 1) * 32)

namespace moe {

// ------------------------------------------------------------------ layout

struct WsLayout {
    size_t ctrl, rgcnt, logits, scores, keys, plan_w, plan_rows, ptrs, g, u, h, gs, us, hs, hsf, down, sd, acc,
        total;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// rows per down-projection task and row group: 32 super-blocks of Q3_K
__host__ __device__ inline int down_rows_per_task(int inter) { return MOE_D_TASK_SB / (inter / MOE_QK); }
// a routed gate/up task: this many rows of the gate matrix and the same rows
// of the up matrix (MOE_G_TASK_SB super-blocks in all)
__host__ __device__ inline int gate_rows_per_task(int dim) { return MOE_G_TASK_SB / 2 / (dim / MOE_QK); }

inline WsLayout ws_layout(const moe_cfg &c)
{
    WsLayout L{};
    size_t M = (size_t)c.max_tokens, cap = M * c.topk, off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    L.ctrl = take(256);
    L.rgcnt = take(sizeof(uint32_t) * (size_t)(c.dim / down_rows_per_task(c.inter)));
    L.logits = take(sizeof(float) * M * c.n_routed);
    L.scores = take(sizeof(float) * M * c.n_routed);
    L.keys = take(sizeof(float) * M * c.n_routed);
    L.plan_w = take(sizeof(float) * cap);
    L.plan_rows = take(sizeof(int32_t) * cap);
    L.ptrs = take(sizeof(uint64_t) * 3 * cap);
    L.g = take(sizeof(float) * cap * c.inter);
    L.u = take(sizeof(float) * cap * c.inter);
    L.h = take(sizeof(float) * cap * c.inter);  // SwiGLU(g, u) per plan pair
    L.gs = take(sizeof(float) * M * c.inter);
    L.us = take(sizeof(float) * M * c.inter);
    L.hs = take(sizeof(uint16_t) * M * c.inter);  // bf16 SwiGLU of the shared expert
    L.hsf = take(sizeof(float) * M * c.inter);    // f32 SwiGLU of a K-quant shared expert
    L.down = take(sizeof(float) * cap * c.dim);
    L.sd = take(sizeof(float) * M * c.dim);
    L.acc = take(sizeof(float) * M * c.dim);
    L.total = off;
    return L;
}

// control words at ws + ctrl
#define MOE_CTRL_TICKET 0
#define MOE_CTRL_STATUS 1
#define MOE_CTRL_GATEUP 2  // 6 words: gate/up task counters (one unused), shared rows done, plan hint

inline int header_words(int m, int k) { return m * (1 + 3 * k) + 2 + 2 * m * k; }

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// n / d and n % d for a divisor known only at run time, by one multiply-high
// with m = ceil(2^32 / d): n m / 2^32 = n / d + n (m d - 2^32) / (d 2^32),
// and the second term stays below 1 / d while n < 2^32 / d, so the floor is
// exact there (task and ring indices are far below it). A plain division by
// a run-time value is a chain of dependent instructions.
struct FastDiv {
    uint32_t d = 1, m = 0;
    __host__ __device__ FastDiv() {}
    // ceil(2^32 / d) = floor((2^32 - 1) / d) + 1 for every d >= 2 (a 32-bit division)
    __host__ __device__ explicit FastDiv(uint32_t dv) : d(dv), m(dv > 1 ? 0xFFFFFFFFu / dv + 1u : 0u) {}
    __device__ __forceinline__ uint32_t div(uint32_t n) const { return d > 1 ? __umulhi(n, m) : n; }
    __device__ __forceinline__ uint32_t mod(uint32_t n) const { return n - div(n) * d; }
};

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase with `parity` of `bar` to complete. Returns false after
// wait_ns nanoseconds and records MOE_WS_TIMEOUT in *status.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *status,
                                          unsigned long long wait_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 63u) == 63u && globaltimer() - t0 > wait_ns) {
            atomicOr(status, (uint32_t)MOE_WS_TIMEOUT);
            return false;
        }
    }
}

// L2 policy for weights that are streamed once: evict first.
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (tx bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Atomic add at GPU scope with acquire-release semantics: releases what the
// calling thread (and, after a CTA barrier, its CTA) wrote before, acquires
// what the earlier adders released. Returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(uint32_t *p, unsigned v)
{
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Fire-and-forget add at GPU scope with release semantics: what the calling
// thread wrote before is visible to whoever acquires the new value.
__device__ __forceinline__ void red_add_release_gpu(uint32_t *p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const uint32_t *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A plain store at GPU scope (to L2) with nothing to wait for: resets a
// counter that no one else touches until a later kernel, which the kernel
// boundary orders after it (an atomic exchange would return a value the
// thread then waits for).
__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, unsigned v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Programmatic dependent launch. wait: block until the preceding kernel in
// the stream has completed and its memory is visible (a no-op without a
// programmatic predecessor). launch_dependents: let the next kernel start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ numbers

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// f32 -> bf16 by round-to-nearest-even on the bit pattern ([moe_v41] fn
// bf16_bytes: add 0x7FFF plus the lowest kept bit, keep the high half).
__device__ __forceinline__ uint16_t f32_to_bf16(float f)
{
    uint32_t b = __float_as_uint(f);
    return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h)
{
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// ------------------------------------------------------------------ token count

// Calls f with the token count as a compile-time constant (IntC<m>), so that
// loops over tokens issue exactly m tokens' work: a loop to MOE_MAX_TOKENS
// with "if (t < m)" is predicated, not branched, and costs all 8.
template <int N>
struct IntC {
    static constexpr int value = N;
};

template <typename F>
__device__ __forceinline__ void with_m(int m, F &&f)
{
    switch (m) {
    case 1: f(IntC<1>{}); break;
    case 2: f(IntC<2>{}); break;
    case 3: f(IntC<3>{}); break;
    case 4: f(IntC<4>{}); break;
    case 5: f(IntC<5>{}); break;
    case 6: f(IntC<6>{}); break;
    case 7: f(IntC<7>{}); break;
    default: f(IntC<8>{}); break;
    }
}

// with_m in a kernel built for one token count: KM > 0 instantiates f for
// that count alone (the kernel's code holds one copy of it), KM = 0 for
// every count
template <int KM, typename F>
__device__ __forceinline__ void with_m_k(int m, F &&f)
{
    if constexpr (KM > 0)
        f(IntC<KM>{});
    else
        with_m(m, f);
}

// s += w . x over one 16-byte chunk of 8 bf16 each, in element order
__device__ __forceinline__ float fma_bf16x8(const uint4 &w, const uint4 &x, float s)
{
    s = fmaf(bf16_lo(w.x), bf16_lo(x.x), s);
    s = fmaf(bf16_hi(w.x), bf16_hi(x.x), s);
    s = fmaf(bf16_lo(w.y), bf16_lo(x.y), s);
    s = fmaf(bf16_hi(w.y), bf16_hi(x.y), s);
    s = fmaf(bf16_lo(w.z), bf16_lo(x.z), s);
    s = fmaf(bf16_hi(w.z), bf16_hi(x.z), s);
    s = fmaf(bf16_lo(w.w), bf16_lo(x.w), s);
    s = fmaf(bf16_hi(w.w), bf16_hi(x.w), s);
    return s;
}

// clamped SwiGLU in f32: silu(min(g, L)) * clamp(u, -L, L); L <= 0: no clamp
__device__ __forceinline__ float swiglu_f32(float g, float u, float limit)
{
    if (limit > 0.0f) {
        g = fminf(g, limit);
        u = fminf(fmaxf(u, -limit), limit);
    }
    float den = __fadd_rn(1.0f, expf(-g));
    return __fmul_rn(__fdiv_rn(g, den), u);
}

}  // namespace moe

// moe_abi.cu -- the extern "C" entry points of libmoe.so (declared and
// documented in include/moe.h): argument checks, workspace layout, launch
// geometry, programmatic dependent launch between the three kernels of a
// layer step, and CUDA-graph capture of whole multi-layer steps.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "moe_common.cuh"

#include "moe_route.cuh"
#include "moe_experts.cuh"
#include "moe_slot.cuh"
#include "moe_prefill.cuh"
#include "moe_runtime.cuh"

using namespace moe;

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

#define CUDA_OK(expr)                                                                          \
    do {                                                                                       \
        cudaError_t e_ = (expr);                                                               \
        if (e_ != cudaSuccess)                                                                 \
            return fail(MOE_ECUDA, "%s: %s (%s)", #expr, cudaGetErrorString(e_), cudaGetErrorName(e_)); \
    } while (0)

bool pow2_in(int v, int lo, int hi)
{
    return v >= lo && v <= hi && (v & (v - 1)) == 0;
}

int check_cfg(const moe_cfg *c)
{
    if (!c)
        return fail(MOE_EINVAL, "cfg is NULL");
    if (c->dim <= 0 || c->inter <= 0 || c->dim % MOE_QK || c->inter % MOE_QK)
        return fail(MOE_EINVAL, "dim (%d) and inter (%d) must be positive multiples of 256", c->dim, c->inter);
    if (c->topk < 1 || c->n_routed < c->topk)
        return fail(MOE_EINVAL, "need 1 <= topk (%d) <= n_routed (%d)", c->topk, c->n_routed);
    if (c->max_tokens < 1)
        return fail(MOE_EINVAL, "max_tokens (%d) must be >= 1", c->max_tokens);
    if (!(c->gate_temp > 0.0f))
        return fail(MOE_EINVAL, "gate_temp must be > 0");
    if (!pow2_in(c->dim, 256, 8192) || !pow2_in(c->inter, 256, 8192))
        return fail(MOE_EUNSUPPORTED, "dim (%d) and inter (%d) must be powers of two in [256, 8192]",
                    c->dim, c->inter);
    if (c->topk > MOE_MAX_TOPK || c->n_routed > MOE_MAX_ROUTED || c->max_tokens > MOE_MAX_TOKENS)
        return fail(MOE_EUNSUPPORTED, "topk <= %d, n_routed <= %d, max_tokens <= %d", MOE_MAX_TOPK,
                    MOE_MAX_ROUTED, MOE_MAX_TOKENS);
    if ((long long)c->max_tokens * c->dim > 32768)
        return fail(MOE_EUNSUPPORTED, "max_tokens * dim must be <= 32768");
    return MOE_OK;
}

int check_m(const moe_cfg *c, int m)
{
    if (m < 0 || m > c->max_tokens)
        return fail(MOE_EINVAL, "m (%d) must be in [0, max_tokens = %d]", m, c->max_tokens);
    return MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DevInfo {
    int sms = 0;
    int smem_optin = 0;
    bool attrs = false;
};

template <int AK>
int tc_attr(int smem_optin)
{
    CUDA_OK(cudaFuncSetAttribute(moe_tc_gemm<AK>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin));
    return MOE_OK;
}

std::mutex g_mu;
DevInfo g_dev[64];

// bound on every wait inside the kernels launched from now on (nanoseconds)
std::atomic<unsigned long long> g_wait_ns{MOE_WAIT_NS};

int dev_info(DevInfo **out)
{
    int d = 0;
    CUDA_OK(cudaGetDevice(&d));
    if (d < 0 || d >= 64)
        return fail(MOE_EUNSUPPORTED, "device ordinal %d", d);
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &I = g_dev[d];
    if (!I.attrs) {
        CUDA_OK(cudaDeviceGetAttribute(&I.sms, cudaDevAttrMultiProcessorCount, d));
        CUDA_OK(cudaDeviceGetAttribute(&I.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d));
        CUDA_OK(cudaFuncSetAttribute(moe_router_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_router_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_router_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_gateup_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_gateup_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_gateup_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_down_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_down_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, I.smem_optin));
        CUDA_OK(cudaFuncSetAttribute(moe_prefill_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     I.smem_optin - 16384));  // beside its static tables
        int rc = tc_attr<0>(I.smem_optin);
        if (rc || (rc = tc_attr<1>(I.smem_optin)) || (rc = tc_attr<2>(I.smem_optin)))
            return rc;
        I.attrs = true;
    }
    *out = &I;
    return MOE_OK;
}

template <typename Args>
int launch(void (*kernel)(Args), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, const Args &a)
{
    cudaLaunchConfig_t lc{};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = pdl ? 1 : 0;
    CUDA_OK(cudaLaunchKernelEx(&lc, kernel, a));
    return MOE_OK;
}

// ------------------------------------------------------------------ geometry

struct Geo {
    int r_rows, r_grid;
    size_t r_smem;
    int g_S, w2r;
    uint32_t g_stage;
    size_t g_smem;
    bool stage_x;
    int d_S, d_pair_cap, d_own_rows;
    uint32_t d_stage;
    size_t d_smem;
    int grid;  // persistent grid of the expert kernels
};

size_t router_smem(int rows, int dim, int m, int n)
{
    size_t main = (size_t)rows * dim * 2 + (size_t)m * dim * 2 + sizeof(float) * rows * m;
    size_t sel = sel_bytes(m, n);
    return 128 + router_pre_bytes(n, rows) + (main > sel ? main : sel);
}

// the most ring stages (up to cap, at least 2) that fit the shared memory
int stages_fit(size_t fixed, uint32_t stage, int cap, size_t limit)
{
    int S = cap;
    while (S > 2 && fixed + ring_head_bytes(S) + (size_t)S * stage + 16 > limit)
        --S;
    return S;
}

// sk: the shared expert's kind (0 none, 1 bf16, 2 K-quant)
int geometry(const moe_cfg &c, int m, int sk, const DevInfo &I, Geo &G)
{
    const int n = c.n_routed, dim = c.dim, inter = c.inter, k = c.topk;
    const size_t limit = (size_t)I.smem_optin;
    // about a third of the SMs compute the router rows, so most of the GPU is
    // free for the gate/up kernel's shared-expert rows while routing runs
    const int r_ctas = std::max(16, I.sms / 3);
    G.r_rows = (n + r_ctas - 1) / r_ctas;
    G.r_grid = (n + G.r_rows - 1) / G.r_rows;
    G.r_smem = router_smem(G.r_rows, dim, m, c.n_routed);
    G.grid = I.sms;
    // gate/up: stages of max(one Q2_K task, one bf16 shared W1 or W3 row, one
    // bf16 W2 row); w2r bf16 W2 rows a task, as many as a stage holds (<= 4,
    // dividing dim). K-quant shared tasks are a routed task's size (W1, W3)
    // or a down task's (W2)
    size_t gst = (size_t)MOE_G_TASK_SB * MOE_Q2K_BYTES;
    if (sk == 1)
        gst = std::max(gst, std::max((size_t)dim * 2, (size_t)inter * 2));
    if (sk == 2)
        gst = std::max(gst, (size_t)MOE_D_TASK_SB * MOE_Q3K_BYTES);
    G.g_stage = (uint32_t)align_up(gst, 128);
    G.w2r = 1;
    while (sk == 1 && G.w2r < 4 && (size_t)G.w2r * 2 * inter * 2 <= G.g_stage && dim % (G.w2r * 2) == 0)
        G.w2r *= 2;
    // bf16 x and hs in shared memory for up to two tokens; beyond, the ring
    // keeps the room and the consumers read them from L2
    G.stage_x = g_stage_x(m);
    size_t g_fixed = align_up((size_t)m * act_row_bytes(dim), 128) +
                     (G.stage_x ? align_up((size_t)m * dim * 2, 128) : 0) + g_hs_bytes(m, inter, sk, G.stage_x) +
                     g_pair_bytes(sk);
    G.g_S = stages_fit(g_fixed, G.g_stage, 32, limit);
    G.g_smem = g_smem_bytes(G.g_S, m, dim, inter, sk, G.stage_x, G.g_stage);
    // down: stages of one Q3_K task (the shared expert is done by the gate/up kernel)
    G.d_stage = (uint32_t)align_up((size_t)MOE_D_TASK_SB * MOE_Q3K_BYTES, 128);
    const int tpr = dim / down_rows_per_task(inter);
    const long long tmax = (long long)m * k * tpr;
    const long long per = (tmax + G.grid - 1) / G.grid;
    int span = (int)((per + tpr - 1) / tpr) + 1;
    G.d_pair_cap = std::min(m * k, span * m);
    G.d_own_rows = 0;
    size_t d_fixed = d_small_bytes(dim, inter) + align_up((size_t)G.d_pair_cap * act_row_bytes(inter), 128);
    G.d_S = stages_fit(d_fixed, G.d_stage, 48, limit);
    // row ownership for a few plan pairs: every CTA quantises all of them but
    // finishes its own rows without tickets, if the ring keeps 16 stages
    if (m * k <= 16) {
        const int own = (tpr + G.grid - 1) / G.grid * down_rows_per_task(inter);
        const size_t fo = d_small_bytes(dim, inter) + align_up((size_t)m * k * act_row_bytes(inter), 128) +
                          align_up(4 * (size_t)m * k * own, 128);
        const int So = stages_fit(fo, G.d_stage, 48, limit);
        if (So >= 16) {
            G.d_own_rows = own;
            G.d_pair_cap = m * k;
            G.d_S = So;
        }
    }
    G.d_smem = d_smem_bytes(G.d_S, G.d_pair_cap, dim, inter, G.d_own_rows, G.d_stage);
    if (G.r_smem > limit || G.g_smem > limit || G.d_smem > limit)
        return fail(MOE_EUNSUPPORTED, "shared memory: router %zu, gate/up %zu, down %zu > %zu bytes", G.r_smem,
                    G.g_smem, G.d_smem, limit);
    return MOE_OK;
}

// ------------------------------------------------------------------ launches

struct Bufs {
    const uint16_t *x;
    float *logits, *scores, *keys;
    int32_t *hdr;
    float *plan_w;
    int32_t *plan_rows;
    unsigned long long *ptrs;
    float *g, *u, *h, *gs, *us, *hsf, *down, *sd, *acc;
    uint16_t *hs;
    uint32_t *ctrl, *rgcnt;
};

Bufs ws_bufs(const moe_cfg &c, void *ws)
{
    const WsLayout L = ws_layout(c);
    char *b = static_cast<char *>(ws);
    Bufs B{};
    B.ctrl = reinterpret_cast<uint32_t *>(b + L.ctrl);
    B.rgcnt = reinterpret_cast<uint32_t *>(b + L.rgcnt);
    B.logits = reinterpret_cast<float *>(b + L.logits);
    B.scores = reinterpret_cast<float *>(b + L.scores);
    B.keys = reinterpret_cast<float *>(b + L.keys);
    B.plan_w = reinterpret_cast<float *>(b + L.plan_w);
    B.plan_rows = reinterpret_cast<int32_t *>(b + L.plan_rows);
    B.ptrs = reinterpret_cast<unsigned long long *>(b + L.ptrs);
    B.g = reinterpret_cast<float *>(b + L.g);
    B.u = reinterpret_cast<float *>(b + L.u);
    B.h = reinterpret_cast<float *>(b + L.h);
    B.gs = reinterpret_cast<float *>(b + L.gs);
    B.us = reinterpret_cast<float *>(b + L.us);
    B.hs = reinterpret_cast<uint16_t *>(b + L.hs);
    B.hsf = reinterpret_cast<float *>(b + L.hsf);
    B.down = reinterpret_cast<float *>(b + L.down);
    B.sd = reinterpret_cast<float *>(b + L.sd);
    B.acc = reinterpret_cast<float *>(b + L.acc);
    return B;
}

// the router and gate/up kernels built for one token and for eight (each
// holds that count's code alone), else for any count
void (*router_kernel_for(int m))(RouteArgs)
{
    return m == 1 ? moe_router_kernel<1> : m == 8 ? moe_router_kernel<8> : moe_router_kernel<0>;
}
void (*gateup_kernel_for(int m))(GArgs)
{
    return m == 1 ? moe_gateup_kernel<1> : m == 8 ? moe_gateup_kernel<8> : moe_gateup_kernel<0>;
}

RouteArgs route_args(const moe_cfg &c, int m)
{
    RouteArgs a{};
    a.dim = c.dim;
    a.n = c.n_routed;
    a.m = m;
    a.temp = c.gate_temp;
    a.route_scale = c.route_scale;
    a.norm = c.norm_topk_prob != 0;
    a.k = c.topk;
    a.wait_ns = g_wait_ns.load();
    return a;
}

void set_arena(RouteArgs &a, const moe_arena &ar)
{
    a.arena_base = static_cast<const char *>(ar.base);
    a.slot_bytes = ar.slot_bytes;
    a.gate_off = ar.gate_off;
    a.up_off = ar.up_off;
    a.down_off = ar.down_off;
}

int check_arena(const moe_arena *ar)
{
    if (!ar || !ar->base)
        return fail(MOE_EINVAL, "arena or arena->base is NULL");
    if (!aligned16(ar->base) || ar->slot_bytes % 16 || ar->gate_off % 16 || ar->up_off % 16 || ar->down_off % 16)
        return fail(MOE_EINVAL, "arena base, slot_bytes and offsets must be 16-byte aligned");
    return MOE_OK;
}

// the two expert kernels of one call. pdl_gateup: the gate/up kernel may start
// before its predecessor ends -- only when that predecessor is the router
// kernel of the same step, which triggers after x is complete (the gate/up
// prologue reads x before its own wait).
int launch_experts(const moe_cfg &c, int m, const Geo &G, const Bufs &B, const uint16_t *x,
                   const unsigned long long *ptrs, const float *plan_w, const int32_t *plan_rows,
                   const int32_t *hdr, int sk, const void *w1, const void *w3, const void *w2,
                   float *acc, float *residual, uint16_t *x_next, cudaStream_t s, bool pdl_gateup,
                   cudaEvent_t *ev = nullptr, bool plan_hint = false)
{
    const int k = c.topk, cap = m * k;
    GArgs ga{};
    ga.x = x;
    ga.w1 = w1;
    ga.w3 = w3;
    ga.w2 = w2;
    ga.sk = sk;
    ga.hs = B.hs;
    ga.hsf = B.hsf;
    ga.sd = B.sd;
    ga.limit = c.swiglu_limit;
    ga.wait_ns = g_wait_ns.load();
    ga.w2r = G.w2r;
    ga.plan_hint = (pdl_gateup || plan_hint) ? 1 : 0;  // only a layer step's router raises the hint
    ga.stage_x = G.stage_x ? 1 : 0;
    ga.hdr = hdr;
    ga.ptrs = ptrs;
    ga.plan_rows = plan_rows;
    ga.g = B.g;
    ga.u = B.u;
    ga.h = B.h;
    ga.gs = B.gs;
    ga.us = B.us;
    ga.status = B.ctrl + MOE_CTRL_STATUS;
    ga.gctr = B.ctrl + MOE_CTRL_GATEUP;
    ga.dim = c.dim;
    ga.inter = c.inter;
    ga.m = m;
    ga.k = k;
    ga.cap = cap;
    ga.plan_off = m * (1 + 3 * k);
    ga.S = G.g_S;
    ga.stage_bytes = G.g_stage;
    int rc = launch(gateup_kernel_for(m), dim3(G.grid), dim3(MOE_THREADS), G.g_smem, s, pdl_gateup, ga);
    if (rc)
        return rc;
    if (ev)
        CUDA_OK(cudaEventRecord(ev[0], s));
    DArgs da{};
    da.hdr = hdr;
    da.ptrs = ptrs;
    da.plan_rows = plan_rows;
    da.plan_w = plan_w;
    da.h = B.h;
    da.has_shared = w2 != nullptr;
    da.down = B.down;
    da.sd = B.sd;
    da.acc = acc;
    da.residual = residual;
    da.x_next = x_next;
    da.rgcnt = B.rgcnt;
    da.status = B.ctrl + MOE_CTRL_STATUS;
    da.gctr = B.ctrl + MOE_CTRL_GATEUP;
    da.limit = c.swiglu_limit;
    da.wait_ns = g_wait_ns.load();
    da.dim = c.dim;
    da.inter = c.inter;
    da.m = m;
    da.k = k;
    da.cap = cap;
    da.plan_off = m * (1 + 3 * k);
    da.S = G.d_S;
    da.pair_cap = G.d_pair_cap;
    da.own_rows = G.d_own_rows;
    da.stage_bytes = G.d_stage;
    if ((rc = launch(G.d_own_rows > 0 ? moe_down_kernel<1> : moe_down_kernel<0>, dim3(G.grid), dim3(MOE_THREADS),
                     G.d_smem, s, ev == nullptr, da)))
        return rc;
    if (ev)
        CUDA_OK(cudaEventRecord(ev[1], s));
    return MOE_OK;
}

int layer_step(const moe_cfg &c, const moe_layer &ly, const moe_arena &ar, const void *x, float *residual,
               void *x_next, int32_t *hdr, int m, void *ws, cudaStream_t s, cudaEvent_t *ev = nullptr)
{
    DevInfo *I;
    int rc = dev_info(&I);
    if (rc)
        return rc;
    const int sk = ly.sh_w1 == nullptr ? 0 : (ly.sh_format == MOE_SHARED_KQUANT ? 2 : 1);
    Geo G;
    if ((rc = geometry(c, m, sk, *I, G)))
        return rc;
    const Bufs B = ws_bufs(c, ws);
    RouteArgs ra = route_args(c, m);
    ra.x = static_cast<const uint16_t *>(x);
    ra.w = static_cast<const uint16_t *>(ly.router_w);
    ra.logits = B.logits;
    ra.scores = B.scores;
    ra.keys = B.keys;
    ra.rows_per_cta = G.r_rows;
    ra.do_select = 1;
    ra.bias = ly.bias;
    ra.slot_row = ly.slot_row;
    set_arena(ra, ar);
    ra.hdr = hdr;
    ra.plan_w = B.plan_w;
    ra.plan_rows = B.plan_rows;
    ra.ptrs = B.ptrs;
    ra.ctrl = B.ctrl;
    const bool pdl = ev == nullptr;
    if (ev)
        CUDA_OK(cudaEventRecord(ev[0], s));
    if ((rc = launch(router_kernel_for(m), dim3(G.r_grid), dim3(256), G.r_smem, s, pdl, ra)))
        return rc;
    if (ev)
        CUDA_OK(cudaEventRecord(ev[1], s));
    return launch_experts(c, m, G, B, static_cast<const uint16_t *>(x), B.ptrs, B.plan_w, B.plan_rows, hdr, sk,
                          ly.sh_w1, ly.sh_w3, ly.sh_w2, B.acc, residual,
                          static_cast<uint16_t *>(x_next), s, pdl, ev ? ev + 2 : nullptr);
}

int check_layer(const moe_cfg &c, const moe_layer *ly)
{
    if (!ly || !ly->router_w || !ly->bias || !ly->slot_row)
        return fail(MOE_EINVAL, "layer, router_w, bias and slot_row must be non-NULL");
    const bool any = ly->sh_w1 || ly->sh_w3 || ly->sh_w2, all = ly->sh_w1 && ly->sh_w3 && ly->sh_w2;
    if (any && !all)
        return fail(MOE_EINVAL, "shared expert: sh_w1, sh_w3 and sh_w2 must be all set or all NULL");
    if (!aligned16(ly->router_w) || (all && (!aligned16(ly->sh_w1) || !aligned16(ly->sh_w3) || !aligned16(ly->sh_w2))))
        return fail(MOE_EINVAL, "router and shared-expert weights must be 16-byte aligned");
    if (ly->sh_format != MOE_SHARED_BF16 && ly->sh_format != MOE_SHARED_KQUANT)
        return fail(MOE_EINVAL, "sh_format (%d) must be MOE_SHARED_BF16 or MOE_SHARED_KQUANT", ly->sh_format);
    (void)c;
    return MOE_OK;
}

// ------------------------------------------------------------------ static workspace
//
// Workspace of moe_layer_step_static: a file-scope device array, so that the
// call needs no device allocation at all. It serves callers that cannot
// allocate device memory: a plain C host program that links only this
// library and has no device allocator of its own, and a serving loop that
// must not allocate once it runs, because cudaMalloc and cudaFree can
// synchronise the whole device and can fail under memory pressure.
// MOE_STATIC_WS_BYTES bounds moe_workspace_bytes of the configurations it
// accepts (4 MiB: dim 4096, inter 2048, 384 routed experts, top-8, 8 tokens
// need 2.5 MB).
#define MOE_STATIC_WS_BYTES (4u << 20)
static __device__ __align__(256) unsigned char g_static_ws[MOE_STATIC_WS_BYTES];

void *g_static_ptr[64];  // per device ordinal, under g_mu

// Address of this device's copy of g_static_ws. The first call on a device
// (with that device current) looks the symbol up and zeroes the whole array
// on `s`, as moe_workspace_init does for a caller's workspace; that set-up
// must not be recorded into a graph, so a first call made while `s` is being
// captured is refused.
int static_ws(cudaStream_t s, void **out)
{
    int d = 0;
    CUDA_OK(cudaGetDevice(&d));
    if (d < 0 || d >= 64)
        return fail(MOE_EUNSUPPORTED, "device ordinal %d", d);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_static_ptr[d]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        CUDA_OK(cudaStreamIsCapturing(s, &cs));
        if (cs != cudaStreamCaptureStatusNone)
            return fail(MOE_EUNSUPPORTED,
                        "moe_layer_step_static: the first call on a device sets up the static workspace and "
                        "must be made outside stream capture");
        void *p = nullptr;
        CUDA_OK(cudaGetSymbolAddress(&p, g_static_ws));
        CUDA_OK(cudaMemsetAsync(p, 0, MOE_STATIC_WS_BYTES, s));
        g_static_ptr[d] = p;
    }
    *out = g_static_ptr[d];
    return MOE_OK;
}

// ------------------------------------------------------------------ tensor maps (TMA descriptors)

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's cuTensorMapEncodeTiled, looked up once through the runtime
// (the library links no driver library)
int encode_tiled(EncodeTiledFn *out)
{
    static EncodeTiledFn fn = nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        CUDA_OK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q));
        if (q != cudaDriverEntryPointSuccess || !p)
            return fail(MOE_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    *out = fn;
    return MOE_OK;
}

// rows x inner 16-bit elements, row stride row_bytes; boxes of box_rows rows
// x 64 elements, 128-byte swizzle (the SW128 K-major operand layout)
int map_rows16(CUtensorMap *m, bool bf16, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
               uint32_t box_rows)
{
    EncodeTiledFn fn;
    int rc = encode_tiled(&fn);
    if (rc)
        return rc;
    const cuuint64_t dims[2] = {inner, rows}, strides[1] = {row_bytes};
    const cuuint32_t box[2] = {64, box_rows}, es[2] = {1, 1};
    const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                          const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ECUDA, "cuTensorMapEncodeTiled (2-D, %llu x %llu) failed: %d", (unsigned long long)rows,
                    (unsigned long long)inner, (int)r);
    return MOE_OK;
}

// The expert arena's blocks of one matrix kind as u32 elements [slot][row]
// [row_bytes / 4]; boxes of 128 rows x raw_row bytes of one slot.
int map_arena(CUtensorMap *m, const void *base, uint64_t row_bytes, uint64_t rows, uint64_t slots,
              uint64_t slot_bytes, uint32_t raw_row)
{
    EncodeTiledFn fn;
    int rc = encode_tiled(&fn);
    if (rc)
        return rc;
    const cuuint64_t dims[3] = {row_bytes / 4, rows, slots}, strides[2] = {row_bytes, slot_bytes};
    const cuuint32_t box[3] = {raw_row / 4, TC_M, 1}, es[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(MOE_ECUDA, "cuTensorMapEncodeTiled (arena, %llu slots) failed: %d", (unsigned long long)slots,
                    (int)r);
    return MOE_OK;
}

// ------------------------------------------------------------------ prefill

struct PfLayout {
    size_t logits, scores, flags, cnt, off, pair_tok, pair_w, pick_pair, tasks, ntasks, status, xg, xg_lo, g, u, hh,
        dw, gs, us, hs, sd, acc, total;
    int P, max_tasks;
};

PfLayout pf_layout(const moe_cfg &c, int m)
{
    PfLayout L{};
    const size_t M = (size_t)m, P = M * c.topk, n = c.n_routed;
    L.P = (int)P;
    L.max_tasks = (int)std::min<size_t>(n, P) + (int)(P / TC_NT) + 1;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    L.logits = take(4 * M * n);
    L.scores = take(4 * M * n);
    L.flags = take(4 * M);
    L.cnt = take(4 * n);
    L.off = take(4 * (n + 1));
    L.pair_tok = take(4 * P);
    L.pair_w = take(4 * P);
    L.pick_pair = take(4 * P);
    L.tasks = take(sizeof(TcTask) * (size_t)L.max_tasks);
    L.ntasks = take(4);
    L.status = take(4);
    L.xg = take(2 * P * c.dim);
    L.xg_lo = take(2 * P * c.dim);
    L.g = take(4 * P * c.inter);
    L.u = take(4 * P * c.inter);
    L.hh = take(2 * P * c.inter);
    L.dw = take(4 * P * c.dim);
    L.gs = take(4 * M * c.inter);
    L.us = take(4 * M * c.inter);
    L.hs = take(2 * M * c.inter);
    L.sd = take(4 * M * c.dim);
    L.acc = take(4 * M * c.dim);
    L.total = off;
    return L;
}

#define MOE_PREFILL_MAX_TOKENS 65536

int check_prefill(const moe_cfg *c, int m)
{
    if (m < 0 || m > MOE_PREFILL_MAX_TOKENS)
        return fail(MOE_EINVAL, "prefill: m (%d) must be in [0, %d]", m, MOE_PREFILL_MAX_TOKENS);
    if (c->dim % 1024 || c->inter % 2048)
        return fail(MOE_EUNSUPPORTED,
                    "prefill: dim (%d) must be a multiple of 1024 and inter (%d) of 2048 (TMA row strides of "
                    "the Q2_K / Q3_K blocks)",
                    c->dim, c->inter);
    return MOE_OK;
}

// one GEMM of the prefill: D[M x N] = A . B^T, out[col * ldo + row]
// the B ring takes the shared memory the A stages and raw stages leave (up
// to TC_SB_MAX full-width stages)
template <int AK>
int launch_tc(const CUtensorMap &am, const CUtensorMap &bm, const CUtensorMap &bm_lo, TcArgs a, dim3 grid,
              cudaStream_t s, int smem_optin)
{
    if (grid.x == 0 || grid.y == 0)
        return MOE_OK;
    // the MMA-completion ring has max(S, SB) barriers, rounded up to even,
    // in room for TC_SB_MAX (an even number)
    if (a.S < 1 || a.S > TC_SB_MAX)
        return fail(MOE_EUNSUPPORTED, "prefill GEMM: %d operand stages (at most %d)", a.S, TC_SB_MAX);
    const size_t fixed = tc_smem_bytes(AK, a.S, a.SR, a.raw_bytes, 0);
    const size_t full = (size_t)TC_SB_MAX * tc_parts(AK) * TC_NT * 128;
    if ((size_t)smem_optin < fixed + 2 * tc_parts(AK) * TC_NT * 128)
        return fail(MOE_EUNSUPPORTED, "prefill GEMM: %zu bytes of shared memory needed", fixed);
    a.b_buf = (uint32_t)std::min(full, ((size_t)smem_optin - fixed) / 2048 * 2048);
    moe_tc_gemm<AK><<<grid, TC_THREADS, fixed + a.b_buf, s>>>(am, bm, bm_lo, a);
    CUDA_OK(cudaGetLastError());
    return MOE_OK;
}

TcArgs tc_args(int M, int N, int K, float *out, int ldo, uint32_t *status)
{
    TcArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.out = out;
    a.ldo = ldo;
    a.S = 3;
    a.SR = 0;
    const int kc = K / TC_KC;  // K-chunks: split over up to four accumulators, evenly
    a.ksplit = kc % 4 == 0 ? 4 : (kc % 2 == 0 ? 2 : 1);
    a.status = status;
    a.wait_ns = g_wait_ns.load();
    return a;
}

// bf16 GEMM out[n * ldo + r] = sum_k A[r, k] B[n, k] (A [M, K], B [N, K] row-major bf16)
int gemm_bf16(const void *A, const void *B, float *out, int M, int N, int K, int ldo, uint32_t *status,
              cudaStream_t s, int smem_optin, int sms)
{
    CUtensorMap am, bm;
    int rc = map_rows16(&am, true, A, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, TC_M);
    if (rc || (rc = map_rows16(&bm, true, B, (uint64_t)K, (uint64_t)N, (uint64_t)K * 2, TC_BROWS)))
        return rc;
    TcArgs a = tc_args(M, N, K, out, ldo, status);
    // narrower column tiles while the grid still fits one wave: a CTA's time
    // hardly depends on its width, so a small grid (the router's 3 row
    // tiles) spreads over more SMs; a second wave would cost a CTA's time
    const int mt = (M + TC_M - 1) / TC_M;
    a.nt = TC_NT;
    while (a.nt > 16 && (long long)mt * ((N + a.nt / 2 - 1) / (a.nt / 2)) <= sms)
        a.nt /= 2;
    return launch_tc<0>(am, bm, bm, a, dim3((N + a.nt - 1) / a.nt, mt), s, smem_optin);
}

// A multi-layer step: the captured graph, and what its eager form needs (the
// layers, buffers and per-layer snapshots), used when capture failed and the
// object runs eagerly, and to rerun the step from a layer.
struct GraphObj {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    bool eager = false;
    moe_cfg cfg{};
    std::vector<moe_layer> layers;
    moe_arena arena{};
    int m = 0, n_layers = 0, hw = 0;
    void *x_a = nullptr, *x_b = nullptr, *ws = nullptr;
    float *residual = nullptr;
    int32_t *headers = nullptr;
    char *snap = nullptr;  // per layer: its input x (bf16) then the residual (f32), or NULL
    size_t x_bytes = 0, res_bytes = 0, hdr_bytes = 0, snap_stride = 0;

    void *x_in(int l) const { return (l % 2 == 0) ? x_a : x_b; }
    void *x_out(int l) const { return (l == n_layers - 1) ? x_a : ((l % 2 == 0) ? x_b : x_a); }
};

size_t snapshot_stride(const moe_cfg &c, int m)
{
    return align_up((size_t)m * c.dim * 2, 256) + align_up((size_t)m * c.dim * 4, 256);
}

// layers `from` .. the last, each preceded by the copy of its input into its
// snapshot (when the object keeps snapshots)
int run_layers(GraphObj &G, int from, cudaStream_t s)
{
    for (int l = from; l < G.n_layers; ++l) {
        if (G.snap) {
            char *sn = G.snap + (size_t)l * G.snap_stride;
            CUDA_OK(cudaMemcpyAsync(sn, G.x_in(l), G.x_bytes, cudaMemcpyDeviceToDevice, s));
            CUDA_OK(cudaMemcpyAsync(sn + align_up(G.x_bytes, 256), G.residual, G.res_bytes, cudaMemcpyDeviceToDevice,
                                    s));
        }
        const int rc = layer_step(G.cfg, G.layers[l], G.arena, G.x_in(l), G.residual, G.x_out(l),
                                  G.headers + (size_t)l * G.hw, G.m, G.ws, s);
        if (rc)
            return rc;
    }
    return MOE_OK;
}

// the inputs of layer l back from its snapshot
int restore_snapshot(GraphObj &G, int l, cudaStream_t s)
{
    const char *sn = G.snap + (size_t)l * G.snap_stride;
    CUDA_OK(cudaMemcpyAsync(G.x_in(l), sn, G.x_bytes, cudaMemcpyDeviceToDevice, s));
    CUDA_OK(cudaMemcpyAsync(G.residual, sn + align_up(G.x_bytes, 256), G.res_bytes, cudaMemcpyDeviceToDevice, s));
    return MOE_OK;
}

// The picks of every token of layer l (header in host memory) made resident.
int cache_ensure(ExpertCache &C, int layer, const int32_t *experts, int n, int *n_fetched, cudaStream_t s)
{
    if (layer < 0 || layer >= C.n_layers || n < 0 || (n > 0 && !experts))
        return fail(MOE_EINVAL, "moe_cache_ensure: layer %d outside [0, %d) or bad experts", layer, C.n_layers);
    std::vector<int> req;
    for (int i = 0; i < n; ++i) {
        const int e = experts[i];
        if (e < 0 || e >= C.n_routed)
            return fail(MOE_EINVAL, "moe_cache_ensure: expert %d outside [0, %d)", e, C.n_routed);
        bool seen = false;
        for (int r : req)
            seen = seen || r == e;
        if (!seen)
            req.push_back(e);
    }
    if ((int)req.size() > C.n_slots)
        return fail(MOE_EUNSUPPORTED, "moe_cache_ensure: %d experts at once, the cache holds %d slots", (int)req.size(),
                    C.n_slots);
    const size_t base = (size_t)layer * C.n_routed;
    // the hits first: most recently used, so no victim below is one of them
    for (int e : req)
        if (C.table[base + e] >= 0) {
            ++C.hits;
            C.touch(C.table[base + e]);
        }
    std::vector<char> dirty(C.n_layers, 0);
    int fetched = 0;
    for (int e : req) {
        if (C.table[base + e] >= 0)
            continue;
        ++C.misses;
        const int v = C.lru.back();
        if (C.owner[v] >= 0) {  // evict the least recently used expert
            ++C.evictions;
            C.table[(size_t)C.owner[v]] = -1;
            dirty[C.owner[v] / C.n_routed] = 1;
        }
        C.owner[v] = (int64_t)(base + e);
        C.table[base + e] = v;
        dirty[layer] = 1;
        C.touch(v);
        if (C.fetch) {
            const int rc = C.fetch(C.user, layer, e, const_cast<char *>(C.arena_base) + (size_t)v * C.slot_bytes,
                                   C.slot_bytes, (moe_stream_t)s);
            if (rc)
                return fail(MOE_ECUDA, "moe_cache_ensure: the expert source failed (%d) for layer %d expert %d", rc,
                            layer, e);
        }
        ++fetched;
    }
    if (C.table_dev)
        for (int l = 0; l < C.n_layers; ++l)
            if (dirty[l])  // pageable source: the copy has taken the row when the call returns
                CUDA_OK(cudaMemcpyAsync(C.table_dev + (size_t)l * C.n_routed, C.table.data() + (size_t)l * C.n_routed,
                                        sizeof(int32_t) * C.n_routed, cudaMemcpyHostToDevice, s));
    if (n_fetched)
        *n_fetched = fetched;
    return MOE_OK;
}

struct HostSource {
    std::vector<const void *> images;  // [layer * n_routed + expert]
    int n_routed = 0;
    uint64_t image_bytes = 0;
};

}  // namespace

// ==================================================================== C ABI

extern "C" {

const char *moe_last_error(void) { return g_err; }

int moe_header_words(const moe_cfg *cfg, int m)
{
    if (!cfg || m < 0 || cfg->topk < 1)
        return fail(MOE_EINVAL, "moe_header_words: bad arguments");
    return header_words(m, cfg->topk);
}

int moe_workspace_bytes(const moe_cfg *cfg, size_t *bytes)
{
    int rc = check_cfg(cfg);
    if (rc)
        return rc;
    if (!bytes)
        return fail(MOE_EINVAL, "bytes is NULL");
    *bytes = ws_layout(*cfg).total;
    return MOE_OK;
}

int moe_workspace_init(void *ws, size_t bytes, moe_stream_t stream)
{
    if (!ws)
        return fail(MOE_EINVAL, "ws is NULL");
    CUDA_OK(cudaMemsetAsync(ws, 0, bytes, (cudaStream_t)stream));
    return MOE_OK;
}

int moe_workspace_view(const moe_cfg *cfg, void *ws, moe_ws_view *v)
{
    int rc = check_cfg(cfg);
    if (rc)
        return rc;
    if (!ws || !v)
        return fail(MOE_EINVAL, "ws and view must be non-NULL");
    const Bufs B = ws_bufs(*cfg, ws);
    v->logits = B.logits;
    v->plan_w = B.plan_w;
    v->plan_rows = B.plan_rows;
    v->ptrs = reinterpret_cast<uint64_t *>(B.ptrs);
    v->g = B.g;
    v->u = B.u;
    v->gs = B.gs;
    v->us = B.us;
    v->down = B.down;
    v->sd = B.sd;
    v->acc = B.acc;
    v->status = B.ctrl + MOE_CTRL_STATUS;
    return MOE_OK;
}

int moe_read_status(void *ws, uint32_t *status, moe_stream_t stream)
{
    if (!ws || !status)
        return fail(MOE_EINVAL, "ws and status must be non-NULL");
    CUDA_OK(cudaMemcpyAsync(status, static_cast<uint32_t *>(ws) + MOE_CTRL_STATUS, 4, cudaMemcpyDeviceToHost,
                            (cudaStream_t)stream));
    CUDA_OK(cudaStreamSynchronize((cudaStream_t)stream));
    return MOE_OK;
}

int moe_set_wait_limit_ns(uint64_t ns)
{
    g_wait_ns.store(ns == 0 ? MOE_WAIT_NS : (unsigned long long)ns);
    return MOE_OK;
}

int moe_expert_step_unreleased(const moe_cfg *cfg, const void *x, const int32_t *header, int m, void *ws,
                               moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)))
        return rc;
    if (m < 1 || !x || !header || !ws || !aligned16(x))
        return fail(MOE_EINVAL, "moe_expert_step_unreleased: bad arguments");
    DevInfo *I;
    if ((rc = dev_info(&I)))
        return rc;
    Geo G;
    if ((rc = geometry(*cfg, m, 0, *I, G)))
        return rc;
    const Bufs B = ws_bufs(*cfg, ws);
    return launch_experts(*cfg, m, G, B, static_cast<const uint16_t *>(x), B.ptrs, B.plan_w, B.plan_rows, header,
                          0, nullptr, nullptr, nullptr, B.acc, nullptr, nullptr, (cudaStream_t)stream, false, nullptr,
                          true);
}

int moe_router_logits(const moe_cfg *cfg, const void *x, const void *w, float *logits, int m,
                      moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)))
        return rc;
    if (m == 0)
        return MOE_OK;
    if (!x || !w || !logits || !aligned16(x) || !aligned16(w))
        return fail(MOE_EINVAL, "x, w (16-byte aligned) and logits must be non-NULL");
    DevInfo *I;
    if ((rc = dev_info(&I)))
        return rc;
    Geo G;
    if ((rc = geometry(*cfg, m, 0, *I, G)))
        return rc;
    RouteArgs a = route_args(*cfg, m);
    a.x = static_cast<const uint16_t *>(x);
    a.w = static_cast<const uint16_t *>(w);
    a.logits = logits;
    a.rows_per_cta = G.r_rows;
    a.do_select = 0;
    return launch(router_kernel_for(m), dim3(G.r_grid), dim3(256), G.r_smem, (cudaStream_t)stream, false, a);
}

int moe_quantize_q8_1(const moe_cfg *cfg, const void *x, int m, void *out, moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)))
        return rc;
    if (m == 0)
        return MOE_OK;
    if (!x || !out)
        return fail(MOE_EINVAL, "x and out must be non-NULL");
    const int nblk = m * cfg->dim / 32;
    const int threads = 256, grid = (nblk * 32 + threads - 1) / threads;
    moe_quantize_q8_1_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>(static_cast<const uint16_t *>(x), nblk,
                                                                         static_cast<uint8_t *>(out));
    CUDA_OK(cudaGetLastError());
    return MOE_OK;
}

int moe_swiglu_q8(const moe_cfg *cfg, const float *g, const float *u, int rows, float *h, void *hq8,
                  moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc)
        return rc;
    if (rows < 0)
        return fail(MOE_EINVAL, "rows must be >= 0");
    if (rows == 0)
        return MOE_OK;
    if (!g || !u || !hq8)
        return fail(MOE_EINVAL, "g, u and hq8 must be non-NULL");
    const int nblk = rows * cfg->inter / 32;
    const int threads = 256, grid = (nblk * 32 + threads - 1) / threads;
    moe_swiglu_q8_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>(g, u, nblk, cfg->swiglu_limit, h,
                                                                     static_cast<uint8_t *>(hq8));
    CUDA_OK(cudaGetLastError());
    return MOE_OK;
}

int moe_route_scores(const moe_cfg *cfg, const float *logits, int count, float *scores, moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc)
        return rc;
    if (count < 0)
        return fail(MOE_EINVAL, "moe_route_scores: count (%d) < 0", count);
    if (count == 0)
        return MOE_OK;
    if (!logits || !scores)
        return fail(MOE_EINVAL, "moe_route_scores: a buffer is NULL");
    ScoreArgs a{logits, scores, cfg->gate_temp, count};
    return launch(moe_score_kernel, dim3((count + MOE_SCORES_PER_CTA - 1) / MOE_SCORES_PER_CTA), dim3(256), 0,
                  (cudaStream_t)stream, false, a);
}

int moe_route_select(const moe_cfg *cfg, const float *logits, const float *bias, const int32_t *slot_row,
                     const moe_arena *arena, int m, int32_t *header, float *plan_w, int32_t *plan_rows,
                     uint64_t *ptrs, moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)) || (rc = check_arena(arena)))
        return rc;
    if (m == 0)
        return MOE_OK;
    if (!logits || !bias || !slot_row || !header || !plan_w || !plan_rows || !ptrs)
        return fail(MOE_EINVAL, "moe_route_select: a buffer is NULL");
    RouteArgs a = route_args(*cfg, m);
    a.logits = const_cast<float *>(logits);
    a.bias = bias;
    a.slot_row = slot_row;
    set_arena(a, *arena);
    a.hdr = header;
    a.plan_w = plan_w;
    a.plan_rows = plan_rows;
    a.ptrs = reinterpret_cast<unsigned long long *>(ptrs);
    DevInfo *I;
    if ((rc = dev_info(&I)))
        return rc;
    const size_t smem = align_up(sel_bytes(m, cfg->n_routed), 128) + sizeof(float) * 2 * (size_t)m * cfg->n_routed +
                        sizeof(int) * (size_t)cfg->n_routed;
    if (smem > (size_t)I->smem_optin)
        return fail(MOE_EUNSUPPORTED, "moe_route_select: %zu bytes of shared memory needed", smem);
    return launch(moe_select_kernel, dim3(1), dim3(256), smem, (cudaStream_t)stream, false, a);
}

int moe_expert_step(const moe_cfg *cfg, const void *x, const uint64_t *ptrs, const float *plan_w,
                    const int32_t *plan_rows, const int32_t *header, int m, float *acc, void *ws,
                    moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)))
        return rc;
    if (m == 0)
        return MOE_OK;
    if (!x || !ptrs || !plan_w || !plan_rows || !header || !acc || !ws || !aligned16(x))
        return fail(MOE_EINVAL, "moe_expert_step: a buffer is NULL or x is not 16-byte aligned");
    DevInfo *I;
    if ((rc = dev_info(&I)))
        return rc;
    Geo G;
    if ((rc = geometry(*cfg, m, 0, *I, G)))
        return rc;
    const Bufs B = ws_bufs(*cfg, ws);
    return launch_experts(*cfg, m, G, B, static_cast<const uint16_t *>(x),
                          reinterpret_cast<const unsigned long long *>(ptrs), plan_w, plan_rows, header, 0, nullptr,
                          nullptr, nullptr, acc, nullptr, nullptr, (cudaStream_t)stream, false);
}

int moe_layer_step(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena, const void *x,
                   float *residual, void *x_next, int32_t *header, int m, void *ws, moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)) || (rc = check_arena(arena)) || (rc = check_layer(*cfg, layer)))
        return rc;
    if (m == 0)
        return MOE_OK;
    if (!x || !residual || !x_next || !header || !ws || !aligned16(x))
        return fail(MOE_EINVAL, "moe_layer_step: a buffer is NULL or x is not 16-byte aligned");
    return layer_step(*cfg, *layer, *arena, x, residual, x_next, header, m, ws, (cudaStream_t)stream);
}

int moe_layer_step_static(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena,
                          const void *x, float *residual, void *x_next, int32_t *header, int m,
                          uint32_t *status_host, moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)) || (rc = check_arena(arena)) || (rc = check_layer(*cfg, layer)))
        return rc;
    const WsLayout L = ws_layout(*cfg);
    if (L.total > MOE_STATIC_WS_BYTES)
        return fail(MOE_EUNSUPPORTED,
                    "moe_layer_step_static: this configuration needs %zu bytes of workspace, the static "
                    "workspace holds %u; use moe_layer_step with a workspace of its own",
                    L.total, (unsigned)MOE_STATIC_WS_BYTES);
    if (m > 0 && (!x || !residual || !x_next || !header || !aligned16(x)))
        return fail(MOE_EINVAL, "moe_layer_step_static: a buffer is NULL or x is not 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    void *ws = nullptr;
    if ((rc = static_ws(s, &ws)))
        return rc;
    // the array keeps the last call's contents: the control words and the
    // row-group counters (everything before the logits) must start at zero,
    // also after a call whose wait ran out and left them set
    CUDA_OK(cudaMemsetAsync(ws, 0, L.logits, s));
    if (m > 0 && (rc = layer_step(*cfg, *layer, *arena, x, residual, x_next, header, m, ws, s)))
        return rc;
    if (status_host)
        CUDA_OK(cudaMemcpyAsync(status_host, static_cast<char *>(ws) + L.ctrl + 4 * MOE_CTRL_STATUS,
                                sizeof(uint32_t), cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

int moe_host_io_bytes(const moe_cfg *cfg, int m, size_t *bytes)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)))
        return rc;
    if (!bytes)
        return fail(MOE_EINVAL, "bytes is NULL");
    const size_t xd = align_up((size_t)m * cfg->dim * 2, 256), rd = align_up((size_t)m * cfg->dim * 4, 256);
    *bytes = 2 * xd + rd + align_up(sizeof(int32_t) * header_words(m, cfg->topk), 256);
    return MOE_OK;
}

int moe_layer_step_host(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena, const void *x_host,
                        float *residual_host, void *x_next_host, int32_t *header_host, int m, void *io,
                        void *ws, moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)) || (rc = check_arena(arena)) || (rc = check_layer(*cfg, layer)))
        return rc;
    if (m == 0)
        return MOE_OK;
    if (!x_host || !residual_host || !x_next_host || !header_host || !io || !ws || !aligned16(io))
        return fail(MOE_EINVAL, "moe_layer_step_host: a buffer is NULL or io is not 16-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    const size_t xb = (size_t)m * cfg->dim * 2, rb = (size_t)m * cfg->dim * 4;
    const size_t xd = align_up(xb, 256), rd = align_up(rb, 256);
    char *p = static_cast<char *>(io);
    void *x_dev = p, *xn_dev = p + xd;
    float *res_dev = reinterpret_cast<float *>(p + 2 * xd);
    int32_t *hdr_dev = reinterpret_cast<int32_t *>(p + 2 * xd + rd);
    const size_t hb = sizeof(int32_t) * header_words(m, cfg->topk);
    CUDA_OK(cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s));
    CUDA_OK(cudaMemcpyAsync(res_dev, residual_host, rb, cudaMemcpyHostToDevice, s));
    if ((rc = layer_step(*cfg, *layer, *arena, x_dev, res_dev, xn_dev, hdr_dev, m, ws, s)))
        return rc;
    CUDA_OK(cudaMemcpyAsync(residual_host, res_dev, rb, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaMemcpyAsync(x_next_host, xn_dev, xb, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaMemcpyAsync(header_host, hdr_dev, hb, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

int moe_slot_table_set(int32_t *table, int n_routed, const int32_t *triples, int n, uint32_t *status,
                       moe_stream_t stream)
{
    if (!table || n_routed < 1 || n_routed > MOE_MAX_ROUTED || n < 0 || (n > 0 && !triples))
        return fail(MOE_EINVAL, "moe_slot_table_set: bad arguments");
    if (n == 0)
        return MOE_OK;
    moe_slot_table_kernel<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(table, n_routed, triples, n, status);
    CUDA_OK(cudaGetLastError());
    return MOE_OK;
}

int moe_dedupe_triples(int32_t *t, int n, int *n_out)
{
    if (n < 0 || (n > 0 && !t) || !n_out)
        return fail(MOE_EINVAL, "moe_dedupe_triples: bad arguments");
    // keep the last triple of each (layer, expert); quadratic, fine for the
    // batch sizes a cache produces between two steps
    std::vector<int32_t> out;
    out.reserve((size_t)n * 3);
    for (int i = 0; i < n; ++i) {
        bool later = false;
        for (int j = i + 1; j < n && !later; ++j)
            later = t[3 * j] == t[3 * i] && t[3 * j + 1] == t[3 * i + 1];
        if (!later) {
            out.push_back(t[3 * i]);
            out.push_back(t[3 * i + 1]);
            out.push_back(t[3 * i + 2]);
        }
    }
    std::memcpy(t, out.data(), out.size() * sizeof(int32_t));
    *n_out = (int)(out.size() / 3);
    return MOE_OK;
}

int moe_parse_header(const moe_cfg *cfg, const int32_t *hdr, int m, int t, int32_t *status, int32_t *picks,
                     float *weights)
{
    if (!cfg || !hdr || t < 0 || t >= m || cfg->topk < 1)
        return fail(MOE_EINVAL, "moe_parse_header: bad arguments");
    const int k = cfg->topk;
    const int32_t *h = hdr + (size_t)t * (1 + 3 * k);
    for (int i = 0; i < k; ++i)
        if (h[1 + i] < 0 || h[1 + i] >= cfg->n_routed)
            return fail(MOE_EINVAL, "route header token %d: pick %d outside 0..%d", t, h[1 + i], cfg->n_routed - 1);
    if (status)
        *status = h[0];
    for (int i = 0; i < k; ++i) {
        if (picks)
            picks[i] = h[1 + i];
        if (weights)
            std::memcpy(&weights[i], &h[1 + k + i], 4);
    }
    return MOE_OK;
}

int moe_graph_snapshot_bytes(const moe_cfg *cfg, int m, int n_layers, size_t *bytes)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)))
        return rc;
    if (n_layers < 1 || !bytes)
        return fail(MOE_EINVAL, "moe_graph_snapshot_bytes: bad arguments");
    *bytes = snapshot_stride(*cfg, m) * (size_t)n_layers;
    return MOE_OK;
}

int moe_graph_create(const moe_cfg *cfg, const moe_layer *layers, int n_layers, const moe_arena *arena, int m,
                     void *x_a, void *x_b, float *residual, int32_t *headers, void *ws, void *snap, unsigned flags,
                     void **graph)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)) || (rc = check_arena(arena)))
        return rc;
    if (!layers || n_layers < 1 || !x_a || !x_b || !residual || !headers || !ws || !graph || m < 1)
        return fail(MOE_EINVAL, "moe_graph_create: bad arguments");
    if ((flags & MOE_GRAPH_SNAPSHOTS) && !snap)
        return fail(MOE_EINVAL, "moe_graph_create: MOE_GRAPH_SNAPSHOTS needs snapshot memory");
    for (int l = 0; l < n_layers; ++l)
        if ((rc = check_layer(*cfg, &layers[l])))
            return rc;
    DevInfo *I;
    if ((rc = dev_info(&I)))
        return rc;
    GraphObj *G = new GraphObj;
    G->cfg = *cfg;
    G->layers.assign(layers, layers + n_layers);
    G->arena = *arena;
    G->m = m;
    G->n_layers = n_layers;
    G->hw = header_words(m, cfg->topk);
    G->x_a = x_a;
    G->x_b = x_b;
    G->ws = ws;
    G->residual = residual;
    G->headers = headers;
    G->snap = (flags & MOE_GRAPH_SNAPSHOTS) ? static_cast<char *>(snap) : nullptr;
    G->snap_stride = snapshot_stride(*cfg, m);
    G->x_bytes = (size_t)m * cfg->dim * 2;
    G->res_bytes = (size_t)m * cfg->dim * 4;
    G->hdr_bytes = sizeof(int32_t) * (size_t)G->hw * n_layers;
    cudaError_t e = cudaSuccess;
    if (flags & MOE_GRAPH_TEST_FAIL_CAPTURE) {
        e = cudaErrorStreamCaptureUnsupported;  // as if the capture had failed
    } else {
        cudaStream_t cs;
        CUDA_OK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
        e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
        if (e == cudaSuccess) {
            rc = run_layers(*G, 0, cs);
            cudaGraph_t g = nullptr;
            cudaError_t e2 = cudaStreamEndCapture(cs, &g);
            if (rc == MOE_OK && e2 == cudaSuccess) {
                G->graph = g;
                e = cudaGraphInstantiate(&G->exec, g, 0);
            } else {
                if (g)
                    cudaGraphDestroy(g);
                e = e2 != cudaSuccess ? e2 : cudaErrorUnknown;
            }
        }
        cudaStreamDestroy(cs);
    }
    if (rc != MOE_OK || e != cudaSuccess) {
        if (G->exec)
            cudaGraphExecDestroy(G->exec);
        if (G->graph)
            cudaGraphDestroy(G->graph);
        G->exec = nullptr;
        G->graph = nullptr;
        if (e != cudaErrorStreamCaptureUnsupported || !(flags & MOE_GRAPH_TEST_FAIL_CAPTURE))
            cudaGetLastError();
        if (!(flags & MOE_GRAPH_EAGER_FALLBACK)) {
            delete G;
            if (rc != MOE_OK)
                return fail(MOE_ECAPTURE, "graph capture failed: %s", g_err);
            return fail(MOE_ECAPTURE, "graph capture failed: %s", cudaGetErrorString(e));
        }
        G->eager = true;  // graph mode off: every launch runs the layers eagerly
    }
    *graph = G;
    return MOE_OK;
}

int moe_graph_is_eager(void *graph, int *eager)
{
    if (!graph || !eager)
        return fail(MOE_EINVAL, "moe_graph_is_eager: bad arguments");
    *eager = static_cast<GraphObj *>(graph)->eager ? 1 : 0;
    return MOE_OK;
}

int moe_graph_rerun_from(void *graph, int layer, moe_stream_t stream)
{
    if (!graph)
        return fail(MOE_EINVAL, "graph is NULL");
    GraphObj *G = static_cast<GraphObj *>(graph);
    if (!G->snap || layer < 0 || layer >= G->n_layers)
        return fail(MOE_EINVAL, "moe_graph_rerun_from: no snapshots, or layer %d outside [0, %d)", layer, G->n_layers);
    const int rc = restore_snapshot(*G, layer, (cudaStream_t)stream);
    return rc ? rc : run_layers(*G, layer, (cudaStream_t)stream);
}

int moe_graph_launch(void *graph, moe_stream_t stream)
{
    if (!graph)
        return fail(MOE_EINVAL, "graph is NULL");
    GraphObj *G = static_cast<GraphObj *>(graph);
    if (G->eager)
        return run_layers(*G, 0, (cudaStream_t)stream);
    CUDA_OK(cudaGraphLaunch(G->exec, (cudaStream_t)stream));
    return MOE_OK;
}

int moe_graph_launch_host(void *graph, const void *x_host, const float *residual_host, void *x_out_host,
                          float *residual_out_host, int32_t *headers_host, moe_stream_t stream)
{
    if (!graph || !x_host || !residual_host || !x_out_host || !residual_out_host || !headers_host)
        return fail(MOE_EINVAL, "moe_graph_launch_host: a buffer is NULL");
    GraphObj *G = static_cast<GraphObj *>(graph);
    cudaStream_t s = (cudaStream_t)stream;
    CUDA_OK(cudaMemcpyAsync(G->x_a, x_host, G->x_bytes, cudaMemcpyHostToDevice, s));
    CUDA_OK(cudaMemcpyAsync(G->residual, residual_host, G->res_bytes, cudaMemcpyHostToDevice, s));
    if (G->eager) {
        const int rc = run_layers(*G, 0, s);
        if (rc)
            return rc;
    } else {
        CUDA_OK(cudaGraphLaunch(G->exec, s));
    }
    CUDA_OK(cudaMemcpyAsync(x_out_host, G->x_a, G->x_bytes, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaMemcpyAsync(residual_out_host, G->residual, G->res_bytes, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaMemcpyAsync(headers_host, G->headers, G->hdr_bytes, cudaMemcpyDeviceToHost, s));
    return MOE_OK;
}

int moe_layer_step_profiled(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena, const void *x,
                            float *residual, void *x_next, int32_t *header, int m, void *ws, moe_stream_t stream,
                            float *ms)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_m(cfg, m)) || (rc = check_arena(arena)) || (rc = check_layer(*cfg, layer)))
        return rc;
    if (m < 1 || !x || !residual || !x_next || !header || !ws || !ms || !aligned16(x))
        return fail(MOE_EINVAL, "moe_layer_step_profiled: bad arguments");
    thread_local cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
    thread_local int ev_dev = -1;
    int d = 0;
    CUDA_OK(cudaGetDevice(&d));
    if (ev_dev != d) {
        for (int i = 0; i < 4; ++i)
            CUDA_OK(cudaEventCreate(&ev[i]));
        ev_dev = d;
    }
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = layer_step(*cfg, *layer, *arena, x, residual, x_next, header, m, ws, s, ev)))
        return rc;
    CUDA_OK(cudaEventSynchronize(ev[3]));
    for (int i = 0; i < 3; ++i)
        CUDA_OK(cudaEventElapsedTime(&ms[i], ev[i], ev[i + 1]));
    return MOE_OK;
}

int moe_gemm_bf16(const void *a, const void *b, float *d, int M, int N, int K, int ldd, moe_stream_t stream)
{
    if (!a || !b || !d || M < 0 || N < 0 || K <= 0 || K % TC_KC || ldd < M || !aligned16(a) || !aligned16(b))
        return fail(MOE_EINVAL, "moe_gemm_bf16: bad arguments (K a positive multiple of 64, ldd >= M, 16-byte "
                                "aligned operands)");
    if (M == 0 || N == 0)
        return MOE_OK;
    DevInfo *I;
    int rc = dev_info(&I);
    if (rc)
        return rc;
    return gemm_bf16(a, b, d, M, N, K, ldd, nullptr, (cudaStream_t)stream, I->smem_optin, I->sms);
}

int moe_prefill_workspace_bytes(const moe_cfg *cfg, int m, size_t *bytes)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_prefill(cfg, m)))
        return rc;
    if (!bytes)
        return fail(MOE_EINVAL, "bytes is NULL");
    *bytes = pf_layout(*cfg, m).total;
    return MOE_OK;
}

}  // extern "C"

namespace {
static int prefill_step(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena, int64_t arena_slots,
                        const void *x, float *residual, void *x_next, int32_t *picks, float *weights, int m,
                        void *ws, size_t ws_bytes, moe_stream_t stream, cudaEvent_t *ev)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_prefill(cfg, m)) || (rc = check_arena(arena)) || (rc = check_layer(*cfg, layer)))
        return rc;
    if (layer->sh_w1 && layer->sh_format != MOE_SHARED_BF16)
        return fail(MOE_EUNSUPPORTED, "prefill: the shared expert must be bf16");
    if (m == 0)
        return MOE_OK;
    if (!x || !residual || !x_next || !picks || !weights || !ws || arena_slots < 1 || !aligned16(x))
        return fail(MOE_EINVAL, "moe_prefill_step: a buffer is NULL, arena_slots < 1 or x not 16-byte aligned");
    const PfLayout L = pf_layout(*cfg, m);
    if (ws_bytes < L.total)
        return fail(MOE_EINVAL, "moe_prefill_step: workspace of %zu bytes, %zu needed", ws_bytes, L.total);
    DevInfo *I;
    if ((rc = dev_info(&I)))
        return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const int n = cfg->n_routed, k = cfg->topk, dim = cfg->dim, inter = cfg->inter, P = L.P;
    char *w = static_cast<char *>(ws);
    float *logits = reinterpret_cast<float *>(w + L.logits), *scores = reinterpret_cast<float *>(w + L.scores);
    int32_t *flags = reinterpret_cast<int32_t *>(w + L.flags), *cnt = reinterpret_cast<int32_t *>(w + L.cnt);
    int32_t *off = reinterpret_cast<int32_t *>(w + L.off), *pair_tok = reinterpret_cast<int32_t *>(w + L.pair_tok);
    float *pair_w = reinterpret_cast<float *>(w + L.pair_w);
    int32_t *pick_pair = reinterpret_cast<int32_t *>(w + L.pick_pair);
    TcTask *tasks = reinterpret_cast<TcTask *>(w + L.tasks);
    int32_t *ntasks = reinterpret_cast<int32_t *>(w + L.ntasks);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + L.status);
    __half *xg = reinterpret_cast<__half *>(w + L.xg), *xg_lo = reinterpret_cast<__half *>(w + L.xg_lo);
    __half *hh = reinterpret_cast<__half *>(w + L.hh);
    float *g = reinterpret_cast<float *>(w + L.g), *u = reinterpret_cast<float *>(w + L.u);
    float *dw = reinterpret_cast<float *>(w + L.dw), *gs = reinterpret_cast<float *>(w + L.gs);
    float *us = reinterpret_cast<float *>(w + L.us), *sd = reinterpret_cast<float *>(w + L.sd);
    float *acc = reinterpret_cast<float *>(w + L.acc);
    uint16_t *hs = reinterpret_cast<uint16_t *>(w + L.hs);
    // stage boundaries for the profiled variant
    auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], s) : cudaSuccess; };
    CUDA_OK(cudaMemsetAsync(status, 0, 4, s));
    CUDA_OK(mark(0));
    // router logits [m, n] on tensor cores, the scores, each token's picks
    if ((rc = gemm_bf16(layer->router_w, x, logits, n, m, dim, n, status, s, I->smem_optin, I->sms)))
        return rc;
    CUDA_OK(mark(1));
    ScoreArgs sa{logits, scores, cfg->gate_temp, m * n};
    if ((rc = launch(moe_score_kernel, dim3((m * n + MOE_SCORES_PER_CTA - 1) / MOE_SCORES_PER_CTA), dim3(256), 0,
                     s, false, sa)))
        return rc;
    PTopArgs ta{logits, scores, layer->bias, picks, flags, weights, m, n, k, cfg->norm_topk_prob != 0,
                cfg->route_scale};
    moe_prefill_topk_kernel<<<(m + 7) / 8, 256, 0, s>>>(ta);
    CUDA_OK(cudaGetLastError());
    // pairs grouped by expert, the column tasks of the routed GEMMs
    PPlanArgs pa{picks, weights, layer->slot_row, m, n, k, cnt, off, pair_tok, pair_w, pick_pair, tasks, ntasks,
                 status};
    const size_t plan_smem = plan_smem_bytes(n, m * k);
    if (plan_smem > (size_t)I->smem_optin - 16384)
        return fail(MOE_EUNSUPPORTED, "prefill plan: %zu bytes of shared memory needed", plan_smem);
    moe_prefill_plan_kernel<<<1, 1024, plan_smem, s>>>(pa);
    CUDA_OK(cudaGetLastError());
    CUDA_OK(mark(2));
    // q8_1 of x, dequantised to fp16, gathered into pair order
    // (x is 16-byte aligned: checked above, the router GEMM's tensor map needs it)
    moe_prefill_xhat_gather_kernel<<<(unsigned)P, 256, 0, s>>>(static_cast<const uint16_t *>(x), pair_tok, P, dim, xg,
                                                               xg_lo);
    CUDA_OK(cudaGetLastError());
    CUDA_OK(mark(3));
    // routed gate and up: Q2_K rows (4 super-blocks a raw stage) x the groups' rows
    const char *ab = static_cast<const char *>(arena->base);
    const uint64_t q2row = (uint64_t)dim / 256 * MOE_Q2K_BYTES, q3row = (uint64_t)inter / 256 * MOE_Q3K_BYTES;
    CUtensorMap gmap, umap, dmap, xmap, xlmap, hmap;
    if ((rc = map_arena(&gmap, ab + arena->gate_off, q2row, inter, arena_slots, arena->slot_bytes,
                        tc_raw_blocks(1) * MOE_Q2K_BYTES)) ||
        (rc = map_arena(&umap, ab + arena->up_off, q2row, inter, arena_slots, arena->slot_bytes,
                        tc_raw_blocks(1) * MOE_Q2K_BYTES)) ||
        (rc = map_arena(&dmap, ab + arena->down_off, q3row, dim, arena_slots, arena->slot_bytes,
                        tc_raw_blocks(2) * MOE_Q3K_BYTES)) ||
        (rc = map_rows16(&xmap, false, xg, dim, P, (uint64_t)dim * 2, TC_BROWS)) ||
        (rc = map_rows16(&xlmap, false, xg_lo, dim, P, (uint64_t)dim * 2, TC_BROWS)) ||
        (rc = map_rows16(&hmap, false, hh, inter, P, (uint64_t)inter * 2, TC_BROWS)))
        return rc;
    TcArgs ga = tc_args(inter, P, dim, g, inter, status);
    ga.tasks = tasks;
    ga.ntasks = ntasks;
    ga.raw_row = tc_raw_blocks(1) * MOE_Q2K_BYTES;
    ga.rk = tc_raw_blocks(1) * 256;
    ga.S = 4;  // A stages in TMEM: 4 x 64 columns (hi and lo) beside two accumulators
    ga.SR = 2;
    ga.ksplit = 2;
    ga.raw_bytes = (uint32_t)(TC_M * ga.raw_row);
    if ((rc = launch_tc<1>(gmap, xmap, xlmap, ga, dim3(L.max_tasks, inter / TC_M), s, I->smem_optin)))
        return rc;
    CUDA_OK(mark(4));
    ga.out = u;
    if ((rc = launch_tc<1>(umap, xmap, xlmap, ga, dim3(L.max_tasks, inter / TC_M), s, I->smem_optin)))
        return rc;
    CUDA_OK(mark(5));
    // h = SwiGLU(g, u), its q8_1, dequantised to fp16
    const int nbh = P * inter / 32;
    moe_prefill_swiglu_kernel<<<(unsigned)(((size_t)nbh * 4 + 255) / 256), 256, 0, s>>>(g, u, nbh, cfg->swiglu_limit,
                                                                                     hh);
    CUDA_OK(cudaGetLastError());
    CUDA_OK(mark(6));
    // routed down: Q3_K rows (8 super-blocks a raw stage), times each pair's weight
    TcArgs da = tc_args(dim, P, inter, dw, dim, status);
    da.colw = pair_w;
    da.tasks = tasks;
    da.ntasks = ntasks;
    da.raw_row = tc_raw_blocks(2) * MOE_Q3K_BYTES;
    da.rk = tc_raw_blocks(2) * 256;
    da.S = 8;  // A stages in TMEM: 8 x 32 columns beside two accumulators
    da.SR = 1;
    da.ksplit = 2;
    da.raw_bytes = (uint32_t)(TC_M * da.raw_row);
    if ((rc = launch_tc<2>(dmap, hmap, hmap, da, dim3(L.max_tasks, dim / TC_M), s, I->smem_optin)))
        return rc;
    CUDA_OK(mark(7));
    // the bf16 shared expert as dense GEMMs
    const float *sdp = nullptr;
    if (layer->sh_w1) {
        if ((rc = gemm_bf16(layer->sh_w1, x, gs, inter, m, dim, inter, status, s, I->smem_optin, I->sms)) ||
            (rc = gemm_bf16(layer->sh_w3, x, us, inter, m, dim, inter, status, s, I->smem_optin, I->sms)))
            return rc;
        const size_t ns = (size_t)m * inter;
        moe_prefill_shared_swiglu_kernel<<<(unsigned)((ns + 255) / 256), 256, 0, s>>>(gs, us, ns, cfg->swiglu_limit,
                                                                                       hs);
        CUDA_OK(cudaGetLastError());
        if ((rc = gemm_bf16(layer->sh_w2, hs, sd, dim, m, inter, dim, status, s, I->smem_optin, I->sms)))
            return rc;
        sdp = sd;
    }
    CUDA_OK(mark(8));
    // acc (pairs in ascending expert id, then sd), residual, x_next
    const size_t nf = (size_t)m * dim;
    const bool v4 = ((reinterpret_cast<uintptr_t>(residual) | reinterpret_cast<uintptr_t>(acc) |
                      reinterpret_cast<uintptr_t>(dw) | reinterpret_cast<uintptr_t>(sdp)) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(x_next) & 7u) == 0;  // dim is a multiple of 4
    if (v4)
        moe_prefill_finish_kernel<4><<<(unsigned)((nf / 4 + 255) / 256), 256, 0, s>>>(
            dw, picks, pick_pair, k, sdp, acc, residual, static_cast<uint16_t *>(x_next), m, dim);
    else
        moe_prefill_finish_kernel<1><<<(unsigned)((nf + 255) / 256), 256, 0, s>>>(
            dw, picks, pick_pair, k, sdp, acc, residual, static_cast<uint16_t *>(x_next), m, dim);
    CUDA_OK(cudaGetLastError());
    CUDA_OK(mark(9));
    (void)cnt;
    (void)off;
    return MOE_OK;
}
}  // namespace

extern "C" {

int moe_prefill_step(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena, int64_t arena_slots,
                     const void *x, float *residual, void *x_next, int32_t *picks, float *weights, int m,
                     void *ws, size_t ws_bytes, moe_stream_t stream)
{
    return prefill_step(cfg, layer, arena, arena_slots, x, residual, x_next, picks, weights, m, ws, ws_bytes, stream,
                        nullptr);
}

int moe_prefill_step_profiled(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena,
                              int64_t arena_slots, const void *x, float *residual, void *x_next, int32_t *picks,
                              float *weights, int m, void *ws, size_t ws_bytes, moe_stream_t stream, float *ms)
{
    if (!ms)
        return fail(MOE_EINVAL, "moe_prefill_step_profiled: ms is NULL");
    thread_local cudaEvent_t ev[10] = {};
    thread_local int ev_dev = -1;
    int d = 0;
    CUDA_OK(cudaGetDevice(&d));
    if (ev_dev != d) {
        for (int i = 0; i < 10; ++i)
            CUDA_OK(cudaEventCreate(&ev[i]));
        ev_dev = d;
    }
    int rc = prefill_step(cfg, layer, arena, arena_slots, x, residual, x_next, picks, weights, m, ws, ws_bytes,
                          stream, ev);
    if (rc)
        return rc;
    if (m == 0) {
        for (int i = 0; i < 9; ++i)
            ms[i] = 0.0f;
        return MOE_OK;
    }
    CUDA_OK(cudaEventSynchronize(ev[9]));
    for (int i = 0; i < 9; ++i)
        CUDA_OK(cudaEventElapsedTime(&ms[i], ev[i], ev[i + 1]));
    return MOE_OK;
}

int moe_prefill_status(const moe_cfg *cfg, int m, void *ws, uint32_t *status_host, moe_stream_t stream)
{
    int rc = check_cfg(cfg);
    if (rc || (rc = check_prefill(cfg, m)))
        return rc;
    if (!ws || !status_host)
        return fail(MOE_EINVAL, "moe_prefill_status: bad arguments");
    const PfLayout L = pf_layout(*cfg, m);
    CUDA_OK(cudaMemcpyAsync(status_host, static_cast<char *>(ws) + L.status, 4, cudaMemcpyDeviceToHost,
                            (cudaStream_t)stream));
    CUDA_OK(cudaStreamSynchronize((cudaStream_t)stream));
    return MOE_OK;
}

int moe_cache_create(int n_layers, int n_routed, int n_slots, const moe_arena *arena, int32_t *slot_table_dev,
                     moe_expert_fetch_fn fetch, void *user, void **cache)
{
    if (n_layers < 1 || n_layers > MOE_SLOT_TABLE_LAYERS || n_routed < 1 || n_routed > MOE_MAX_ROUTED ||
        n_slots < 1 || !arena || !cache)
        return fail(MOE_EINVAL, "moe_cache_create: bad arguments");
    ExpertCache *C = new ExpertCache;
    C->init(n_layers, n_routed, n_slots, arena, slot_table_dev, fetch, user);
    if (slot_table_dev)
        CUDA_OK(cudaMemcpy(slot_table_dev, C->table.data(), sizeof(int32_t) * C->table.size(),
                           cudaMemcpyHostToDevice));
    *cache = C;
    return MOE_OK;
}

int moe_cache_destroy(void *cache)
{
    delete static_cast<ExpertCache *>(cache);
    return MOE_OK;
}

int moe_cache_ensure(void *cache, int layer, const int32_t *experts_host, int n, int *n_fetched, moe_stream_t stream)
{
    if (!cache)
        return fail(MOE_EINVAL, "cache is NULL");
    return cache_ensure(*static_cast<ExpertCache *>(cache), layer, experts_host, n, n_fetched, (cudaStream_t)stream);
}

int moe_cache_slot_of(void *cache, int layer, int expert, int32_t *slot)
{
    if (!cache || !slot)
        return fail(MOE_EINVAL, "moe_cache_slot_of: bad arguments");
    ExpertCache *C = static_cast<ExpertCache *>(cache);
    if (layer < 0 || layer >= C->n_layers || expert < 0 || expert >= C->n_routed)
        return fail(MOE_EINVAL, "moe_cache_slot_of: (%d, %d) outside the table", layer, expert);
    *slot = C->table[(size_t)layer * C->n_routed + expert];
    return MOE_OK;
}

int moe_cache_stats(void *cache, uint64_t *hits, uint64_t *misses, uint64_t *evictions)
{
    if (!cache)
        return fail(MOE_EINVAL, "cache is NULL");
    ExpertCache *C = static_cast<ExpertCache *>(cache);
    if (hits)
        *hits = C->hits;
    if (misses)
        *misses = C->misses;
    if (evictions)
        *evictions = C->evictions;
    return MOE_OK;
}

int moe_host_source_create(const void *const *images_host, int n_layers, int n_routed, uint64_t image_bytes,
                           void **source)
{
    if (!images_host || n_layers < 1 || n_routed < 1 || image_bytes == 0 || !source)
        return fail(MOE_EINVAL, "moe_host_source_create: bad arguments");
    HostSource *H = new HostSource;
    H->images.assign(images_host, images_host + (size_t)n_layers * n_routed);
    H->n_routed = n_routed;
    H->image_bytes = image_bytes;
    *source = H;
    return MOE_OK;
}

int moe_host_source_destroy(void *source)
{
    delete static_cast<HostSource *>(source);
    return MOE_OK;
}

int moe_fetch_host_images(void *source, int layer, int expert, void *slot_dev, uint64_t slot_bytes, moe_stream_t stream)
{
    HostSource *H = static_cast<HostSource *>(source);
    if (!H || !slot_dev || H->image_bytes > slot_bytes)
        return MOE_EINVAL;
    const void *img = H->images[(size_t)layer * H->n_routed + expert];
    if (!img)
        return MOE_EINVAL;
    return cudaMemcpyAsync(slot_dev, img, H->image_bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream) == cudaSuccess
               ? MOE_OK
               : MOE_ECUDA;
}

// the distinct picks of every token of one layer's header
static std::vector<int32_t> header_picks(const int32_t *h, int m, int k)
{
    std::vector<int32_t> v;
    for (int t = 0; t < m; ++t)
        for (int i = 0; i < k; ++i)
            v.push_back(h[(size_t)t * (1 + 3 * k) + 1 + i]);
    return v;
}

static bool header_miss(const int32_t *h, int m, int k)
{
    for (int t = 0; t < m; ++t)
        if (h[(size_t)t * (1 + 3 * k)] & MOE_HDR_MISS)
            return true;
    return false;
}

int moe_graph_step_cached(void *graph, void *cache, int32_t *headers_host, int *layers_rerun, moe_stream_t stream)
{
    if (!graph || !cache || !headers_host)
        return fail(MOE_EINVAL, "moe_graph_step_cached: bad arguments");
    GraphObj *G = static_cast<GraphObj *>(graph);
    ExpertCache *C = static_cast<ExpertCache *>(cache);
    if (!G->snap)
        return fail(MOE_EINVAL, "moe_graph_step_cached: the graph keeps no snapshots (MOE_GRAPH_SNAPSHOTS)");
    if (C->n_layers < G->n_layers || C->n_routed != G->cfg.n_routed)
        return fail(MOE_EINVAL, "moe_graph_step_cached: the cache covers %d layers of %d experts", C->n_layers,
                    C->n_routed);
    for (int l = 0; l < G->n_layers; ++l)
        if (!C->table_dev || G->layers[l].slot_row != C->table_dev + (size_t)l * C->n_routed)
            return fail(MOE_EINVAL, "moe_graph_step_cached: layer %d does not use row %d of the cache's table", l, l);
    cudaStream_t s = (cudaStream_t)stream;
    const int k = G->cfg.topk, m = G->m, hw = G->hw;
    int rc = moe_graph_launch(graph, stream);
    if (rc)
        return rc;
    CUDA_OK(cudaMemcpyAsync(headers_host, G->headers, G->hdr_bytes, cudaMemcpyDeviceToHost, s));
    CUDA_OK(cudaStreamSynchronize(s));
    int first = -1;
    for (int l = 0; l < G->n_layers && first < 0; ++l)
        if (header_miss(headers_host + (size_t)l * hw, m, k))
            first = l;
    if (layers_rerun)
        *layers_rerun = 0;
    if (first < 0)
        return MOE_OK;
    // from the first layer with a miss: its picks made resident, its input
    // back from the snapshot, then layer by layer eagerly, each layer's
    // misses fetched and the layer run again from its snapshot
    for (int l = first; l < G->n_layers; ++l) {
        int32_t *h = headers_host + (size_t)l * hw;
        for (int attempt = 0;; ++attempt) {
            if (attempt > 0 || l == first) {
                const std::vector<int32_t> p = header_picks(h, m, k);
                if ((rc = cache_ensure(*C, l, p.data(), (int)p.size(), nullptr, s)))
                    return rc;
                if ((rc = restore_snapshot(*G, l, s)))
                    return rc;
            }
            if (G->snap) {
                char *sn = G->snap + (size_t)l * G->snap_stride;
                CUDA_OK(cudaMemcpyAsync(sn, G->x_in(l), G->x_bytes, cudaMemcpyDeviceToDevice, s));
                CUDA_OK(cudaMemcpyAsync(sn + align_up(G->x_bytes, 256), G->residual, G->res_bytes,
                                        cudaMemcpyDeviceToDevice, s));
            }
            if ((rc = layer_step(G->cfg, G->layers[l], G->arena, G->x_in(l), G->residual, G->x_out(l),
                                 G->headers + (size_t)l * hw, m, G->ws, s)))
                return rc;
            CUDA_OK(cudaMemcpyAsync(h, G->headers + (size_t)l * hw, sizeof(int32_t) * hw, cudaMemcpyDeviceToHost, s));
            CUDA_OK(cudaStreamSynchronize(s));
            if (!header_miss(h, m, k))
                break;
            if (attempt >= 1)
                return fail(MOE_EUNSUPPORTED, "moe_graph_step_cached: layer %d still misses after a fetch", l);
        }
    }
    if (layers_rerun)
        *layers_rerun = G->n_layers - first;
    return MOE_OK;
}

int moe_graph_destroy(void *graph)
{
    if (!graph)
        return MOE_OK;
    GraphObj *G = static_cast<GraphObj *>(graph);
    if (G->exec)
        cudaGraphExecDestroy(G->exec);
    if (G->graph)
        cudaGraphDestroy(G->graph);
    delete G;
    return MOE_OK;
}

}  // extern "C"

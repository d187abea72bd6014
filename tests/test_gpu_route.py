"""GPU parity of the inputs, the q8_1 quantiser, the router logits, the
selection and the slot table, through the C ABI, against the CPU oracle.

Selection parity follows the design of page
spark_model/layers/moe_v41/device_route.rs, fn device_route_check: the host
chain runs on the same logits the device used, and the picks, the weight
bits, the plan weights and the pointer table must be equal.
"""
import numpy as np
import pytest
import torch

import moe_decode_quantized_gb300 as moe
import oracle
from moe_decode_quantized_gb300 import synth, synth_gpu
from moe_decode_quantized_gb300.workload import bf16_tensor, x_tensor

from helpers import (assert_logits_close, decode_cfg, gpu, new_header, ocfg, tiny_cfg, tiny_workload)
from moe_decode_quantized_gb300.workload import Workload

pytestmark = gpu


# ------------------------------------------------------------------ generator twin

@pytest.mark.parametrize("nblocks", [1, 7, 1000])
def test_synth_device_twin_matches_host_generator(nblocks):
    key = synth.tensor_key(3, 1, synth.T_GATE, 5)
    d = torch.zeros(nblocks * 84 + 16, dtype=torch.uint8, device="cuda")
    synth_gpu.q2k(d, nblocks, key)
    np.testing.assert_array_equal(d.cpu().numpy()[:nblocks * 84], synth.q2k_blocks(key, nblocks).ravel())
    assert not d[nblocks * 84:].any()
    d3 = torch.zeros(nblocks * 110 + 16, dtype=torch.uint8, device="cuda")
    synth_gpu.q3k(d3, nblocks, key)
    np.testing.assert_array_equal(d3.cpu().numpy()[:nblocks * 110], synth.q3k_blocks(key, nblocks).ravel())
    n = nblocks * 37 + 3
    b = torch.zeros(n, dtype=torch.int16, device="cuda")
    synth_gpu.normal_bf16(b, n, key, 0.02)
    np.testing.assert_array_equal(b.cpu().numpy().view(np.uint16), synth.normal_bf16(key, n, 0.02))
    f = torch.zeros(n, dtype=torch.float32, device="cuda")
    synth_gpu.uniform_f32(f, n, key, -0.1, 0.1)
    np.testing.assert_array_equal(f.cpu().numpy().view(np.uint32), synth.uniform_f32(key, n, -0.1, 0.1).view(np.uint32))


def test_decode_workload_matches_host_images():
    cfg = decode_cfg()
    wl = Workload(cfg, n_layers=1, seed=5, shared=True)
    for e in (0, 191, 383):
        off = e * wl.shape.slot_bytes
        dev = wl.arena_t[off:off + wl.shape.slot_bytes].cpu().numpy()
        host = wl.host_expert(0, e)
        for lo, n in ((wl.shape.gate_off, wl.shape.gate_bytes), (wl.shape.up_off, wl.shape.up_bytes),
                      (wl.shape.down_off, wl.shape.down_bytes)):
            np.testing.assert_array_equal(dev[lo:lo + n], host[lo:lo + n])
    np.testing.assert_array_equal(wl.router[0].cpu().numpy().view(np.uint16), wl.host_router(0))
    np.testing.assert_array_equal(wl.bias[0].cpu().numpy(), wl.host_bias(0))
    for dv, hv in zip(wl.sh[0], wl.host_shared(0)):
        np.testing.assert_array_equal(dv.cpu().numpy().view(np.uint16), hv)


# ------------------------------------------------------------------ q8_1

@pytest.mark.parametrize("m,dim", [(1, 256), (3, 4096), (8, 4096)])
def test_quantize_q8_1_is_bit_exact(m, dim):
    cfg = moe.Config(dim=dim, inter=256, n_routed=16, topk=2, max_tokens=m)
    x = synth.x_bf16(7, m, m, dim)
    x[0, :32] = 0                         # an all-zero block
    x[-1, 32:64] = 0x3F80                 # a constant block (all 1.0)
    xd = bf16_tensor(x, "cuda")
    out = torch.zeros(m * dim // 32 * 36, dtype=torch.uint8, device="cuda")
    moe.quantize_q8_1(cfg, xd, m, out)
    torch.cuda.synchronize()
    want = oracle.quant_q8_1((x.astype(np.uint32) << 16).view(np.float32))
    np.testing.assert_array_equal(out.cpu().numpy().reshape(-1, 36), want)


def test_swiglu_q8_against_oracle():
    cfg = moe.Config(dim=256, inter=2048, n_routed=16, topk=2, swiglu_limit=7.0)
    rng = np.random.default_rng(9)
    rows = 3
    g = (rng.standard_normal((rows, 2048)) * 4).astype(np.float32)
    u = (rng.standard_normal((rows, 2048)) * 4).astype(np.float32)
    g[0, :40] = np.linspace(-20, 20, 40)           # both sides of the clamp
    u[0, :40] = np.linspace(-20, 20, 40)
    gd, ud = torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda()
    h = torch.zeros_like(gd)
    hq = torch.zeros(rows * 2048 // 32 * 36, dtype=torch.uint8, device="cuda")
    moe.swiglu_q8(cfg, gd, ud, rows, h, hq)
    torch.cuda.synchronize()
    hv = h.cpu().numpy()
    ref = np.vectorize(lambda a, b: oracle.swiglu(a, b, 7.0))(g.astype(np.float64), u.astype(np.float64))
    assert np.abs(hv - ref).max() <= 4e-7 * max(1.0, np.abs(ref).max())
    # the q8_1 decisions are taken in f32 on the kernel's own h: bit-exact
    np.testing.assert_array_equal(hq.cpu().numpy().reshape(-1, 36), oracle.quant_q8_1(hv))


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("which,m", [("tiny", 1), ("decode", 1), ("decode", 8)])
def test_router_logits(which, m):
    cfg = tiny_cfg(m) if which == "tiny" else decode_cfg(m)
    seed = 21
    w = synth.router_bf16(seed, 0, cfg.n_routed, cfg.dim)
    x = synth.x_bf16(seed, 1, m, cfg.dim)
    logits = torch.zeros((m, cfg.n_routed), dtype=torch.float32, device="cuda")
    moe.router_logits(cfg, bf16_tensor(x, "cuda"), bf16_tensor(w, "cuda"), logits, m)
    torch.cuda.synchronize()
    assert_logits_close(logits.cpu().numpy(), oracle.router_logits(x, w))


# ------------------------------------------------------------------ selection

def _select(cfg, logits_np, bias_np, slot_row_np, m, arena):
    hdr = new_header(cfg, m)
    cap = m * cfg.topk
    pw = torch.zeros(cap, dtype=torch.float32, device="cuda")
    pr = torch.zeros(cap, dtype=torch.int32, device="cuda")
    ptrs = torch.zeros(3 * cap, dtype=torch.int64, device="cuda")
    moe.route_select(cfg, torch.from_numpy(logits_np).cuda(), torch.from_numpy(bias_np).cuda(),
                     torch.from_numpy(slot_row_np).cuda(), arena, m, hdr, pw, pr, ptrs)
    torch.cuda.synchronize()
    return hdr.cpu().numpy(), pw.cpu().numpy(), pr.cpu().numpy(), ptrs.cpu().numpy().view(np.uint64)


def _same_f32_bits(got, want):
    """Bit-identical f32, except that any NaN equals any NaN (payloads carry no meaning)."""
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    both_nan = np.isnan(got) & np.isnan(want)
    np.testing.assert_array_equal(np.where(both_nan, 0, got.view(np.uint32)),
                                  np.where(both_nan, 0, want.view(np.uint32)))


def _check_selection(cfg, logits, bias, slot_row, m, arena_tuple, hdr, pw, pr, ptrs):
    """The device header / plan / pointer table against the oracle's (selection
    and plan layout) on the same logits: every word the layout defines."""
    k, n = cfg.topk, cfg.n_routed
    picks, weights, _, flags = oracle.route(ocfg(cfg), logits, bias)
    rhdr, rpw, rpr, rptrs, ne = oracle.plan(picks[:m], weights[:m], flags[:m], slot_row, arena_tuple, n)
    hw, cap = 1 + 3 * k, m * k
    po = m * hw
    for t in range(m):
        row = hdr[t * hw:(t + 1) * hw]
        assert list(row[:1 + k]) == list(rhdr[t * hw:t * hw + 1 + k]), (t, row, rhdr[t * hw:(t + 1) * hw])
        _same_f32_bits(row[1 + k:1 + 2 * k].view(np.float32), rhdr[t * hw + 1 + k:t * hw + 1 + 2 * k].view(np.float32))
        assert list(row[1 + 2 * k:]) == list(rhdr[t * hw + 1 + 2 * k:(t + 1) * hw]), t
    assert int(hdr[po]) == ne
    assert list(hdr[po + 1:po + 2 + ne]) == list(rhdr[po + 1:po + 2 + ne])
    assert list(hdr[po + 2 + cap:po + 2 + cap + ne]) == list(rhdr[po + 2 + cap:po + 2 + cap + ne])
    assert list(pr[:cap]) == list(rpr)
    _same_f32_bits(pw[:cap], rpw)
    for off in (0, cap, 2 * cap):
        assert list(ptrs[off:off + ne]) == list(rptrs[off:off + ne])


def _arena(size=1 << 20):
    t = torch.zeros(size, dtype=torch.uint8, device="cuda")
    a = moe.Arena(t, 4096, 0, 1024, 2048)
    return t, a, (t.data_ptr(), 4096, 0, 1024, 2048)


# ------------------------------------------------------------------ the score

def _oracle_scores(logits, temp):
    """The oracle's scores (the f32 chain, each step rounded from long double)
    and the mask of scores with a step within 2^-56 of an f32 midpoint."""
    n = 1024
    lg = np.asarray(logits, np.float32)
    pad = (-len(lg)) % n
    rows = np.concatenate([lg, np.zeros(pad, np.float32)]).reshape(-1, n)
    c = oracle.cfg(256, 256, n, 1, True, temp, 1.0, 0.0)
    _, _, scores, flags = oracle.route(c, rows, np.zeros(n, np.float32))
    near = np.zeros(rows.shape, bool)
    for r in np.nonzero(flags & 4)[0]:  # rows holding a near-midpoint score
        for j in range(n):
            near[r, j] = oracle.score(float(rows[r, j]), temp)[1]
    return scores.ravel()[:len(lg)], near.ravel()[:len(lg)]


@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_route_scores_are_correctly_rounded(temp):
    """Page moe_v41.rs fn softplus / fn route_from_logits: the score is the
    f32 chain sqrt(ln_1p(exp(l / temp))), each step correctly rounded; the
    device's float-float decisions (double and double-double precision near
    midpoints) equal the oracle's long-double roundings bit for bit."""
    rng = np.random.default_rng(11)
    parts = [rng.normal(0.0, 3.0, 1 << 19),
             rng.uniform(-60.0, 30.0, 1 << 18),
             rng.uniform(19.9, 20.1, 1 << 14) * temp,       # around the x > 20 cut
             rng.uniform(-17.6, -17.0, 1 << 14) * temp,     # e around 2^-25: ln(1 + e) rounds to e below
             rng.uniform(-104.5, -86.0, 1 << 16) * temp,    # e^t subnormal, and rounding to 0 below -103.97
             rng.uniform(-175.0, -40.0, 1 << 15) * temp,
             rng.uniform(-1.0, 1.0, 1 << 14) * 2.0 ** -20,  # e near 1
             rng.normal(0.0, 1e-3, 1 << 14),
             np.array([0.0, -0.0, 20.0 * temp, -104.0 * temp, -103.97 * temp, 1e-30, -1e-30, 88.0, -88.0,
                       300.0, -300.0, np.inf, -np.inf])]
    lg = np.concatenate(parts).astype(np.float32)
    d_in = torch.from_numpy(lg).cuda()
    d_out = torch.full_like(d_in, float("nan"))
    cfg = tiny_cfg(1, gate_temp=temp)
    moe.route_scores(cfg, d_in, d_out, len(lg))
    torch.cuda.synchronize()
    got = d_out.cpu().numpy()
    ref, near = _oracle_scores(lg, temp)
    ok = (got.view(np.uint32) == ref.view(np.uint32)) | near
    bad = np.nonzero(~ok)[0]
    assert len(bad) == 0, [(float(lg[i]), float(got[i]), float(ref[i])) for i in bad[:5]]
    assert near.sum() < 50


@pytest.mark.parametrize("case", ["tiny", "decode_m1", "decode_m8", "tie_m8", "no_norm", "top1",
                                  "temp", "wide_bias"])
def test_route_select_bit_exact(case):
    m = 8 if case in ("decode_m8", "tie_m8") else 1
    kw = {}
    if case == "no_norm":
        kw = dict(norm_topk_prob=False)
    if case == "top1":
        kw = dict(topk=1)
    if case == "temp":
        kw = dict(gate_temp=0.7)
    cfg = tiny_cfg(m) if case == "tiny" else decode_cfg(m, **kw)
    seed = 31 + len(case)
    n = cfg.n_routed
    logits = synth.normal_f32(synth.tensor_key(seed, 0, synth.T_LOGITS), m * n, 1.3).reshape(m, n)
    bias = synth.bias_f32(seed, 0, n, *((-1.0, 1.0) if case == "wide_bias" else (-0.1, 0.1)))
    if case == "tie_m8":
        logits = synth.tie_logits(seed, 0, m, n)
        bias = synth.round_to_grid(bias)
    slot_row = np.arange(n, dtype=np.int32)[::-1].copy()
    t, arena, at = _arena()
    hdr, pw, pr, ptrs = _select(cfg, logits, bias, slot_row, m, arena)
    _check_selection(cfg, logits, bias, slot_row, m, at, hdr, pw, pr, ptrs)


def test_route_select_ties_everywhere():
    """All logits equal and bias on a coarse grid: the picks are the lowest ids of the
    best bias class, in id order."""
    cfg = decode_cfg(2)
    n = cfg.n_routed
    logits = np.zeros((2, n), np.float32)
    logits[1] = 0.5
    bias = np.zeros(n, np.float32)
    bias[100:110] = 0.0625
    slot_row = np.arange(n, dtype=np.int32)
    t, arena, at = _arena()
    hdr, pw, pr, ptrs = _select(cfg, logits, bias, slot_row, 2, arena)
    _check_selection(cfg, logits, bias, slot_row, 2, at, hdr, pw, pr, ptrs)
    assert list(hdr[1:7]) == [100, 101, 102, 103, 104, 105]


def test_route_select_miss_and_nonfinite_flags():
    cfg = decode_cfg(3)
    n = cfg.n_routed
    logits = synth.normal_f32(synth.tensor_key(41, 0, synth.T_LOGITS), 3 * n, 1.3).reshape(3, n)
    bias = synth.bias_f32(41, 0, n)
    logits[1, 17] = np.nan
    logits[1, 18] = np.inf
    logits[2, :] = np.nan
    logits[2, 5] = 2.0
    logits[2, 9] = -np.inf
    picks0, _, _, _ = oracle.route(ocfg(cfg), logits[:1], bias)
    slot_row = np.arange(n, dtype=np.int32)
    slot_row[picks0[0][2]] = -1                 # token 0: one pick not resident
    t, arena, at = _arena()
    hdr, pw, pr, ptrs = _select(cfg, logits, bias, slot_row, 3, arena)
    _check_selection(cfg, logits, bias, slot_row, 3, at, hdr, pw, pr, ptrs)
    hw = 1 + 3 * cfg.topk
    assert hdr[0] & moe.MOE_HDR_MISS
    assert hdr[hw] & moe.MOE_HDR_NONFINITE and hdr[2 * hw] & moe.MOE_HDR_NONFINITE
    assert hdr[hw + 1] == 18                    # +inf key ranks first


def test_router_then_select_in_one_launch_matches_separate_calls():
    """The layer step's fused router + last-CTA selection writes the same header as
    moe_router_logits followed by moe_route_select."""
    cfg = decode_cfg(8)
    wl = Workload(cfg, n_layers=1, seed=51, shared=False, fill_experts=False)
    m = 8
    x = x_tensor(51, 0, m, cfg.dim)
    logits = torch.zeros((m, cfg.n_routed), dtype=torch.float32, device="cuda")
    moe.router_logits(cfg, x, wl.router[0], logits, m)
    hdr_a = new_header(cfg, m)
    cap = m * cfg.topk
    pw = torch.zeros(cap, dtype=torch.float32, device="cuda")
    pr = torch.zeros(cap, dtype=torch.int32, device="cuda")
    ptrs = torch.zeros(3 * cap, dtype=torch.int64, device="cuda")
    moe.route_select(cfg, logits, wl.bias[0], wl.slot_table[0], wl.arena, m, hdr_a, pw, pr, ptrs)
    res = torch.zeros((m, cfg.dim), dtype=torch.float32, device="cuda")
    xn = torch.empty_like(x)
    hdr_b = new_header(cfg, m)
    # experts are not filled: only the routing outputs are compared here
    moe.layer_step(cfg, wl.layer(0), wl.arena, x, res, xn, hdr_b, m, wl.ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hdr_a.cpu().numpy(), hdr_b.cpu().numpy())
    v = moe.workspace_view(cfg, wl.ws)
    off = v["logits"] - wl.ws.data_ptr()
    ws_logits = wl.ws[off:off + 4 * m * cfg.n_routed].view(torch.float32).reshape(m, cfg.n_routed)
    np.testing.assert_array_equal(ws_logits.cpu().numpy(), logits.cpu().numpy())
    assert moe.read_status(wl.ws) == 0


def test_slot_table_set():
    n = 384
    table = torch.full((moe.SLOT_TABLE_LAYERS, n), -1, dtype=torch.int32, device="cuda")
    trip = np.array([[0, 1, 10], [3, 383, 7], [63, 0, 5], [0, 1, 11], [64, 0, 1], [2, 384, 1]], np.int32)
    trip = moe.dedupe_triples(trip)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    td = torch.from_numpy(trip).cuda()
    moe.slot_table_set(table, n, td, trip.shape[0], status)
    torch.cuda.synchronize()
    t = table.cpu().numpy()
    assert t[0, 1] == 11 and t[3, 383] == 7 and t[63, 0] == 5
    assert (t != -1).sum() == 3
    assert status.item() & moe.MOE_WS_TRIPLE

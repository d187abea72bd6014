"""GPU parity of the expert GEMVs and the whole layer step, through the C ABI,
against the CPU oracle on the same seeded inputs.

Page spark_model/layers/moe_v41.rs (module doc, fn shared_side): routed
experts as K-quant GEMVs on raw Q2_K / Q3_K blocks with a q8_1 activation and
clamped SwiGLU, the bf16 shared expert added after them, the residual.
"""
import numpy as np
import pytest
import torch

import moe_decode_quantized_gb300 as moe
import oracle
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import Workload, bf16_tensor, x_tensor

from helpers import (GU_RTOL, OUT_RTOL, THREADS, bf16_vals, compare_layer as _compare_layer, decode_cfg,
                     expert_image, gpu, near_tie, new_header, ocfg, rel_inf, run_layer as _run_layer, tiny_cfg,
                     tiny_workload, ws_view as _view)

pytestmark = gpu


@pytest.fixture(scope="module")
def decode_wl():
    cfg = decode_cfg(8)
    wl = Workload(cfg, n_layers=1, seed=1, shared=True)
    torch.cuda.synchronize()
    yield wl
    del wl
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ tiny layer

@pytest.mark.parametrize("m", [1, 2])
def test_tiny_layer_step(m):
    cfg = tiny_cfg(m)
    wl = tiny_workload(cfg, seed=0)
    x_bits = synth.x_bf16(0, 0, m, cfg.dim)
    x = bf16_tensor(x_bits, "cuda")
    res, xn, hdr = _run_layer(wl, cfg, 0, x, m)
    _compare_layer(wl, cfg, x_bits, m, res, xn, hdr)


def test_tiny_expert_intermediates():
    """g, u against the oracle's exact dots; down against the oracle fed the same h."""
    cfg = tiny_cfg(1)
    wl = tiny_workload(cfg, seed=2)
    x_bits = synth.x_bf16(2, 0, 1, cfg.dim)
    res, xn, hdr = _run_layer(wl, cfg, 0, bf16_tensor(x_bits, "cuda"), 1)
    h = hdr.cpu().numpy()
    k = cfg.topk
    po = 1 + 3 * k
    ne = int(h[po])
    plan = list(h[po + 2 + k:po + 2 + k + ne])
    g = _view(wl, cfg, "g", k * cfg.inter).reshape(k, cfg.inter)
    u = _view(wl, cfg, "u", k * cfg.inter).reshape(k, cfg.inter)
    dn = _view(wl, cfg, "down", k * cfg.dim).reshape(k, cfg.dim)
    xq = oracle.quant_q8_1(bf16_vals(x_bits[0]))
    shp = wl.shape
    for p, e in enumerate(plan):
        img = expert_image(wl, 0, int(e))
        ref = oracle.expert_token(ocfg(cfg), img[shp.gate_off:], img[shp.up_off:], img[shp.down_off:], xq)
        assert rel_inf(g[p], ref["g"]) <= GU_RTOL
        assert rel_inf(u[p], ref["u"]) <= GU_RTOL
        assert rel_inf(dn[p], ref["down"]) <= OUT_RTOL


def test_tiny_layer_without_renorm_and_top1():
    for kw in (dict(norm_topk_prob=False), dict(topk=1)):
        cfg = tiny_cfg(1, **kw)
        wl = tiny_workload(cfg, seed=3)
        x_bits = synth.x_bf16(3, 0, 1, cfg.dim)
        res, xn, hdr = _run_layer(wl, cfg, 0, bf16_tensor(x_bits, "cuda"), 1)
        _compare_layer(wl, cfg, x_bits, 1, res, xn, hdr)


# ------------------------------------------------------------------ decode layer (384 x 6, shared)

def test_decode_layer_step_m1(decode_wl):
    cfg = decode_cfg(1)
    cfg.max_tokens = decode_wl.cfg.max_tokens
    for batch in range(2):
        x_bits = synth.x_bf16(1, 100 + batch, 1, cfg.dim)
        res0 = (synth.normal_f32(synth.tensor_key(1, batch, synth.T_F32), cfg.dim, 0.5)
                .reshape(1, cfg.dim))
        res = torch.from_numpy(res0.copy()).cuda()
        res, xn, hdr = _run_layer(decode_wl, cfg, 0, bf16_tensor(x_bits, "cuda"), 1, res)
        _compare_layer(decode_wl, cfg, x_bits, 1, res, xn, hdr, residual0=res0)


def test_decode_expert_intermediates(decode_wl):
    cfg = decode_cfg(1)
    cfg.max_tokens = decode_wl.cfg.max_tokens
    x_bits = synth.x_bf16(1, 7, 1, cfg.dim)
    res, xn, hdr = _run_layer(decode_wl, cfg, 0, bf16_tensor(x_bits, "cuda"), 1)
    h = hdr.cpu().numpy()
    k = cfg.topk
    po = 1 + 3 * k
    plan = list(h[po + 2 + k:po + 2 + 2 * k])
    g = _view(decode_wl, cfg, "g", k * cfg.inter).reshape(k, cfg.inter)
    u = _view(decode_wl, cfg, "u", k * cfg.inter).reshape(k, cfg.inter)
    dn = _view(decode_wl, cfg, "down", k * cfg.dim).reshape(k, cfg.dim)
    xq = oracle.quant_q8_1(bf16_vals(x_bits[0]))
    shp = decode_wl.shape
    for p in (0, k - 1):
        img = decode_wl.host_expert(0, int(plan[p]))
        ref = oracle.expert_token(ocfg(cfg), img[shp.gate_off:], img[shp.up_off:], img[shp.down_off:], xq,
                                  threads=THREADS)
        assert rel_inf(g[p], ref["g"]) <= GU_RTOL
        assert rel_inf(u[p], ref["u"]) <= GU_RTOL
        assert rel_inf(dn[p], ref["down"]) <= OUT_RTOL
    gs = _view(decode_wl, cfg, "gs", cfg.inter)
    sd = _view(decode_wl, cfg, "sd", cfg.dim)
    sref = oracle.shared_token(ocfg(cfg), *decode_wl.host_shared(0), x_bits[0], threads=THREADS)
    assert rel_inf(gs, sref["gs"]) <= GU_RTOL
    assert rel_inf(sd, sref["sd"]) <= OUT_RTOL


def test_decode_small_batch_m8(decode_wl):
    cfg = decode_wl.cfg
    m = 8
    x_bits = synth.x_bf16(1, 200, m, cfg.dim)
    res, xn, hdr = _run_layer(decode_wl, cfg, 0, bf16_tensor(x_bits, "cuda"), m)
    _compare_layer(decode_wl, cfg, x_bits, m, res, xn, hdr)


def test_batch_invariance_and_determinism(decode_wl):
    """Row t of the m = 8 step equals the m = 1 step on x_t, bit for bit; repeated
    runs give identical bytes."""
    cfg = decode_wl.cfg
    m = 8
    x_bits = synth.x_bf16(1, 300, m, cfg.dim)
    x = bf16_tensor(x_bits, "cuda")
    res8, xn8, hdr8 = _run_layer(decode_wl, cfg, 0, x, m)
    res8b, xn8b, hdr8b = _run_layer(decode_wl, cfg, 0, x, m)
    assert torch.equal(res8, res8b) and torch.equal(xn8, xn8b) and torch.equal(hdr8, hdr8b)
    h8 = hdr8.cpu().numpy()
    for t in range(m):
        r1, x1, h1 = _run_layer(decode_wl, cfg, 0, x[t:t + 1].contiguous(), 1)
        assert torch.equal(r1[0], res8[t])
        assert torch.equal(x1[0], xn8[t])
        hw = 1 + 3 * cfg.topk
        np.testing.assert_array_equal(h1.cpu().numpy()[:hw], h8[t * hw:(t + 1) * hw])


def test_expert_step_routed_only(decode_wl):
    """moe_route_select + moe_expert_step: acc = the routed sum alone."""
    cfg = decode_wl.cfg
    m = 2
    x_bits = synth.x_bf16(1, 400, m, cfg.dim)
    x = bf16_tensor(x_bits, "cuda")
    logits = torch.zeros((m, cfg.n_routed), dtype=torch.float32, device="cuda")
    moe.router_logits(cfg, x, decode_wl.router[0], logits, m)
    hdr = new_header(cfg, m)
    cap = m * cfg.topk
    pw = torch.zeros(cap, dtype=torch.float32, device="cuda")
    pr = torch.zeros(cap, dtype=torch.int32, device="cuda")
    ptrs = torch.zeros(3 * cap, dtype=torch.int64, device="cuda")
    moe.route_select(cfg, logits, decode_wl.bias[0], decode_wl.slot_table[0], decode_wl.arena, m, hdr, pw,
                     pr, ptrs)
    acc = torch.zeros((m, cfg.dim), dtype=torch.float32, device="cuda")
    moe.expert_step(cfg, x, ptrs, pw, pr, hdr, m, acc, decode_wl.ws)
    torch.cuda.synchronize()
    assert moe.read_status(decode_wl.ws) == 0
    oc = ocfg(cfg)
    ref = oracle.layer(oc, x_bits, decode_wl.host_router(0), decode_wl.host_bias(0),
                       {int(e): decode_wl.host_expert(0, int(e))
                        for e in np.unique(oracle.route(oc, logits.cpu().numpy(), decode_wl.host_bias(0))[0])},
                       (decode_wl.shape.gate_off, decode_wl.shape.up_off, decode_wl.shape.down_off), None,
                       threads=THREADS)
    a = acc.cpu().numpy()
    for t in range(m):
        if not near_tie(cfg, ref["logits"], decode_wl.host_bias(0), t):
            assert rel_inf(a[t], ref["acc"][t]) <= OUT_RTOL


def test_host_buffer_entry_point_matches_device_path(decode_wl):
    cfg = decode_wl.cfg
    m = 2
    x_bits = synth.x_bf16(1, 500, m, cfg.dim)
    res0 = np.full((m, cfg.dim), 0.125, np.float32)
    # device path
    r_dev, xn_dev, h_dev = _run_layer(decode_wl, cfg, 0, bf16_tensor(x_bits, "cuda"), m,
                                      torch.from_numpy(res0.copy()).cuda())
    # host path
    io = torch.empty(moe.host_io_bytes(cfg, m), dtype=torch.uint8, device="cuda")
    xh = torch.from_numpy(x_bits.view(np.int16).copy()).pin_memory()
    rh = torch.from_numpy(res0.copy()).pin_memory()
    xnh = torch.zeros((m, cfg.dim), dtype=torch.int16).pin_memory()
    hh = torch.zeros(moe.header_words(cfg, m), dtype=torch.int32).pin_memory()
    moe.layer_step_host(cfg, decode_wl.layer(0), decode_wl.arena, xh, rh, xnh, hh, m, io, decode_wl.ws)
    torch.cuda.synchronize()
    assert torch.equal(rh, r_dev.cpu())
    assert torch.equal(xnh, xn_dev.cpu())
    assert torch.equal(hh, h_dev.cpu())


def test_miss_flag_points_absent_experts_at_slot_zero():
    """A slot-table entry of -1: the header flags the miss and the pointers use slot 0
    (page spark_model/layers/moe_v41/device_route.rs, module doc)."""
    cfg = tiny_cfg(1)
    wl = tiny_workload(cfg, seed=4)
    x_bits = synth.x_bf16(4, 0, 1, cfg.dim)
    x = bf16_tensor(x_bits, "cuda")
    _, _, hdr = _run_layer(wl, cfg, 0, x, 1)
    picks = moe.parse_header(cfg, hdr.cpu().numpy(), 1, 0)[1]
    gone = int(picks[0])
    wl.slot_table[0, gone] = -1
    res, xn, hdr2 = _run_layer(wl, cfg, 0, x, 1)
    h2 = hdr2.cpu().numpy()
    assert h2[0] & moe.MOE_HDR_MISS
    # the absent expert's compute used slot 0 (expert 0's blocks): compare with the
    # oracle given that substitution
    imgs = {int(e): expert_image(wl, 0, int(e)) for e in picks}
    imgs[gone] = expert_image(wl, 0, 0)
    ref = oracle.layer(ocfg(cfg), x_bits, wl.host_router(0), wl.host_bias(0), imgs,
                       (wl.shape.gate_off, wl.shape.up_off, wl.shape.down_off))
    assert rel_inf(res.cpu().numpy(), ref["acc"]) <= OUT_RTOL


def test_empty_batch_is_a_no_op(decode_wl):
    cfg = decode_wl.cfg
    x = torch.zeros((1, cfg.dim), dtype=torch.int16, device="cuda")
    res = torch.full((1, cfg.dim), 3.0, device="cuda")
    xn = torch.zeros_like(x)
    hdr = new_header(cfg, 1)
    moe.layer_step(cfg, decode_wl.layer(0), decode_wl.arena, x, res, xn, hdr, 0, decode_wl.ws)
    torch.cuda.synchronize()
    assert torch.all(res == 3.0) and not hdr.any()


def test_invalid_arguments_are_rejected_before_launch(decode_wl):
    cfg = decode_wl.cfg
    x = torch.zeros((1, cfg.dim), dtype=torch.int16, device="cuda")
    res = torch.zeros((1, cfg.dim), device="cuda")
    hdr = new_header(cfg, 1)
    with pytest.raises(moe.MoeError) as e:
        moe.layer_step(cfg, decode_wl.layer(0), decode_wl.arena, x, res, x, hdr, 9, decode_wl.ws)
    assert e.value.code == -1
    bad = moe.Arena(decode_wl.arena_t.data_ptr() + 4, decode_wl.arena.slot_bytes, 0, 0, 0)
    with pytest.raises(moe.MoeError):
        moe.layer_step(cfg, decode_wl.layer(0), bad, x, res, x, hdr, 1, decode_wl.ws)


# ------------------------------------------------------------------ K-quant shared expert

@pytest.mark.parametrize("m", [1, 2, 3])
def test_tiny_layer_kquant_shared(m):
    """Page moe_v41.rs MoeV41LayerWeights: the shared w1, w3 as Q2_K and w2 as
    Q3_K blocks on the routed experts' kernels (struct MoeV41 sh_q8: its own
    q8_1 of the SwiGLU output), added after the routed sum."""
    cfg = tiny_cfg(m)
    wl = tiny_workload(cfg, seed=60 + m, shared=True, shared_kquant=True)
    x_bits = synth.x_bf16(60 + m, 0, m, cfg.dim)
    res, xn, hdr = _run_layer(wl, cfg, 0, bf16_tensor(x_bits, "cuda"), m)
    _compare_layer(wl, cfg, x_bits, m, res, xn, hdr)
    # the shared expert's own intermediates against the oracle's routed-expert math
    gs = _view(wl, cfg, "gs", m * cfg.inter).reshape(m, cfg.inter)
    sd = _view(wl, cfg, "sd", m * cfg.dim).reshape(m, cfg.dim)
    w1, w3, w2 = wl.host_shared(0)
    for t in range(m):
        xq = oracle.quant_q8_1(bf16_vals(x_bits[t]))
        ref = oracle.expert_token(ocfg(cfg), w1, w3, w2, xq)
        assert rel_inf(gs[t], ref["g"]) <= GU_RTOL
        assert rel_inf(sd[t], ref["down"]) <= OUT_RTOL


@pytest.mark.parametrize("m", [1, 8])
def test_decode_layer_kquant_shared(m):
    cfg = decode_cfg(m)
    wl = Workload(cfg, n_layers=1, seed=64, shared=True, shared_kquant=True)
    x_bits = synth.x_bf16(64, 1, m, cfg.dim)
    res, xn, hdr = _run_layer(wl, cfg, 0, bf16_tensor(x_bits, "cuda"), m)
    _compare_layer(wl, cfg, x_bits, m, res, xn, hdr)
    del wl
    torch.cuda.empty_cache()

"""Pins of the oracle's expert, shared-expert and layer composition (no GPU).

Page spark_model/layers/moe_v41.rs (module doc, MoeV41Cfg, fn shared_side)
and page spark_model/layers/moe_v41/device_route.rs (plan in ascending id).
The dense reference below dequantises whole matrices with the pinned block
decoders and multiplies with numpy's matmul, so an indexing mistake in the
oracle's GEMV loops (row stride, block order, transposed operand) fails here.
"""
import math

import numpy as np
import pytest

import oracle
from moe_decode_quantized_gb300 import synth


def _bf16_vals(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# Clamped SwiGLU, h = silu(min(g, L)) * clamp(u, -L, L), silu(z) = z / (1 + e^-z),
# no clamp for L <= 0 (page moe_v41.rs, MoeV41Cfg swiglu_limit). Values worked
# by hand from e^-1 = 0.36787944117144232160, e = 2.71828182845904523536,
# e^-2 = 0.13533528323661269189, e^-7 = 0.00091188196555451621,
# e^-10 = 0.00004539992976248485, e^-3 = 0.04978706836786394298:
SWIGLU_CASES = [
    # g, u, L, h
    (1.0, 1.0, 7.0, 0.73105857863000487925),       # 1 / (1 + e^-1)
    (-1.0, 2.0, 7.0, -0.53788284273999024150),     # -2 / (1 + e)
    (10.0, 3.0, 7.0, 20.980867924917586447),       # g clamped to 7: 3 * 7 / (1 + e^-7)
    (7.0, 7.0, 7.0, 48.955358491474368377),        # g and u at the limit: 7 * 7 / (1 + e^-7)
    (2.0, 9.0, 7.0, 12.331159091690354217),        # u clamped to +7: 7 * 2 / (1 + e^-2)
    (2.0, -9.0, 7.0, -12.331159091690354217),      # u clamped to -7
    (10.0, 3.0, 0.0, 29.998638063938926968),       # L = 0: no clamp, 3 * 10 / (1 + e^-10)
    (10.0, 3.0, -1.0, 29.998638063938926968),      # L < 0: no clamp
    (-30.0, 2.0, 7.0, -5.6145737813035793723e-12),  # g below -L is not clamped: 2 * -30 / (1 + e^30)
    (0.0, 5.0, 7.0, 0.0),
    (3.0, -20.0, 1.5, -1.8395425714356982341),     # both clamped: -1.5 * 1.5 / (1 + e^-1.5)
]


@pytest.mark.parametrize("g,u,limit,h", SWIGLU_CASES)
def test_swiglu_hand_worked_values(g, u, limit, h):
    assert oracle.swiglu(g, u, limit) == pytest.approx(h, rel=1e-14, abs=1e-300)


def test_swiglu_clamp_bounds():
    """With L >= 1, |h| <= L^2 (silu(z) <= z for z > 0, |silu(z)| < 0.28 for
    z < 0); without a clamp h grows with g u."""
    rng = np.random.default_rng(30)
    for g, u in rng.standard_normal((400, 2)) * 12:
        assert abs(oracle.swiglu(g, u, 7.0)) <= 49.0
        assert abs(oracle.swiglu(g, u, 1.5)) <= 2.25
    assert oracle.swiglu(40.0, 40.0, 0.0) > 1500.0


def _dense(blocks, rows, nb, q3):
    dq = oracle.dequant_q3k if q3 else oracle.dequant_q2k
    return dq(blocks.reshape(rows * nb, -1)).reshape(rows, nb * 256)


@pytest.mark.parametrize("dim,inter", [(256, 256), (512, 768)])
def test_expert_chain_against_dense_matmul(dim, inter):
    c = oracle.cfg(dim, inter, 8, 2)
    shp = synth.LayerShape(dim, inter, 8)
    img = synth.expert_bytes(5, 0, 3, shp)
    gate = img[shp.gate_off:shp.gate_off + shp.gate_bytes]
    up = img[shp.up_off:shp.up_off + shp.up_bytes]
    down = img[shp.down_off:shp.down_off + shp.down_bytes]
    x = _bf16_vals(synth.x_bf16(5, 0, 1, dim)[0]).astype(np.float32)
    xq = oracle.quant_q8_1(x)
    out = oracle.expert_token(c, gate, up, down, xq)
    xv = oracle.dequant_q8_1(xq).ravel()
    Wg = _dense(gate, inter, dim // 256, False)
    Wu = _dense(up, inter, dim // 256, False)
    Wd = _dense(down, dim, inter // 256, True)
    g = Wg @ xv
    u = Wu @ xv
    np.testing.assert_allclose(out["g"], g.astype(np.float32), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(out["u"], u.astype(np.float32), rtol=1e-6, atol=1e-6)
    h = np.array([oracle.swiglu(a, b, 7.0) for a, b in zip(g, u)], np.float32)
    np.testing.assert_array_equal(out["h"], h)
    np.testing.assert_array_equal(out["h_q8"], oracle.quant_q8_1(h))
    hv = oracle.dequant_q8_1(out["h_q8"]).ravel()
    np.testing.assert_allclose(out["down"], (Wd @ hv).astype(np.float32), rtol=1e-6, atol=1e-6)


def test_shared_expert_against_dense_matmul():
    dim, inter = 512, 256
    c = oracle.cfg(dim, inter, 8, 2)
    w1, w3, w2 = synth.shared_bf16(6, 0, dim, inter)
    x = synth.x_bf16(6, 0, 1, dim)[0]
    out = oracle.shared_token(c, w1, w3, w2, x)
    xv = _bf16_vals(x)
    gs = _bf16_vals(w1) @ xv
    us = _bf16_vals(w3) @ xv
    np.testing.assert_allclose(out["gs"], gs.astype(np.float32), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(out["us"], us.astype(np.float32), rtol=1e-6, atol=1e-7)
    hs_f32 = np.array([oracle.swiglu(a, b, 7.0) for a, b in zip(gs, us)], np.float32)
    import torch
    hs = torch.from_numpy(hs_f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out["hs"], hs)
    np.testing.assert_allclose(out["sd"], (_bf16_vals(w2) @ _bf16_vals(hs)).astype(np.float32),
                               rtol=1e-6, atol=1e-7)


def _tiny_layer(seed, dim=256, inter=256, n=16, k=2, norm=True, scale=2.5):
    c = oracle.cfg(dim, inter, n, k, norm, 1.0, scale, 7.0)
    shp = synth.LayerShape(dim, inter, n)
    experts = {e: synth.expert_bytes(seed, 0, e, shp) for e in range(n)}
    x = synth.x_bf16(seed, 0, 2, dim)
    w = synth.router_bf16(seed, 0, n, dim)
    b = synth.bias_f32(seed, 0, n)
    return c, shp, experts, x, w, b


def test_layer_single_pick_no_renorm_closed_form():
    """k = 1, no renormalisation, no shared expert: acc = f32(route_scale * score) * down."""
    c, shp, experts, x, w, b = _tiny_layer(40, k=1, norm=False, scale=1.75)
    out = oracle.layer(c, x, w, b, experts, (shp.gate_off, shp.up_off, shp.down_off))
    for t in range(2):
        e = int(out["picks"][t, 0])
        s, _ = oracle.score(float(out["logits"][t, e]))
        wt = np.float32(s * np.float32(1.75))
        assert out["weights"][t, 0] == wt
        xq = oracle.quant_q8_1(_bf16_vals(x[t]).astype(np.float32))
        img = experts[e]
        dn = oracle.expert_token(c, img[shp.gate_off:], img[shp.up_off:], img[shp.down_off:], xq)["down"]
        np.testing.assert_array_equal(out["acc"][t], (np.float32(0) + wt * dn).astype(np.float32))


def test_layer_zero_experts_leave_only_the_shared_expert():
    dim, inter, n = 256, 256, 16
    c, shp, _, x, w, b = _tiny_layer(41)
    experts = {e: np.zeros(shp.slot_bytes, np.uint8) for e in range(n)}   # d = 0 everywhere
    sh = synth.shared_bf16(41, 0, dim, inter)
    res0 = np.ones((2, dim), np.float32) * np.float32(0.25)
    out = oracle.layer(c, x, w, b, experts, (shp.gate_off, shp.up_off, shp.down_off), sh, res0)
    for t in range(2):
        sd = oracle.shared_token(c, *sh, x[t])["sd"]
        np.testing.assert_array_equal(out["acc"][t], sd)
        np.testing.assert_array_equal(out["residual"][t], res0[t] + sd)
    import torch
    xn = torch.from_numpy(out["residual"]).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(out["x_next"], xn)


def test_layer_accumulates_in_ascending_id_then_shared():
    c, shp, experts, x, w, b = _tiny_layer(42, k=3)
    sh = synth.shared_bf16(42, 0, 256, 256)
    out = oracle.layer(c, x, w, b, experts, (shp.gate_off, shp.up_off, shp.down_off), sh)
    for t in range(2):
        xq = oracle.quant_q8_1(_bf16_vals(x[t]).astype(np.float32))
        pairs = sorted(zip(out["picks"][t], out["weights"][t]))
        acc = np.zeros(256, np.float32)
        for e, wt in pairs:
            img = experts[int(e)]
            dn = oracle.expert_token(c, img[shp.gate_off:], img[shp.up_off:], img[shp.down_off:], xq)["down"]
            acc = (acc + np.float32(wt) * dn).astype(np.float32)
        acc = (acc + oracle.shared_token(c, *sh, x[t])["sd"]).astype(np.float32)
        np.testing.assert_array_equal(out["acc"][t], acc)


def test_layer_kquant_shared_expert_is_a_routed_expert_of_weight_one():
    """Page moe_v41.rs MoeV41LayerWeights: the shared w1, w3 may be Q2_K and w2
    Q3_K blocks, run on the routed experts' kernels (struct MoeV41: sh_q8, its
    own q8_1 of the SwiGLU output). acc = the routed sum in ascending id, then
    the shared expert's down output (weight 1) added last; its blocks are
    checked against dense matmuls by test_expert_chain_against_dense_matmul."""
    c, shp, experts, x, w, b = _tiny_layer(45, k=2)
    img = np.frombuffer(synth.expert_bytes(45, 0, 999, shp), np.uint8)
    sh = (img[shp.gate_off:shp.gate_off + shp.gate_bytes], img[shp.up_off:shp.up_off + shp.up_bytes],
          img[shp.down_off:shp.down_off + shp.down_bytes])
    res0 = np.full((2, 256), 0.5, np.float32)
    out = oracle.layer(c, x, w, b, experts, (shp.gate_off, shp.up_off, shp.down_off), sh, res0,
                       shared_kquant=True)
    base = oracle.layer(c, x, w, b, experts, (shp.gate_off, shp.up_off, shp.down_off), None, res0)
    for t in range(2):
        xq = oracle.quant_q8_1(_bf16_vals(x[t]).astype(np.float32))
        sd = oracle.expert_token(c, sh[0], sh[1], sh[2], xq)["down"]
        np.testing.assert_array_equal(out["acc"][t], (base["acc"][t] + sd).astype(np.float32))
        np.testing.assert_array_equal(out["sd"][t], sd)
        np.testing.assert_array_equal(out["residual"][t], (res0[t] + out["acc"][t]).astype(np.float32))
    assert np.abs(sd).max() > 0


def test_layer_missing_expert_is_an_error():
    c, shp, experts, x, w, b = _tiny_layer(43)
    with pytest.raises(KeyError):
        oracle.layer(c, x, w, b, {}, (shp.gate_off, shp.up_off, shp.down_off))


def test_threads_do_not_change_results():
    c, shp, experts, x, w, b = _tiny_layer(44, dim=512, inter=512)
    a = oracle.layer(c, x, w, b, experts, (shp.gate_off, shp.up_off, shp.down_off), threads=1)
    d = oracle.layer(c, x, w, b, experts, (shp.gate_off, shp.up_off, shp.down_off), threads=4)
    np.testing.assert_array_equal(a["acc"], d["acc"])

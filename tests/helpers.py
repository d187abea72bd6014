"""Shared helpers of the GPU parity tests: configurations, tolerances, and the
oracle run on the same seeded inputs the device workload holds."""
import os

import numpy as np
import pytest
import torch

import moe_decode_quantized_gb300 as moe
import oracle
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import Workload, x_tensor

THREADS = max(1, min(16, os.cpu_count() or 1))

# matching rules (stated for this engine): logits |d| <= 1e-5 max(|l|, rms(l));
# picks, slots, pointers and weight bits exact; layer outputs max|d| / max|ref| <= 2e-3
LOGIT_RTOL = 1e-5
OUT_RTOL = 2e-3
# intermediates that see only f32 scale arithmetic (no re-quantisation)
GU_RTOL = 1e-5


def tiny_cfg(m=1, **kw):
    base = dict(dim=256, inter=256, n_routed=16, topk=2, norm_topk_prob=True, max_tokens=m,
                gate_temp=1.0, route_scale=2.5, swiglu_limit=7.0)
    base.update(kw)
    return moe.Config(**base)


def decode_cfg(m=1, **kw):
    base = dict(dim=4096, inter=2048, n_routed=384, topk=6, norm_topk_prob=True, max_tokens=m,
                gate_temp=1.0, route_scale=2.5, swiglu_limit=7.0)
    base.update(kw)
    return moe.Config(**base)


def ocfg(cfg: moe.Config):
    return oracle.cfg(cfg.dim, cfg.inter, cfg.n_routed, cfg.topk, cfg.norm_topk_prob, cfg.gate_temp,
                      cfg.route_scale, cfg.swiglu_limit)


def tiny_workload(cfg, seed=0, n_layers=1, shared=False, shared_kquant=False):
    """The tiny layer: experts quantised from N(0, 0.02) with the oracle's quantisers."""
    wl = Workload(cfg, n_layers=n_layers, seed=seed, shared=shared, fill_experts=False,
                  shared_kquant=shared_kquant)
    wl.images = {}
    for l in range(n_layers):
        for e in range(cfg.n_routed):
            img = oracle.quantised_expert_image(seed, l, e, wl.shape)
            wl.images[(l, e)] = img
            wl.set_expert_image(l, e, img)
    return wl


def expert_image(wl, l, e):
    imgs = getattr(wl, "images", None)
    if imgs is not None and (l, e) in imgs:
        return imgs[(l, e)]
    return wl.host_expert(l, e)


def bf16_vals(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def rel_inf(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def assert_bf16_within_one_ulp(got_bits, ref_bits, slack):
    """x_next = bf16(residual): the two residuals differ by rounding, so a value that
    lies near a bf16 rounding boundary may land one bf16 ulp apart."""
    got = bf16_vals(got_bits).astype(np.float64)
    ref = bf16_vals(ref_bits).astype(np.float64)
    mag = np.maximum(np.abs(ref), np.finfo(np.float32).tiny)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    bad = np.abs(got - ref) > ulp + slack
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], ref[bad][:5])


def assert_logits_close(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    for t in range(ref.shape[0]):
        rms = np.sqrt(np.mean(ref[t] ** 2))
        bound = LOGIT_RTOL * np.maximum(np.abs(ref[t]), rms)
        assert np.all(np.abs(got[t] - ref[t]) <= bound), (t, np.abs(got[t] - ref[t]).max())


def assert_weights_close(cfg, w, ref_w, dl):
    """Routing weights against the oracle's when the logits differ by at most dl.

    d ln(sqrt(softplus(x))) / dx = sigmoid(x) / (2 softplus(x)) <= 1/2, since
    ln(1 + y) >= y / (1 + y); above the x > 20 cut the score is sqrt(x), slope
    1/(2x). So each score moves by at most dl / (2 temp) relatively, and a
    renormalised weight (a score over the sum of k scores) by at most twice
    that; the f32 roundings of each score's three steps (exp, ln_1p, sqrt:
    together within 2 ulp of the exact chain, once on each side) and of the
    sum, quotient and product add k + 8 ulp."""
    w = np.asarray(w, np.float64)
    ref_w = np.asarray(ref_w, np.float64)
    rel = dl / cfg.gate_temp + (cfg.topk + 8) * 2.0 ** -24
    assert np.all(np.abs(w - ref_w) <= rel * np.abs(ref_w)), (w, ref_w, dl)


def keys_of(cfg, logits, bias):
    """Exact-rounded keys as the oracle defines them (for near-tie detection)."""
    _, _, scores, _ = oracle.route(ocfg(cfg), logits, bias)
    return (scores + np.asarray(bias, np.float32)).astype(np.float32)


def _close_gaps(cfg, logits, bias, t):
    """Token t's keys in descending order, and for each adjacent pair whether the
    two are closer than the logit error bound allows us to resolve."""
    key = keys_of(cfg, logits[t:t + 1], bias)[0].astype(np.float64)
    order = np.sort(key)[::-1]
    rms = np.sqrt(np.mean(np.asarray(logits[t], np.float64) ** 2))
    eps = LOGIT_RTOL * max(float(np.abs(logits[t]).max()), rms)
    close = (order[:-1] - order[1:]) <= 2.0 * (0.5 * eps + 4e-7 * np.abs(order[:-1]))
    return order, close


def near_tie(cfg, logits, bias, t):
    """True when token t's k-th and (k+1)-th keys are closer than the logit error
    bound allows us to resolve (the end-to-end picked set may then legitimately
    differ)."""
    order, close = _close_gaps(cfg, logits, bias, t)
    k = cfg.topk
    return k < len(order) and bool(close[k - 1])


def order_near_tie(cfg, logits, bias, t):
    """True when two adjacent keys among token t's k best are that close: the
    set of picks is fixed, their order may legitimately differ."""
    _, close = _close_gaps(cfg, logits, bias, t)
    return bool(np.any(close[:cfg.topk - 1]))


def match_picks(cfg, picks, weights, ref_picks, ref_weights, logits, bias, t):
    """Asserts the picks equal the oracle's -- in order, or as a set when two
    of the k best keys are too close to order -- and returns both sides'
    weights in the same pick order."""
    picks, ref_picks = list(picks), list(ref_picks)
    if not order_near_tie(cfg, logits, bias, t):
        assert picks == ref_picks, (t, picks, ref_picks)
        return np.asarray(weights), np.asarray(ref_weights)
    assert sorted(picks) == sorted(ref_picks), (t, picks, ref_picks)
    a, b = np.argsort(picks), np.argsort(ref_picks)
    return np.asarray(weights)[a], np.asarray(ref_weights)[b]


def oracle_layer(wl, cfg, l, x_bits, residual=None):
    """The oracle's layer step on the workload's host inputs (experts materialised
    for every pick the oracle makes)."""
    oc = ocfg(cfg)
    router = wl.host_router(l)
    bias = wl.host_bias(l)
    logits = oracle.router_logits(x_bits, router)
    picks, _, _, _ = oracle.route(oc, logits, bias)
    experts = {int(e): expert_image(wl, l, int(e)) for e in np.unique(picks)}
    out = oracle.layer(oc, x_bits, router, bias, experts,
                       (wl.shape.gate_off, wl.shape.up_off, wl.shape.down_off), wl.host_shared(l),
                       residual, threads=THREADS, shared_kquant=getattr(wl, "shared_kquant", False))
    out["experts"] = experts
    return out


def new_header(cfg, m, n_layers=1):
    return torch.zeros(n_layers * moe.header_words(cfg, m), dtype=torch.int32, device="cuda")


def parse_all(cfg, hdr_np, m):
    out = []
    for t in range(m):
        out.append(moe.parse_header(cfg, hdr_np, m, t))
    return out


def ws_view(wl, cfg, name, count, dtype=torch.float32):
    v = moe.workspace_view(cfg, wl.ws)
    off = v[name] - wl.ws.data_ptr()
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return wl.ws[off:off + nbytes].view(dtype).cpu().numpy()


def run_layer(wl, cfg, l, x, m, residual=None):
    res = torch.zeros((m, cfg.dim), dtype=torch.float32, device="cuda") if residual is None else residual
    xn = torch.empty_like(x)
    hdr = new_header(cfg, m)
    moe.layer_step(cfg, wl.layer(l), wl.arena, x, res, xn, hdr, m, wl.ws)
    torch.cuda.synchronize()
    assert moe.read_status(wl.ws) == 0
    return res, xn, hdr


def compare_layer(wl, cfg, x_bits, m, res, xn, hdr, residual0=None, l=0):
    ref = oracle_layer(wl, cfg, l, x_bits, residual0)
    h = hdr.cpu().numpy()
    ws_logits = ws_view(wl, cfg, "logits", m * cfg.n_routed).reshape(m, cfg.n_routed)
    compared = 0
    acc = ws_view(wl, cfg, "acc", m * cfg.dim).reshape(m, cfg.dim)
    for t, (st, picks, w) in enumerate(parse_all(cfg, h, m)):
        if near_tie(cfg, ref["logits"], wl.host_bias(l), t):
            continue  # the picks may legitimately differ; reported by the test below
        # the weights: bit-exact on the device's logits (below), and against the
        # oracle's within what the logits' own difference allows
        w1, w2 = match_picks(cfg, picks, w, ref["picks"][t], ref["weights"][t], ref["logits"], wl.host_bias(l), t)
        dl = float(np.abs(ws_logits[t].astype(np.float64) - ref["logits"][t]).max())
        assert_weights_close(cfg, w1, w2, dl)
        assert rel_inf(acc[t], ref["acc"][t]) <= OUT_RTOL, (t, rel_inf(acc[t], ref["acc"][t]))
        compared += 1
    assert compared >= max(1, m - 1)
    # selection on the device's own logits is exact (the device_route_check design)
    opicks, oweights, _, _ = oracle.route(ocfg(cfg), ws_logits, wl.host_bias(l))
    for t, (st, picks, w) in enumerate(parse_all(cfg, h, m)):
        assert list(picks) == list(opicks[t])
        np.testing.assert_array_equal(w.view(np.uint32), oweights[t].view(np.uint32))
    r = res.cpu().numpy()
    assert rel_inf(r, ref["residual"]) <= OUT_RTOL
    assert_bf16_within_one_ulp(xn.cpu().numpy().view(np.uint16), ref["x_next"],
                               OUT_RTOL * np.abs(ref["residual"]).max())
    return ref


gpu = pytest.mark.gpu

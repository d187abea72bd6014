"""GPU tests of the captured multi-layer step (page
spark_model/layers/deepseek_v41_layer/step_seg.rs, module doc: the step as
CUDA graphs, replayed, headers read once after the launch).

- a captured graph equals the same layer steps launched eagerly, bit for bit;
- replays continue from the previous replay's output (the graph writes its
  output back into its input buffer);
- the 40-layer decode chain follows the oracle layer by layer until the first
  token-layer whose top-k boundary is closer than the logit error bound.
"""
import numpy as np
import pytest
import torch

import moe_decode_quantized_gb300 as moe
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import Workload, bf16_tensor

from helpers import (OUT_RTOL, bf16_vals, decode_cfg, gpu, match_picks, near_tie, new_header, oracle_layer,
                     parse_all, rel_inf, tiny_cfg, tiny_workload)

pytestmark = gpu


def _eager_chain(wl, cfg, x0, res0, m, n_layers, replays=1):
    x = x0.clone()
    res = res0.clone()
    hw = moe.header_words(cfg, m)
    hdr = new_header(cfg, m, n_layers)
    for _ in range(replays):
        for l in range(n_layers):
            xn = torch.empty_like(x)
            moe.layer_step(cfg, wl.layer(l), wl.arena, x, res, xn, hdr[l * hw:(l + 1) * hw], m, wl.ws)
            x = xn
    torch.cuda.synchronize()
    return x, res, hdr


def _graph_chain(wl, cfg, x0, res0, m, n_layers, replays=1):
    xa = x0.clone()
    xb = torch.empty_like(xa)
    res = res0.clone()
    hdr = new_header(cfg, m, n_layers)
    g = moe.Graph(cfg, [wl.layer(l) for l in range(n_layers)], wl.arena, m, xa, xb, res, hdr, wl.ws)
    for _ in range(replays):
        g.launch()
    torch.cuda.synchronize()
    g.close()
    return xa, res, hdr


@pytest.mark.parametrize("m,n_layers,replays", [(1, 3, 2), (2, 4, 1)])
def test_tiny_graph_equals_eager(m, n_layers, replays):
    cfg = tiny_cfg(m)
    wl = tiny_workload(cfg, seed=6, n_layers=n_layers)
    x0 = bf16_tensor(synth.x_bf16(6, 0, m, cfg.dim), "cuda")
    r0 = torch.zeros((m, cfg.dim), device="cuda")
    xe, re, he = _eager_chain(wl, cfg, x0, r0, m, n_layers, replays)
    xg, rg, hg = _graph_chain(wl, cfg, x0, r0, m, n_layers, replays)
    assert torch.equal(xe, xg) and torch.equal(re, rg) and torch.equal(he, hg)
    assert moe.read_status(wl.ws) == 0


def test_decode_graph_equals_eager_and_replays_advance():
    cfg = decode_cfg(1)
    n_layers = 4
    wl = Workload(cfg, n_layers=n_layers, seed=8, shared=True)
    x0 = bf16_tensor(synth.x_bf16(8, 0, 1, cfg.dim), "cuda")
    r0 = torch.zeros((1, cfg.dim), device="cuda")
    xe, re, he = _eager_chain(wl, cfg, x0, r0, 1, n_layers, replays=3)
    xg, rg, hg = _graph_chain(wl, cfg, x0, r0, 1, n_layers, replays=3)
    assert torch.equal(xe, xg) and torch.equal(re, rg) and torch.equal(he, hg)
    # one replay vs three: the input advanced, so the routing differs
    x1, r1, h1 = _graph_chain(wl, cfg, x0, r0, 1, n_layers, replays=1)
    assert not torch.equal(h1, hg)
    assert moe.read_status(wl.ws) == 0


def test_forty_layer_chain_against_oracle():
    """40 stacked decode layers (the 40-layer step's shape), one token.

    Layer by layer on the oracle's own chain: layer l of the device gets the
    oracle's x_l and residual_l (inputs may come from the oracle, never the
    reverse) and must match the oracle's layer l output. Two free-running chains
    are not compared element by element: each side rounds x = bf16(residual)
    from residuals that differ by rounding, an occasional one-ulp flip changes
    the next layer's input, and these unnormalised synthetic layers amplify it.
    Then the captured 40-layer graph equals the eager 40-layer chain bit for bit."""
    cfg = decode_cfg(1)
    n_layers = 40
    free, _ = torch.cuda.mem_get_info()
    need = n_layers * synth.LayerShape(cfg.dim, cfg.inter, cfg.n_routed).slot_bytes * cfg.n_routed
    if free < need + (8 << 30):
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, {free / 2**30:.0f} GiB available")
    wl = Workload(cfg, n_layers=n_layers, seed=9, shared=True)
    hw = moe.header_words(cfg, 1)
    x_bits = synth.x_bf16(9, 0, 1, cfg.dim)
    ox, ores = x_bits, np.zeros((1, cfg.dim), np.float32)
    errs, skipped = [], 0
    for l in range(n_layers):
        ref = oracle_layer(wl, cfg, l, ox, ores)
        x = bf16_tensor(ox, "cuda")
        res = torch.from_numpy(ores.copy()).cuda()
        xn = torch.empty_like(x)
        hdr = new_header(cfg, 1)
        moe.layer_step(cfg, wl.layer(l), wl.arena, x, res, xn, hdr, 1, wl.ws)
        torch.cuda.synchronize()
        if near_tie(cfg, ref["logits"], wl.host_bias(l), 0):
            skipped += 1
        else:
            _, picks, w = parse_all(cfg, hdr.cpu().numpy(), 1)[0]
            match_picks(cfg, picks, w, ref["picks"][0], ref["weights"][0], ref["logits"], wl.host_bias(l), 0)
            acc = moe_acc(wl, cfg)
            err = rel_inf(acc, ref["acc"])
            errs.append(err)
            assert err <= OUT_RTOL, (l, err)
            assert rel_inf(res.cpu().numpy(), ref["residual"]) <= OUT_RTOL, l
        ox, ores = ref["x_next"], ref["residual"]
    assert skipped <= 4, skipped
    print(f"40-layer chain, layer by layer: max acc rel error {max(errs):.2e} over {len(errs)} layers, "
          f"{skipped} near-tie layers skipped")
    x0 = bf16_tensor(x_bits, "cuda")
    r0 = torch.zeros((1, cfg.dim), device="cuda")
    xe, re, he = _eager_chain(wl, cfg, x0, r0, 1, n_layers)
    xg, rg, hg = _graph_chain(wl, cfg, x0, r0, 1, n_layers)
    assert torch.equal(xg, xe) and torch.equal(rg, re) and torch.equal(hg, he)
    assert moe.read_status(wl.ws) == 0


def moe_acc(wl, cfg):
    v = moe.workspace_view(cfg, wl.ws)
    off = v["acc"] - wl.ws.data_ptr()
    return wl.ws[off:off + 4 * cfg.dim].view(torch.float32).cpu().numpy()[None]

"""GPU tests of the step's fallback paths (page
spark_model/layers/deepseek_v41_layer/step_seg.rs, module doc and fn step_seg:
per-layer snapshots, a replay whose header carries the miss flag restored and
finished eagerly; fn close_or_disable: graph mode off when capture fails) and
of expert residency through the LRU cache (page spark_model/layers/moe_v41.rs
module doc, page .../moe_v41/device_route.rs fn slot_table_update).

Every result is compared bit for bit with the same layers run eagerly with
every expert resident: residency changes where an expert's blocks live, not
what is computed."""
import numpy as np
import pytest
import torch

import moe_decode_quantized_gb300 as moe
import oracle
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import bf16_tensor

from helpers import gpu, new_header, tiny_cfg, tiny_workload

pytestmark = gpu


def _eager(wl, cfg, x0, r0, m, L, rounds=1):
    x, res = x0.clone(), r0.clone()
    hw = moe.header_words(cfg, m)
    hdr = new_header(cfg, m, L)
    for _ in range(rounds):
        for l in range(L):
            xn = torch.empty_like(x)
            moe.layer_step(cfg, wl.layer(l), wl.arena, x, res, xn, hdr[l * hw:(l + 1) * hw], m, wl.ws)
            x = xn
    torch.cuda.synchronize()
    return x, res, hdr


def _graph(wl, cfg, x0, r0, m, L, flags, layers=None, arena=None):
    xa, xb, res = x0.clone(), torch.empty_like(x0), r0.clone()
    hdr = new_header(cfg, m, L)
    snap = torch.empty(moe.graph_snapshot_bytes(cfg, m, L), dtype=torch.uint8, device="cuda")
    g = moe.Graph(cfg, layers or [wl.layer(l) for l in range(L)], arena or wl.arena, m, xa, xb, res, hdr, wl.ws,
                  snapshots=snap, flags=flags | moe.MOE_GRAPH_SNAPSHOTS)
    return g, xa, res, hdr


def test_capture_failure_falls_back_to_eager():
    cfg = tiny_cfg(2)
    L = 3
    wl = tiny_workload(cfg, seed=70, n_layers=L)
    x0 = bf16_tensor(synth.x_bf16(70, 0, 2, cfg.dim), "cuda")
    r0 = torch.zeros((2, cfg.dim), device="cuda")
    xe, re, he = _eager(wl, cfg, x0, r0, 2, L, rounds=2)
    g, xa, res, hdr = _graph(wl, cfg, x0, r0, 2, L, moe.MOE_GRAPH_EAGER_FALLBACK | moe.MOE_GRAPH_TEST_FAIL_CAPTURE)
    assert g.eager
    g.launch()
    g.launch()
    torch.cuda.synchronize()
    assert torch.equal(xa, xe) and torch.equal(res, re) and torch.equal(hdr, he)
    g.close()
    with pytest.raises(moe.MoeError) as e:  # without the fallback a failed capture is an error
        _graph(wl, cfg, x0, r0, 2, L, moe.MOE_GRAPH_TEST_FAIL_CAPTURE)
    assert e.value.code == -4


@pytest.mark.parametrize("layer", [0, 2])
def test_rerun_from_a_snapshot_repeats_the_step(layer):
    cfg = tiny_cfg(1)
    L = 4
    wl = tiny_workload(cfg, seed=71, n_layers=L)
    x0 = bf16_tensor(synth.x_bf16(71, 0, 1, cfg.dim), "cuda")
    r0 = torch.zeros((1, cfg.dim), device="cuda")
    g, xa, res, hdr = _graph(wl, cfg, x0, r0, 1, L, 0)
    assert not g.eager
    g.launch()
    torch.cuda.synchronize()
    x1, r1, h1 = xa.clone(), res.clone(), hdr.clone()
    g.rerun_from(layer)
    torch.cuda.synchronize()
    assert torch.equal(xa, x1) and torch.equal(res, r1) and torch.equal(hdr, h1)
    xe, re, _ = _eager(wl, cfg, x0, r0, 1, L)
    assert torch.equal(x1, xe) and torch.equal(r1, re)


@pytest.mark.parametrize("m,slots", [(1, 6), (2, 8)])
def test_graph_step_with_expert_cache_matches_all_resident(m, slots):
    """3 layers x 16 experts (48 expert images in pinned host memory), an
    arena of a few slots, tokens one after another: misses are fetched, the
    step rerun from the first layer with a miss, and every token's result
    equals the all-resident eager run bit for bit."""
    cfg = tiny_cfg(m)
    L, n = 3, cfg.n_routed
    ref = tiny_workload(cfg, seed=72, n_layers=L)  # every expert resident
    shp = ref.shape
    images = [[torch.from_numpy(oracle.quantised_expert_image(72, l, e, shp)).pin_memory() for e in range(n)]
              for l in range(L)]
    src = moe.HostSource(images, L, n, shp.slot_bytes)
    arena_t = torch.zeros(slots * shp.slot_bytes, dtype=torch.uint8, device="cuda")
    arena = moe.Arena(arena_t, shp.slot_bytes, shp.gate_off, shp.up_off, shp.down_off)
    table = torch.full((moe.SLOT_TABLE_LAYERS, n), -1, dtype=torch.int32, device="cuda")
    cache = moe.ExpertCache(L, n, slots, arena, table, src)
    layers = [moe.Layer(ref.router[l], ref.bias[l], table[l]) for l in range(L)]
    xa = torch.empty((m, cfg.dim), dtype=torch.int16, device="cuda")
    xb, res = torch.empty_like(xa), torch.zeros((m, cfg.dim), device="cuda")
    hdr = new_header(cfg, m, L)
    snap = torch.empty(moe.graph_snapshot_bytes(cfg, m, L), dtype=torch.uint8, device="cuda")
    g = moe.Graph(cfg, layers, arena, m, xa, xb, res, hdr, ref.ws, snapshots=snap, flags=moe.MOE_GRAPH_SNAPSHOTS)
    hh = np.zeros(L * moe.header_words(cfg, m), np.int32)
    reruns = []
    for tok in range(6):
        x0 = bf16_tensor(synth.x_bf16(72, 10 + tok, m, cfg.dim), "cuda")
        r0 = torch.zeros((m, cfg.dim), device="cuda")
        xa.copy_(x0)
        res.copy_(r0)
        reruns.append(g.step_cached(cache, hh))
        xe, re, he = _eager(ref, cfg, x0, r0, m, L)
        assert torch.equal(xa, xe) and torch.equal(res, re), tok
        hw = moe.header_words(cfg, m)
        for l in range(L):  # the final headers: the all-resident picks, no miss left
            got = hh[l * hw:(l + 1) * hw].copy()
            want = he[l * hw:(l + 1) * hw].cpu().numpy()
            for t in range(m):
                assert not (got[t * (1 + 3 * cfg.topk)] & moe.MOE_HDR_MISS)
                row = slice(t * (1 + 3 * cfg.topk) + 1, t * (1 + 3 * cfg.topk) + 1 + 2 * cfg.topk)
                assert list(got[row]) == list(want[row])  # picks and weight bits
    hits, misses, evictions = cache.stats()
    assert reruns[0] == L and misses > 0 and evictions > 0
    g.close()
    cache.close()

"""GPU parity of the batched (prefill) arm, through the C ABI, against the CPU
oracle on the same seeded inputs.

Page spark_model/layers/moe_v41.rs, struct Kernels (gather, scatter_add,
sum_rows, quant_d2s6 / quant_d4, mmq_q2k_*, mmq_q3k_*, gemm): many tokens
through the layer at once, the routed experts as GEMMs over each expert's
group of tokens. The layer's arithmetic is the decode step's, so the oracle
is oracle.layer on the same tokens; the tensor-core GEMMs take fp16-rounded
dequantised operands (about 2^-12 relative per operand), inside the layer
tolerance. Expert load is skewed by a correction bias ~U(-1, 1), as in the
prefill workload."""
import numpy as np
import pytest
import torch

import moe_decode_quantized_gb300 as moe
import oracle
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import Workload, bf16_tensor

from helpers import (OUT_RTOL, assert_bf16_within_one_ulp, assert_logits_close, gpu, match_picks, near_tie, ocfg,
                     oracle_layer, rel_inf)

pytestmark = gpu


@pytest.fixture(autouse=True)
def short_waits():
    moe.set_wait_limit_ns(500_000_000)  # a stalled pipeline gives up within half a second
    yield
    moe.set_wait_limit_ns(0)


def _bf16(rng, shape, scale):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("M,N,K,ldd", [(384, 200, 4096, 384), (256, 17, 128, 300), (2048, 512, 1024, 2048),
                                       (130, 1, 64, 130)])
def test_gemm_bf16_against_exact_products(M, N, K, ldd):
    """d[n, r] = sum_k a[r, k] b[n, k]: bf16 products are exact in f32, so the
    only error is f32 accumulation, bounded here by 2^-20 sum |a b|."""
    rng = np.random.default_rng(70 + M + N)
    a = _bf16(rng, (M, K), 1.0)
    b = _bf16(rng, (N, K), 0.5)
    d = torch.full((N, ldd), float("nan"), device="cuda")
    moe.gemm_bf16(a.view(torch.int16).cuda(), b.view(torch.int16).cuda(), d, M, N, K, ldd)
    torch.cuda.synchronize()
    a64, b64 = a.double().numpy(), b.double().numpy()
    ref = b64 @ a64.T                       # [N, M]
    mag = np.abs(b64) @ np.abs(a64).T
    got = d.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got[:, :M] - ref) <= 2.0 ** -20 * mag + 1e-30)
    if ldd > M:
        assert np.isnan(got[:, M:]).all()  # columns beyond M are not written


def _run_prefill(wl, cfg, x_bits, m):
    x = bf16_tensor(x_bits, "cuda")
    res = torch.zeros((m, cfg.dim), dtype=torch.float32, device="cuda")
    xn = torch.empty_like(x)
    picks = torch.full((m, cfg.topk), -1, dtype=torch.int32, device="cuda")
    weights = torch.zeros((m, cfg.topk), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.prefill_workspace_bytes(cfg, m), dtype=torch.uint8, device="cuda")
    moe.prefill_step(cfg, wl.layer(0), wl.arena, cfg.n_routed, x, res, xn, picks, weights, m, ws)
    torch.cuda.synchronize()
    assert moe.prefill_status(cfg, m, ws) == 0
    # the router GEMM alone on the same inputs (the same kernel: the same bits)
    logits = torch.zeros((m, cfg.n_routed), dtype=torch.float32, device="cuda")
    moe.gemm_bf16(wl.router[0], x, logits, cfg.n_routed, m, cfg.dim, cfg.n_routed)
    torch.cuda.synchronize()
    return res.cpu().numpy(), xn.cpu().numpy().view(np.uint16), picks.cpu().numpy(), weights.cpu().numpy(), \
        logits.cpu().numpy()


def _compare(wl, cfg, x_bits, m, sample):
    res, xn, picks, weights, logits = _run_prefill(wl, cfg, x_bits, m)
    # the selection is exact on the device's own logits
    opicks, oweights, _, _ = oracle.route(ocfg(cfg), logits, wl.host_bias(0))
    np.testing.assert_array_equal(picks, opicks)
    np.testing.assert_array_equal(weights.view(np.uint32), oweights.view(np.uint32))
    # the layer against the oracle on a sample of the tokens (rows are independent)
    ref = oracle_layer(wl, cfg, 0, x_bits[sample])
    assert_logits_close(logits[sample], ref["logits"])
    compared = 0
    for j, t in enumerate(sample):
        if near_tie(cfg, ref["logits"], wl.host_bias(0), j):
            continue
        match_picks(cfg, picks[t], weights[t], ref["picks"][j], ref["weights"][j], ref["logits"], wl.host_bias(0), j)
        assert rel_inf(res[t], ref["residual"][j]) <= OUT_RTOL, (t, rel_inf(res[t], ref["residual"][j]))
        assert_bf16_within_one_ulp(xn[t], ref["x_next"][j], OUT_RTOL * np.abs(ref["residual"][j]).max())
        compared += 1
    assert compared >= len(sample) - 2
    return picks


@pytest.mark.parametrize("m", [1, 37, 100])
def test_prefill_small_layer(m):
    """dim 1024, inter 2048, 32 experts, top 4, shared expert: every token checked."""
    cfg = moe.Config(dim=1024, inter=2048, n_routed=32, topk=4, max_tokens=1)
    wl = Workload(cfg, n_layers=1, seed=80 + m, shared=True, bias_range=(-1.0, 1.0))
    x_bits = synth.x_bf16(80 + m, 0, m, cfg.dim)
    _compare(wl, cfg, x_bits, m, list(range(m)))


def test_prefill_groups_wider_than_a_tile():
    """8 experts, top 2, 300 tokens: groups of more than 128 tokens span
    several column tiles of the routed GEMMs (and a ragged last one)."""
    cfg = moe.Config(dim=1024, inter=2048, n_routed=8, topk=2, max_tokens=1)
    wl = Workload(cfg, n_layers=1, seed=86, shared=True, bias_range=(-1.0, 1.0))
    x_bits = synth.x_bf16(86, 0, 300, cfg.dim)
    picks = _compare(wl, cfg, x_bits, 300, list(range(0, 300, 7)))
    counts = np.bincount(picks.ravel(), minlength=cfg.n_routed)
    assert counts.max() > 128 and counts.max() % 128 != 0


def test_prefill_without_shared_expert():
    cfg = moe.Config(dim=1024, inter=2048, n_routed=16, topk=2, max_tokens=1)
    wl = Workload(cfg, n_layers=1, seed=85, shared=False, bias_range=(-1.0, 1.0))
    x_bits = synth.x_bf16(85, 0, 40, cfg.dim)
    _compare(wl, cfg, x_bits, 40, list(range(40)))


def test_prefill_decode_layer_512_tokens():
    """The prefill workload: 512 tokens through the decode layer (dim 4096,
    inter 2048, 384 x top 6, bf16 shared expert), bias ~U(-1, 1); the
    oracle checks a sample of 12 tokens (the other rows are computed the
    same way and independently)."""
    cfg = moe.Config(dim=4096, inter=2048, n_routed=384, topk=6, max_tokens=1)
    wl = Workload(cfg, n_layers=1, seed=90, shared=True, bias_range=(-1.0, 1.0))
    x_bits = synth.x_bf16(90, 0, 512, cfg.dim)
    sample = [0, 1, 63, 64, 127, 128, 200, 255, 256, 383, 500, 511]
    picks = _compare(wl, cfg, x_bits, 512, sample)
    counts = np.bincount(picks.ravel(), minlength=cfg.n_routed)
    assert (counts == 0).sum() > cfg.n_routed // 2 and counts.max() > 3 * counts.mean()  # skewed groups
    del wl
    torch.cuda.empty_cache()


def _prefill_once(wl, cfg, x, res, xn, m):
    picks = torch.zeros((m, cfg.topk), dtype=torch.int32, device="cuda")
    weights = torch.zeros((m, cfg.topk), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.prefill_workspace_bytes(cfg, m), dtype=torch.uint8, device="cuda")
    moe.prefill_step(cfg, wl.layer(0), wl.arena, cfg.n_routed, x, res, xn, picks, weights, m, ws)
    torch.cuda.synchronize()
    assert moe.prefill_status(cfg, m, ws) == 0


def test_prefill_unaligned_residual_and_x_next_give_the_same_bits():
    """residual only 4-byte and x_next only 2-byte aligned: the finish takes
    one element a thread instead of four; the outputs are the aligned run's,
    bit for bit (the same sums in the same order)."""
    cfg = moe.Config(dim=1024, inter=2048, n_routed=32, topk=4, max_tokens=1)
    wl = Workload(cfg, n_layers=1, seed=87, shared=True, bias_range=(-1.0, 1.0))
    m = 20
    x = bf16_tensor(synth.x_bf16(87, 0, m, cfg.dim), "cuda")
    res0 = torch.full((m, cfg.dim), 0.25, dtype=torch.float32, device="cuda")
    xn0 = torch.empty_like(x)
    _prefill_once(wl, cfg, x, res0, xn0, m)
    rbuf = torch.full((m * cfg.dim + 1,), 0.25, dtype=torch.float32, device="cuda")
    xbuf = torch.zeros((m * cfg.dim + 1,), dtype=x.dtype, device="cuda")
    res1, xn1 = rbuf[1:].view(m, cfg.dim), xbuf[1:].view(m, cfg.dim)
    assert res1.data_ptr() % 16 == 4 and xn1.data_ptr() % 8 == 2
    _prefill_once(wl, cfg, x, res1, xn1, m)
    assert torch.equal(res0, res1) and torch.equal(xn0, xn1)


def test_prefill_rejects_an_unaligned_x_before_any_launch():
    """x must be 16-byte aligned (the router GEMM reads it through a tensor
    map): an offset view is refused on the host, and the next step runs."""
    cfg = moe.Config(dim=1024, inter=2048, n_routed=32, topk=4, max_tokens=1)
    wl = Workload(cfg, n_layers=1, seed=88, shared=True, bias_range=(-1.0, 1.0))
    m = 4
    xbuf = bf16_tensor(synth.x_bf16(88, 0, m * cfg.dim + 8, 1).reshape(-1), "cuda")
    x_bad = xbuf[1:1 + m * cfg.dim].view(m, cfg.dim)
    assert x_bad.data_ptr() % 16 == 2
    res = torch.zeros((m, cfg.dim), dtype=torch.float32, device="cuda")
    xn = torch.empty((m, cfg.dim), dtype=x_bad.dtype, device="cuda")
    with pytest.raises(moe.MoeError):
        _prefill_once(wl, cfg, x_bad, res, xn, m)
    _prefill_once(wl, cfg, xbuf[8:8 + m * cfg.dim].view(m, cfg.dim), res, xn, m)


def test_prefill_plan_beyond_its_shared_memory_tables():
    """1000 tokens x top 6 = 6000 picks, more than the plan kernel builds in
    shared memory: the pair tables are written straight to global memory;
    a sample of the tokens checked against the oracle."""
    cfg = moe.Config(dim=1024, inter=2048, n_routed=32, topk=6, max_tokens=1)
    wl = Workload(cfg, n_layers=1, seed=89, shared=True, bias_range=(-1.0, 1.0))
    m = 1000
    x_bits = synth.x_bf16(89, 0, m, cfg.dim)
    picks = _compare(wl, cfg, x_bits, m, list(range(0, m, 41)) + [m - 1])
    assert m * cfg.topk > 5120 and (picks >= 0).all()

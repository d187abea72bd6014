"""GPU parity at the edges of what the C ABI accepts, against the CPU oracle
on the same seeded inputs: SwiGLU without a clamp (swiglu_limit <= 0), the
largest plan (top 8 of 1024 experts), the widest rows (dim or inter 8192),
and both sides of the down kernel's switch from row ownership (at most 16
plan pairs) to row-group tickets (more).

Page spark_model/layers/moe_v41.rs, MoeV41Cfg (dim, inter, n_routed, topk,
swiglu_limit, max_tokens) and module doc (the layer's math)."""
import pytest
import torch

import moe_decode_quantized_gb300 as moe
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import Workload, bf16_tensor

from helpers import compare_layer, gpu, run_layer, tiny_cfg, tiny_workload

pytestmark = gpu


def _layer_case(cfg, m, seed, shared=False, tiny=False):
    wl = tiny_workload(cfg, seed=seed, shared=shared) if tiny else Workload(cfg, n_layers=1, seed=seed,
                                                                             shared=shared)
    x_bits = synth.x_bf16(seed, 0, m, cfg.dim)
    res, xn, hdr = run_layer(wl, cfg, 0, bf16_tensor(x_bits, "cuda"), m)
    compare_layer(wl, cfg, x_bits, m, res, xn, hdr)
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("limit", [0.0, -1.0])
def test_swiglu_without_clamp(limit):
    """L <= 0: h = silu(g) u with nothing clamped (reading F4); the tiny
    layer's experts give |g|, |u| up to a few units, a larger x scale makes
    them exceed any small limit."""
    cfg = tiny_cfg(2, swiglu_limit=limit)
    _layer_case(cfg, 2, seed=41, shared=True, tiny=True)


def test_swiglu_clamp_active():
    """A limit small enough that the clamp changes most of h (L = 0.05)."""
    cfg = tiny_cfg(1, swiglu_limit=0.05)
    _layer_case(cfg, 1, seed=42, shared=True, tiny=True)


@pytest.mark.parametrize("m", [1, 2])
def test_top8_of_1024_experts(m):
    """The largest selection: 1024 routed experts, top 8 (at m = 2, 16 plan
    pairs: the down kernel's row ownership at its limit)."""
    cfg = moe.Config(dim=256, inter=256, n_routed=1024, topk=8, max_tokens=m)
    _layer_case(cfg, m, seed=43)


@pytest.mark.parametrize("dim,inter,m", [(8192, 1024, 1), (8192, 1024, 4), (1024, 8192, 2)])
def test_widest_rows(dim, inter, m):
    """dim 8192 (two-row gate/up tasks) or inter 8192 (two-row down tasks);
    m = 4 at dim 8192 is the m * dim = 32768 bound."""
    cfg = moe.Config(dim=dim, inter=inter, n_routed=32, topk=4, max_tokens=m)
    _layer_case(cfg, m, seed=44, shared=True)


@pytest.mark.parametrize("m,k", [(2, 8), (3, 6)])
def test_down_kernel_path_switch(m, k):
    """m k = 16 plan pairs: each down CTA owns whole row groups; m k = 18: the
    expert-major ranges with row-group tickets. The decode-layer shape (dim
    4096, inter 2048) with 64 experts."""
    cfg = moe.Config(dim=4096, inter=2048, n_routed=64, topk=k, max_tokens=m)
    _layer_case(cfg, m, seed=45 + m, shared=True)

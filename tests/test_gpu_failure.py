"""Failure handling on the GPU without a fault: a bounded device wait that
can only run out returns an error status the host reads, the context stays
usable, and after moe_workspace_init the next step matches the oracle.

No GPU is faulted, trapped or hung here: the wait is a poll on a word that
nothing raises (the selection's plan-ready word with no router kernel
before the expert kernels), bounded at 1 ms by moe_set_wait_limit_ns."""
import time

import torch

import moe_decode_quantized_gb300 as moe
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import bf16_tensor

from helpers import compare_layer, gpu, new_header, run_layer, tiny_cfg, tiny_workload

pytestmark = gpu


def test_wait_that_runs_out_sets_timeout_and_the_next_step_is_exact():
    cfg = tiny_cfg(1)
    wl = tiny_workload(cfg, seed=51)
    x_bits = synth.x_bf16(51, 0, 1, cfg.dim)
    x = bf16_tensor(x_bits, "cuda")
    ref = run_layer(wl, cfg, 0, x, 1)  # a normal step first: every kernel loaded
    hdr = new_header(cfg, 1)  # an empty plan: no expert is read
    torch.cuda.synchronize()
    moe.set_wait_limit_ns(1_000_000)
    try:
        t0 = time.perf_counter()
        moe.expert_step_unreleased(cfg, x, hdr, 1, wl.ws)
        status = moe.read_status(wl.ws)  # synchronises the stream
        dt = time.perf_counter() - t0
    finally:
        moe.set_wait_limit_ns(0)
    assert status & moe.MOE_WS_TIMEOUT
    assert dt < 1.0  # ended by the 1 ms bound, not the 2 s default
    # the context is usable and, once the workspace is initialised again, the
    # layer step is exact
    moe.workspace_init(wl.ws)
    res, xn, hdr = run_layer(wl, cfg, 0, x, 1)
    compare_layer(wl, cfg, x_bits, 1, res, xn, hdr)
    for a, b in zip(ref, (res, xn, hdr)):
        assert torch.equal(a, b)


def test_wait_limit_does_not_change_a_normal_step():
    """A short bound that no wait of a normal step reaches (100 ms) leaves the
    step's result unchanged."""
    cfg = tiny_cfg(2)
    wl = tiny_workload(cfg, seed=52, shared=True)
    x = bf16_tensor(synth.x_bf16(52, 0, 2, cfg.dim), "cuda")
    ref = run_layer(wl, cfg, 0, x, 2)
    moe.set_wait_limit_ns(100_000_000)
    try:
        got = run_layer(wl, cfg, 0, x, 2)
    finally:
        moe.set_wait_limit_ns(0)
    for a, b in zip(ref, got):
        assert torch.equal(a, b)

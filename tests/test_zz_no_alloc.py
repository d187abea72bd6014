"""moe_layer_step_static: the layer step on the library's own static device
workspace, for callers that cannot allocate device memory.

The pages have no counterpart of this call; it must give exactly what
moe_layer_step gives on a workspace of the caller's (the kernels are
deterministic, so bit for bit), and it must not allocate device memory. This
file is named to be collected last, so that the static array has already
seen other calls' data (and the tests here also pass alone)."""
import numpy as np
import pytest
import torch

import moe_decode_quantized_gb300 as moe
from moe_decode_quantized_gb300 import synth
from moe_decode_quantized_gb300.workload import Workload, bf16_tensor

from helpers import decode_cfg, new_header, tiny_cfg, tiny_workload

STATIC_WS_BYTES = 4 << 20


def test_static_rejects_a_workspace_beyond_its_size():
    """Host-side check, before any device call."""
    cfg = moe.Config(dim=4096, inter=8192, n_routed=1024, topk=8, max_tokens=8)
    assert moe.workspace_bytes(cfg) > STATIC_WS_BYTES
    arena = moe.Arena(base=1 << 20, slot_bytes=1 << 20, gate_off=0, up_off=1 << 16, down_off=1 << 17)
    layer = moe.Layer(router_w=1 << 20, bias=1 << 20, slot_row=1 << 20)
    with pytest.raises(moe.MoeError) as e:
        moe.layer_step_static(cfg, layer, arena, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1, stream=0)
    assert e.value.code == -2 and "static workspace holds" in str(e.value)


def _two_steps(step, cfg, x0, r0, m):
    """Two layer steps in a row, the second on the first one's output."""
    x = x0.clone()
    res = r0.clone()
    outs = []
    for _ in range(2):
        xn = torch.empty_like(x)
        hdr = new_header(cfg, m)
        step(x, res, xn, hdr)
        torch.cuda.synchronize()
        outs.append((xn.clone(), res.clone(), hdr.clone()))
        x = xn
    return outs


def _compare(cfg, wl, m, x0, r0):
    ly = wl.layer(0)

    def with_ws(x, res, xn, hdr):
        moe.layer_step(cfg, ly, wl.arena, x, res, xn, hdr, m, wl.ws)

    status = np.full(1, 0xFFFFFFFF, np.uint32)

    def static(x, res, xn, hdr):
        status[0] = 0xFFFFFFFF
        moe.layer_step_static(cfg, ly, wl.arena, x, res, xn, hdr, m, status)
        torch.cuda.synchronize()
        assert status[0] == 0

    ref = _two_steps(with_ws, cfg, x0, r0, m)
    got = _two_steps(static, cfg, x0, r0, m)
    for (xr, rr, hr), (xg, rg, hg) in zip(ref, got):
        assert torch.equal(hr, hg)  # picks, weights and slots
        assert torch.equal(rg, rr)  # the same kernels on the same inputs: bit for bit
        assert torch.equal(xg, xr)
    assert moe.read_status(wl.ws) == 0

    # no device allocation: with every buffer in place and the array set up by
    # the calls above, further calls leave the device's free memory unchanged
    x, res, xn, hdr = x0.clone(), r0.clone(), torch.empty_like(x0), new_header(cfg, m)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(4):
        moe.layer_step_static(cfg, ly, wl.arena, x, res, xn, hdr, m, status)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


@pytest.mark.gpu
def test_static_matches_workspace_path_tiny():
    cfg = tiny_cfg(2)
    wl = tiny_workload(cfg, seed=21, shared=True)
    x0 = bf16_tensor(synth.x_bf16(21, 0, 2, cfg.dim), "cuda")
    r0 = torch.zeros((2, cfg.dim), device="cuda")
    _compare(cfg, wl, 2, x0, r0)


@pytest.mark.gpu
@pytest.mark.parametrize("m", [1, 8])
def test_static_matches_workspace_path_decode(m):
    cfg = decode_cfg(m)
    wl = Workload(cfg, n_layers=1, seed=22, shared=True)
    x0 = bf16_tensor(synth.x_bf16(22, 0, m, cfg.dim), "cuda")
    r0 = torch.zeros((m, cfg.dim), device="cuda")
    _compare(cfg, wl, m, x0, r0)

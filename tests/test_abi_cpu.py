"""The C ABI without a GPU: both libraries build and load, export every symbol
their headers declare, and reject bad arguments on the host (no compute)."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

import moe_decode_quantized_gb300 as moe
from moe_decode_quantized_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", src)))


def _exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True, check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_libraries_build():
    paths = build.build()
    for p in paths:
        assert os.path.exists(p)


@pytest.mark.parametrize("header,lib", [("moe.h", build.LIBMOE), ("moe_synth.h", build.LIBSYNTH)])
def test_every_declared_symbol_is_exported(header, lib):
    names = _declared(header)
    assert len(names) >= 4
    exp = _exported(lib)
    missing = [n for n in names if n not in exp]
    assert not missing, missing


def test_binding_declares_every_symbol():
    assert set(_declared("moe.h")) == set(_lib.MOE_SYMBOLS)
    assert set(_declared("moe_synth.h")) == set(_lib.SYNTH_SYMBOLS)


def test_library_loads_without_gpu():
    L = _lib.moe()
    assert L.moe_last_error() is not None


def test_host_side_validation():
    cfg = moe.Config(dim=4096, inter=2048, n_routed=384, topk=6, max_tokens=8)
    assert moe.header_words(cfg, 1) == 19 + 2 + 12
    assert moe.workspace_bytes(cfg) > 0
    bad = moe.Config(dim=300, inter=2048, n_routed=384, topk=6)
    with pytest.raises(moe.MoeError) as e:
        moe.workspace_bytes(bad)
    assert e.value.code == -1
    odd = moe.Config(dim=7168, inter=2048, n_routed=384, topk=6)
    with pytest.raises(moe.MoeError) as e:
        moe.workspace_bytes(odd)
    assert e.value.code == -2
    with pytest.raises(moe.MoeError):
        moe.workspace_bytes(moe.Config(dim=4096, inter=2048, n_routed=384, topk=9))
    with pytest.raises(moe.MoeError):
        moe.workspace_bytes(moe.Config(dim=4096, inter=2048, n_routed=4, topk=6))


def test_dedupe_triples_last_write_wins():
    t = np.array([[0, 5, 1], [1, 5, 2], [0, 5, -1], [0, 7, 3], [0, 5, 9]], np.int32)
    d = moe.dedupe_triples(t)
    assert sorted(map(tuple, d.tolist())) == [(0, 5, 9), (0, 7, 3), (1, 5, 2)]


def test_parse_header_checks_picks():
    cfg = moe.Config(dim=256, inter=256, n_routed=16, topk=2)
    h = np.zeros(moe.header_words(cfg, 1), np.int32)
    h[0] = 1
    h[1:3] = [3, 7]
    h[3:5] = np.array([0.25, 0.5], np.float32).view(np.int32)
    st, picks, w = moe.parse_header(cfg, h, 1, 0)
    assert st == 1 and list(picks) == [3, 7] and list(w) == [0.25, 0.5]
    h[2] = 16
    with pytest.raises(moe.MoeError):
        moe.parse_header(cfg, h, 1, 0)

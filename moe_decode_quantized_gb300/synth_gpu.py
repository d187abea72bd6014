"""Device-side fills with the seeded input generator (libmoe_synth.so, the
twin of synth.py): the same bytes as the host generator, written in place.
Inputs only -- none of the layer's arithmetic."""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import _lib, synth
from . import _stream, _ptr


def _ok(rc):
    if rc != 0:
        raise RuntimeError(f"libmoe_synth: CUDA error {rc}")


def q2k(dst, nblocks: int, key: int, stream=None):
    _ok(_lib.synth().moe_synth_q2k(_ptr(dst), nblocks, key, _stream(stream)))


def q3k(dst, nblocks: int, key: int, stream=None):
    _ok(_lib.synth().moe_synth_q3k(_ptr(dst), nblocks, key, _stream(stream)))


def normal_bf16(dst, n: int, key: int, sigma: float, stream=None):
    _ok(_lib.synth().moe_synth_normal_bf16(_ptr(dst), n, key, float(synth.normal_scale(sigma)),
                                            _stream(stream)))


def uniform_f32(dst, n: int, key: int, lo: float, hi: float, stream=None):
    a = np.float32(np.float32(hi) - np.float32(lo))
    _ok(_lib.synth().moe_synth_uniform_f32(_ptr(dst), n, key, float(np.float32(lo)), float(a),
                                            _stream(stream)))


def fill_expert(base_ptr: int, seed: int, layer: int, expert: int, shp: synth.LayerShape, stream=None):
    """Writes expert `expert` of `layer` into the slot image at device address base_ptr."""
    nq2 = shp.gate_bytes // synth.Q2K_BYTES
    nq3 = shp.down_bytes // synth.Q3K_BYTES
    q2k(base_ptr + shp.gate_off, nq2, synth.tensor_key(seed, layer, synth.T_GATE, expert), stream)
    q2k(base_ptr + shp.up_off, nq2, synth.tensor_key(seed, layer, synth.T_UP, expert), stream)
    q3k(base_ptr + shp.down_off, nq3, synth.tensor_key(seed, layer, synth.T_DOWN, expert), stream)

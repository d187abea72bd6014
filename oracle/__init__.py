"""Python access to the CPU oracle (oracle/moe_oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only tests/, the smoke check in
__graft_entry__ and the benchmark's CPU-baseline leg import this package. The
product path (moe_decode_quantized_gb300) never imports it and shares no code
with it.

The C file is compiled on demand with gcc (-O2, no fast-math,
-ffp-contract=off) into oracle/liboracle.so; every function below only
marshals numpy arrays into the C routines.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain C11, -O2, no FMA contraction)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= max(
            os.path.getmtime(SRC), os.path.getmtime(os.path.join(HERE, "moe_oracle.h"))):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-D_GNU_SOURCE", "-o", tmp, SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


class Cfg(C.Structure):
    _fields_ = [("dim", C.c_int32), ("inter", C.c_int32), ("n_routed", C.c_int32),
                ("topk", C.c_int32), ("norm_topk_prob", C.c_int32), ("gate_temp", C.c_float),
                ("route_scale", C.c_float), ("swiglu_limit", C.c_float)]


def cfg(dim, inter, n_routed, topk, norm_topk_prob=True, gate_temp=1.0, route_scale=2.5,
        swiglu_limit=7.0) -> Cfg:
    return Cfg(dim, inter, n_routed, topk, int(bool(norm_topk_prob)), gate_temp, route_scale,
               swiglu_limit)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(LIB)
            P = C.c_void_p
            L.orc_bf16_from_f32.restype = C.c_uint16
            L.orc_bf16_from_f32.argtypes = [C.c_float]
            L.orc_bf16_to_f64.restype = C.c_double
            L.orc_bf16_to_f64.argtypes = [C.c_uint16]
            L.orc_f16_to_f64.restype = C.c_double
            L.orc_f16_to_f64.argtypes = [C.c_uint16]
            L.orc_f16_from_f32.restype = C.c_uint16
            L.orc_f16_from_f32.argtypes = [C.c_float]
            for f in ("orc_dequant_q2k", "orc_dequant_q3k", "orc_dequant_q8_1",
                      "orc_quantize_q2k", "orc_quantize_q3k"):
                getattr(L, f).restype = None
                getattr(L, f).argtypes = [P, P]
            L.orc_quant_q8_1.restype = None
            L.orc_quant_q8_1.argtypes = [P, C.c_int, P]
            L.orc_router_logits.restype = None
            L.orc_router_logits.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P]
            L.orc_score.restype = C.c_float
            L.orc_score.argtypes = [C.c_float, C.c_float, C.POINTER(C.c_int)]
            L.orc_route.restype = C.c_int
            L.orc_route.argtypes = [C.POINTER(Cfg), P, P, C.c_int, P, P, P, P]
            L.orc_plan.restype = C.c_int
            L.orc_plan.argtypes = [C.c_int, C.c_int, C.c_int, P, P, P, P, C.c_uint64, C.c_uint64,
                                   C.c_uint64, C.c_uint64, C.c_uint64, P, P, P, P]
            L.orc_swiglu.restype = C.c_double
            L.orc_swiglu.argtypes = [C.c_double, C.c_double, C.c_double]
            L.orc_expert_token.restype = None
            L.orc_expert_token.argtypes = [C.POINTER(Cfg), P, P, P, P, P, P, P, P, P, C.c_int]
            L.orc_shared_token.restype = None
            L.orc_shared_token.argtypes = [C.POINTER(Cfg), P, P, P, P, P, P, P, P, C.c_int]
            L.orc_layer.restype = C.c_int
            L.orc_layer.argtypes = [C.POINTER(Cfg), C.c_int, P, P, P, P, C.c_uint64, C.c_uint64,
                                    C.c_uint64, P, P, P, C.c_int, P, P, P, P, P, P, P, P, C.c_int]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ------------------------------------------------------------------ numbers

def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    L = lib()
    x = _f32(x)
    return np.array([L.orc_bf16_from_f32(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    L = lib()
    h = _u16(h)
    return np.array([L.orc_bf16_to_f64(int(v)) for v in h.ravel()]).reshape(h.shape)


def f16_from_f32(x: np.ndarray) -> np.ndarray:
    L = lib()
    x = _f32(x)
    return np.array([L.orc_f16_from_f32(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def f16_to_f64(h: np.ndarray) -> np.ndarray:
    L = lib()
    h = _u16(h)
    return np.array([L.orc_f16_to_f64(int(v)) for v in h.ravel()]).reshape(h.shape)


# ------------------------------------------------------------------ blocks

def dequant_q2k(blocks: np.ndarray) -> np.ndarray:
    """(nb, 84) raw bytes -> (nb, 256) f64 weights."""
    L = lib()
    b = _u8(blocks).reshape(-1, 84)
    out = np.zeros((b.shape[0], 256))
    for i in range(b.shape[0]):
        row = np.ascontiguousarray(b[i])
        o = np.zeros(256)
        L.orc_dequant_q2k(_p(row), _p(o))
        out[i] = o
    return out


def dequant_q3k(blocks: np.ndarray) -> np.ndarray:
    L = lib()
    b = _u8(blocks).reshape(-1, 110)
    out = np.zeros((b.shape[0], 256))
    for i in range(b.shape[0]):
        row = np.ascontiguousarray(b[i])
        o = np.zeros(256)
        L.orc_dequant_q3k(_p(row), _p(o))
        out[i] = o
    return out


def quant_q8_1(x: np.ndarray) -> np.ndarray:
    """f32 values (multiple of 32) -> raw q8_1 bytes, shape (n/32, 36)."""
    x = _f32(x).ravel()
    out = np.zeros((x.size // 32, 36), dtype=np.uint8)
    lib().orc_quant_q8_1(_p(x), x.size, _p(out))
    return out


def dequant_q8_1(blocks: np.ndarray) -> np.ndarray:
    L = lib()
    b = _u8(blocks).reshape(-1, 36)
    out = np.zeros((b.shape[0], 32))
    for i in range(b.shape[0]):
        row = np.ascontiguousarray(b[i])
        o = np.zeros(32)
        L.orc_dequant_q8_1(_p(row), _p(o))
        out[i] = o
    return out


def quantize_q2k(x: np.ndarray) -> np.ndarray:
    """f32 values (multiple of 256) -> raw Q2_K blocks (n/256, 84)."""
    x = _f32(x).reshape(-1, 256)
    out = np.zeros((x.shape[0], 84), dtype=np.uint8)
    L = lib()
    for i in range(x.shape[0]):
        xi = np.ascontiguousarray(x[i])
        o = np.zeros(84, dtype=np.uint8)
        L.orc_quantize_q2k(_p(xi), _p(o))
        out[i] = o
    return out


def quantize_q3k(x: np.ndarray) -> np.ndarray:
    x = _f32(x).reshape(-1, 256)
    out = np.zeros((x.shape[0], 110), dtype=np.uint8)
    L = lib()
    for i in range(x.shape[0]):
        xi = np.ascontiguousarray(x[i])
        o = np.zeros(110, dtype=np.uint8)
        L.orc_quantize_q3k(_p(xi), _p(o))
        out[i] = o
    return out


# ------------------------------------------------------------------ routing

def router_logits(x_bf16: np.ndarray, w_bf16: np.ndarray) -> np.ndarray:
    x = _u16(x_bf16)
    w = _u16(w_bf16)
    m, dim = x.shape
    n = w.shape[0]
    out = np.zeros((m, n), dtype=np.float32)
    lib().orc_router_logits(_p(x), _p(w), dim, n, m, _p(out))
    return out


def score(logit: float, temp: float = 1.0):
    nm = C.c_int(0)
    s = lib().orc_score(float(logit), float(temp), C.byref(nm))
    return np.float32(s), bool(nm.value)


def route(c: Cfg, logits: np.ndarray, bias: np.ndarray):
    """-> picks (m,k) int32 in pick order, weights (m,k) f32, scores (m,n) f32, flags (m,)."""
    lg = _f32(logits).reshape(-1, c.n_routed)
    m = lg.shape[0]
    b = _f32(bias)
    picks = np.zeros((m, c.topk), dtype=np.int32)
    weights = np.zeros((m, c.topk), dtype=np.float32)
    scores = np.zeros((m, c.n_routed), dtype=np.float32)
    flags = np.zeros(m, dtype=np.int32)
    rc = lib().orc_route(C.byref(c), _p(lg), _p(b), m, _p(picks), _p(weights), _p(scores), _p(flags))
    assert rc == 0
    return picks, weights, scores, flags


def header_words(m: int, k: int) -> int:
    """Words of the route header of m tokens: m rows of 1 + 3k, then the plan
    tail (ne, m k + 1 pair starts, m k plan experts)."""
    return m * (1 + 3 * k) + 2 + 2 * m * k


def plan(picks, weights, flags, slot_row, arena, n_routed: int, fill: int = -7):
    """The header, plan weights / rows and pointer table of m tokens (see
    orc_plan). arena = (base, slot_bytes, gate_off, up_off, down_off). Header
    words the layout leaves unused keep `fill`. -> (hdr, plan_w, plan_rows,
    ptrs, ne)."""
    pk = np.ascontiguousarray(picks, dtype=np.int32)
    m, k = pk.shape
    w = _f32(weights).reshape(m, k)
    fl = np.ascontiguousarray(flags if flags is not None else np.zeros(m), dtype=np.int32)
    sr = np.ascontiguousarray(slot_row, dtype=np.int32)
    hdr = np.full(header_words(m, k), fill, np.int32)
    pw = np.zeros(m * k, np.float32)
    pr = np.zeros(m * k, np.int32)
    ptrs = np.zeros(3 * m * k, np.uint64)
    base, sb, go, uo, do = (int(v) for v in arena)
    ne = lib().orc_plan(m, k, int(n_routed), _p(pk), _p(w), _p(fl), _p(sr), base, sb, go, uo, do,
                        _p(hdr), _p(pw), _p(pr), _p(ptrs))
    return hdr, pw, pr, ptrs, ne


def swiglu(g: float, u: float, limit: float) -> float:
    return lib().orc_swiglu(float(g), float(u), float(limit))


# ------------------------------------------------------------------ experts / layer

def expert_token(c: Cfg, gate: np.ndarray, up: np.ndarray, down: np.ndarray, x_q8: np.ndarray,
                 threads: int = 1):
    """-> dict(g, u, h, h_q8, down) for one token through one routed expert."""
    g = np.zeros(c.inter, np.float32)
    u = np.zeros(c.inter, np.float32)
    h = np.zeros(c.inter, np.float32)
    hq = np.zeros((c.inter // 32, 36), np.uint8)
    dn = np.zeros(c.dim, np.float32)
    gate, up, down, xq = _u8(gate), _u8(up), _u8(down), _u8(x_q8)
    lib().orc_expert_token(C.byref(c), _p(gate), _p(up), _p(down), _p(xq), _p(g), _p(u), _p(h),
                           _p(hq), _p(dn), threads)
    return dict(g=g, u=u, h=h, h_q8=hq, down=dn)


def shared_token(c: Cfg, w1, w3, w2, x_bf16, threads: int = 1):
    gs = np.zeros(c.inter, np.float32)
    us = np.zeros(c.inter, np.float32)
    hs = np.zeros(c.inter, np.uint16)
    sd = np.zeros(c.dim, np.float32)
    w1, w3, w2, x = _u16(w1), _u16(w3), _u16(w2), _u16(x_bf16)
    lib().orc_shared_token(C.byref(c), _p(w1), _p(w3), _p(w2), _p(x), _p(gs), _p(us), _p(hs),
                           _p(sd), threads)
    return dict(gs=gs, us=us, hs=hs, sd=sd)


def layer(c: Cfg, x_bf16, router_w, bias, experts: dict, offsets, shared=None, residual=None,
          threads: int = 1, shared_kquant: bool = False):
    """One layer step over m tokens.

    experts: {expert id: slot image (uint8)}; offsets = (gate_off, up_off, down_off);
    shared = (w1, w3, w2) bf16 bit arrays, or with shared_kquant the Q2_K w1,
    w3 and Q3_K w2 blocks as uint8 arrays, or None; residual f32 (m, dim)
    (default zeros).
    Returns dict(logits, picks, weights, flags, acc, sd, residual, x_next).
    """
    x = _u16(x_bf16)
    m = x.shape[0]
    w = _u16(router_w)
    b = _f32(bias)
    keep = [_u8(experts[e]) if e in experts else None for e in range(c.n_routed)]
    table = (C.c_void_p * c.n_routed)(*[None if a is None else a.ctypes.data for a in keep])
    res = np.zeros((m, c.dim), np.float32) if residual is None else _f32(residual).copy()
    xn = np.zeros((m, c.dim), np.uint16)
    logits = np.zeros((m, c.n_routed), np.float32)
    picks = np.zeros((m, c.topk), np.int32)
    weights = np.zeros((m, c.topk), np.float32)
    flags = np.zeros(m, np.int32)
    acc = np.zeros((m, c.dim), np.float32)
    sd = np.zeros((m, c.dim), np.float32)
    if shared is not None:
        w1, w3, w2 = (_u8(a) if shared_kquant else _u16(a) for a in shared)
    else:
        w1 = w3 = w2 = None
    rc = lib().orc_layer(C.byref(c), m, _p(x), _p(w), _p(b), C.cast(table, C.c_void_p),
                         int(offsets[0]), int(offsets[1]), int(offsets[2]), _p(w1), _p(w3), _p(w2),
                         int(bool(shared_kquant)), _p(res), _p(xn), _p(logits), _p(picks), _p(weights), _p(flags), _p(acc),
                         _p(sd), threads)
    if rc != 0:
        raise KeyError("oracle layer: a picked expert has no host image")
    return dict(logits=logits, picks=picks, weights=weights, flags=flags, acc=acc, sd=sd,
                residual=res, x_next=xn)


# ------------------------------------------------------------------ tiny-layer inputs

def quantised_expert_image(seed: int, layer: int, expert: int, shp) -> np.ndarray:
    """One expert's slot image for the tiny layer: N(0, 0.02) weights from the seeded
    generator, quantised with the oracle's Q2_K (gate, up) and Q3_K (down) quantisers."""
    from moe_decode_quantized_gb300 import synth
    img = np.zeros(shp.slot_bytes, np.uint8)
    parts = ((shp.gate_off, shp.gate_bytes, quantize_q2k, 84, synth.T_GATE),
             (shp.up_off, shp.up_bytes, quantize_q2k, 84, synth.T_UP),
             (shp.down_off, shp.down_bytes, quantize_q3k, 110, synth.T_DOWN))
    for off, nbytes, quant, bb, t in parts:
        nw = nbytes // bb * 256
        w = synth.normal_f32(synth.tensor_key(seed, layer, synth.T_F32, 16 * t + expert), nw, 0.02)
        img[off:off + nbytes] = quant(w).ravel()
    return img

"""GB300-native engine for one decode step of a DeepSeek-style MoE layer whose
routed experts stay in raw Q2_K / Q3_K blocks.

Thin Python binding of libmoe.so (include/moe.h): every function only turns
torch tensors into device pointers and calls the C ABI function of the same
name; all arithmetic runs in the CUDA kernels. Tensors must live on the
current CUDA device; work is enqueued on the current torch stream unless a
`stream` (torch.cuda.Stream or raw handle) is given.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from . import _lib

MOE_HDR_MISS = 1
MOE_HDR_NONFINITE = 2
MOE_WS_TIMEOUT = 1
MOE_WS_PLAN = 2
MOE_WS_TRIPLE = 4
MOE_SHARED_BF16 = 0
MOE_SHARED_KQUANT = 1
MOE_GRAPH_SNAPSHOTS = 1
MOE_GRAPH_EAGER_FALLBACK = 2
MOE_GRAPH_TEST_FAIL_CAPTURE = 4
SLOT_TABLE_LAYERS = 64

__all__ = ["Config", "Arena", "Layer", "MoeError", "header_words", "workspace_bytes",
           "workspace_init", "router_logits", "quantize_q8_1", "route_select", "expert_step",
           "swiglu_q8", "layer_step", "host_io_bytes", "layer_step_host", "workspace_view",
           "read_status", "layer_step_profiled", "layer_step_static", "route_scores", "set_wait_limit_ns",
           "expert_step_unreleased", "gemm_bf16", "prefill_workspace_bytes", "prefill_step", "prefill_step_profiled", "prefill_status", "graph_snapshot_bytes", "HostSource",
           "ExpertCache", "slot_table_set", "dedupe_triples", "parse_header", "Graph"]


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def _check(rc: int):
    if rc != 0:
        raise MoeError(rc, _lib.moe().moe_last_error().decode())


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _ptr(t):
    """Device (or host) address of a tensor / array / int; None stays NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return C.c_void_p(t)
    if isinstance(t, np.ndarray):
        return C.c_void_p(t.ctypes.data)
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return C.c_void_p(t.data_ptr())


@dataclass
class Config:
    """Layer configuration (page spark_model/layers/moe_v41.rs, struct MoeV41Cfg)."""
    dim: int
    inter: int
    n_routed: int
    topk: int
    norm_topk_prob: bool = True
    max_tokens: int = 1
    gate_temp: float = 1.0
    route_scale: float = 2.5
    swiglu_limit: float = 7.0

    def c(self) -> _lib.MoeCfg:
        return _lib.MoeCfg(self.dim, self.inter, self.n_routed, self.topk, int(bool(self.norm_topk_prob)),
                           self.max_tokens, self.gate_temp, self.route_scale, self.swiglu_limit)


@dataclass
class Arena:
    """Device expert arena (page .../moe_v41/device_route.rs, fn arena_of)."""
    base: object
    slot_bytes: int
    gate_off: int
    up_off: int
    down_off: int

    def c(self) -> _lib.MoeArena:
        return _lib.MoeArena(_ptr(self.base), self.slot_bytes, self.gate_off, self.up_off, self.down_off)


@dataclass
class Layer:
    """One layer's resident weights (page spark_model/layers/moe_v41.rs, MoeV41LayerWeights).
    sh_format: MOE_SHARED_BF16 (bf16 w1, w3, w2) or MOE_SHARED_KQUANT (Q2_K w1,
    w3 and Q3_K w2 blocks, laid out as a routed expert's gate, up, down)."""
    router_w: object
    bias: object
    slot_row: object
    sh_w1: object = None
    sh_w3: object = None
    sh_w2: object = None
    sh_format: int = 0

    def c(self) -> _lib.MoeLayer:
        return _lib.MoeLayer(_ptr(self.router_w), _ptr(self.bias), _ptr(self.slot_row), _ptr(self.sh_w1),
                             _ptr(self.sh_w3), _ptr(self.sh_w2), int(self.sh_format))


class HostSource:
    """Expert slot images in host memory (include/moe.h, moe_host_source_create):
    images[layer][expert] -> a host array (pinned torch tensor or numpy), kept alive here."""

    def __init__(self, images, n_layers: int, n_routed: int, image_bytes: int):
        self._keep = images
        ptrs = (C.c_void_p * (n_layers * n_routed))()
        for l in range(n_layers):
            for e in range(n_routed):
                img = images[l][e]
                ptrs[l * n_routed + e] = img.data_ptr() if hasattr(img, "data_ptr") else img.ctypes.data
        h = C.c_void_p()
        _check(_lib.moe().moe_host_source_create(C.cast(ptrs, C.c_void_p), n_layers, n_routed, image_bytes,
                                                 C.byref(h)))
        self._h = h

    def close(self):
        if self._h:
            _lib.moe().moe_host_source_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ExpertCache:
    """LRU expert slots over an arena (include/moe.h, moe_cache_create). source:
    a HostSource (its fetch runs in the library), or a Python callable
    fetch(layer, expert, slot_address, slot_bytes, stream) -> int, or None."""

    def __init__(self, n_layers: int, n_routed: int, n_slots: int, arena: Arena, slot_table=None, source=None):
        lib = _lib.moe()
        self._keep = (arena, slot_table, source)
        if isinstance(source, HostSource):
            fn = C.cast(lib.moe_fetch_host_images, C.c_void_p)
            user = source._h
        elif source is not None:
            self._cb = _lib.FETCH_FN(lambda u, l, e, d, b, s: int(source(l, e, d, b, s)))
            fn = C.cast(self._cb, C.c_void_p)
            user = None
        else:
            fn, user = None, None
        h = C.c_void_p()
        _check(lib.moe_cache_create(n_layers, n_routed, n_slots, C.byref(arena.c()), _ptr(slot_table), fn, user,
                                    C.byref(h)))
        self._h = h

    def ensure(self, layer: int, experts, stream=None) -> int:
        e = np.ascontiguousarray(experts, dtype=np.int32)
        n = C.c_int(0)
        _check(_lib.moe().moe_cache_ensure(self._h, layer, C.c_void_p(e.ctypes.data), e.size, C.byref(n),
                                           _stream(stream)))
        return n.value

    def slot_of(self, layer: int, expert: int) -> int:
        sl = C.c_int32(0)
        _check(_lib.moe().moe_cache_slot_of(self._h, layer, expert, C.byref(sl)))
        return sl.value

    def stats(self):
        h, m, ev = C.c_uint64(0), C.c_uint64(0), C.c_uint64(0)
        _check(_lib.moe().moe_cache_stats(self._h, C.byref(h), C.byref(m), C.byref(ev)))
        return h.value, m.value, ev.value

    def close(self):
        if self._h:
            _lib.moe().moe_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def header_words(cfg: Config, m: int) -> int:
    n = _lib.moe().moe_header_words(C.byref(cfg.c()), m)
    if n < 0:
        _check(n)
    return n


def workspace_bytes(cfg: Config) -> int:
    b = C.c_size_t(0)
    _check(_lib.moe().moe_workspace_bytes(C.byref(cfg.c()), C.byref(b)))
    return b.value


def workspace_init(ws, stream=None):
    _check(_lib.moe().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def router_logits(cfg: Config, x, w, logits, m: int, stream=None):
    _check(_lib.moe().moe_router_logits(C.byref(cfg.c()), _ptr(x), _ptr(w), _ptr(logits), m, _stream(stream)))


def quantize_q8_1(cfg: Config, x, m: int, out, stream=None):
    _check(_lib.moe().moe_quantize_q8_1(C.byref(cfg.c()), _ptr(x), m, _ptr(out), _stream(stream)))


def route_select(cfg: Config, logits, bias, slot_row, arena: Arena, m: int, header, plan_w, plan_rows, ptrs,
                 stream=None):
    _check(_lib.moe().moe_route_select(C.byref(cfg.c()), _ptr(logits), _ptr(bias), _ptr(slot_row),
                                       C.byref(arena.c()), m, _ptr(header), _ptr(plan_w), _ptr(plan_rows),
                                       _ptr(ptrs), _stream(stream)))


def expert_step(cfg: Config, x, ptrs, plan_w, plan_rows, header, m: int, acc, ws, stream=None):
    _check(_lib.moe().moe_expert_step(C.byref(cfg.c()), _ptr(x), _ptr(ptrs), _ptr(plan_w), _ptr(plan_rows),
                                      _ptr(header), m, _ptr(acc), _ptr(ws), _stream(stream)))


def swiglu_q8(cfg: Config, g, u, rows: int, h, hq8, stream=None):
    _check(_lib.moe().moe_swiglu_q8(C.byref(cfg.c()), _ptr(g), _ptr(u), rows, _ptr(h), _ptr(hq8),
                                    _stream(stream)))


def layer_step(cfg: Config, layer: Layer, arena: Arena, x, residual, x_next, header, m: int, ws, stream=None):
    _check(_lib.moe().moe_layer_step(C.byref(cfg.c()), C.byref(layer.c()), C.byref(arena.c()), _ptr(x),
                                     _ptr(residual), _ptr(x_next), _ptr(header), m, _ptr(ws), _stream(stream)))


def layer_step_static(cfg: Config, layer: Layer, arena: Arena, x, residual, x_next, header, m: int,
                      status=None, stream=None):
    """layer_step on the library's own static device workspace (no allocation).
    status: None, or a host uint32 array of one element that receives the
    workspace status once the stream reaches the end of the call."""
    _check(_lib.moe().moe_layer_step_static(C.byref(cfg.c()), C.byref(layer.c()), C.byref(arena.c()), _ptr(x),
                                            _ptr(residual), _ptr(x_next), _ptr(header), m, _ptr(status),
                                            _stream(stream)))


def set_wait_limit_ns(ns: int):
    """Bound (ns) on every wait inside kernels enqueued from now on; 0 = 2 s."""
    _check(_lib.moe().moe_set_wait_limit_ns(int(ns)))


def expert_step_unreleased(cfg: Config, x, header, m: int, ws, stream=None):
    """The expert kernels with no router before them: their wait for the plan
    can only run out (a failure-handling check; see include/moe.h)."""
    _check(_lib.moe().moe_expert_step_unreleased(C.byref(cfg.c()), _ptr(x), _ptr(header), m, _ptr(ws),
                                                 _stream(stream)))


def route_scores(cfg: Config, logits, scores, count: int, stream=None):
    """scores[i] = the f32 chain sqrt(ln_1p(exp(logits[i] / gate_temp))), each step correctly rounded."""
    _check(_lib.moe().moe_route_scores(C.byref(cfg.c()), _ptr(logits), count, _ptr(scores), _stream(stream)))


def host_io_bytes(cfg: Config, m: int) -> int:
    b = C.c_size_t(0)
    _check(_lib.moe().moe_host_io_bytes(C.byref(cfg.c()), m, C.byref(b)))
    return b.value


def layer_step_host(cfg: Config, layer: Layer, arena: Arena, x_host, residual_host, x_next_host, header_host,
                    m: int, io, ws, stream=None):
    """Host buffers (pinned torch CPU tensors or numpy arrays) in and out."""
    _check(_lib.moe().moe_layer_step_host(C.byref(cfg.c()), C.byref(layer.c()), C.byref(arena.c()),
                                          _ptr(x_host), _ptr(residual_host), _ptr(x_next_host),
                                          _ptr(header_host), m, _ptr(io), _ptr(ws), _stream(stream)))


def layer_step_profiled(cfg: Config, layer: Layer, arena: Arena, x, residual, x_next, header, m: int, ws,
                        stream=None):
    """-> [ms router+select, ms gate/up, ms down] for one layer step (kernels not overlapped)."""
    ms = np.zeros(3, np.float32)
    _check(_lib.moe().moe_layer_step_profiled(C.byref(cfg.c()), C.byref(layer.c()), C.byref(arena.c()), _ptr(x),
                                              _ptr(residual), _ptr(x_next), _ptr(header), m, _ptr(ws),
                                              _stream(stream), C.c_void_p(ms.ctypes.data)))
    return ms


def workspace_view(cfg: Config, ws) -> dict:
    v = _lib.MoeWsView()
    _check(_lib.moe().moe_workspace_view(C.byref(cfg.c()), _ptr(ws), C.byref(v)))
    return {name: getattr(v, name) for name, _ in _lib.MoeWsView._fields_}


def read_status(ws, stream=None) -> int:
    s = C.c_uint32(0)
    _check(_lib.moe().moe_read_status(_ptr(ws), C.byref(s), _stream(stream)))
    return s.value


def slot_table_set(table, n_routed: int, triples, n: int, status=None, stream=None):
    _check(_lib.moe().moe_slot_table_set(_ptr(table), n_routed, _ptr(triples), n, _ptr(status),
                                         _stream(stream)))


def dedupe_triples(triples: np.ndarray) -> np.ndarray:
    """Last-write-wins dedupe of (layer, expert, slot) triples (host)."""
    t = np.ascontiguousarray(triples, dtype=np.int32).reshape(-1, 3).copy()
    n = C.c_int(0)
    _check(_lib.moe().moe_dedupe_triples(C.c_void_p(t.ctypes.data), t.shape[0], C.byref(n)))
    return t[:n.value].copy()


def parse_header(cfg: Config, header_host: np.ndarray, m: int, t: int):
    """-> (status, picks, weights) of token t from a header copied to the host."""
    h = np.ascontiguousarray(header_host, dtype=np.int32)
    st = np.zeros(1, np.int32)
    picks = np.zeros(cfg.topk, np.int32)
    w = np.zeros(cfg.topk, np.float32)
    _check(_lib.moe().moe_parse_header(C.byref(cfg.c()), C.c_void_p(h.ctypes.data), m, t,
                                       C.c_void_p(st.ctypes.data), C.c_void_p(picks.ctypes.data),
                                       C.c_void_p(w.ctypes.data)))
    return int(st[0]), picks, w


def gemm_bf16(a, b, d, M: int, N: int, K: int, ldd: int, stream=None):
    """d[n * ldd + r] = sum_k a[r, k] b[n, k] on the tensor cores (bf16 in, f32 out)."""
    _check(_lib.moe().moe_gemm_bf16(_ptr(a), _ptr(b), _ptr(d), M, N, K, ldd, _stream(stream)))


def prefill_workspace_bytes(cfg: Config, m: int) -> int:
    b = C.c_size_t(0)
    _check(_lib.moe().moe_prefill_workspace_bytes(C.byref(cfg.c()), m, C.byref(b)))
    return b.value


def prefill_step(cfg: Config, layer: Layer, arena: Arena, arena_slots: int, x, residual, x_next, picks, weights,
                 m: int, ws, stream=None):
    """The batched (prefill) layer step for m tokens (include/moe.h, moe_prefill_step)."""
    _check(_lib.moe().moe_prefill_step(C.byref(cfg.c()), C.byref(layer.c()), C.byref(arena.c()), int(arena_slots),
                                       _ptr(x), _ptr(residual), _ptr(x_next), _ptr(picks), _ptr(weights), m,
                                       _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def prefill_step_profiled(cfg: Config, layer: Layer, arena: Arena, arena_slots: int, x, residual, x_next, picks,
                          weights, m: int, ws, stream=None):
    """-> ms of the nine stages of one prefill step (include/moe.h, moe_prefill_step_profiled)."""
    ms = np.zeros(9, np.float32)
    _check(_lib.moe().moe_prefill_step_profiled(C.byref(cfg.c()), C.byref(layer.c()), C.byref(arena.c()),
                                                int(arena_slots), _ptr(x), _ptr(residual), _ptr(x_next), _ptr(picks),
                                                _ptr(weights), m, _ptr(ws), ws.numel() * ws.element_size(),
                                                _stream(stream), C.c_void_p(ms.ctypes.data)))
    return ms


def prefill_status(cfg: Config, m: int, ws, stream=None) -> int:
    s = C.c_uint32(0)
    _check(_lib.moe().moe_prefill_status(C.byref(cfg.c()), m, _ptr(ws), C.byref(s), _stream(stream)))
    return s.value


def graph_snapshot_bytes(cfg: Config, m: int, n_layers: int) -> int:
    b = C.c_size_t(0)
    _check(_lib.moe().moe_graph_snapshot_bytes(C.byref(cfg.c()), m, n_layers, C.byref(b)))
    return b.value


class Graph:
    """A captured multi-layer step (include/moe.h, moe_graph_create). snapshots:
    device memory of graph_snapshot_bytes (with MOE_GRAPH_SNAPSHOTS in flags)."""

    def __init__(self, cfg: Config, layers, arena: Arena, m: int, x_a, x_b, residual, headers, ws, snapshots=None,
                 flags: int = 0):
        arr = (_lib.MoeLayer * len(layers))(*[ly.c() for ly in layers])
        self._keep = (layers, arena, x_a, x_b, residual, headers, ws, snapshots)
        h = C.c_void_p()
        _check(_lib.moe().moe_graph_create(C.byref(cfg.c()), C.cast(arr, C.c_void_p), len(layers),
                                           C.byref(arena.c()), m, _ptr(x_a), _ptr(x_b), _ptr(residual),
                                           _ptr(headers), _ptr(ws), _ptr(snapshots), flags, C.byref(h)))
        self._h = h

    @property
    def eager(self) -> bool:
        e = C.c_int(0)
        _check(_lib.moe().moe_graph_is_eager(self._h, C.byref(e)))
        return bool(e.value)

    def rerun_from(self, layer: int, stream=None):
        _check(_lib.moe().moe_graph_rerun_from(self._h, layer, _stream(stream)))

    def step_cached(self, cache: "ExpertCache", headers_host: np.ndarray, stream=None) -> int:
        """One launch with misses fetched and the rest rerun (moe_graph_step_cached);
        -> layers rerun. headers_host: int32 numpy array of the graph's header rows."""
        n = C.c_int(0)
        _check(_lib.moe().moe_graph_step_cached(self._h, cache._h, C.c_void_p(headers_host.ctypes.data),
                                                C.byref(n), _stream(stream)))
        return n.value

    def launch(self, stream=None):
        _check(_lib.moe().moe_graph_launch(self._h, _stream(stream)))

    def launch_host(self, x_host, residual_host, x_out_host, residual_out_host, headers_host, stream=None):
        _check(_lib.moe().moe_graph_launch_host(self._h, _ptr(x_host), _ptr(residual_host), _ptr(x_out_host),
                                                _ptr(residual_out_host), _ptr(headers_host), _stream(stream)))

    def close(self):
        if self._h:
            _lib.moe().moe_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

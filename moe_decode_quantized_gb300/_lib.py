"""ctypes declarations of libmoe.so (include/moe.h) and libmoe_synth.so
(include/moe_synth.h). Loading fails loudly when a library is missing: there
is no fallback path."""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

_lock = threading.Lock()
_moe = None
_synth = None

P = C.c_void_p
I32 = C.c_int32
U64 = C.c_uint64
SZ = C.c_size_t


class MoeCfg(C.Structure):
    _fields_ = [("dim", I32), ("inter", I32), ("n_routed", I32), ("topk", I32),
                ("norm_topk_prob", I32), ("max_tokens", I32), ("gate_temp", C.c_float),
                ("route_scale", C.c_float), ("swiglu_limit", C.c_float)]


class MoeArena(C.Structure):
    _fields_ = [("base", P), ("slot_bytes", U64), ("gate_off", U64), ("up_off", U64),
                ("down_off", U64)]


class MoeLayer(C.Structure):
    _fields_ = [("router_w", P), ("bias", P), ("slot_row", P), ("sh_w1", P), ("sh_w3", P),
                ("sh_w2", P), ("sh_format", C.c_int32)]


class MoeWsView(C.Structure):
    _fields_ = [("logits", P), ("plan_w", P), ("plan_rows", P), ("ptrs", P), ("g", P), ("u", P),
                ("gs", P), ("us", P), ("down", P), ("sd", P), ("acc", P), ("status", P)]


# the type of an expert fetch callback (include/moe.h, moe_expert_fetch_fn)
FETCH_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_uint64, C.c_void_p)

# name -> (restype, argtypes); every symbol include/moe.h declares
MOE_SYMBOLS = {
    "moe_header_words": (C.c_int, [C.POINTER(MoeCfg), C.c_int]),
    "moe_workspace_bytes": (C.c_int, [C.POINTER(MoeCfg), C.POINTER(SZ)]),
    "moe_workspace_init": (C.c_int, [P, SZ, P]),
    "moe_router_logits": (C.c_int, [C.POINTER(MoeCfg), P, P, P, C.c_int, P]),
    "moe_quantize_q8_1": (C.c_int, [C.POINTER(MoeCfg), P, C.c_int, P, P]),
    "moe_route_select": (C.c_int, [C.POINTER(MoeCfg), P, P, P, C.POINTER(MoeArena), C.c_int, P, P,
                                   P, P, P]),
    "moe_route_scores": (C.c_int, [C.POINTER(MoeCfg), P, C.c_int, P, P]),
    "moe_expert_step": (C.c_int, [C.POINTER(MoeCfg), P, P, P, P, P, C.c_int, P, P, P]),
    "moe_swiglu_q8": (C.c_int, [C.POINTER(MoeCfg), P, P, C.c_int, P, P, P]),
    "moe_layer_step": (C.c_int, [C.POINTER(MoeCfg), C.POINTER(MoeLayer), C.POINTER(MoeArena), P, P,
                                 P, P, C.c_int, P, P]),
    "moe_layer_step_static": (C.c_int, [C.POINTER(MoeCfg), C.POINTER(MoeLayer), C.POINTER(MoeArena),
                                        P, P, P, P, C.c_int, P, P]),
    "moe_host_io_bytes": (C.c_int, [C.POINTER(MoeCfg), C.c_int, C.POINTER(SZ)]),
    "moe_layer_step_host": (C.c_int, [C.POINTER(MoeCfg), C.POINTER(MoeLayer), C.POINTER(MoeArena),
                                      P, P, P, P, C.c_int, P, P, P]),
    "moe_workspace_view": (C.c_int, [C.POINTER(MoeCfg), P, C.POINTER(MoeWsView)]),
    "moe_read_status": (C.c_int, [P, C.POINTER(C.c_uint32), P]),
    "moe_slot_table_set": (C.c_int, [P, C.c_int, P, C.c_int, P, P]),
    "moe_dedupe_triples": (C.c_int, [P, C.c_int, C.POINTER(C.c_int)]),
    "moe_parse_header": (C.c_int, [C.POINTER(MoeCfg), P, C.c_int, C.c_int, P, P, P]),
    "moe_graph_snapshot_bytes": (C.c_int, [C.POINTER(MoeCfg), C.c_int, C.c_int, C.POINTER(SZ)]),
    "moe_graph_create": (C.c_int, [C.POINTER(MoeCfg), P, C.c_int, C.POINTER(MoeArena), C.c_int, P,
                                   P, P, P, P, P, C.c_uint, C.POINTER(P)]),
    "moe_graph_is_eager": (C.c_int, [P, C.POINTER(C.c_int)]),
    "moe_graph_rerun_from": (C.c_int, [P, C.c_int, P]),
    "moe_cache_create": (C.c_int, [C.c_int, C.c_int, C.c_int, C.POINTER(MoeArena), P, P, P, C.POINTER(P)]),
    "moe_cache_destroy": (C.c_int, [P]),
    "moe_cache_ensure": (C.c_int, [P, C.c_int, P, C.c_int, C.POINTER(C.c_int), P]),
    "moe_cache_slot_of": (C.c_int, [P, C.c_int, C.c_int, C.POINTER(C.c_int32)]),
    "moe_cache_stats": (C.c_int, [P, C.POINTER(U64), C.POINTER(U64), C.POINTER(U64)]),
    "moe_host_source_create": (C.c_int, [P, C.c_int, C.c_int, U64, C.POINTER(P)]),
    "moe_host_source_destroy": (C.c_int, [P]),
    "moe_fetch_host_images": (C.c_int, [P, C.c_int, C.c_int, P, U64, P]),
    "moe_graph_step_cached": (C.c_int, [P, P, P, C.POINTER(C.c_int), P]),
    "moe_graph_launch": (C.c_int, [P, P]),
    "moe_graph_destroy": (C.c_int, [P]),
    "moe_graph_launch_host": (C.c_int, [P, P, P, P, P, P, P]),
    "moe_layer_step_profiled": (C.c_int, [C.POINTER(MoeCfg), C.POINTER(MoeLayer), C.POINTER(MoeArena), P,
                                          P, P, P, C.c_int, P, P, P]),
    "moe_set_wait_limit_ns": (C.c_int, [U64]),
    "moe_expert_step_unreleased": (C.c_int, [C.POINTER(MoeCfg), P, P, C.c_int, P, P]),
    "moe_gemm_bf16": (C.c_int, [P, P, P, C.c_int, C.c_int, C.c_int, C.c_int, P]),
    "moe_prefill_workspace_bytes": (C.c_int, [C.POINTER(MoeCfg), C.c_int, C.POINTER(SZ)]),
    "moe_prefill_step": (C.c_int, [C.POINTER(MoeCfg), C.POINTER(MoeLayer), C.POINTER(MoeArena), C.c_int64, P, P,
                                   P, P, P, C.c_int, P, SZ, P]),
    "moe_prefill_step_profiled": (C.c_int, [C.POINTER(MoeCfg), C.POINTER(MoeLayer), C.POINTER(MoeArena),
                                            C.c_int64, P, P, P, P, P, C.c_int, P, SZ, P, P]),
    "moe_prefill_status": (C.c_int, [C.POINTER(MoeCfg), C.c_int, P, C.POINTER(C.c_uint32), P]),
    "moe_last_error": (C.c_char_p, []),
}

SYNTH_SYMBOLS = {
    "moe_synth_q2k": (C.c_int, [P, U64, U64, P]),
    "moe_synth_q3k": (C.c_int, [P, U64, U64, P]),
    "moe_synth_normal_bf16": (C.c_int, [P, U64, U64, C.c_float, P]),
    "moe_synth_uniform_f32": (C.c_int, [P, U64, U64, C.c_float, C.c_float, P]),
}


def _open(path: str, symbols: dict):
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is not built: call "
                           "moe_decode_quantized_gb300.build.build() (nvcc, sm_103a)")
    lib = C.CDLL(path)
    for name, (res, args) in symbols.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def moe():
    global _moe
    with _lock:
        if _moe is None:
            if not os.path.exists(_build.LIBMOE):
                _build.build()
            _moe = _open(_build.LIBMOE, MOE_SYMBOLS)
    return _moe


def synth():
    global _synth
    with _lock:
        if _synth is None:
            if not os.path.exists(_build.LIBSYNTH):
                _build.build()
            _synth = _open(_build.LIBSYNTH, SYNTH_SYMBOLS)
    return _synth

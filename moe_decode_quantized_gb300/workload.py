"""Synthetic decode workloads on the device, built from the seeded generator.

A Workload holds n_layers independent MoE layers of one shape: one expert
arena with n_layers * n_routed slots (slot of (layer l, expert e) =
l * n_routed + e, so every expert is resident), the [64, n_routed] slot table,
and per layer the bf16 router, the f32 correction bias and (optionally) the
shared expert, bf16 or K-quant. Values follow synth.py: router ~N(0, 0.02),
bias ~U(-0.1, 0.1) (or a caller range), bf16 shared ~N(0, 0.02), experts
(and a K-quant shared expert) random Q2_K / Q3_K blocks. No arithmetic of the
layer lives here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (MOE_SHARED_BF16, MOE_SHARED_KQUANT, Arena, Config, Layer, SLOT_TABLE_LAYERS, synth, synth_gpu,
               workspace_bytes, workspace_init)

SHARED_KQ_INDEX = synth.SHARED_KQ_INDEX  # the K-quant shared expert's blocks: this expert index


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(device)


class Workload:
    def __init__(self, cfg: Config, n_layers: int = 1, seed: int = 0, shared: bool = True,
                 device="cuda", bias_range=(-0.1, 0.1), fill_experts: bool = True, shared_kquant: bool = False):
        assert n_layers <= SLOT_TABLE_LAYERS
        self.cfg, self.n_layers, self.seed, self.shared = cfg, n_layers, seed, shared
        self.shared_kquant = shared and shared_kquant
        self.device = torch.device(device)
        self.shape = shp = synth.LayerShape(cfg.dim, cfg.inter, cfg.n_routed)
        n = cfg.n_routed
        self.arena_t = torch.empty(n_layers * n * shp.slot_bytes, dtype=torch.uint8, device=self.device)
        self.arena = Arena(self.arena_t, shp.slot_bytes, shp.gate_off, shp.up_off, shp.down_off)
        table = np.full((SLOT_TABLE_LAYERS, n), -1, np.int32)
        for l in range(n_layers):
            table[l] = np.arange(l * n, (l + 1) * n, dtype=np.int32)
        self.slot_table = torch.from_numpy(table).to(self.device)
        self.router, self.bias, self.sh = [], [], []
        base = self.arena_t.data_ptr()
        for l in range(n_layers):
            w = torch.empty((n, cfg.dim), dtype=torch.int16, device=self.device)
            synth_gpu.normal_bf16(w, w.numel(), synth.tensor_key(seed, l, synth.T_ROUTER), 0.02)
            b = torch.empty(n, dtype=torch.float32, device=self.device)
            synth_gpu.uniform_f32(b, n, synth.tensor_key(seed, l, synth.T_BIAS), *bias_range)
            self.router.append(w)
            self.bias.append(b)
            if self.shared_kquant:
                # Q2_K w1, w3 and Q3_K w2 laid out as an expert slot (synthetic
                # blocks of expert index SHARED_KQ_INDEX)
                buf = torch.empty(shp.slot_bytes, dtype=torch.uint8, device=self.device)
                synth_gpu.fill_expert(buf.data_ptr(), seed, l, SHARED_KQ_INDEX, shp)
                self.sh.append((buf[shp.gate_off:], buf[shp.up_off:], buf[shp.down_off:]))
                self.sh_bufs = getattr(self, "sh_bufs", []) + [buf]
            elif shared:
                w1 = torch.empty((cfg.inter, cfg.dim), dtype=torch.int16, device=self.device)
                w3 = torch.empty((cfg.inter, cfg.dim), dtype=torch.int16, device=self.device)
                w2 = torch.empty((cfg.dim, cfg.inter), dtype=torch.int16, device=self.device)
                synth_gpu.normal_bf16(w1, w1.numel(), synth.tensor_key(seed, l, synth.T_SH_W1), 0.02)
                synth_gpu.normal_bf16(w3, w3.numel(), synth.tensor_key(seed, l, synth.T_SH_W3), 0.02)
                synth_gpu.normal_bf16(w2, w2.numel(), synth.tensor_key(seed, l, synth.T_SH_W2), 0.02)
                self.sh.append((w1, w3, w2))
            if fill_experts:
                for e in range(n):
                    synth_gpu.fill_expert(base + (l * n + e) * shp.slot_bytes, seed, l, e, shp)
        self.bias_range = bias_range
        self.ws = torch.empty(workspace_bytes(cfg), dtype=torch.uint8, device=self.device)
        workspace_init(self.ws)

    # ------------------------------------------------------------------ views
    def layer(self, l: int) -> Layer:
        sh = self.sh[l] if self.shared else (None, None, None)
        return Layer(self.router[l], self.bias[l], self.slot_table[l], *sh,
                     sh_format=MOE_SHARED_KQUANT if self.shared_kquant else MOE_SHARED_BF16)

    def slot_of(self, l: int, e: int) -> int:
        return l * self.cfg.n_routed + e

    def set_expert_image(self, l: int, e: int, img: np.ndarray):
        """Overwrite one slot with a host-made image (e.g. the tiny layer's quantised experts)."""
        off = self.slot_of(l, e) * self.shape.slot_bytes
        self.arena_t[off:off + self.shape.slot_bytes].copy_(torch.from_numpy(np.ascontiguousarray(img)))

    # host copies of the same inputs (for the oracle)
    def host_router(self, l: int) -> np.ndarray:
        return synth.router_bf16(self.seed, l, self.cfg.n_routed, self.cfg.dim)

    def host_bias(self, l: int) -> np.ndarray:
        return synth.bias_f32(self.seed, l, self.cfg.n_routed, *self.bias_range)

    def host_shared(self, l: int):
        """bf16 (w1, w3, w2) bit arrays, or the K-quant blocks as uint8 arrays."""
        if self.shared_kquant:
            img = np.frombuffer(synth.expert_bytes(self.seed, l, SHARED_KQ_INDEX, self.shape), np.uint8)
            shp = self.shape
            return (img[shp.gate_off:shp.gate_off + shp.gate_bytes], img[shp.up_off:shp.up_off + shp.up_bytes],
                    img[shp.down_off:shp.down_off + shp.down_bytes])
        return synth.shared_bf16(self.seed, l, self.cfg.dim, self.cfg.inter) if self.shared else None

    def host_expert(self, l: int, e: int) -> np.ndarray:
        return synth.expert_bytes(self.seed, l, e, self.shape)


def x_tensor(seed: int, batch: int, m: int, dim: int, device="cuda") -> torch.Tensor:
    return bf16_tensor(synth.x_bf16(seed, batch, m, dim), device)

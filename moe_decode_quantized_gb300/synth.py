"""Seeded synthetic inputs for the MoE decode layer (host side).

This module makes INPUTS only. It holds none of the layer's arithmetic: no
dequantisation, no dot products, no routing. Both the CUDA path and the CPU
oracle consume what it produces; `csrc/synth.cu` is its device twin, which
writes the same bytes straight into device memory for the multi-GB expert
arenas (the twin is checked byte-for-byte against this module by the tests).

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used in counter mode. Every tensor has its
own 64-bit key, derived from (seed, layer, tensor id, index); word i of that
tensor is mix64(key + (i + 1) * GOLDEN). All derived values use integer
operations or single IEEE-rounded f32 operations, so host and device agree bit
for bit.

Value recipes (the shapes follow the DeepSeek-style decode layer the pages
describe: bf16 activations and router, f32 correction bias, raw Q2_K / Q3_K
expert blocks):

* approx-normal f32: the four 16-bit fields of one word summed (Irwin-Hall,
  n = 4), centred, times an f32 scale so the standard deviation is `sigma`;
  tails are cut at 3.46 sigma.
* bf16: the approx-normal f32 rounded to nearest-even bf16.
* uniform f32 in [lo, hi): the top 24 bits of a word as u * 2^-24, then
  lo + (hi - lo) * u with two f32 roundings.
* Q2_K blocks (84 B), centred like quantised weights: random quants, each
  sub-block's scale sc in 0..5 with min 3 sc, f16 `d` in [2^-9, 2^-8) and
  `dmin` = d / 2, so every weight is d * sc * (q - 1.5) (uniform random bytes
  everywhere would make biased weights whose dot products grow with the
  length instead of its square root).
* random Q3_K blocks (110 B): uniform random bytes, except that the high byte
  of the f16 `d` field is forced into [2^-12, 2^-11).
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
M64 = (1 << 64) - 1

# tensor ids inside a key
T_X = 1
T_ROUTER = 2
T_BIAS = 3
T_SH_W1 = 4
T_SH_W3 = 5
T_SH_W2 = 6
T_GATE = 7
T_UP = 8
T_DOWN = 9
T_F32 = 10        # plain approx-normal f32 (inputs to the oracle's quantiser)
SHARED_KQ_INDEX = 4095  # expert index in the generator's keys of a K-quant shared expert
T_LOGITS = 11     # synthetic logits fed straight to the selection

# the Irwin-Hall (n=4) standard deviation of a sum of four u16 fields
IH4_SIGMA = float(np.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0))
IH4_MEAN2 = 131070  # 4 * 65535 / 2

Q2K_BYTES = 84
Q3K_BYTES = 110
QK = 256


def _mix64_int(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * MIX1) & M64
    z = ((z ^ (z >> 27)) * MIX2) & M64
    return z ^ (z >> 31)


def tensor_key(seed: int, layer: int, tensor: int, index: int = 0) -> int:
    """64-bit key of one tensor: mix64(mix64(seed*GOLDEN + 1) ^ packed id)."""
    base = _mix64_int((seed * GOLDEN + 1) & M64)
    packed = ((layer & 0xFFFFFF) << 40) | ((tensor & 0xFF) << 32) | (index & 0xFFFFFFFF)
    return _mix64_int(base ^ packed)


def words(key: int, start: int, count: int) -> np.ndarray:
    """Words start .. start+count-1 of the tensor keyed `key` (uint64)."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(key) + i * np.uint64(GOLDEN)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        return z ^ (z >> np.uint64(31))


def normal_scale(sigma: float) -> np.float32:
    """The f32 factor that turns a centred Irwin-Hall sum into std `sigma`."""
    return np.float32(sigma / IH4_SIGMA)


def normal_f32(key: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    w = words(key, start, n)
    s = ((w & np.uint64(0xFFFF)) + ((w >> np.uint64(16)) & np.uint64(0xFFFF))
         + ((w >> np.uint64(32)) & np.uint64(0xFFFF)) + (w >> np.uint64(48)))
    v = s.astype(np.int64) - IH4_MEAN2           # |v| < 2^18: exact in f32
    return v.astype(np.float32) * normal_scale(sigma)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even f32 -> bf16 bit patterns (uint16)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) & np.uint64(0xFFFF)
    return r.astype(np.uint16)


def normal_bf16(key: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    """bf16 bit patterns (uint16) of approx-normal values."""
    return f32_to_bf16_bits(normal_f32(key, n, sigma, start))


def uniform_f32(key: int, n: int, lo: float, hi: float, start: int = 0) -> np.ndarray:
    w = words(key, start, n)
    u = (w >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    a = np.float32(np.float32(hi) - np.float32(lo))
    return (u * a) + np.float32(lo)


def random_bytes(key: int, nbytes: int) -> np.ndarray:
    nw = (nbytes + 7) // 8
    return words(key, 0, nw).view(np.uint8)[:nbytes].copy()


def q2k_blocks(key: int, nblocks: int) -> np.ndarray:
    """`nblocks` random Q2_K super-blocks as raw bytes, shape (nblocks, 84),
    centred like quantised weights: every sub-block's min is 3x its scale
    (scale sc in 0..5, min 3 sc) and dmin = d / 2, so that each weight is
    d * sc * (q - 1.5); random quants, d in [2^-9, 2^-8)."""
    r = random_bytes(key, nblocks * Q2K_BYTES).reshape(nblocks, Q2K_BYTES)
    b = r.copy()
    sc = ((r[:, :16] & 0x0F).astype(np.uint32) * 6) >> 4                  # 0..5
    b[:, :16] = (sc | ((3 * sc) << 4)).astype(np.uint8)                  # scale | min << 4
    b[:, 81] = (r[:, 81] & 0x03) | 0x18                                    # d in [2^-9, 2^-8)
    b[:, 82] = r[:, 80]                                                    # dmin = d / 2:
    b[:, 83] = (r[:, 81] & 0x03) | 0x14                                    # exponent one lower
    return b


def q3k_blocks(key: int, nblocks: int) -> np.ndarray:
    """`nblocks` random Q3_K super-blocks as raw bytes, shape (nblocks, 110)."""
    b = random_bytes(key, nblocks * Q3K_BYTES).reshape(nblocks, Q3K_BYTES)
    b[:, 109] = (b[:, 109] & 0x03) | 0x0C  # d in [2^-12, 2^-11)
    return b


# ---------------------------------------------------------------- layer recipe

class LayerShape:
    """Sizes of one MoE layer and of its expert slot in the arena."""

    def __init__(self, dim: int, inter: int, n_routed: int):
        assert dim % QK == 0 and inter % QK == 0
        self.dim, self.inter, self.n_routed = dim, inter, n_routed
        self.gate_bytes = inter * (dim // QK) * Q2K_BYTES
        self.up_bytes = self.gate_bytes
        self.down_bytes = dim * (inter // QK) * Q3K_BYTES
        a = lambda v: (v + 255) // 256 * 256
        self.gate_off = 0
        self.up_off = a(self.gate_bytes)
        self.down_off = self.up_off + a(self.up_bytes)
        self.slot_bytes = a(self.down_off + self.down_bytes)


def expert_bytes(seed: int, layer: int, expert: int, shp: LayerShape) -> bytes:
    """One expert's slot image: gate | up | down raw blocks at their offsets."""
    out = np.zeros(shp.slot_bytes, dtype=np.uint8)
    nq2 = shp.gate_bytes // Q2K_BYTES
    nq3 = shp.down_bytes // Q3K_BYTES
    out[shp.gate_off:shp.gate_off + shp.gate_bytes] = q2k_blocks(
        tensor_key(seed, layer, T_GATE, expert), nq2).ravel()
    out[shp.up_off:shp.up_off + shp.up_bytes] = q2k_blocks(
        tensor_key(seed, layer, T_UP, expert), nq2).ravel()
    out[shp.down_off:shp.down_off + shp.down_bytes] = q3k_blocks(
        tensor_key(seed, layer, T_DOWN, expert), nq3).ravel()
    return out


def x_bf16(seed: int, batch: int, m: int, dim: int) -> np.ndarray:
    """m activation rows ~N(0, 1) (approx), bf16 bits, shape (m, dim)."""
    return normal_bf16(tensor_key(seed, batch, T_X), m * dim, 1.0).reshape(m, dim)


def router_bf16(seed: int, layer: int, n_routed: int, dim: int) -> np.ndarray:
    return normal_bf16(tensor_key(seed, layer, T_ROUTER), n_routed * dim, 0.02).reshape(n_routed, dim)


def bias_f32(seed: int, layer: int, n_routed: int, lo: float = -0.1, hi: float = 0.1) -> np.ndarray:
    return uniform_f32(tensor_key(seed, layer, T_BIAS), n_routed, lo, hi)


def shared_bf16(seed: int, layer: int, dim: int, inter: int):
    """Shared expert (w1 [inter,dim], w3 [inter,dim], w2 [dim,inter]) ~N(0, 0.02)."""
    w1 = normal_bf16(tensor_key(seed, layer, T_SH_W1), inter * dim, 0.02).reshape(inter, dim)
    w3 = normal_bf16(tensor_key(seed, layer, T_SH_W3), inter * dim, 0.02).reshape(inter, dim)
    w2 = normal_bf16(tensor_key(seed, layer, T_SH_W2), dim * inter, 0.02).reshape(dim, inter)
    return w1, w3, w2


def tie_logits(seed: int, batch: int, m: int, n_routed: int, step: float = 2.0 ** -4) -> np.ndarray:
    """Logits on a 2^-4 grid (many exact ties), shape (m, n_routed), f32."""
    v = normal_f32(tensor_key(seed, batch, T_LOGITS), m * n_routed, 1.3)
    return (np.rint(v / np.float32(step)) * np.float32(step)).astype(np.float32).reshape(m, n_routed)


def round_to_grid(v: np.ndarray, step: float = 2.0 ** -4) -> np.ndarray:
    return (np.rint(v / np.float32(step)) * np.float32(step)).astype(np.float32)

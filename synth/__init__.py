"""Seeded synthetic inputs for the MXFP4 routed-expert MoE layer.

This module only draws random numbers and lays them out in the boundary's
storage formats (bf16 bit patterns, packed E2M1 nibbles, E8M0 scale bytes).
It holds none of the layer's arithmetic: no quantisation, no dot products,
no routing.  Both the oracle tests and the CUDA tests take their inputs from
here, so neither side ever produces the other's inputs.

Generator: a counter-based SplitMix64.  Every tensor of a layer owns a stream
id; element ``i`` of that stream is ``mix(base(seed, stream) + i * GAMMA)``, so
any slice of any tensor (one expert, one token) can be drawn on its own and
always gets the same values.

Workload recipe (the shapes are the MoE layer of the DeepSeek-V4-Flash pages:
256 routed experts, top-6, hidden 4096, expert intermediate 2048):
  * router weights N(0, 0.02), fp32 (tiny layer) or bf16;
  * expert gate/up/down weights: uniform random 4-bit E2M1 codes, two per
    byte, plus one E8M0 byte per 32 values with exponent uniform in [-4, 0]
    (byte 123..127);
  * activations N(0, 1), fp32 (tiny layer) or bf16;
  * optional router-logit bias ln p_e with p a Zipf(s) law over a seeded
    permutation of the experts (skewed "concurrent serving" routing).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)

# stream ids
S_ROUTER = 1
S_X = 2
S_PERM = 3
S_EXPERT0 = 16  # expert e, tensor j in [0, 6): S_EXPERT0 + 8 * e + j
S_SHARED0 = 8   # the shared expert, tensor j in [0, 6): S_SHARED0 + j
T_WG, T_SG, T_WU, T_SU, T_WD, T_SD = range(6)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Elements [start, start+count) of one SplitMix64 counter stream."""
    with np.errstate(over="ignore"):
        base = _mix(np.array([seed], dtype=np.uint64) * GAMMA
                    + np.array([stream], dtype=np.uint64) * _STREAM_MUL)[0]
        idx = np.arange(start, start + count, dtype=np.uint64)
        return _mix(base + idx * GAMMA)


def uniform01(seed, stream, start, count) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (raw_u64(seed, stream, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed, stream, start, count, std=1.0) -> np.ndarray:
    """Box-Muller normals; sample i uses counters 2i and 2i+1."""
    r = raw_u64(seed, stream, 2 * start, 2 * count)
    u1 = ((r[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (r[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return std * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def random_bytes(seed, stream, nbytes: int) -> np.ndarray:
    """nbytes uniform random bytes (8 per counter value)."""
    n64 = (nbytes + 7) // 8
    return raw_u64(seed, stream, 0, n64).view(np.uint8)[:nbytes].copy()


def e8m0_bytes(seed, stream, count: int, lo: int = -4, hi: int = 0) -> np.ndarray:
    """E8M0 scale bytes 127 + e with e uniform in [lo, hi]."""
    span = np.uint64(hi - lo + 1)
    r = raw_u64(seed, stream, 0, count) >> np.uint64(32)
    e = ((r * span) >> np.uint64(32)).astype(np.int64) + lo
    return (127 + e).astype(np.uint8)


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """Shape and storage types of one MoE layer.

    H hidden size, E routed experts, k experts per token, I expert
    intermediate size.  x_dtype / wr_dtype are "f32" or "bf16".
    """
    H: int
    E: int
    k: int
    I: int
    x_dtype: str = "bf16"
    wr_dtype: str = "bf16"
    seed: int = 0
    zipf_s: float | None = None  # router-logit bias ln p_e, p ~ Zipf(s)

    @property
    def expert_bytes(self) -> int:
        H, I = self.H, self.I
        return 2 * (I * H // 2 + I * H // 32) + (H * I // 2 + H * I // 32)


# The workloads of the pages' layer (DeepSeek-V4-Flash routed experts).
TINY = LayerSpec(H=256, E=8, k=2, I=128, x_dtype="f32", wr_dtype="f32")
DSV4 = LayerSpec(H=4096, E=256, k=6, I=2048, x_dtype="bf16", wr_dtype="bf16")
DSV4_ZIPF = dataclasses.replace(DSV4, zipf_s=1.1)


def router_weights(spec: LayerSpec) -> np.ndarray:
    """[E, H] router weights N(0, 0.02); float32, or uint16 bf16 bits."""
    w = normal(spec.seed, S_ROUTER, 0, spec.E * spec.H, std=0.02).astype(np.float32)
    w = w.reshape(spec.E, spec.H)
    return f32_to_bf16_bits(w) if spec.wr_dtype == "bf16" else w


def router_bias(spec: LayerSpec) -> np.ndarray | None:
    """Per-expert logit bias ln p_e, p = Zipf(s) over a seeded permutation."""
    if spec.zipf_s is None:
        return None
    keys = raw_u64(spec.seed, S_PERM, 0, spec.E)
    perm = np.argsort(keys, kind="stable")  # perm[rank] = expert id
    rank = np.empty(spec.E, dtype=np.int64)
    rank[perm] = np.arange(spec.E)
    p = (rank + 1.0) ** (-spec.zipf_s)
    p /= p.sum()
    return np.log(p).astype(np.float32)


def activations(spec: LayerSpec, T: int, token0: int = 0) -> np.ndarray:
    """[T, H] activations N(0, 1) for tokens token0..token0+T-1."""
    x = normal(spec.seed, S_X, token0 * spec.H, T * spec.H).astype(np.float32).reshape(T, spec.H)
    return f32_to_bf16_bits(x) if spec.x_dtype == "bf16" else x


@dataclasses.dataclass
class ExpertWeights:
    """One routed expert in boundary layout (row-major, K contiguous).

    wg, wu: [I, H/2] uint8, element 2c in the low nibble of byte c, 2c+1 high.
    sg, su: [I, H/32] uint8 E8M0.  wd: [H, I/2] uint8, sd: [H, I/32] uint8.
    """
    wg: np.ndarray
    sg: np.ndarray
    wu: np.ndarray
    su: np.ndarray
    wd: np.ndarray
    sd: np.ndarray


def expert(spec: LayerSpec, e: int) -> ExpertWeights:
    H, I, s = spec.H, spec.I, spec.seed
    base = S_EXPERT0 + 8 * e
    return ExpertWeights(
        wg=random_bytes(s, base + T_WG, I * H // 2).reshape(I, H // 2),
        sg=e8m0_bytes(s, base + T_SG, I * H // 32).reshape(I, H // 32),
        wu=random_bytes(s, base + T_WU, I * H // 2).reshape(I, H // 2),
        su=e8m0_bytes(s, base + T_SU, I * H // 32).reshape(I, H // 32),
        wd=random_bytes(s, base + T_WD, H * I // 2).reshape(H, I // 2),
        sd=e8m0_bytes(s, base + T_SD, H * I // 32).reshape(H, I // 32),
    )


def shared_expert(spec: LayerSpec) -> ExpertWeights:
    """The layer's shared expert: the routed experts' format and shape, drawn
    from its own streams."""
    H, I, s = spec.H, spec.I, spec.seed
    return ExpertWeights(
        wg=random_bytes(s, S_SHARED0 + T_WG, I * H // 2).reshape(I, H // 2),
        sg=e8m0_bytes(s, S_SHARED0 + T_SG, I * H // 32).reshape(I, H // 32),
        wu=random_bytes(s, S_SHARED0 + T_WU, I * H // 2).reshape(I, H // 2),
        su=e8m0_bytes(s, S_SHARED0 + T_SU, I * H // 32).reshape(I, H // 32),
        wd=random_bytes(s, S_SHARED0 + T_WD, H * I // 2).reshape(H, I // 2),
        sd=e8m0_bytes(s, S_SHARED0 + T_SD, H * I // 32).reshape(H, I // 32),
    )


def int8_codes(seed, stream, rows, cols, lo=-127, hi=127) -> np.ndarray:
    """Uniform int8 codes in [lo, hi] (stage tests feed these as Q8 values)."""
    span = np.uint64(hi - lo + 1)
    r = raw_u64(seed, stream, 0, rows * cols) >> np.uint64(32)
    return (((r * span) >> np.uint64(32)).astype(np.int64) + lo).astype(np.int8).reshape(rows, cols)


def positive_scales(seed, stream, rows, cols, lo=1e-3, hi=1e-1) -> np.ndarray:
    """Log-uniform fp32 scales in [lo, hi]."""
    u = uniform01(seed, stream, 0, rows * cols)
    return np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo))).astype(np.float32).reshape(rows, cols)

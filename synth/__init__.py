"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the method (no activation, selection,
projection or quantisation step). It only draws numbers and shapes them like
the workloads the pages evaluate on, so that both sides of a parity test read
the same bf16 values.

Generator (counter based, identical on every machine):

* ``splitmix64`` finaliser (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014): ``z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9; z ^= z >> 27; z *= 0x94D049BB133111EB;
  z ^= z >> 31`` on uint64, wrapping.
* A stream is named by ``(seed, layer, tensor_id)``. Its key is
  ``k = mix(mix(mix(seed + G) ^ ((layer + 1) * G)) ^ ((tensor_id + 1) * G))``
  with ``G = 0x9E3779B97F4A7C15``; element ``i`` of the stream draws
  ``u_i = ((mix(k + (i + 1) * G) >> 11) + 0.5) * 2**-53``, uniform on (0, 1).
* Normals use the Box-Muller transform on consecutive pairs
  ``(u_{2m}, u_{2m+1})``: ``r = sqrt(-2 ln u_{2m})``, element ``2m`` is
  ``r cos(2 pi u_{2m+1})`` and element ``2m+1`` is ``r sin(2 pi u_{2m+1})``,
  computed in float64.
* bf16 values are produced from float64 by rounding to float32 (numpy,
  round-to-nearest-even) and then to bf16 (round-to-nearest-even on the bit
  pattern). Arrays of bf16 are returned as ``uint16`` bit patterns.

Workloads follow the FFN shapes of Llama3.2-1B/3B, Qwen2.5-3B and
Llama-3.1-8B that the SelectInfer and SpAx pages evaluate: weights
~N(0, 0.02), each gate row scaled by a per-neuron LogNormal(0, sigma) factor,
tokens ~N(0, 1).
"""
from __future__ import annotations

import dataclasses
import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids of the streams; fixed so that every consumer draws the same data
T_WGATE, T_WUP, T_WDOWN, T_GATE_SCALE = 1, 2, 3, 4
T_CALIB, T_PROMPT, T_DECODE = 5, 6, 7
T_ABSACT, T_SCORES_A, T_SCORES_B, T_SPAX_A, T_MISC = 8, 9, 10, 11, 12


def _mix(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z ^ (z >> np.uint64(30))
        z = z * _M1
        z = z ^ (z >> np.uint64(27))
        z = z * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, layer: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = _mix(np.uint64(seed) + _G)
        k = _mix(k ^ (np.uint64(layer + 1) * _G))
        k = _mix(k ^ (np.uint64(tensor_id + 1) * _G))
    return np.uint64(k)


def uniform(seed: int, layer: int, tensor_id: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` uniforms on (0, 1), elements ``offset .. offset+n-1`` of the stream."""
    k = stream_key(seed, layer, tensor_id)
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix(k + i * _G)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, layer: int, tensor_id: int, n: int, chunk: int = 1 << 24) -> np.ndarray:
    """``n`` standard normals (float64) of stream ``(seed, layer, tensor_id)``."""
    out = np.empty(n, dtype=np.float64)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, chunk):
        p1 = min(npairs, p0 + chunk)
        u = uniform(seed, layer, tensor_id, 2 * (p1 - p0), offset=2 * p0)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = 2.0 * np.pi * u2
        pair = np.empty(2 * (p1 - p0), dtype=np.float64)
        pair[0::2] = r * np.cos(th)
        pair[1::2] = r * np.sin(th)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = pair[: hi - lo]
    return out


def to_bf16_bits(x) -> np.ndarray:
    """float64/float32 -> bf16 bit patterns (uint16), via float32, both steps RNE."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16).reshape(f.shape)


def bf16_bits_to_f32(h) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact widening)."""
    h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------- workloads


@dataclasses.dataclass(frozen=True)
class Workload:
    """One of the evaluated FFN shapes and its selection parameters."""

    name: str
    d: int            # hidden size
    N: int            # FFN intermediate size d_ff (number of neurons)
    L: int            # layers
    gamma: float      # loaded ratio
    delta: float      # static (base) ratio
    phi: float        # computed ratio, phi = delta + epsilon
    alpha: int        # per-token top-alpha count
    T: int            # prompt tokens per sequence
    B: int            # sequences
    decode_tokens: int
    calib_tokens: int
    sigma: float      # gate-row LogNormal(0, sigma) scale
    spax: bool = False
    top_frac: float = 0.0
    mid_frac: float = 0.0
    group: int = 128
    bits: int = 4


WORKLOADS = {
    "tiny-d256": Workload("tiny-d256 (single FFN layer d=256, d_ff=1024)", 256, 1024, 1,
                          0.7, 0.2, 0.4, 64, 32, 1, 16, 128, 1.0),
    "llama3.2-1b": Workload("Llama3.2-1B FFN stack (16 x d=2048, d_ff=8192)", 2048, 8192, 16,
                            0.7, 0.2, 0.4, 1024, 512, 1, 256, 4096, 1.0),
    "llama3.2-3b": Workload("Llama3.2-3B FFN stack (28 x d=3072, d_ff=8192)", 3072, 8192, 28,
                            0.7, 0.25, 0.5, 1024, 1024, 1, 512, 4096, 1.0),
    "qwen2.5-3b": Workload("Qwen2.5-3B FFN stack (36 x d=2048, d_ff=11008), 8 prompts", 2048, 11008, 36,
                           0.8, 0.25, 0.5, 1024, 256, 8, 256, 4096, 1.5),
    "llama3.1-8b-spax": Workload("Llama-3.1-8B FFN stack (32 x d=4096, d_ff=14336), SpAx tiers", 4096, 14336, 32,
                                 1.0, 0.0, 1.0, 0, 512, 1, 256, 0, 1.0,
                                 spax=True, top_frac=0.3, mid_frac=0.3),
}


def layer_weights(seed: int, layer: int, d: int, N: int, sigma: float = 1.0, std: float = 0.02):
    """HF-layout bf16 weights of one SwiGLU FFN layer.

    Returns ``(Wg [N x d], Wu [N x d], Wd [d x N])`` as uint16 bf16 bit patterns.
    Gate row n is multiplied by ``exp(sigma * z_n)``, ``z_n ~ N(0,1)``, before the
    single rounding to bf16.
    """
    z = normal(seed, layer, T_GATE_SCALE, N)
    scale = np.exp(sigma * z)
    wg = normal(seed, layer, T_WGATE, N * d).reshape(N, d) * std * scale[:, None]
    wu = normal(seed, layer, T_WUP, N * d).reshape(N, d) * std
    wd = normal(seed, layer, T_WDOWN, d * N).reshape(d, N) * std
    return to_bf16_bits(wg), to_bf16_bits(wu), to_bf16_bits(wd)


def tokens(seed: int, layer: int, tensor_id: int, rows: int, d: int) -> np.ndarray:
    """``rows`` tokens of width ``d`` drawn N(0,1), as bf16 bits ``[rows x d]``."""
    return to_bf16_bits(normal(seed, layer, tensor_id, rows * d).reshape(rows, d))


def tie_heavy_absact(seed: int, rows: int, n: int, levels: int = 16) -> np.ndarray:
    """Non-negative float32 matrix whose entries take only ``levels`` distinct values.

    Used to force many ties in selection tests.
    """
    u = uniform(seed, 0, T_ABSACT, rows * n)
    q = np.floor(u * levels).astype(np.float32)
    return (q / np.float32(4.0)).reshape(rows, n).astype(np.float32)


def lognormal_absact(seed: int, rows: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """Non-negative float32 matrix shaped like |silu(g) u| magnitudes (heavy tailed)."""
    z = normal(seed, 1, T_ABSACT, rows * n)
    s = normal(seed, 2, T_ABSACT, n)
    v = np.abs(z).reshape(rows, n) * np.exp(sigma * s)[None, :]
    return v.astype(np.float32)

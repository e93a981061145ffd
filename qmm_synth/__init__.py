"""Seeded synthetic inputs for the group-quantized 4-bit matmul workloads.

This module draws random numbers and lays them out as the raw inputs of the
method (nibble-packed weights, fp16 scales and biases, activations). It holds
none of the method's arithmetic: no packing, no rotation, no quantization, no
partials. Both the CPU oracle and the CUDA path consume what it returns.

Generator: the SplitMix64 output function (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) applied to
``key + (i + 1) * GAMMA``. Element ``i`` of a stream therefore depends only on
``(seed, stream name, i)``, so any sampled subset of a large tensor can be
regenerated on its own.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream_key(seed: int, stream: str) -> np.uint64:
    """64-bit key of a named stream: FNV-1a of the name, mixed with the seed."""
    h = 0xCBF29CE484222325
    for ch in stream.encode():
        h = ((h ^ ch) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    with np.errstate(over="ignore"):
        base = np.array([h ^ ((seed * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF)], dtype=np.uint64)
    return _mix64(base)[0]


def draws(seed: int, stream: str, count: int, start: int = 0) -> np.ndarray:
    """``count`` 64-bit draws of a stream, elements ``start .. start+count-1``."""
    key = _stream_key(seed, stream)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * GAMMA)


def draws_at(seed: int, stream: str, index: np.ndarray) -> np.ndarray:
    """Draws at arbitrary element indices of a stream."""
    key = _stream_key(seed, stream)
    idx = np.asarray(index, dtype=np.uint64) + np.uint64(1)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * GAMMA)


def unit_uniform(d: np.ndarray) -> np.ndarray:
    """Map 64-bit draws to float64 in [0, 1) (top 53 bits)."""
    return (d >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


# ---------------------------------------------------------------- tensors


def nibble_bytes(seed: int, stream: str, N: int, K: int) -> np.ndarray:
    """[N][K/2] bytes of uniformly random nibbles (low nibble = even k).

    Read as 4-bit two's complement the values are uniform on [-8, 7]; read as
    unsigned they are uniform on [0, 15].
    """
    assert K % 2 == 0
    nbytes = N * (K // 2)
    d = draws(seed, stream, (nbytes + 7) // 8)
    return d.astype("<u8").view(np.uint8)[:nbytes].reshape(N, K // 2).copy()


def codebook_i8(seed: int, stream: str) -> np.ndarray:
    """16 distinct int8 levels in [-127, 127], ascending.

    The first 16 distinct values of the uniform draws mapped onto [-127, 127]
    (a non-uniform level set, so that no entry is an affine function of its
    index).
    """
    d = draws(seed, stream, 256)
    vals = (d % np.uint64(255)).astype(np.int64) - 127
    _, first = np.unique(vals, return_index=True)
    picked = vals[np.sort(first)[:16]]
    assert picked.size == 16
    return np.sort(picked).astype(np.int8)


def uniform_f32(seed: int, stream: str, lo: float, hi: float) -> float:
    """One fp32 U(lo, hi) draw (rounded to nearest even), as a Python float."""
    u = unit_uniform(draws(seed, stream, 1))[0]
    return float(np.float32(lo + (hi - lo) * u))


def uniform_f16(seed: int, stream: str, shape, lo: float, hi: float) -> np.ndarray:
    """fp16 bit patterns (uint16) of U(lo, hi) draws rounded to nearest even."""
    n = int(np.prod(shape))
    u = unit_uniform(draws(seed, stream, n))
    v = (lo + (hi - lo) * u).astype(np.float16)
    return v.view(np.uint16).reshape(shape)


def normal(seed: int, stream: str, n: int) -> np.ndarray:
    """n standard normal float64 values by the Box-Muller transform."""
    pairs = (n + 1) // 2
    d = draws(seed, stream, 2 * pairs)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = unit_uniform(d[1::2])
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return z[:n]


def orthogonal_f32(seed: int, stream: str, K: int) -> np.ndarray:
    """[K][K] float32 random orthogonal matrix: Q of the QR factorization of a
    matrix of N(0,1) draws (signs fixed by diag(R) > 0), rounded to fp32."""
    A = normal(seed, stream, K * K).reshape(K, K)
    Q, Rm = np.linalg.qr(A)
    Q = Q * np.where(np.diag(Rm) < 0, -1.0, 1.0)[None, :]
    return Q.astype(np.float32)


def activations_f32(seed: int, stream: str, M: int, K: int, outlier_frac: float = 0.0,
                    outlier_mag: float = 20.0) -> np.ndarray:
    """[M][K] float32 activations: N(0,1), plus optional outliers.

    With ``outlier_frac`` > 0 each row gets ``round(outlier_frac*K)`` distinct
    positions, chosen uniformly (partial Fisher-Yates), set to +-outlier_mag
    with a random sign.
    """
    x = normal(seed, stream, M * K).astype(np.float32).reshape(M, K)
    cnt = int(round(outlier_frac * K))
    if cnt:
        for m in range(M):
            d = draws(seed, f"{stream}/outliers/{m}", 2 * cnt)
            perm = np.arange(K)
            for i in range(cnt):
                j = i + int(d[i] % np.uint64(K - i))
                perm[i], perm[j] = perm[j], perm[i]
            sign = np.where((d[cnt:] & np.uint64(1)) == 1, 1.0, -1.0)
            x[m, perm[:cnt]] = (sign * outlier_mag).astype(np.float32)
    return x


def activations_f16(seed: int, stream: str, M: int, K: int) -> np.ndarray:
    """[M][K] fp16 bit patterns of N(0,1) draws rounded to nearest even."""
    return normal(seed, stream, M * K).astype(np.float16).view(np.uint16).reshape(M, K)


# ---------------------------------------------------------------- workloads

W4A8 = 0
AFFINE = 1
CQ4 = 2


@dataclass
class Layer:
    """One quantized linear layer of a workload: y = W x with W [N][K]."""
    name: str
    variant: int
    N: int
    K: int
    group: int
    hadamard: int            # 0 or the rotation size (== group)
    scale_lo: float = 0.005
    scale_hi: float = 0.02
    bias_lo: float = -0.1
    bias_hi: float = 0.1
    outlier_frac: float = 0.0


@dataclass
class Workload:
    name: str
    layers: list
    Ms: list
    seed: int = 0
    notes: str = ""
    extra: dict = field(default_factory=dict)


def workloads() -> dict:
    """The five synthetic workloads, by name."""
    return {
        "gemv_k1024_n1024": Workload(
            "gemv_k1024_n1024",
            [Layer("w", W4A8, 1024, 1024, 64, 0)], [1],
            notes="W4A8 GEMV, int4 U[-8,7], g64, fp16 scales U(0.005,0.02), x N(0,1), no rotation"),
        "gemma_decode": Workload(
            "gemma_decode",
            [Layer("gate_up", W4A8, 12288, 1536, 64, 64, outlier_frac=0.01),
             Layer("down", W4A8, 1536, 6144, 64, 64, outlier_frac=0.01),
             Layer("q", W4A8, 2048, 1536, 64, 64, outlier_frac=0.01),
             Layer("o", W4A8, 1536, 2048, 64, 64, outlier_frac=0.01)], [1],
            notes="Gemma-shaped decoder projections, M=1, W4A8 g64, Hadamard-64, x N(0,1) + 1% +-20 outliers"),
        "prefill_gemm": Workload(
            "prefill_gemm",
            [Layer("gate_up", W4A8, 12288, 1536, 64, 64)], [16, 64, 128, 512, 1068],
            notes="W4A8 prefill GEMM K=1536 N=12288 g64 Hadamard-64, x N(0,1)"),
        "affine_gemm": Workload(
            "affine_gemm",
            [Layer("gate_up", AFFINE, 34816, 5120, 64, 0)], [64, 65, 128],
            notes="affine 4-bit w = s*q + b, q in [0,15], g64, x fp16 N(0,1)"),
        "lm_head": Workload(
            "lm_head",
            [Layer("lm_head", W4A8, 262144, 1536, 128, 128)], [1, 2, 4, 8, 16, 32],
            notes="lm_head / batched decode sweep, W4A8 g128, Hadamard-128"),
    }


def layer_weights(seed: int, prefix: str, layer: Layer):
    """(q_bytes [N][K/2] u8, scales [N][G] fp16 bits, biases [N][G] fp16 bits or None)."""
    G = layer.K // layer.group
    q = nibble_bytes(seed, f"{prefix}/q", layer.N, layer.K)
    s = uniform_f16(seed, f"{prefix}/scales", (layer.N, G), layer.scale_lo, layer.scale_hi)
    b = None
    if layer.variant == AFFINE:
        b = uniform_f16(seed, f"{prefix}/biases", (layer.N, G), layer.bias_lo, layer.bias_hi)
    return q, s, b


def layer_codebook(seed: int, prefix: str):
    """(codebook int8 [16], cb_scale fp32) of a codebook-4-bit layer.

    cb_scale ~ U(0.04, 0.08) puts cb_scale * max|C| near the symmetric
    variant's largest level (8), so weights span the same range.
    """
    return codebook_i8(seed, f"{prefix}/codebook"), uniform_f32(seed, f"{prefix}/cb_scale", 0.04, 0.08)


def layer_activations(seed: int, prefix: str, layer: Layer, M: int):
    """W4A8: float32 [M][K]; affine: fp16 bits [M][K]."""
    if layer.variant == AFFINE:
        return activations_f16(seed, f"{prefix}/x", M, layer.K)
    return activations_f32(seed, f"{prefix}/x", M, layer.K, layer.outlier_frac)

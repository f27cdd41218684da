"""Seeded synthetic inputs for the block-scaled fp8 GEMM path.

This module is shared by the tests, the smoke check and the bench, on both the
CUDA side and the oracle side.  It holds none of the method's arithmetic (no
quantisation, no GEMM): it only draws numbers.

Generator (counter based, so any element can be drawn independently):
  * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014) used in counter mode: the finaliser applied to
    key + (index + 1) * 0x9E3779B97F4A7C15, key = finaliser(seed*2^32 + stream
    + 0x9E3779B97F4A7C15);
  * uniform u in (0, 1): the top 53 bits, (v >> 11) * 2^-53 + 2^-54;
  * normals: Box-Muller on the uniform pair (2i, 2i + 1) of a stream;
  * outliers: element i is multiplied by `factor` when uniform(outlier stream)[i] < p.

Workloads (shapes, distributions and seeds of the five configurations):
  c0  W8A8        M=1,            N=512,   K=1024  x~N(0,1), 1% x20 outliers     seed 0
  c1  weight-only M=16,           N=4096,  K=4096  x~N(0,1)                       seed 1
  c2  W8A8 fused  M in 1..16,     N=12288, K=4096  x~N(0,1), 0.5% x50 outliers   seed 2
  c3  expert MLP  M=8, H=4096, I=1536, H_out=4096  x~N(0,1)                       seed 3
  c4  W8A8 fused  M in {32,64,128,255,8192}, N=K=4096, x~N(0,1)                  seed 4
Weights are fp32 ~N(0, 0.02) master copies; the library quantises them.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids
S_ACT = 1
S_OUTLIER = 2
S_WEIGHT = 3          # + 16 * tensor id


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def _key(seed: int, stream: int) -> np.uint64:
    k = np.array([((int(seed) & 0xFFFFFFFF) << 32) | (int(stream) & 0xFFFFFFFF)], dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(k + _GOLDEN)[0]


def uniform(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n uniforms in (0, 1) (float64) for counters offset .. offset+n-1."""
    with np.errstate(over="ignore"):
        c = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = _key(seed, stream) + c * _GOLDEN
        v = _mix(z)
    return (v >> np.uint64(11)).astype(np.float64) * (2.0 ** -53) + 2.0 ** -54


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals (float64); normal i uses uniform pair (2*(i//2), 2*(i//2)+1)."""
    out = np.empty(n, dtype=np.float64)
    chunk = 1 << 22                               # even, so pairs never straddle chunks
    for start in range(0, n, chunk):
        cnt = min(chunk, n - start)
        pairs = (cnt + 1) // 2
        u = uniform(seed, stream, 2 * pairs, offset=start)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        z = np.empty(2 * pairs, dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        out[start:start + cnt] = z[:cnt]
    return out


def activations(seed: int, M: int, K: int, outlier_p: float = 0.0, outlier_x: float = 1.0,
                tensor: int = 0) -> np.ndarray:
    """fp32 [M][K] activations ~N(0,1), each entry independently scaled by
    outlier_x with probability outlier_p.  The caller rounds to bf16."""
    n = M * K
    x = normal(seed, S_ACT + 16 * tensor, n)
    if outlier_p > 0.0:
        mask = uniform(seed, S_OUTLIER + 16 * tensor, n) < outlier_p
        x[mask] *= outlier_x
    return x.astype(np.float32).reshape(M, K)


def weights(seed: int, N: int, K: int, std: float = 0.02, tensor: int = 0) -> np.ndarray:
    """fp32 [N][K] master weights ~N(0, std)."""
    return (normal(seed, S_WEIGHT + 16 * tensor, N * K) * std).astype(np.float32).reshape(N, K)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 with torch's round-to-nearest-even cast; returns uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


CONFIGS = {
    "c0": dict(kind="w8a8", M=[1], N=512, K=1024, p=0.01, factor=20.0, seed=0),
    "c1": dict(kind="w8bf16", M=[16], N=4096, K=4096, p=0.0, factor=1.0, seed=1),
    "c2": dict(kind="w8a8", M=[1, 2, 4, 8, 16], N=12288, K=4096, p=0.005, factor=50.0, seed=2),
    "c3": dict(kind="mlp", M=[8], H=4096, I=1536, H_out=4096, p=0.0, factor=1.0, seed=3),
    "c4": dict(kind="w8a8", M=[32, 64, 128, 255, 8192], N=4096, K=4096, p=0.0, factor=1.0, seed=4),
}

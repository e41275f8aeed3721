"""Seeded synthetic inputs for the Hyper-Connection gated residual.

This module only draws random numbers and rounds them to the storage types.
It holds none of the method's arithmetic, so both the CUDA library and the
fp64 oracle can be fed from it without sharing any computation.

Generator: SplitMix64 on a counter (value ``i`` of stream ``key`` is
``splitmix64(base(key) + (i + 1) * 0x9E3779B97F4A7C15)``), 53-bit uniforms in
(0, 1], Box-Muller pairs for normals and ``Z / sqrt(chi2_3 / 3)`` for the
Student-t (nu = 3) draws of the wide workload.  Every tensor has its own
stream, so a tensor's values depend only on (seed, tensor, element index):
row ``m`` of an activation tensor is the same whatever ``M`` is generated.

Workload shapes and distributions follow the pages' benchmark setup
(aiter PR #5913, "Performance": HC=4, HS=2560, lowrank 320, bf16) and the
wide variant (HC=8, HS=4096, r=512, heavy-tailed R, y scaled by 10).
"""
from __future__ import annotations

import dataclasses

import numpy as np

SEED = 20261202

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20

# stream ids, one per tensor
_ID = {"Wnorm": 1, "Wd": 2, "Wi": 3, "Wu": 4, "R": 5, "y": 6, "inj": 7}


@dataclasses.dataclass(frozen=True)
class Shape:
    """One workload shape: HC streams of width HS, low rank r."""

    HC: int = 4
    HS: int = 2560
    r: int = 320
    eps: float = 1e-6
    heavy_tailed: bool = False   # R ~ Student-t(3), y ~ 10 * N(0, 1)

    @property
    def K(self) -> int:
        return self.HC * self.HS


DEFAULT = Shape()
WIDE = Shape(HC=8, HS=4096, r=512, heavy_tailed=True)


def _stream_base(seed: int, key: int) -> np.uint64:
    return np.uint64((seed * 0x100000001B3 + key * (1 << 40)) & 0xFFFFFFFFFFFFFFFF)


def uniforms(seed: int, key: int, start: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1] from counter positions start .. start+n-1."""
    out = np.empty(n, dtype=np.float64)
    base = _stream_base(seed, key)
    for c0 in range(0, n, _CHUNK):
        m = min(_CHUNK, n - c0)
        z = np.arange(start + c0 + 1, start + c0 + 1 + m, dtype=np.uint64)
        z *= _GAMMA
        z += base
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
        z >>= np.uint64(11)
        o = out[c0:c0 + m]
        np.add(z, 1.0, out=o, casting="unsafe")
        o *= 1.0 / 9007199254740992.0
    return out


def normals(seed: int, key: int, start: int, n: int) -> np.ndarray:
    """n standard normals; normal i uses uniforms 2*(i//2) and 2*(i//2)+1."""
    p0 = start // 2
    p1 = (start + n + 1) // 2
    u = uniforms(seed, key, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
    rad = np.sqrt(-2.0 * np.log(u[:, 0]))
    ang = (2.0 * np.pi) * u[:, 1]
    z = np.empty((p1 - p0, 2), dtype=np.float64)
    z[:, 0] = rad * np.cos(ang)
    z[:, 1] = rad * np.sin(ang)
    z = z.reshape(-1)
    off = start - 2 * p0
    return z[off:off + n]


def student_t3(seed: int, key: int, start: int, n: int) -> np.ndarray:
    """n Student-t draws with 3 degrees of freedom, 4 normals per draw."""
    z = normals(seed, key, 4 * start, 4 * n).reshape(n, 4)
    chi2 = z[:, 1] ** 2 + z[:, 2] ** 2 + z[:, 3] ** 2
    return z[:, 0] / np.sqrt(chi2 / 3.0)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round to bfloat16 (via float32, round-to-nearest-even); uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u += np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    bits = (u >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        bits[nan] = 0x7FC0
    return bits


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bfloat16 bit patterns as float64."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def weights(shape: Shape = DEFAULT, seed: int = SEED) -> dict:
    """Wnorm [K], Wd [r, K], Wi [HC, K], Wu [K, r] as bf16 bit arrays.

    Wnorm ~ N(0, 0.1), Wd and Wi ~ N(0, 1/sqrt(K)), Wu ~ N(0, 1/sqrt(r)).
    """
    K, r, HC = shape.K, shape.r, shape.HC
    out = {
        "Wnorm": 0.1 * normals(seed, _ID["Wnorm"], 0, K),
        "Wd": normals(seed, _ID["Wd"], 0, r * K).reshape(r, K) / np.sqrt(K),
        "Wi": normals(seed, _ID["Wi"], 0, HC * K).reshape(HC, K) / np.sqrt(K),
        "Wu": normals(seed, _ID["Wu"], 0, K * r).reshape(K, r) / np.sqrt(r),
    }
    return {k: to_bf16_bits(v) for k, v in out.items()}


def activation_rows(start: int, stop: int, shape: Shape = DEFAULT, seed: int = SEED) -> dict:
    """Rows start .. stop-1 of R [., HC, HS] bf16, y [., HS] bf16 and inj [., HC]
    float32 -- exactly the rows ``activations`` gives for any M >= stop.

    R, y ~ N(0, 1) (wide workload: R ~ Student-t(3), y ~ 10 N(0, 1)) and
    inj ~ N(0, 2) (std 2).  Row m of a tensor reads counter positions
    m * row_length onwards of that tensor's stream, so any row range can be
    drawn on its own (for instance by several processes in parallel).
    """
    HC, HS, K = shape.HC, shape.HS, shape.K
    n = stop - start
    if shape.heavy_tailed:
        R = student_t3(seed, _ID["R"], start * K, n * K)
        y = 10.0 * normals(seed, _ID["y"], start * HS, n * HS)
    else:
        R = normals(seed, _ID["R"], start * K, n * K)
        y = normals(seed, _ID["y"], start * HS, n * HS)
    inj = 2.0 * normals(seed, _ID["inj"], start * HC, n * HC)
    return {"R": to_bf16_bits(R).reshape(n, HC, HS), "y": to_bf16_bits(y).reshape(n, HS),
            "inj": inj.astype(np.float32).reshape(n, HC)}


def activations(M: int, shape: Shape = DEFAULT, seed: int = SEED,
                distinct_rows: int | None = None) -> dict:
    """R [M, HC, HS] bf16, y [M, HS] bf16, inj [M, HC] float32 (rows 0 .. M-1
    of ``activation_rows``).

    With ``distinct_rows`` set, row m holds the generator's row
    ``m % distinct_rows``: the benchmark uses it to build very large inputs
    quickly (timing does not depend on the values); parity tests draw every
    row.
    """
    G = M if distinct_rows is None else min(M, distinct_rows)
    a = activation_rows(0, G, shape, seed)
    if G < M:
        idx = np.arange(M) % G
        a = {k: v[idx] for k, v in a.items()}
    return a

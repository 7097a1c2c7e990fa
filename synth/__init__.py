"""Seeded synthetic inputs for the depth-routing read.

This module is shared by the CPU oracle and by the CUDA path; it holds none of
the routing arithmetic. It only draws random numbers from a counter-based
generator (Philox-4x64, numpy's implementation of the published definition),
scales them as the workload recipe says and rounds them to the storage dtype,
so that both sides see bit-identical inputs.

Workload recipe (synthetic stand-ins for the trained models of the
"Multi-Head Attention Residuals" page, Table 5 / Appendix E, and the
"Low-Rank Attention Residuals" page, Appendix I):

* sublayer output ``o_j`` (``j >= 1``) ~ N(0, 1) / sqrt(ceil(j / 2)), i.e.
  scaled by one over the square root of the layer that wrote it; the token
  embedding ``o_0`` ~ N(0, 1);
* routing queries ``q`` ~ N(0, 0.02^2) (the pages' initialiser std);
* RMSNorm weight ``g`` = 1 (``kind="ones"``), or 1 + N(0, 0.1^2)
  (``kind="random"``, used by tests so that q and g cannot be confused);
* upstream gradient dL/dout ~ N(0, 1), a fresh draw per routing site.

Every tensor has its own Philox key, derived from (seed, tag, index), so a
tensor does not depend on which other tensors were drawn before it.
"""

from __future__ import annotations

import hashlib
import math

import numpy as np

__all__ = [
    "philox",
    "normal_f32",
    "to_storage",
    "storage_to_f64",
    "storage_to_f32",
    "bf16_bits_from_f32",
    "sublayer_output",
    "sublayer_outputs",
    "site_query",
    "site_norm_weight",
    "site_dout",
    "DTYPES",
]

DTYPES = ("f32", "bf16")

_TAGS = {"source": 1, "query": 2, "normw": 3, "dout": 4, "misc": 5}


def philox(seed: int, *ids: int) -> np.random.Generator:
    """A Philox-4x64 stream keyed by ``(seed, *ids)``."""
    h = hashlib.blake2b(digest_size=16)
    h.update(int(seed).to_bytes(8, "little", signed=True))
    for i in ids:
        h.update(int(i).to_bytes(8, "little", signed=True))
    key = int.from_bytes(h.digest(), "little")
    return np.random.Generator(np.random.Philox(key=key))


def normal_f32(seed: int, ids: tuple, shape, std: float = 1.0) -> np.ndarray:
    x = philox(seed, *ids).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16. Inputs must be finite.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array -> storage array (uint16 bf16 patterns, or float32)."""
    if dtype == "bf16":
        return bf16_bits_from_f32(x)
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def storage_to_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of stored values to float64."""
    return storage_to_f32(a, dtype).astype(np.float64)


def layer_scale(j: int) -> float:
    """1/sqrt(layer) for sublayer output j (layer = ceil(j/2)); 1 for j = 0."""
    if j == 0:
        return 1.0
    return 1.0 / math.sqrt((j + 1) // 2)


def sublayer_output(seed: int, j: int, T: int, d: int, dtype: str) -> np.ndarray:
    """Storage array [T, d] for sublayer output j (j = 0 is the embedding)."""
    x = normal_f32(seed, (_TAGS["source"], j), (T, d), layer_scale(j))
    return to_storage(x, dtype)


def sublayer_outputs(seed: int, count: int, T: int, d: int, dtype: str) -> np.ndarray:
    """Storage array [count, T, d]: outputs 0..count-1."""
    sd = np.uint16 if dtype == "bf16" else np.float32
    out = np.empty((count, T, d), dtype=sd)
    for j in range(count):
        out[j] = sublayer_output(seed, j, T, d, dtype)
    return out


def site_query(seed: int, site: int, r: int, std: float = 0.02) -> np.ndarray:
    """float32 [r] query of one routing site."""
    return normal_f32(seed, (_TAGS["query"], site), (r,), std)


def site_norm_weight(seed: int, site: int, r: int, kind: str = "ones") -> np.ndarray:
    """float32 [r] RMSNorm weight of one routing site."""
    if kind == "ones":
        return np.ones(r, dtype=np.float32)
    if kind == "random":
        return np.float32(1.0) + normal_f32(seed, (_TAGS["normw"], site), (r,), 0.1)
    raise ValueError(f"unknown norm-weight kind {kind!r}")


def site_dout(seed: int, site: int, T: int, d: int, dtype: str) -> np.ndarray:
    """Storage array [T, d]: upstream gradient dL/dout of one routing site."""
    return to_storage(normal_f32(seed, (_TAGS["dout"], site), (T, d)), dtype)


def misc_normal(seed: int, tag: int, shape, std: float = 1.0) -> np.ndarray:
    """A float32 draw for tests that need extra independent values."""
    return normal_f32(seed, (_TAGS["misc"], tag), shape, std)

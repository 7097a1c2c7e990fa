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


# ---- device-side generation for full-size workloads -----------------------------
# Full-size microbatches hold billions of values; they are drawn on the GPU by
# torch's seeded Philox generator, one generator per tensor (keyed like the host
# streams above). The oracle side of a parity check reads the same values back
# for the tokens it samples, so both sides still see identical bits.

def _key64(seed: int, *ids: int) -> int:
    h = hashlib.blake2b(digest_size=8)
    h.update(int(seed).to_bytes(8, "little", signed=True))
    for i in ids:
        h.update(int(i).to_bytes(8, "little", signed=True))
    return int.from_bytes(h.digest(), "little") & ((1 << 63) - 1)


class DeviceInputs:
    """Seeded synthetic inputs drawn on a CUDA device (same recipe as above).

    Methods return torch tensors on ``device``; ``dtype`` is "bf16" or "f32"
    (rounded to nearest even by torch's conversion)."""

    def __init__(self, seed: int = 0, device="cuda", q_std: float = 0.02,
                 g_kind: str = "ones"):
        import torch
        self.torch = torch
        self.seed, self.device, self.q_std, self.g_kind = seed, torch.device(device), q_std, g_kind

    def _randn(self, shape, *ids):
        torch = self.torch
        g = torch.Generator(device=self.device)
        g.manual_seed(_key64(self.seed, *ids))
        return torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)

    def _cast(self, x, dtype):
        return x.to(self.torch.bfloat16 if dtype == "bf16" else self.torch.float32)

    def output(self, j: int, T: int, d: int, dtype: str):
        return self._cast(self._randn((T, d), _TAGS["source"], j) * layer_scale(j), dtype)

    def query(self, site: int, r: int):
        return self._randn((r,), _TAGS["query"], site) * self.q_std

    def norm_weight(self, site: int, r: int):
        if self.g_kind == "ones":
            return None
        return 1.0 + 0.1 * self._randn((r,), _TAGS["normw"], site)

    def dout(self, site: int, T: int, d: int, dtype: str):
        return self._cast(self._randn((T, d), _TAGS["dout"], site), dtype)


class HostInputs:
    """The host (numpy Philox) streams above, served as CUDA tensors.

    Same interface as ``DeviceInputs``; ``host_*`` methods return the float64
    values the oracle consumes (exact widenings of the stored values)."""

    def __init__(self, seed: int = 0, device="cuda", q_std: float = 0.02,
                 g_kind: str = "ones"):
        import torch
        self.torch = torch
        self.seed, self.device, self.q_std, self.g_kind = seed, torch.device(device), q_std, g_kind

    def _to_dev(self, a: np.ndarray, dtype: str):
        torch = self.torch
        if dtype == "bf16":
            t = torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32).copy())
        return t.to(self.device)

    def output(self, j, T, d, dtype):
        return self._to_dev(sublayer_output(self.seed, j, T, d, dtype), dtype)

    def query(self, site, r):
        return self._to_dev(site_query(self.seed, site, r, self.q_std), "f32")

    def norm_weight(self, site, r):
        if self.g_kind == "ones":
            return None
        return self._to_dev(site_norm_weight(self.seed, site, r, self.g_kind), "f32")

    def dout(self, site, T, d, dtype):
        return self._to_dev(site_dout(self.seed, site, T, d, dtype), dtype)

    # float64 views for the oracle
    def host_output(self, j, T, d, dtype):
        return storage_to_f64(sublayer_output(self.seed, j, T, d, dtype), dtype)

    def host_query(self, site, r):
        return site_query(self.seed, site, r, self.q_std).astype(np.float64)

    def host_norm_weight(self, site, r):
        if self.g_kind == "ones":
            return None
        return site_norm_weight(self.seed, site, r, self.g_kind).astype(np.float64)

    def host_dout(self, site, T, d, dtype):
        return storage_to_f64(site_dout(self.seed, site, T, d, dtype), dtype)

"""Storage rounding of bank rows (oracle side).

A block-routing partial sum is formed at full precision and stored once in the
bank's dtype ("Low-Rank Attention Residuals", Sec. 3.3, partial-block routing:
accumulation precedes slicing and normalisation; the stored tensor is the
rounded sum). The oracle rounds float64 values itself:

* ``bf16``: 8 significant bits, round to nearest with ties to even, written
  from the format's definition with ``frexp``/``rint`` (no float32 detour);
* ``f32`` : IEEE single precision (numpy's correctly rounded cast).

Values below the bfloat16 normal range are not handled (the synthetic inputs
never reach them).
"""

from __future__ import annotations

import numpy as np

__all__ = ["round_to_storage", "storage_bits", "block_bank"]


def round_to_storage(x, dtype: str) -> np.ndarray:
    """float64 values rounded to the nearest value of the storage dtype."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    if dtype == "bf16":
        m, e = np.frexp(x)                    # x = m * 2**e, 0.5 <= |m| < 1
        return np.ldexp(np.rint(m * 256.0), e - 8)
    raise ValueError(f"unknown dtype {dtype!r}")


def storage_bits(x, dtype: str) -> np.ndarray:
    """Bit patterns of values that are exactly representable in the dtype."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return x32.view(np.uint32)
    if dtype == "bf16":
        u = x32.view(np.uint32)
        if np.any(u & np.uint32(0xFFFF)):
            raise ValueError("values are not bfloat16-representable")
        return (u >> np.uint32(16)).astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def block_bank(outputs, plan: dict, dtype: str) -> list[np.ndarray]:
    """Bank rows of block routing from sublayer outputs (float64 arrays).

    ``outputs[t]`` is o_t (t = 0 the embedding), already representable in the
    storage dtype; ``plan`` comes from ``schedule.block_plan``.
    """
    rows: list[np.ndarray] = []
    for op in plan["row_ops"]:
        if op[0] == "emb":
            rows.append(np.asarray(outputs[0], dtype=np.float64))
        elif op[0] == "copy":
            rows.append(np.asarray(outputs[op[1]], dtype=np.float64))
        else:
            _, p, t = op
            rows.append(round_to_storage(rows[p] + outputs[t], dtype))
    return rows

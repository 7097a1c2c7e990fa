"""CPU oracle for the depth-routing read — test infrastructure only.

Only ``tests/``, the package smoke check and the benchmark's CPU-baseline leg
may import this package. The product path never does: it shares no code with
the oracle and fails loudly when its CUDA library is missing.

The arithmetic lives in ``ar_oracle.c`` (plain float64 C, one token at a
time, compiled with gcc); this module only marshals numpy arrays to it and
holds the source-schedule bookkeeping (``schedule.py``) and the storage
rounding of accumulated block sums (``storage.py``).

Every function here is pinned by ``tests/test_oracle_*.py`` against brute
force (the routing equations term by term in numpy), torch autograd,
finite differences and the invariants the pages state.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

from . import schedule, storage  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ar_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIBPATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ar_oracle.c`` with gcc (OpenMP when the compiler has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIBPATH)
            and os.path.getmtime(_LIBPATH) >= os.path.getmtime(_SRC)):
        return _LIBPATH
    tmp = _LIBPATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIBPATH)
    return _LIBPATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            L.orc_max_threads.restype = i32
            L.orc_inv_rms.argtypes = [P, i64, i32, i32, i32, f64, P]
            L.orc_inv_rms.restype = i32
            L.orc_route_fwd.argtypes = [P, i32, i64, i32, i32, i32, i32, f64, P, P, P, P, P]
            L.orc_route_fwd.restype = i32
            L.orc_route_bwd.argtypes = [P, i32, i64, i32, i32, i32, i32, f64, P, P, P, P, P, P]
            L.orc_route_bwd.restype = i32
            _lib = L
    return _lib


def threads() -> int:
    """Number of OpenMP threads the oracle uses."""
    return int(lib().orc_max_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs):
    arr = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return arr


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle rejected the call (code {rc})")


def inv_rms(x, r: int | None = None, eps: float = 1e-6, full_width: bool = False) -> np.ndarray:
    """Inverse RMS per token of one [T, d] source over its key coordinates."""
    x = _f64(x)
    T, d = x.shape
    r = d if r is None else r
    out = np.empty(T, dtype=np.float64)
    _check(lib().orc_inv_rms(_ptr(x), T, d, r, int(full_width), eps, _ptr(out)))
    return out


def route_fwd(sources, q, g, H: int, r: int | None = None, eps: float = 1e-6,
              full_width: bool = False, want_alpha: bool = False):
    """Forward of one routing site.

    sources: sequence of N float64 arrays [T, d]; q, g: [r] (g may be None).
    Returns ``(out [T,d], lse [T,H])`` or, with ``want_alpha``,
    ``(out, lse, alpha [T,N,H])``.
    """
    srcs = [_f64(s) for s in sources]
    N = len(srcs)
    T, d = srcs[0].shape
    r = d if r is None else r
    qq = _f64(q)
    gg = None if g is None else _f64(g)
    out = np.empty((T, d), dtype=np.float64)
    lse = np.empty((T, H), dtype=np.float64)
    alpha = np.empty((T, N, H), dtype=np.float64) if want_alpha else None
    _check(lib().orc_route_fwd(_ptr_array(srcs), N, T, d, r, H, int(full_width), eps,
                               _ptr(qq), None if gg is None else _ptr(gg),
                               _ptr(out), _ptr(lse),
                               None if alpha is None else _ptr(alpha)))
    return (out, lse, alpha) if want_alpha else (out, lse)


def route_bwd(sources, q, g, dout, H: int, r: int | None = None, eps: float = 1e-6,
              full_width: bool = False, dsrc=None):
    """Backward of one routing site.

    Returns ``(dsrc, dq, dg)``: ``dsrc`` a list of N float64 [T, d] arrays
    holding dL/ds_n (if ``dsrc`` is given, the site's gradients are ADDED to
    those arrays in place), ``dq`` and ``dg`` float64 [r].
    """
    srcs = [_f64(s) for s in sources]
    N = len(srcs)
    T, d = srcs[0].shape
    r = d if r is None else r
    if dsrc is None:
        dsrc = [np.zeros((T, d), dtype=np.float64) for _ in range(N)]
    for a in dsrc:
        if a.dtype != np.float64 or not a.flags.c_contiguous or a.shape != (T, d):
            raise ValueError("dsrc entries must be C-contiguous float64 [T, d]")
    qq = _f64(q)
    gg = None if g is None else _f64(g)
    G = _f64(dout)
    dq = np.empty(r, dtype=np.float64)
    dg = np.empty(r, dtype=np.float64)
    _check(lib().orc_route_bwd(_ptr_array(srcs), N, T, d, r, H, int(full_width), eps,
                               _ptr(qq), None if gg is None else _ptr(gg), _ptr(G),
                               _ptr_array(dsrc), _ptr(dq), _ptr(dg)))
    return dsrc, dq, dg


def route_fwd_delta(sources, q, g, H: int, partial, alpha: float, r: int | None = None,
                    eps: float = 1e-6, full_width: bool = False):
    """Delta form of one site ("Multi-Head Attention Residuals", Sec. 3.3,
    identity-preserving conversion): h = partial + alpha * routed.
    Returns ``(h, routed, lse)``."""
    routed, lse = route_fwd(sources, q, g, H, r=r, eps=eps, full_width=full_width)
    return _f64(partial) + float(alpha) * routed, routed, lse


def route_bwd_delta(sources, q, g, dout, H: int, alpha: float, r: int | None = None,
                    eps: float = 1e-6, full_width: bool = False, dsrc=None):
    """Backward of ``route_fwd_delta``: the routed read receives alpha * dout.
    Returns ``(dsrc, dq, dg, dalpha, dpartial)`` with dalpha = sum <dout, routed>
    and dpartial = dout."""
    G = _f64(dout)
    routed, _ = route_fwd(sources, q, g, H, r=r, eps=eps, full_width=full_width)
    dsrc, dq, dg = route_bwd(sources, q, g, float(alpha) * G, H, r=r, eps=eps,
                             full_width=full_width, dsrc=dsrc)
    return dsrc, dq, dg, float(np.sum(G * routed)), G


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))

"""CPU oracle for the depth-routing read — test infrastructure only.

Only ``tests/``, the package smoke check and the benchmark's CPU-baseline leg
may import this package. The product path never does: it shares no code with
the oracle and fails loudly when its CUDA library is missing.

The arithmetic lives in ``ar_oracle.c`` (plain C, one token at a time,
compiled with gcc as a float64 library, the parity reference, and from the
same source as a float32 library, the CPU baseline the benchmark times); this
module only marshals numpy arrays to it and
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
# float64: the parity reference; float32: the same source built with
# -DORC_FLOAT, the CPU baseline the benchmark times
_LIBPATHS = {"f64": os.path.join(_BUILD, "liboracle.so"),
             "f32": os.path.join(_BUILD, "liboracle_f32.so")}
_LIBPATH = _LIBPATHS["f64"]
_NP = {"f64": np.float64, "f32": np.float32}
_lock = threading.Lock()
_libs = {}


def _build_one(path: str, defines, force: bool) -> str:
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", *defines, "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, path)
    return path


def build(force: bool = False) -> str:
    """Compile ``ar_oracle.c`` with gcc (OpenMP when the compiler has it), as
    the float64 library and the float32 one. Returns the float64 library's path."""
    os.makedirs(_BUILD, exist_ok=True)
    _build_one(_LIBPATHS["f32"], ["-DORC_FLOAT"], force)
    return _build_one(_LIBPATHS["f64"], [], force)


def lib(precision: str = "f64"):
    with _lock:
        if precision not in _libs:
            if precision not in _LIBPATHS:
                raise ValueError(f"unknown precision {precision!r}")
            build()
            L = ctypes.CDLL(_LIBPATHS[precision])
            P = ctypes.c_void_p
            i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            L.orc_max_threads.restype = i32
            L.orc_real_bytes.restype = i32
            L.orc_inv_rms.argtypes = [P, i64, i32, i32, i32, f64, P]
            L.orc_inv_rms.restype = i32
            L.orc_route_fwd.argtypes = [P, i32, i64, i32, i32, i32, i32, f64, P, P, P, P, P]
            L.orc_route_fwd.restype = i32
            L.orc_route_bwd.argtypes = [P, i32, i64, i32, i32, i32, i32, f64, P, P, P, P, P, P, P]
            L.orc_route_bwd.restype = i32
            if L.orc_real_bytes() != np.dtype(_NP[precision]).itemsize:
                raise RuntimeError(f"{_LIBPATHS[precision]} is not the {precision} build")
            _libs[precision] = L
    return _libs[precision]


def threads() -> int:
    """Number of OpenMP threads the oracle uses."""
    return int(lib().orc_max_threads())


def _arr(a, precision: str = "f64") -> np.ndarray:
    return np.ascontiguousarray(a, dtype=_NP[precision])


def _f64(a) -> np.ndarray:
    return _arr(a, "f64")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs):
    arr = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return arr


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle rejected the call (code {rc})")


def inv_rms(x, r: int | None = None, eps: float = 1e-6, full_width: bool = False,
            precision: str = "f64") -> np.ndarray:
    """Inverse RMS per token of one [T, d] source over its key coordinates."""
    x = _arr(x, precision)
    T, d = x.shape
    r = d if r is None else r
    out = np.empty(T, dtype=_NP[precision])
    _check(lib(precision).orc_inv_rms(_ptr(x), T, d, r, int(full_width), eps, _ptr(out)))
    return out


def route_fwd(sources, q, g, H: int, r: int | None = None, eps: float = 1e-6,
              full_width: bool = False, want_alpha: bool = False, precision: str = "f64"):
    """Forward of one routing site.

    sources: sequence of N arrays [T, d]; q, g: [r] (g may be None).
    Returns ``(out [T,d], lse [T,H])`` or, with ``want_alpha``,
    ``(out, lse, alpha [T,N,H])``, in the arithmetic type of ``precision``
    ("f64", the parity reference, or "f32").
    """
    dt = _NP[precision]
    srcs = [_arr(s, precision) for s in sources]
    N = len(srcs)
    T, d = srcs[0].shape
    r = d if r is None else r
    qq = _arr(q, precision)
    gg = None if g is None else _arr(g, precision)
    out = np.empty((T, d), dtype=dt)
    lse = np.empty((T, H), dtype=dt)
    alpha = np.empty((T, N, H), dtype=dt) if want_alpha else None
    _check(lib(precision).orc_route_fwd(_ptr_array(srcs), N, T, d, r, H, int(full_width), eps,
                               _ptr(qq), None if gg is None else _ptr(gg),
                               _ptr(out), _ptr(lse),
                               None if alpha is None else _ptr(alpha)))
    return (out, lse, alpha) if want_alpha else (out, lse)


def route_bwd(sources, q, g, dout, H: int, r: int | None = None, eps: float = 1e-6,
              full_width: bool = False, dsrc=None, precision: str = "f64", fwd_out=None):
    """Backward of one routing site.

    Returns ``(dsrc, dq, dg)``: ``dsrc`` a list of N [T, d] arrays holding
    dL/ds_n (if ``dsrc`` is given, the site's gradients are ADDED to those
    arrays in place), ``dq`` and ``dg`` [r]; all in the arithmetic type of
    ``precision`` ("f64", the parity reference, or "f32").
    ``fwd_out`` ([T, d] or None): the forward output whose per-head dot with
    dout couples the sources in the routing feedback. None recomputes it (the
    definition); given, it is taken as is (the stored output a one-pass
    backward reads, e.g. rounded to bf16).
    """
    dt = _NP[precision]
    srcs = [_arr(s, precision) for s in sources]
    N = len(srcs)
    T, d = srcs[0].shape
    r = d if r is None else r
    if dsrc is None:
        dsrc = [np.zeros((T, d), dtype=dt) for _ in range(N)]
    for a in dsrc:
        if a.dtype != dt or not a.flags.c_contiguous or a.shape != (T, d):
            raise ValueError(f"dsrc entries must be C-contiguous {np.dtype(dt).name} [T, d]")
    qq = _arr(q, precision)
    gg = None if g is None else _arr(g, precision)
    G = _arr(dout, precision)
    dq = np.empty(r, dtype=dt)
    dg = np.empty(r, dtype=dt)
    fo = None if fwd_out is None else _arr(fwd_out, precision)
    if fo is not None and fo.shape != (T, d):
        raise ValueError("fwd_out must be [T, d]")
    _check(lib(precision).orc_route_bwd(_ptr_array(srcs), N, T, d, r, H, int(full_width), eps,
                               _ptr(qq), None if gg is None else _ptr(gg), _ptr(G),
                               None if fo is None else _ptr(fo),
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

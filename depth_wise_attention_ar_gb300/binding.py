"""ctypes binding of libattnres_gb300.so (include/attnres.h).

The ``ar_*`` functions mirror the C entry points one to one and only marshal
arguments (tensors -> device pointers, lists -> int32 arrays, streams ->
cudaStream_t). ``Bank`` is a convenience owner of the buffers a bank needs,
allocated with torch; every computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing, importing this module raises.

With AR_CHECKED=1 in the environment the range-checked build of the same
library (libattnres_gb300_checked.so, include/attnres.h: ar_checked_fault) is
loaded instead; it has the same entry points.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
CHECKED = os.environ.get("AR_CHECKED", "") == "1"
LIBPATH = os.path.join(HERE, "libattnres_gb300_checked.so" if CHECKED else "libattnres_gb300.so")

AR_OK = 0
STATUS = {0: "AR_OK", 1: "AR_ERR_INVALID_ARG", 2: "AR_ERR_SHAPE", 3: "AR_ERR_ALIGN",
          4: "AR_ERR_CAPACITY", 5: "AR_ERR_ORDER", 6: "AR_ERR_CUDA", 7: "AR_ERR_TIMEOUT",
          8: "AR_ERR_UNSUPPORTED", 9: "AR_ERR_BOUNDS"}
AR_F32, AR_BF16 = 0, 1
AR_NORM_KEY, AR_NORM_FULL = 0, 1
AR_MAX_SOURCES = 256
AR_MAX_QUERIES = 8
AR_DEVERR_WAIT_TIMEOUT = 1
AR_DEVERR_BOUNDS = 2

# Every function the header declares, with its ctypes signature.
_P, _I32, _I64, _F32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_I32P, _I64P, _U32P, _SZP = (ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64),
                             ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_size_t))
class ArSite(ctypes.Structure):
    """struct ar_site: a routing site with strided query / norm weight."""
    _fields_ = [("rows", ctypes.POINTER(ctypes.c_int32)), ("n_src", ctypes.c_int32),
                ("H", ctypes.c_int32), ("q", ctypes.c_void_p), ("q_stride", ctypes.c_int64),
                ("g", ctypes.c_void_p), ("g_stride", ctypes.c_int64),
                ("site_id", ctypes.c_int32)]


_SITEP = ctypes.POINTER(ArSite)
SIGNATURES = {
    "ar_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "ar_inv_rms_floats": ([_I64, _I32, _I64P], ctypes.c_int),
    "ar_bank_create": ([ctypes.POINTER(_P), _I64, _I32, _I32, _I32, ctypes.c_int, ctypes.c_int,
                        _F32, _P, _P, _P], ctypes.c_int),
    "ar_bank_destroy": ([_P], ctypes.c_int),
    "ar_bank_row_count": ([_P, _I32P], ctypes.c_int),
    "ar_bank_row_ptr": ([_P, _I32, ctypes.POINTER(_P)], ctypes.c_int),
    "ar_bank_append": ([_P, _P, _I32, _I32P, _P], ctypes.c_int),
    "ar_bank_append_strided": ([_P, _P, _I64, _I64, _I32, _I32P, _P], ctypes.c_int),
    "ar_route_fwd_site": ([_P, _SITEP, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "ar_route_bwd_site": ([_P, _SITEP, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "ar_bank_zero_grad": ([_P], ctypes.c_int),
    "ar_bank_reset": ([_P], ctypes.c_int),
    "ar_route_fwd": ([_P, _I32P, _I32, _I32, _P, _P, _P, _P, _I32, _P], ctypes.c_int),
    "ar_route_fwd_append": ([_P, _P, _I32, _I32P, _I32P, _I32, _I32, _P, _P, _P, _P, _I32, _I32P,
                             _P], ctypes.c_int),
    "ar_route_fwd_delta": ([_P, _I32P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _P],
                           ctypes.c_int),
    "ar_route_bwd_delta": ([_P, _I32P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                            _I32, _P], ctypes.c_int),
    "ar_bank_append_broadcast": ([_P, _P, _I32P, _P], ctypes.c_int),
    "ar_bank_grad_token_sum": ([_P, _I32, _P, _P], ctypes.c_int),
    "ar_route_bwd_workspace": ([_P, _I32, _SZP], ctypes.c_int),
    "ar_route_bwd": ([_P, _I32P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I32, _P],
                     ctypes.c_int),
    "ar_route_bwd_noalloc": ([_P, _I32P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _P],
                             ctypes.c_int),
    "ar_noalloc_scratch_bytes": ([_SZP], ctypes.c_int),
    "ar_bank_grad_fold": ([_P, _I32, _I32, _P], ctypes.c_int),
    "ar_route_merge": ([_P, _I32, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "ar_route_fwd_multi": ([_P, _I32P, _I32, _I32, _I32, _P, _P, _P, _P, _P], ctypes.c_int),
    "ar_block_schedule": ([_I32, _I32, _I32P, _I32P, _I32P, _I64, _I64P], ctypes.c_int),
    "ar_device_error": ([_U32P], ctypes.c_int),
    "ar_device_status": ([], ctypes.c_int),
    "ar_route_fwd_lost_copies": ([_P, _I32P, _I32, _I32, _P, _P, _P, _P, ctypes.c_uint32, _P],
                                 ctypes.c_int),
    "ar_route_bwd_exact": ([_P, _SITEP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "ar_checked_fault": ([_I32P, ctypes.POINTER(ctypes.c_uint64), _U32P, _U32P], ctypes.c_int),
    "ar_checked_trim_out": ([_I64], ctypes.c_int),
}

if not os.path.exists(LIBPATH):
    raise ImportError(
        f"{LIBPATH} is not built; run depth_wise_attention_ar_gb300.build.build("
        f"{'checked=True' if CHECKED else ''}) "
        "(nvcc, sm_103a). There is no CPU fallback.")

_lib = ctypes.CDLL(LIBPATH)
for _name, (_args, _res) in SIGNATURES.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class ARError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{fn}: {self.name}")


def _check(fn: str, st: int):
    if st != AR_OK:
        raise ARError(fn, st)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


def _rows(rows):
    arr = (ctypes.c_int32 * max(1, len(rows)))(*[int(r) for r in rows])
    return arr, len(rows)


# ---- one-to-one wrappers of the C ABI ------------------------------------------

def ar_status_string(status: int) -> str:
    return _lib.ar_status_string(status).decode()


def ar_inv_rms_floats(T: int, capacity: int) -> int:
    n = ctypes.c_int64()
    _check("ar_inv_rms_floats", _lib.ar_inv_rms_floats(T, capacity, ctypes.byref(n)))
    return n.value


def ar_bank_create(T, d, r, capacity, dtype, norm, eps, rows, inv_rms, grad):
    h = ctypes.c_void_p()
    _check("ar_bank_create", _lib.ar_bank_create(ctypes.byref(h), T, d, r, capacity, dtype, norm,
                                                 eps, _ptr(rows), _ptr(inv_rms), _ptr(grad)))
    return h


def ar_bank_destroy(bank):
    _check("ar_bank_destroy", _lib.ar_bank_destroy(bank))


def ar_bank_row_count(bank) -> int:
    n = ctypes.c_int32()
    _check("ar_bank_row_count", _lib.ar_bank_row_count(bank, ctypes.byref(n)))
    return n.value


def ar_bank_row_ptr(bank, row: int) -> int:
    p = ctypes.c_void_p()
    _check("ar_bank_row_ptr", _lib.ar_bank_row_ptr(bank, row, ctypes.byref(p)))
    return p.value or 0


def ar_bank_append(bank, src, accumulate_from: int = -1, stream=None) -> int:
    row = ctypes.c_int32(-1)
    _check("ar_bank_append", _lib.ar_bank_append(bank, _ptr(src), accumulate_from,
                                                 ctypes.byref(row), _stream(stream)))
    return row.value


def ar_bank_append_strided(bank, src, token_stride: int, elem_stride: int,
                           accumulate_from: int = -1, stream=None) -> int:
    row = ctypes.c_int32(-1)
    _check("ar_bank_append_strided",
           _lib.ar_bank_append_strided(bank, _ptr(src), token_stride, elem_stride,
                                       accumulate_from, ctypes.byref(row), _stream(stream)))
    return row.value


def make_site(rows, H, q, g=None, site_id=0, q_stride=None, g_stride=None):
    """An ArSite (plus the row array it points to, which must stay alive).
    Strides default to those of the q / g tensors."""
    arr, n = _rows(rows)
    qs = q_stride if q_stride is not None else (q.stride(0) if isinstance(q, torch.Tensor) else 1)
    gs = g_stride if g_stride is not None else (
        g.stride(0) if isinstance(g, torch.Tensor) else 1)
    site = ArSite(ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32)), n, H, _ptr(q), qs, _ptr(g),
                  gs, site_id)
    site._keep = arr
    return site


def ar_route_fwd_site(bank, site: ArSite, partial, alpha, out, routed, lse, stream=None):
    _check("ar_route_fwd_site", _lib.ar_route_fwd_site(bank, ctypes.byref(site), _ptr(partial),
                                                       _ptr(alpha), _ptr(out), _ptr(routed),
                                                       _ptr(lse), _stream(stream)))


def ar_route_bwd_site(bank, site: ArSite, out, dout, lse, alpha, dq, dg, dalpha, ws, ws_bytes,
                      stream=None):
    _check("ar_route_bwd_site", _lib.ar_route_bwd_site(bank, ctypes.byref(site), _ptr(out),
                                                       _ptr(dout), _ptr(lse), _ptr(alpha),
                                                       _ptr(dq), _ptr(dg), _ptr(dalpha), _ptr(ws),
                                                       ws_bytes, _stream(stream)))


def ar_route_bwd_exact(bank, site: ArSite, out, dout, lse, alpha, coupling, dq, dg, dalpha, ws,
                       ws_bytes, stream=None):
    _check("ar_route_bwd_exact", _lib.ar_route_bwd_exact(bank, ctypes.byref(site), _ptr(out),
                                                         _ptr(dout), _ptr(lse), _ptr(alpha),
                                                         _ptr(coupling), _ptr(dq), _ptr(dg),
                                                         _ptr(dalpha), _ptr(ws), ws_bytes,
                                                         _stream(stream)))


def ar_bank_zero_grad(bank):
    _check("ar_bank_zero_grad", _lib.ar_bank_zero_grad(bank))


def ar_bank_reset(bank):
    _check("ar_bank_reset", _lib.ar_bank_reset(bank))


def ar_route_fwd(bank, rows, H, q, g, out, lse, site_id, stream=None):
    arr, n = _rows(rows)
    _check("ar_route_fwd", _lib.ar_route_fwd(bank, arr, n, H, _ptr(q), _ptr(g), _ptr(out),
                                             _ptr(lse), site_id, _stream(stream)))


def ar_route_fwd_append(bank, src, accumulate_from, rows, H, q, g, out, lse, site_id,
                        stream=None):
    """Append + forward in one call; returns (new row, fused)."""
    arr, n = _rows(rows)
    row, fused = ctypes.c_int32(-1), ctypes.c_int32(0)
    _check("ar_route_fwd_append",
           _lib.ar_route_fwd_append(bank, _ptr(src), accumulate_from, ctypes.byref(row), arr, n,
                                    H, _ptr(q), _ptr(g), _ptr(out), _ptr(lse), site_id,
                                    ctypes.byref(fused), _stream(stream)))
    return row.value, bool(fused.value)


def ar_route_fwd_delta(bank, rows, H, q, g, partial, alpha, out, routed, lse, site_id,
                       stream=None):
    arr, n = _rows(rows)
    _check("ar_route_fwd_delta", _lib.ar_route_fwd_delta(bank, arr, n, H, _ptr(q), _ptr(g),
                                                         _ptr(partial), _ptr(alpha), _ptr(out),
                                                         _ptr(routed), _ptr(lse), site_id,
                                                         _stream(stream)))


def ar_route_bwd_delta(bank, rows, H, q, g, routed, dout, lse, alpha, dq, dg, dalpha, ws,
                       ws_bytes, site_id, stream=None):
    arr, n = _rows(rows)
    _check("ar_route_bwd_delta", _lib.ar_route_bwd_delta(bank, arr, n, H, _ptr(q), _ptr(g),
                                                         _ptr(routed), _ptr(dout), _ptr(lse),
                                                         _ptr(alpha), _ptr(dq), _ptr(dg),
                                                         _ptr(dalpha), _ptr(ws), ws_bytes,
                                                         site_id, _stream(stream)))


def ar_bank_append_broadcast(bank, vec, stream=None) -> int:
    row = ctypes.c_int32(-1)
    _check("ar_bank_append_broadcast", _lib.ar_bank_append_broadcast(bank, _ptr(vec),
                                                                     ctypes.byref(row),
                                                                     _stream(stream)))
    return row.value


def ar_bank_grad_token_sum(bank, row, out, stream=None):
    _check("ar_bank_grad_token_sum", _lib.ar_bank_grad_token_sum(bank, row, _ptr(out),
                                                                 _stream(stream)))


def ar_route_bwd_workspace(bank, H) -> int:
    b = ctypes.c_size_t()
    _check("ar_route_bwd_workspace", _lib.ar_route_bwd_workspace(bank, H, ctypes.byref(b)))
    return b.value


def ar_route_bwd(bank, rows, H, q, g, out, dout, lse, dq, dg, ws, ws_bytes, site_id, stream=None):
    arr, n = _rows(rows)
    _check("ar_route_bwd", _lib.ar_route_bwd(bank, arr, n, H, _ptr(q), _ptr(g), _ptr(out),
                                             _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dg), _ptr(ws),
                                             ws_bytes, site_id, _stream(stream)))


def ar_route_bwd_noalloc(bank, rows, H, q, g, out, dout, lse, dq, dg, site_id, stream=None):
    arr, n = _rows(rows)
    _check("ar_route_bwd_noalloc", _lib.ar_route_bwd_noalloc(bank, arr, n, H, _ptr(q), _ptr(g),
                                                             _ptr(out), _ptr(dout), _ptr(lse),
                                                             _ptr(dq), _ptr(dg), site_id,
                                                             _stream(stream)))


def ar_noalloc_scratch_bytes() -> int:
    b = ctypes.c_size_t()
    _check("ar_noalloc_scratch_bytes", _lib.ar_noalloc_scratch_bytes(ctypes.byref(b)))
    return b.value


def ar_bank_grad_fold(bank, dst_row: int, src_row: int, stream=None):
    _check("ar_bank_grad_fold", _lib.ar_bank_grad_fold(bank, dst_row, src_row, _stream(stream)))


def ar_route_merge(bank, H, out_a, lse_a, out_b, lse_b, out, lse, stream=None):
    _check("ar_route_merge", _lib.ar_route_merge(bank, H, _ptr(out_a), _ptr(lse_a), _ptr(out_b),
                                                 _ptr(lse_b), _ptr(out), _ptr(lse),
                                                 _stream(stream)))


def _ptr_array(xs):
    arr = (ctypes.c_void_p * max(1, len(xs)))(*[_ptr(x) for x in xs])
    return arr, ctypes.cast(arr, ctypes.c_void_p)


def ar_route_fwd_multi(bank, rows, H, qs, gs, outs, lses, stream=None):
    arr, n = _rows(rows)
    qa, qp = _ptr_array(qs)
    ga, gp = _ptr_array(gs) if gs is not None else (None, None)
    oa, op = _ptr_array(outs)
    la, lp = _ptr_array(lses)
    _check("ar_route_fwd_multi", _lib.ar_route_fwd_multi(bank, arr, n, H, len(qs), qp, gp, op, lp,
                                                         _stream(stream)))


def ar_block_schedule(M: int, NB: int | None):
    """Returns (acc_from [M+1], sites: list of M+1 row lists)."""
    acc = (ctypes.c_int32 * (M + 1))()
    ptr = (ctypes.c_int32 * (M + 2))()
    need = ctypes.c_int64()
    nb = 0 if NB is None else NB
    st = _lib.ar_block_schedule(M, nb, acc, ptr, None, 0, ctypes.byref(need))
    if st not in (AR_OK, 4):
        _check("ar_block_schedule", st)
    flat = (ctypes.c_int32 * max(1, need.value))()
    _check("ar_block_schedule", _lib.ar_block_schedule(M, nb, acc, ptr, flat, need.value,
                                                       ctypes.byref(need)))
    sites = [list(flat[ptr[t]:ptr[t + 1]]) for t in range(M + 1)]
    return list(acc), sites


def ar_device_error() -> int:
    bits = ctypes.c_uint32()
    _check("ar_device_error", _lib.ar_device_error(ctypes.byref(bits)))
    return bits.value


def ar_device_status():
    """Raises ARError (AR_ERR_BOUNDS) if a checked build refused an access,
    else (AR_ERR_TIMEOUT) if a device-side wait ran out, since the last read
    of the device error word; clears the word."""
    _check("ar_device_status", _lib.ar_device_status())


def ar_route_fwd_lost_copies(bank, rows, H, q, g, out, lse, poll_limit: int, stream=None):
    arr, n = _rows(rows)
    _check("ar_route_fwd_lost_copies",
           _lib.ar_route_fwd_lost_copies(bank, arr, n, H, _ptr(q), _ptr(g), _ptr(out), _ptr(lse),
                                         poll_limit, _stream(stream)))


def ar_checked_fault():
    """(checked, address, bytes, kind) of the first access a checked build
    refused since the last call (kind 0: none); clears the record. checked
    is 0 in the unchecked library, which touches no device here."""
    c, a, b, k = ctypes.c_int32(), ctypes.c_uint64(), ctypes.c_uint32(), ctypes.c_uint32()
    _check("ar_checked_fault", _lib.ar_checked_fault(ctypes.byref(c), ctypes.byref(a),
                                                     ctypes.byref(b), ctypes.byref(k)))
    return c.value, a.value, b.value, k.value


def ar_checked_trim_out(nbytes: int):
    _check("ar_checked_trim_out", _lib.ar_checked_trim_out(nbytes))


# ---- convenience owner of a bank's buffers -------------------------------------

_TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
_AR_DT = {"bf16": AR_BF16, "f32": AR_F32}


class Bank:
    """A bank plus the torch buffers it points into (see ar_bank_create)."""

    def __init__(self, T: int, d: int, r: int | None = None, capacity: int = 1,
                 dtype: str = "bf16", norm: str = "key", eps: float = 1e-6,
                 with_grad: bool = True, device=None, grad: torch.Tensor | None = None):
        """grad: optional caller-owned [capacity, T, d] fp32 gradient rows
        (16-byte aligned; any view of that shape with unit inner strides)."""
        r = d if r is None else r
        dev = torch.device("cuda" if device is None else device)
        self.T, self.d, self.r, self.capacity, self.dtype = T, d, r, capacity, dtype
        self.torch_dtype = _TORCH_DT[dtype]
        self.rows = torch.empty((capacity, T, d), dtype=self.torch_dtype, device=dev)
        self.inv_ld = (capacity + 3) // 4 * 4
        self.inv = torch.empty(max(1, ar_inv_rms_floats(T, capacity)), dtype=torch.float32,
                               device=dev)
        if grad is not None:
            if (tuple(grad.shape) != (capacity, T, d) or grad.dtype != torch.float32
                    or not grad.is_contiguous()):
                raise ValueError("grad must be a contiguous fp32 [capacity, T, d] tensor")
            self.grad = grad
        else:
            self.grad = (torch.empty((capacity, T, d), dtype=torch.float32, device=dev)
                         if with_grad else None)
        self.handle = ar_bank_create(T, d, r, capacity, _AR_DT[dtype],
                                     AR_NORM_FULL if norm == "full" else AR_NORM_KEY, eps,
                                     self.rows, self.inv, self.grad)
        self._ws = {}

    def close(self):
        if self.handle is not None:
            ar_bank_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def count(self) -> int:
        return ar_bank_row_count(self.handle)

    def slot(self, row: int) -> torch.Tensor:
        return self.rows[row]

    def append(self, src: torch.Tensor, accumulate_from: int = -1, stream=None) -> int:
        """Append a [T, d] source; a strided view goes through ar_bank_append_strided."""
        if isinstance(src, torch.Tensor) and not src.is_contiguous() and src.dim() == 2:
            self._check_tensor(src, (self.T, self.d), self.torch_dtype, "src", contiguous=False)
            return ar_bank_append_strided(self.handle, src, src.stride(0), src.stride(1),
                                          accumulate_from, stream)
        self._check_tensor(src, (self.T, self.d), self.torch_dtype, "src")
        return ar_bank_append(self.handle, src, accumulate_from, stream)

    def zero_grad(self):
        ar_bank_zero_grad(self.handle)

    def reset(self):
        ar_bank_reset(self.handle)

    def inv_rms(self) -> torch.Tensor:
        """The cache as [T, capacity] (token-major view)."""
        return self.inv[: self.T * self.inv_ld].view(self.T, self.inv_ld)[:, : self.capacity]

    def route_fwd(self, rows, H, q, g=None, out=None, lse=None, site_id=0, stream=None):
        dev = self.rows.device
        if out is None:
            out = torch.empty((self.T, self.d), dtype=self.torch_dtype, device=dev)
        if lse is None:
            lse = torch.empty((self.T, H), dtype=torch.float32, device=dev)
        self._check_tensor(out, (self.T, self.d), self.torch_dtype, "out")
        self._check_tensor(lse, (self.T, H), torch.float32, "lse")
        self._check_tensor(q, (self.r,), torch.float32, "q", contiguous=False)
        if g is not None:
            self._check_tensor(g, (self.r,), torch.float32, "g", contiguous=False)
        if _strided(q, g):
            ar_route_fwd_site(self.handle, make_site(rows, H, q, g, site_id), None, None, out,
                              None, lse, stream)
        else:
            ar_route_fwd(self.handle, rows, H, q, g, out, lse, site_id, stream)
        return out, lse

    def route_fwd_append(self, src, accumulate_from, rows, H, q, g=None, out=None, lse=None,
                         site_id=0, stream=None):
        """Append src as the next row, then read the site (see ar_route_fwd_append);
        returns (out, lse, row, fused)."""
        dev = self.rows.device
        if out is None:
            out = torch.empty((self.T, self.d), dtype=self.torch_dtype, device=dev)
        if lse is None:
            lse = torch.empty((self.T, H), dtype=torch.float32, device=dev)
        self._check_tensor(src, (self.T, self.d), self.torch_dtype, "src")
        self._check_tensor(out, (self.T, self.d), self.torch_dtype, "out")
        self._check_tensor(lse, (self.T, H), torch.float32, "lse")
        self._check_tensor(q, (self.r,), torch.float32, "q")
        if g is not None:
            self._check_tensor(g, (self.r,), torch.float32, "g")
        row, fused = ar_route_fwd_append(self.handle, src, accumulate_from, rows, H, q, g, out,
                                         lse, site_id, stream)
        return out, lse, row, fused

    def route_fwd_delta(self, rows, H, q, g, partial, alpha, out=None, routed=None, lse=None,
                        site_id=0, stream=None):
        """Delta form: out = partial + alpha * routed (see ar_route_fwd_delta)."""
        dev = self.rows.device
        shape = (self.T, self.d)
        out = torch.empty(shape, dtype=self.torch_dtype, device=dev) if out is None else out
        routed = torch.empty(shape, dtype=self.torch_dtype, device=dev) if routed is None else routed
        lse = torch.empty((self.T, H), dtype=torch.float32, device=dev) if lse is None else lse
        for t, sh, dt, nm in ((partial, shape, self.torch_dtype, "partial"),
                              (out, shape, self.torch_dtype, "out"),
                              (routed, shape, self.torch_dtype, "routed"),
                              (lse, (self.T, H), torch.float32, "lse"),
                              (alpha, (1,), torch.float32, "alpha")):
            self._check_tensor(t, sh, dt, nm)
        ar_route_fwd_delta(self.handle, rows, H, q, g, partial, alpha, out, routed, lse, site_id,
                           stream)
        return out, routed, lse

    def route_bwd_delta(self, rows, H, q, g, routed, dout, lse, alpha, dq=None, dg=None,
                        dalpha=None, site_id=0, stream=None, ws=None):
        dev = self.rows.device
        dq = torch.empty(self.r, dtype=torch.float32, device=dev) if dq is None else dq
        if dg is None and g is not None:
            dg = torch.empty(self.r, dtype=torch.float32, device=dev)
        dalpha = torch.empty(1, dtype=torch.float32, device=dev) if dalpha is None else dalpha
        ws = self.workspace(H) if ws is None else ws
        ar_route_bwd_delta(self.handle, rows, H, q, g, routed, dout, lse, alpha, dq, dg, dalpha,
                           ws, ws.numel() * 4, site_id, stream)
        return dq, dg, dalpha

    def route_fwd_multi(self, rows, H, qs, gs=None, outs=None, lses=None, stream=None):
        """Reads of several sites over one row list in one pass (see
        ar_route_fwd_multi); returns (outs, lses)."""
        dev = self.rows.device
        if outs is None:
            outs = [torch.empty((self.T, self.d), dtype=self.torch_dtype, device=dev) for _ in qs]
        if lses is None:
            lses = [torch.empty((self.T, H), dtype=torch.float32, device=dev) for _ in qs]
        for i, q in enumerate(qs):
            self._check_tensor(q, (self.r,), torch.float32, f"q[{i}]")
            if gs is not None and gs[i] is not None:
                self._check_tensor(gs[i], (self.r,), torch.float32, f"g[{i}]")
            self._check_tensor(outs[i], (self.T, self.d), self.torch_dtype, f"out[{i}]")
            self._check_tensor(lses[i], (self.T, H), torch.float32, f"lse[{i}]")
        ar_route_fwd_multi(self.handle, rows, H, qs, gs, outs, lses, stream)
        return outs, lses

    def append_broadcast(self, vec, stream=None) -> int:
        self._check_tensor(vec, (self.d,), self.torch_dtype, "vec")
        return ar_bank_append_broadcast(self.handle, vec, stream)

    def grad_token_sum(self, row, out=None, stream=None):
        out = torch.empty(self.d, dtype=torch.float32, device=self.rows.device) if out is None else out
        ar_bank_grad_token_sum(self.handle, row, out, stream)
        return out

    def workspace(self, H) -> torch.Tensor:
        nbytes = ar_route_bwd_workspace(self.handle, H)
        ws = self._ws.get(H)
        if ws is None or ws.numel() * 4 < nbytes:
            ws = torch.empty(max(4, nbytes // 4), dtype=torch.float32, device=self.rows.device)
            self._ws[H] = ws
        return ws

    def route_bwd(self, rows, H, q, g, out, dout, lse, dq=None, dg=None, site_id=0,
                  stream=None, ws=None, exact=False):
        """exact=True: the coupling term summed over the sources first
        (ar_route_bwd_exact), into a [T, H] scratch allocated here."""
        dev = self.rows.device
        strided = _strided(q, g)
        if dq is None:  # laid out like q (dq is written with q's stride)
            dq = torch.empty_strided((self.r,), (q.stride(0),), dtype=torch.float32, device=dev)
        if dg is None and g is not None:
            dg = torch.empty_strided((self.r,), (g.stride(0),), dtype=torch.float32, device=dev)
        for t, shape, dt, nm in ((out, (self.T, self.d), self.torch_dtype, "out"),
                                 (dout, (self.T, self.d), self.torch_dtype, "dout"),
                                 (lse, (self.T, H), torch.float32, "lse")):
            self._check_tensor(t, shape, dt, nm)
        for t, ref, nm in ((q, q, "q"), (dq, q, "dq"), (g, g, "g"), (dg, g, "dg")):
            if t is not None:
                self._check_tensor(t, (self.r,), torch.float32, nm, contiguous=False)
                if ref is not None and t.stride(0) != ref.stride(0):
                    raise ValueError(f"{nm} must have the stride of {'q' if nm[-1] == 'q' else 'g'}")
        if ws is None:
            ws = self.workspace(H)
        if exact:
            coupling = torch.empty((self.T, H), dtype=torch.float32, device=dev)
            ar_route_bwd_exact(self.handle, make_site(rows, H, q, g, site_id), out, dout, lse,
                               None, coupling, dq, dg, None, ws, ws.numel() * 4, stream)
            return dq, dg
        if strided:
            ar_route_bwd_site(self.handle, make_site(rows, H, q, g, site_id), out, dout, lse, None,
                              dq, dg, None, ws, ws.numel() * 4, stream)
        else:
            ar_route_bwd(self.handle, rows, H, q, g, out, dout, lse, dq, dg, ws, ws.numel() * 4,
                         site_id, stream)
        return dq, dg

    @staticmethod
    def _check_tensor(t, shape, dtype, name, contiguous=True):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype or (contiguous and
                                                                  not t.is_contiguous()):
            raise ValueError(f"{name}: expected {'contiguous ' if contiguous else ''}{dtype} "
                             f"{tuple(shape)}, got {t.dtype} {tuple(t.shape)}")
        if not contiguous and any(st < 1 for st in t.stride()[-1:]):
            raise ValueError(f"{name}: element stride must be positive")


def _strided(q, g) -> bool:
    return q.stride(0) != 1 or (g is not None and g.stride(0) != 1)

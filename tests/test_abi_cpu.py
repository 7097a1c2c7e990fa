"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/attnres.h declares, its schedule bookkeeping matches
the oracle bit for bit, and argument checks fail before any launch."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attnres.h")


@pytest.fixture(scope="module")
def B():
    from depth_wise_attention_ar_gb300 import build
    build.build()
    from depth_wise_attention_ar_gb300 import binding
    return binding


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(ar_[a-z0-9_]+)\s*\(", txt)))


def test_library_exports_every_declared_symbol(B):
    names = _declared()
    assert len(names) >= 14
    lib = ctypes.CDLL(B.LIBPATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.SIGNATURES) == names


def test_status_strings(B):
    for code, name in B.STATUS.items():
        assert B.ar_status_string(code) == name


def test_inv_rms_floats(B):
    assert B.ar_inv_rms_floats(10, 73) == 10 * 76
    assert B.ar_inv_rms_floats(0, 1) == 0
    with pytest.raises(B.ARError):
        B.ar_inv_rms_floats(5, 0)


@pytest.mark.parametrize("M,NB", [(1, None), (4, None), (6, 3), (5, 2), (48, 5), (64, 8),
                                  (72, None), (7, 7), (9, 1), (13, 4)])
def test_block_schedule_matches_oracle(B, M, NB):
    from oracle import schedule
    acc, sites = B.ar_block_schedule(M, NB)
    plan = schedule.block_plan(M, NB)
    assert sites == plan["sites"]
    exp_acc = [-1 if op[0] in ("emb", "copy") else op[1] for op in plan["row_ops"]]
    assert acc == exp_acc


def test_block_schedule_errors(B):
    with pytest.raises(B.ARError) as e:
        B.ar_block_schedule(0, 1)
    assert e.value.name == "AR_ERR_INVALID_ARG"


FAKE = 1 << 20  # an aligned address that is never dereferenced by these calls


def _bank(B, T=16, d=512, r=None, cap=4, dtype=1, grad=True):
    return B.ar_bank_create(T, d, d if r is None else r, cap, dtype, 0, 1e-6, FAKE, FAKE,
                            FAKE if grad else None)


def test_bank_create_checks(B):
    def code(*a):
        with pytest.raises(B.ARError) as e:
            B.ar_bank_create(*a)
        return e.value.name
    assert code(16, 512, 512, 4, 1, 0, 1e-6, None, FAKE, FAKE) == "AR_ERR_INVALID_ARG"
    assert code(16, 512, 512, 0, 1, 0, 1e-6, FAKE, FAKE, FAKE) == "AR_ERR_INVALID_ARG"
    assert code(16, 512, 1024, 4, 1, 0, 1e-6, FAKE, FAKE, FAKE) == "AR_ERR_SHAPE"
    assert code(16, 500, 500, 4, 1, 0, 1e-6, FAKE, FAKE, FAKE) == "AR_ERR_SHAPE"
    assert code(16, 512, 512, 4, 1, 0, 1e-6, FAKE + 8, FAKE, FAKE) == "AR_ERR_ALIGN"
    assert code(16, 512, 512, 4, 7, 0, 1e-6, FAKE, FAKE, FAKE) == "AR_ERR_INVALID_ARG"
    h = _bank(B)
    assert B.ar_bank_row_count(h) == 0
    assert B.ar_bank_row_ptr(h, 2) == FAKE + 2 * 16 * 512 * 2
    with pytest.raises(B.ARError):
        B.ar_bank_row_ptr(h, 4)
    B.ar_bank_destroy(h)


def _err(fn, *a, **k):
    from depth_wise_attention_ar_gb300 import binding
    with pytest.raises(binding.ARError) as e:
        fn(*a, **k)
    return e.value.name


def test_route_argument_checks_precede_launch(B):
    h = _bank(B)
    q = FAKE
    # nothing appended: any row is out of range
    assert _err(B.ar_route_fwd, h, [0], 4, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_fwd, h, [], 4, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_fwd, h, list(range(257)), 4, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_fwd, h, [0], 3, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_SHAPE"
    assert _err(B.ar_route_fwd, h, [0], 64, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_UNSUPPORTED"
    assert _err(B.ar_route_fwd, h, [0], 4, None, None, FAKE, FAKE, 1, 0) == "AR_ERR_INVALID_ARG"
    B.ar_bank_destroy(h)
    for d, r, H in ((8192, 8192, 2), (1024, 760, 8), (8192, 1024, 8), (1000, 1000, 8),
                    (16384, 16384, 8), (512, 256, 64)):
        h = _bank(B, d=d, r=r)
        assert _err(B.ar_route_fwd, h, [0], H, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_UNSUPPORTED"
        B.ar_bank_destroy(h)
    # the delta form is served by the full-key and four-warp kernels only
    h = _bank(B, d=1280, r=256)
    assert _err(B.ar_route_fwd_delta, h, [0], 8, q, None, FAKE, FAKE, FAKE, FAKE, FAKE, 1,
                0) == "AR_ERR_INVALID_ARG"   # nothing appended yet
    B.ar_bank_destroy(h)


def test_failed_append_leaves_bank_unchanged_without_gpu(B):
    import torch
    if torch.cuda.is_available():
        pytest.skip("this check needs a machine without a GPU")
    h = _bank(B)
    assert _err(B.ar_bank_append, h, FAKE, -1, 0) == "AR_ERR_CUDA"
    assert B.ar_bank_row_count(h) == 0
    assert _err(B.ar_bank_append, h, FAKE, 0, 0) == "AR_ERR_INVALID_ARG"   # row 0 not appended
    assert _err(B.ar_bank_append, h, FAKE + 4, -1, 0) == "AR_ERR_ALIGN"
    B.ar_bank_destroy(h)


def test_backward_without_gradient_rows_is_rejected(B):
    h = _bank(B, grad=False)
    assert _err(B.ar_route_bwd, h, [0], 4, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20,
                0, 0) == "AR_ERR_INVALID_ARG"
    B.ar_bank_destroy(h)

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


def test_block_schedule_matches_oracle_sweep(B):
    from oracle import schedule
    for M in range(1, 41):
        for NB in list(range(1, M + 1)) + [None]:
            acc, sites = B.ar_block_schedule(M, NB)
            plan = schedule.block_plan(M, NB)
            assert sites == plan["sites"], (M, NB)
            assert acc == [-1 if op[0] in ("emb", "copy") else op[1] for op in plan["row_ops"]]


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
    assert code(16, 0, 0, 4, 1, 0, 1e-6, FAKE, FAKE, FAKE) == "AR_ERR_SHAPE"
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
    # H = 64 over d = 512 is served (by the scalar-access kernels): the row check fails
    assert _err(B.ar_route_fwd, h, [0], 64, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_fwd, h, [0], 4, None, None, FAKE, FAKE, 1, 0) == "AR_ERR_INVALID_ARG"
    B.ar_bank_destroy(h)
    # every shape has a kernel family unless the scalar-access kernels' per-warp
    # [n_src, H] arrays outgrow shared memory
    for d, r, H, n in ((8192, 8192, 8192, 4), (4096, 4096, 1024, 32), (2048, 2048, 2048, 16)):
        h = _bank(B, d=d, r=r)
        assert _err(B.ar_route_fwd, h, list(range(n)), H, q, None, FAKE, FAKE, 1,
                    0) == "AR_ERR_UNSUPPORTED"
        # a repeated row counts once
        assert _err(B.ar_route_fwd, h, [0] * n, H, q, None, FAKE, FAKE, 1,
                    0) == "AR_ERR_INVALID_ARG"
        B.ar_bank_destroy(h)
    for d, r, H in ((8192, 8192, 2), (1024, 760, 8), (8192, 1024, 8), (1000, 1000, 8),
                    (513, 513, 1), (513, 128, 1), (520, 260, 5)):
        h = _bank(B, d=d, r=r)
        assert _err(B.ar_route_fwd, h, [0], H, q, None, FAKE, FAKE, 1, 0) == "AR_ERR_INVALID_ARG"
        B.ar_bank_destroy(h)
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
    assert _err(B.ar_bank_append, h, FAKE + 1, -1, 0) == "AR_ERR_ALIGN"
    B.ar_bank_destroy(h)


def test_backward_without_gradient_rows_is_rejected(B):
    h = _bank(B, grad=False)
    assert _err(B.ar_route_bwd, h, [0], 4, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 20,
                0, 0) == "AR_ERR_INVALID_ARG"
    B.ar_bank_destroy(h)


def test_site_descriptor_and_strided_append_checks(B):
    h = _bank(B)
    site = B.make_site([0], 4, FAKE, None, 1, q_stride=1, g_stride=1)
    assert _err(B.ar_route_fwd_site, h, site, None, None, FAKE, None, FAKE, 0) == "AR_ERR_INVALID_ARG"
    bad = B.make_site([0], 4, FAKE, None, 1, q_stride=0, g_stride=1)
    assert _err(B.ar_route_fwd_site, h, bad, None, None, FAKE, None, FAKE, 0) == "AR_ERR_INVALID_ARG"
    # the delta pointers come all together or not at all
    assert _err(B.ar_route_fwd_site, h, site, FAKE, None, FAKE, None, FAKE,
                0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_bwd_site, h, site, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, FAKE,
                1 << 20, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_bank_append_strided, h, FAKE, -1, 1, -1, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_bank_append_strided, h, FAKE, 512, 0, -1, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_bank_append_strided, h, FAKE + 1, 512, 1, -1, 0) == "AR_ERR_ALIGN"
    B.ar_bank_destroy(h)


def test_site_struct_layout_matches_the_header(B, tmp_path):
    """ctypes' ArSite has the field offsets and size gcc gives struct ar_site."""
    import ctypes
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stddef.h>\n#include <stdio.h>\n#include "attnres.h"\n'
        'int main(void) { printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(ar_site),'
        ' offsetof(ar_site, rows), offsetof(ar_site, n_src), offsetof(ar_site, H),'
        ' offsetof(ar_site, q), offsetof(ar_site, q_stride), offsetof(ar_site, g),'
        ' offsetof(ar_site, g_stride), offsetof(ar_site, site_id)); return 0; }\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    S = B.ArSite
    want = [ctypes.sizeof(S)] + [getattr(S, f).offset for f, _ in S._fields_]
    assert got == want


def test_multi_query_read_argument_checks(B):
    h = _bank(B)
    # nothing appended: a row out of range; query count out of range; null query
    assert _err(B.ar_route_fwd_multi, h, [0], 4, [FAKE], None, [FAKE], [FAKE], 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_fwd_multi, h, [0], 4, [], None, [], [], 0) == "AR_ERR_INVALID_ARG"
    nine = [FAKE] * (B.AR_MAX_QUERIES + 1)
    assert _err(B.ar_route_fwd_multi, h, [0], 4, nine, None, nine, nine, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_fwd_multi, h, [0], 3, [FAKE], None, [FAKE], [FAKE], 0) == "AR_ERR_SHAPE"
    B.ar_bank_destroy(h)


def test_route_fwd_append_checks_precede_launch(B):
    """ar_route_fwd_append runs the append's and the site's checks before it
    appends or launches anything: on each refusal the bank is unchanged."""
    import torch
    h = _bank(B, cap=2)
    fa = B.ar_route_fwd_append
    # the site lists a row past the new one (the new row is 0)
    assert _err(fa, h, FAKE, -1, [0, 1], 4, FAKE, None, FAKE, FAKE, 0, 0) == "AR_ERR_INVALID_ARG"
    # accumulation onto a row that does not exist
    assert _err(fa, h, FAKE, 0, [0], 4, FAKE, None, FAKE, FAKE, 0, 0) == "AR_ERR_INVALID_ARG"
    assert _err(fa, h, FAKE + 1, -1, [0], 4, FAKE, None, FAKE, FAKE, 0, 0) == "AR_ERR_ALIGN"
    assert _err(fa, h, FAKE, -1, [0], 3, FAKE, None, FAKE, FAKE, 0, 0) == "AR_ERR_SHAPE"
    assert _err(fa, h, FAKE, -1, [0], 4, FAKE, None, None, FAKE, 0, 0) == "AR_ERR_INVALID_ARG"
    assert _err(fa, h, FAKE, -1, [0], 4, None, None, FAKE, FAKE, 0, 0) == "AR_ERR_INVALID_ARG"
    assert _err(fa, h, FAKE, -1, [], 4, FAKE, None, FAKE, FAKE, 0, 0) == "AR_ERR_INVALID_ARG"
    assert B.ar_bank_row_count(h) == 0
    if not torch.cuda.is_available():
        # a valid call reaches the launch, which fails without a GPU
        assert _err(fa, h, FAKE, -1, [0], 4, FAKE, None, FAKE, FAKE, 0, 0) == "AR_ERR_CUDA"
        assert B.ar_bank_row_count(h) == 0
    B.ar_bank_destroy(h)


def test_binding_refuses_to_import_without_the_library(tmp_path):
    """No fallback: the package's Python, copied without the compiled library,
    raises on import of the binding and on any package name it provides."""
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "depth_wise_attention_ar_gb300")
    dst = tmp_path / "depth_wise_attention_ar_gb300"
    dst.mkdir()
    for name in os.listdir(src):
        if name.endswith(".py"):
            shutil.copy(os.path.join(src, name), dst / name)
    for stmt in ("import depth_wise_attention_ar_gb300.binding",
                 "import depth_wise_attention_ar_gb300 as p; p.Bank"):
        p = subprocess.run([sys.executable, "-c", stmt],
                           cwd=tmp_path, capture_output=True, text=True,
                           env={**os.environ, "PYTHONPATH": str(tmp_path)})
        assert p.returncode != 0
        assert "ImportError" in p.stderr and "is not built" in p.stderr


def test_noalloc_scratch_size_is_reported_by_the_library(B):
    """The no-alloc backward's fixed scratch size comes from the library (the
    header's AR_NOALLOC_SCRATCH_BYTES), so callers and tests need no copy of it."""
    assert B.ar_noalloc_scratch_bytes() == 8 << 20
    txt = open(HEADER).read()
    assert "#define AR_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)" in txt


def test_device_status_without_gpu(B):
    """Reading the device error word needs a device: without one the call
    reports AR_ERR_CUDA (and never AR_ERR_TIMEOUT)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("this check needs a machine without a GPU")
    assert _err(B.ar_device_status) == "AR_ERR_CUDA"


def test_lost_copy_hook_checks_precede_launch(B):
    h = _bank(B)
    # nothing appended: the site's rows are out of range
    assert _err(B.ar_route_fwd_lost_copies, h, [0], 4, FAKE, None, FAKE, FAKE, 100,
                0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_fwd_lost_copies, h, [0], 3, FAKE, None, FAKE, FAKE, 100,
                0) == "AR_ERR_SHAPE"
    B.ar_bank_destroy(h)


def test_unchecked_library_reports_no_range_checks(B):
    """The library the binding loads by default is built without the range
    checks: ar_checked_fault says so without touching a device, and the
    trim hook of the checks is refused."""
    if B.CHECKED:
        pytest.skip("the range-checked build is loaded")
    assert B.ar_checked_fault() == (0, 0, 0, 0)
    assert _err(B.ar_checked_trim_out, 64) == "AR_ERR_UNSUPPORTED"


def test_checked_build_has_its_own_library_and_objects():
    """The range-checked variant builds from the same sources into its own
    library and object folder, so the two never overwrite each other."""
    from depth_wise_attention_ar_gb300 import build
    assert build.LIB != build.LIB_CHECKED and build.BUILD != build.BUILD_CHECKED
    assert os.path.dirname(build.LIB_CHECKED) == os.path.dirname(build.LIB)


def test_exact_backward_checks_precede_launch(B):
    """ar_route_bwd_exact refuses a missing or misaligned coupling buffer, and
    the delta form, before anything is launched."""
    h = _bank(B)
    site = B.make_site([0], 4, FAKE, None, 0)
    assert _err(B.ar_route_bwd_exact, h, site, FAKE, FAKE, FAKE, None, None, FAKE, None, None,
                FAKE, 1 << 20, 0) == "AR_ERR_INVALID_ARG"
    assert _err(B.ar_route_bwd_exact, h, site, FAKE, FAKE, FAKE, None, FAKE + 2, FAKE, None, None,
                FAKE, 1 << 20, 0) == "AR_ERR_ALIGN"
    assert _err(B.ar_route_bwd_exact, h, site, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE,
                FAKE, 1 << 20, 0) == "AR_ERR_UNSUPPORTED"      # the delta form
    B.ar_bank_destroy(h)


def test_binding_signatures_match_the_header_parameter_counts(B):
    """Every ctypes signature in the binding takes as many arguments as its C
    declaration in include/attnres.h has parameters (a parameter added on one
    side only would shift every argument after it)."""
    txt = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    decls = dict(re.findall(r"\b(ar_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", txt))
    for name, (argtypes, _) in B.SIGNATURES.items():
        params = " ".join(decls[name].split())
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert n == len(argtypes), (name, n, len(argtypes))

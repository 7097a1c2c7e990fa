"""The range-checked build (a stand-in for a memory checker; see
include/attnres.h, ar_checked_fault).

test_gpu_suite_under_range_checks builds libattnres_gb300_checked.so and runs
the GPU tests again in a child process that loads it (AR_CHECKED=1): every
kernel access is checked against its launch's buffers, and the suite's
conftest fails any test after which an access was refused. The other tests
here run only in that child: they shorten the declared extent of an output
buffer (inside the real allocation, so nothing leaves real memory) and check
that the stores into the cut-off tail are refused, recorded and skipped,
while everything else the kernel writes still matches the oracle.
"""

import os
import subprocess
import sys

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKED = os.environ.get("AR_CHECKED", "") == "1"


def test_gpu_suite_under_range_checks():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    if CHECKED:
        pytest.skip("already inside the checked run")
    from depth_wise_attention_ar_gb300 import build
    build.build(checked=True)
    env = dict(os.environ, AR_CHECKED="1")
    cmd = [sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=2400)
    print(p.stdout[-4000:])
    print(p.stderr[-2000:])
    assert p.returncode == 0
    last = p.stdout.strip().splitlines()[-1]
    assert " passed" in last and "failed" not in last


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    if not CHECKED:
        pytest.skip("runs in the range-checked build (AR_CHECKED=1)")
    from depth_wise_attention_ar_gb300 import build
    build.build(checked=True)
    from depth_wise_attention_ar_gb300 import binding
    assert binding.CHECKED
    return binding


def _nmax(x, ref):
    x = np.asarray(x, dtype=np.float64)
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


# (d, r, H): one shape per forward family — one-warp full keys, the
# two-tokens-per-warp kernel, four warps per row with full and sliced keys,
# one-warp sliced keys, scalar accesses
SHAPES = [(1280, 1280, 8), (512, 512, 4), (4096, 4096, 8), (4096, 1024, 8), (1280, 256, 8),
          (520, 520, 4)]


@pytest.mark.parametrize("d,r,H", SHAPES)
def test_stores_past_a_shortened_output_are_refused(B, orc, d, r, H):
    import torch
    T, N, dt = 333, 5, "bf16"
    es = 2
    inp = synth.HostInputs(seed=71 + d + r, q_std=0.5, g_kind="random")
    bank = B.Bank(T, d, r, N, dt)
    for j in range(N):
        bank.append(inp.output(j, T, d, dt))
    rows = list(range(N))
    q, g = inp.query(0, r), inp.norm_weight(0, r)
    out = torch.full((T, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), 7.0, device="cuda")
    B.ar_device_status()
    assert B.ar_checked_fault()[3] == 0
    B.ar_checked_trim_out(d * es)                 # the last token's row is cut off
    try:
        bank.route_fwd(rows, H, q, g, out=out, lse=lse, site_id=0)
    finally:
        B.ar_checked_trim_out(0)
    checked, addr, nbytes, kind = B.ar_checked_fault()
    assert checked == 1 and kind == 2             # a refused global store
    base = out.data_ptr() + (T - 1) * d * es
    assert base <= addr < base + d * es and addr + nbytes <= base + d * es
    with pytest.raises(B.ARError) as e:
        B.ar_device_status()
    assert e.value.name == "AR_ERR_BOUNDS"
    assert torch.all(out[T - 1] == 7.0)           # refused stores were not made
    host = [inp.host_output(j, T, d, dt) for j in rows]
    ref_out, ref_lse = orc.route_fwd(host, inp.host_query(0, r), inp.host_norm_weight(0, r), H, r=r)
    got = out[: T - 1].double().cpu().numpy()
    assert _nmax(got, ref_out[: T - 1]) < 2e-2
    assert _nmax(lse.double().cpu().numpy(), ref_lse) < 2e-2
    bank.close()


def test_multi_query_stores_past_a_shortened_output_are_refused(B, orc):
    import torch
    T, d, H, N, nq = 257, 1280, 8, 4, 3
    inp = synth.HostInputs(seed=83, q_std=0.5, g_kind="random")
    bank = B.Bank(T, d, d, N, "bf16")
    for j in range(N):
        bank.append(inp.output(j, T, d, "bf16"))
    rows = list(range(N))
    qs = [inp.query(i, d) for i in range(nq)]
    gs = [inp.norm_weight(i, d) for i in range(nq)]
    outs = [torch.full((T, d), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(nq)]
    lses = [torch.full((T, H), 7.0, device="cuda") for _ in range(nq)]
    B.ar_device_status()
    B.ar_checked_trim_out(d * 2)
    try:
        bank.route_fwd_multi(rows, H, qs, gs, outs=outs, lses=lses)
    finally:
        B.ar_checked_trim_out(0)
    checked, addr, nbytes, kind = B.ar_checked_fault()
    assert checked == 1 and kind == 2
    tails = [o.data_ptr() + (T - 1) * d * 2 for o in outs]
    assert any(t <= addr < t + d * 2 for t in tails)
    with pytest.raises(B.ARError) as e:
        B.ar_device_status()
    assert e.value.name == "AR_ERR_BOUNDS"
    host = [inp.host_output(j, T, d, "bf16") for j in rows]
    for i in range(nq):
        assert torch.all(outs[i][T - 1] == 7.0)
        ref_out, ref_lse = orc.route_fwd(host, inp.host_query(i, d), inp.host_norm_weight(i, d), H)
        assert _nmax(outs[i][: T - 1].double().cpu().numpy(), ref_out[: T - 1]) < 2e-2
        assert _nmax(lses[i].double().cpu().numpy(), ref_lse) < 2e-2
    bank.close()


@pytest.mark.parametrize("d,H", [(1280, 8), (520, 4)])
def test_merge_stores_past_a_shortened_output_are_refused(B, orc, d, H):
    """The same check on a kernel that takes its buffer table as a parameter
    of its own (the merge of two partial reads): the vector path (d = 1280)
    and the one-column path (d = 520)."""
    import torch
    T, N, dt = 301, 4, "bf16"
    inp = synth.HostInputs(seed=97 + d, q_std=0.5, g_kind="random")
    bank = B.Bank(T, d, d, N, dt)
    for j in range(N):
        bank.append(inp.output(j, T, d, dt))
    q, g = inp.query(0, d), inp.norm_weight(0, d)
    out_a, lse_a = bank.route_fwd([0, 1, 2], H, q, g, site_id=0)
    out_b, lse_b = bank.route_fwd([3], H, q, g, site_id=1)
    out = torch.full((T, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), 7.0, device="cuda")
    B.ar_device_status()
    assert B.ar_checked_fault()[3] == 0
    B.ar_checked_trim_out(d * 2)
    try:
        B.ar_route_merge(bank.handle, H, out_a, lse_a, out_b, lse_b, out, lse)
    finally:
        B.ar_checked_trim_out(0)
    checked, addr, nbytes, kind = B.ar_checked_fault()
    assert checked == 1 and kind == 2
    base = out.data_ptr() + (T - 1) * d * 2
    assert base <= addr < base + d * 2
    with pytest.raises(B.ARError) as e:
        B.ar_device_status()
    assert e.value.name == "AR_ERR_BOUNDS"
    assert torch.all(out[T - 1] == 7.0)
    host = [inp.host_output(j, T, d, dt) for j in range(N)]
    ref_out, ref_lse = orc.route_fwd(host, inp.host_query(0, d), inp.host_norm_weight(0, d), H)
    assert _nmax(out[: T - 1].double().cpu().numpy(), ref_out[: T - 1]) < 2e-2
    assert _nmax(lse.double().cpu().numpy(), ref_lse) < 2e-2
    bank.close()

"""Failure detection on the device, without a fault: a bounded wait that runs
out is reported through the device error word and the host turns it into
AR_ERR_TIMEOUT; the context stays usable.

The forward used here arms every shared-memory stage for its row's bytes and
issues no copy (ar_route_fwd_lost_copies), so each warp's first wait runs out
after a short poll limit with nothing in flight. Nothing traps and nothing
waits without a bound. Also here: a call made while another device is current
than the bank's is refused before any launch (needs two GPUs).
"""

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from depth_wise_attention_ar_gb300 import build
    build.build()
    from depth_wise_attention_ar_gb300 import binding
    return binding


def _nmax(x, ref):
    x = x.detach().double().cpu().numpy()
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def test_lost_copy_wait_runs_out_and_reports_timeout(B, orc):
    import torch
    T, d, H, N = 4099, 1280, 8, 3
    inp = synth.HostInputs(seed=61, q_std=0.5, g_kind="random")
    bank = B.Bank(T, d, d, N, "bf16")
    for j in range(N):
        bank.rows[j].copy_(inp.output(j, T, d, "bf16"))
        bank.append(bank.rows[j])
    q, g = inp.query(0, d), inp.norm_weight(0, d)
    rows = list(range(N))
    B.ar_device_status()                       # a clean error word to start from
    out = torch.full((T, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, H), 7.0, device="cuda")
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    B.ar_route_fwd_lost_copies(bank.handle, rows, H, q, g, out, lse, 2000)
    t1.record()
    torch.cuda.synchronize()
    # bounded: at most 2000 polls for the lost wait and per armed stage, each
    # sleeping at most the kernels' suspend hint (10 us)
    ms = t0.elapsed_time(t1)
    print(f"lost-copy forward: {ms:.2f} ms")
    assert ms < 1000.0
    with pytest.raises(B.ARError) as e:
        B.ar_device_status()
    assert e.value.name == "AR_ERR_TIMEOUT"
    assert torch.all(out == 7.0) and torch.all(lse == 7.0)   # the warps left before writing
    B.ar_device_status()                       # reading cleared the word
    # the context is still usable: the same site's real forward matches the oracle
    out2, lse2 = bank.route_fwd(rows, H, q, g, site_id=0)
    torch.cuda.synchronize()
    B.ar_device_status()
    host = [inp.host_output(j, T, d, "bf16") for j in rows]
    ref_out, ref_lse = orc.route_fwd(host, inp.host_query(0, d), inp.host_norm_weight(0, d), H)
    assert _nmax(out2, ref_out) < 2e-2 and _nmax(lse2, ref_lse) < 2e-2


def test_lost_copy_hook_serves_only_the_one_warp_forward(B):
    import torch
    q = torch.zeros(512, device="cuda")
    bank = B.Bank(16, 512, 512, 1, "bf16")
    bank.append(torch.zeros((16, 512), dtype=torch.bfloat16, device="cuda"))
    out = torch.empty((16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((16, 4), device="cuda")
    with pytest.raises(B.ARError) as e:         # two tokens per warp at 512 columns, H = 4
        B.ar_route_fwd_lost_copies(bank.handle, [0], 4, q, None, out, lse, 100)
    assert e.value.name == "AR_ERR_UNSUPPORTED"
    with pytest.raises(B.ARError) as e:
        B.ar_route_fwd_lost_copies(bank.handle, [0], 8, q, None, out, lse, 0)
    assert e.value.name == "AR_ERR_INVALID_ARG"


def test_calls_on_another_device_are_refused(B):
    import torch
    if torch.cuda.device_count() < 2:
        pytest.skip("needs two GPUs")
    with torch.cuda.device(0):
        bank = B.Bank(64, 512, 512, 2, "bf16", device="cuda:0")
        bank.append(torch.zeros((64, 512), dtype=torch.bfloat16, device="cuda:0"))
    with torch.cuda.device(1):
        with pytest.raises(B.ARError) as e:
            B.ar_bank_append(bank.handle, bank.rows[1].data_ptr(), -1)
        assert e.value.name == "AR_ERR_INVALID_ARG"
        assert B.ar_bank_row_count(bank.handle) == 1

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _no_refused_access():
    """Under the range-checked build (AR_CHECKED=1), fail any test after which
    the library reports an access its checks refused. Tests that provoke a
    refusal on purpose read and clear the record themselves."""
    yield
    if os.environ.get("AR_CHECKED", "") != "1":
        return
    b = sys.modules.get("depth_wise_attention_ar_gb300.binding")
    if b is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    checked, addr, nbytes, kind = b.ar_checked_fault()
    assert checked == 1, "AR_CHECKED=1 but the unchecked library is loaded"
    assert kind == 0, f"a kernel access was refused: kind {kind}, {nbytes} bytes at {addr:#x}"

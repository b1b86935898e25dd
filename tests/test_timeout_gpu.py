"""Bounded device waits run out without a fault.

A test hook (GBCE_TEST_STALL_COPY=1) makes CTA 0 of the streaming or the
register-resident kernel leave its first bulk copy out, so the wait for it
gives up after GBCE_WAIT_TIMEOUT_MS. The call must report CE_ERR_TIMEOUT
through the device status word, and the context must stay usable: the same
call without the hook then matches the oracle. Nothing here traps, faults or
hangs the GPU."""
import pytest

import workloads
from ce_gpu import run_cuda

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


@pytest.mark.parametrize("kernel,V", [("4", 4096), ("4", 32000), ("2", 65536), ("6", 131072)])
@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_wait_runs_out_then_context_usable(monkeypatch, kernel, V, reduction):
    from softmax_cross_entropy_gb300 import _lib
    from test_parity_gpu import check_full
    monkeypatch.setenv("GBCE_KERNEL", kernel)
    monkeypatch.setenv("GBCE_WAIT_TIMEOUT_MS", "20")
    # no ignored rows: CTA 0 owns row 0 (48 rows, one or a few a CTA), and an
    # ignored row would leave it no copy to leave out
    case = workloads.random_case(17, 48, V, dtype="bf16", ignore_frac=0.0, reduction=reduction,
                                 softcap=30.0 if kernel == "6" else None)
    monkeypatch.setenv("GBCE_TEST_STALL_COPY", "1")
    out = run_cuda(case)
    assert out["status"] == _lib.CE_ERR_TIMEOUT
    monkeypatch.delenv("GBCE_TEST_STALL_COPY")
    check_full(case)

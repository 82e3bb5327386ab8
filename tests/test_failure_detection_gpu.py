"""Failure detection on the GPU without a fault: a bounded wait on a barrier that
nothing completes gives up after its limit, the kernel returns, the host reads
W4A16_ERR_TIMEOUT from the error word, and the same context then runs a correct GEMM
on the same workspace (error word and split-K counters cleared)."""
import numpy as np
import pytest

from tests.parity import check_within
from weight_only_int4_02_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def w():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_02_gb300 import w4a16
    w4a16.lib()
    return w4a16


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("own_workspace", [False, True])
def test_bounded_wait_times_out_and_the_context_stays_usable(w, oracle_mod, own_workspace):
    M, N, K, G = 1, 4096, 4096, 128          # a split plan: the counters are in use
    ws = None if own_workspace else torch.zeros(w.workspace_bytes(M, N, K, G), dtype=torch.uint8, device="cuda")
    assert w.check_device_status(ws) == w.OK
    w.selftest_wait_timeout(2_000_000, workspace=ws)          # 2 ms
    assert w.check_device_status(ws) == w.ERR_TIMEOUT
    assert w.check_device_status(ws) == w.OK                  # read once, then cleared
    x, q, s = inputs.problem(M, K, N, G, 3)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    if own_workspace:
        y = w.gemm(to_dev(x), packed, sp, N, G)
    else:
        y = w.gemm_ws(to_dev(x), packed, sp, N, G, ws)
    torch.cuda.synchronize()
    assert w.check_device_status(ws) == w.OK
    y_ref, absum = oracle_mod.gemm(x, q, s, G)
    check_within(y.cpu().numpy(), y_ref, absum, "GEMM after a timed-out wait")


def test_timeout_takes_about_its_limit(w):
    ws = torch.zeros(4096 * 2, dtype=torch.uint8, device="cuda")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    w.selftest_wait_timeout(20_000_000, workspace=ws)         # 20 ms
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    assert 19.0 <= ms <= 200.0, ms
    assert w.check_device_status(ws) == w.ERR_TIMEOUT

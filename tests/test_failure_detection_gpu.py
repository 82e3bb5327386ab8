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


def test_gemm_waits_run_out_in_every_kernel_then_the_context_recovers(w, oracle_mod):
    """The GEMM kernels' own bounded waits, made to run out: with the wait limit at
    1 ns, a wait that is not satisfied at once gives up; its CTA stops issuing, waits
    (with a fixed bound) for the copies and MMAs it has in flight, frees its tensor
    memory and returns, and the host reads W4A16_ERR_TIMEOUT. Every kernel is one
    CTA (no clusters, no writes between CTAs), so this path touches nothing another
    CTA still uses. A long-K layer (18432 deep, one 128-column tile per SM) keeps
    waits of microseconds in every kernel: the tensor-core tiles of 16 to 256 rows,
    the CUDA-core kernel and the decode kernel (8 and 16 rows of X). With the limit restored, the same context and
    workspace compute the same GEMMs correctly (checked against the oracle on
    sampled rows and columns)."""
    K, N, G = 18432, 19456, 128
    q = inputs.codes(K, N, 7)
    s = inputs.scales(K, N, G, 7, "halfnormal", 0.01)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    runs = [(1, 1), (16, 2), (32, 2), (64, 2), (128, 2), (256, 2), (1, 3), (16, 3)]   # (M, forced path)
    xs = {M: inputs.activations(M, K, 70 + M) for M, _ in runs}
    assert w.check_device_status() == w.OK
    prev = w.set_wait_limit_ns(1)
    try:
        for M, path in runs:
            prev_path = w.force_path(path)
            try:
                for attempt in range(3):
                    w.gemm(to_dev(xs[M]), packed, sp, N, G)
                    torch.cuda.synchronize()
                    status = w.check_device_status()
                    if status == w.ERR_TIMEOUT:
                        break
                assert status == w.ERR_TIMEOUT, (M, path, status)
                assert w.check_device_status() == w.OK          # read once, then cleared
            finally:
                w.force_path(prev_path)
    finally:
        w.set_wait_limit_ns(prev)
    rs = np.random.default_rng(8)
    cols = np.sort(rs.choice(N, 192, replace=False))
    for M, path in runs:
        prev_path = w.force_path(path)
        try:
            y = w.gemm(to_dev(xs[M]), packed, sp, N, G)
            torch.cuda.synchronize()
        finally:
            w.force_path(prev_path)
        assert w.check_device_status() == w.OK
        rows = np.unique(rs.integers(0, M, size=6))
        y_ref, absum = oracle_mod.gemm_sample(xs[M], q, s, G, rows, cols)
        check_within(y.cpu().numpy()[np.ix_(rows, cols)], y_ref, absum, "M=%d path %d after timeouts" % (M, path))

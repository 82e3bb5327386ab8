"""The no-allocation entry point, for callers that may not allocate device memory
(plug-ins whose host framework owns all GPU memory, latency-critical loops that
cannot take cudaMalloc's device-wide synchronisation).

Its results are checked against the CPU oracle, within the same bound as every
other parity test, on two calls in a row (the second reuses the fixed scratch
array the first one left behind), and bit for bit against the regular entry
point. This file is collected last so that a run stopping at its first failure
has run every other test first; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from tests.parity import check_within
from weight_only_int4_02_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [
    (16, 4096, 4096),    # 16-row tensor-core tiles, every tile split across CTAs: the scratch is used
    (17, 4096, 4096),    # 32-row tiles with a 17-row tail, split tiles
    (3, 4096, 4096),     # three rows: the decode kernel, no scratch at all
    (1, 4096, 4096),     # one row: the decode kernel
])
def test_no_alloc_matches_the_oracle_on_two_calls(oracle_mod, M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_02_gb300 import w4a16
    G = 128
    q = inputs.codes(K, N, seed=21)
    s = inputs.scales(K, N, G, seed=21)
    packed, sp = w4a16.pack(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), G)
    for call, seed in enumerate((31, 32)):
        x = inputs.activations(M, K, seed=seed)
        xd = torch.from_numpy(x).cuda()
        y = w4a16.gemm_noalloc(xd, packed, sp, N, G)
        torch.cuda.synchronize()
        y_ref, absum = oracle_mod.gemm(x, q, s, G)
        check_within(y.cpu().numpy(), y_ref, absum, "no-alloc M=%d call %d" % (M, call + 1))
        assert torch.equal(y, w4a16.gemm(xd, packed, sp, N, G))
    assert w4a16.check_device_status() == w4a16.OK


def test_no_alloc_rejects_shapes_beyond_its_array():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_02_gb300 import w4a16
    M, N, K, G = 128, 22016, 4096, 128         # 152 CTAs of 128-row partials: about 20 MB of scratch
    packed, sp = w4a16.pack(torch.zeros((K, N), dtype=torch.uint8, device="cuda"),
                            torch.ones((K // G, N), dtype=torch.float16, device="cuda"), G)
    x = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    with pytest.raises(w4a16.W4A16Error) as e:
        w4a16.gemm_noalloc(x, packed, sp, N, G)
    assert e.value.status == w4a16.ERR_WORKSPACE

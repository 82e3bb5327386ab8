"""GPU parity of the fused epilogue y = act(x @ dequant(W) + bias) + residual
(w4a16_gemm_fused) against the oracle's GEMM followed by its FP64 epilogue.

Shapes cover the direct store of unsplit tiles and the split-K fix-up, 16- to
256-row tiles, ragged M/N/K, an in-place residual (residual is y), and a full-size
decode layer on sampled outputs."""
import numpy as np
import pytest

from tests.parity import check_within_fused
from tests.test_oracle import hand_inputs
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


def epilogue_inputs(M, N, seed):
    rng = np.random.default_rng(seed)
    bias = rng.standard_normal(N).astype(np.float16)
    resid = (rng.standard_normal((M, N)) * 0.5).astype(np.float16)
    return bias, resid


def run_case(w, oracle_mod, M, N, K, G, activation, use_bias, use_resid, in_place=False, seed=11):
    x, q, s = inputs.problem(M, K, N, G, seed)
    bias, resid = epilogue_inputs(M, N, seed + 1)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    b_d = to_dev(bias) if use_bias else None
    r_d = to_dev(resid) if use_resid else None
    if in_place:
        y = w.gemm_fused(to_dev(x), packed, sp, N, G, bias=b_d, residual=r_d, activation=activation, y=r_d)
        assert y.data_ptr() == r_d.data_ptr()
    else:
        y = w.gemm_fused(to_dev(x), packed, sp, N, G, bias=b_d, residual=r_d, activation=activation)
    torch.cuda.synchronize()
    z, absum = oracle_mod.gemm(x, q, s, G)
    y_ref = oracle_mod.epilogue(z, bias=bias if use_bias else None, residual=resid if use_resid else None,
                                activation=activation)
    b_abs = np.abs(bias.astype(np.float64))[None, :] if use_bias else 0.0
    r_abs = np.abs(resid.astype(np.float64)) if use_resid else 0.0
    check_within_fused(y.cpu().numpy(), y_ref, z, absum, b_abs, r_abs,
                       "M=%d N=%d K=%d %s bias=%d resid=%d" % (M, N, K, activation, use_bias, use_resid))


SHAPES = [
    (16, 32768, 1024, 128),   # split region first, then whole tiles (more tiles than SMs)
    (100, 40000, 512, 64),    # the same with 128-row tiles, ragged M
    (1, 256, 16384, 128),     # split-K, 16-row tile
    (3, 136, 200, 200),       # ragged, one group per column
    (17, 4096, 4000, 64),     # 32-row tile, ragged K
    (64, 512, 1024, 128),     # 64-row tile pair (cluster)
    (128, 1024, 2048, 32),    # 128-row tile pair, groups of 32
    (300, 264, 136, 32),      # 256-row tiles, two row tiles
]


@pytest.mark.parametrize("M,N,K,G", SHAPES)
@pytest.mark.parametrize("activation", ["none", "silu", "relu"])
def test_fused_parity(w, oracle_mod, M, N, K, G, activation):
    run_case(w, oracle_mod, M, N, K, G, activation, True, True)


@pytest.mark.parametrize("use_bias,use_resid", [(False, False), (True, False), (False, True)])
def test_fused_parts(w, oracle_mod, use_bias, use_resid):
    for (M, N, K, G) in [(1, 256, 16384, 128), (64, 512, 1024, 128)]:
        run_case(w, oracle_mod, M, N, K, G, "silu", use_bias, use_resid)


def test_fused_in_place_residual(w, oracle_mod):
    for (M, N, K, G) in [(1, 256, 16384, 128), (17, 4096, 4000, 64), (300, 264, 136, 32)]:
        run_case(w, oracle_mod, M, N, K, G, "silu", True, True, in_place=True)


def test_fused_without_epilogue_equals_plain_gemm(w):
    x, q, s = inputs.problem(16, 4096, 4096, 128, 5)
    packed, sp = w.pack(to_dev(q), to_dev(s), 128)
    a = w.gemm(to_dev(x), packed, sp, 4096, 128)
    b = w.gemm_fused(to_dev(x), packed, sp, 4096, 128)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_fused_hand_example_is_bit_exact(w):
    """1x8x8, G = K = 8, bias b[n] = n/2, ReLU: every value is exact in FP16."""
    x, q, s = hand_inputs(8)
    packed, sp = w.pack(to_dev(q), to_dev(s), 8)
    b = (np.arange(8) / 2.0).astype(np.float16)
    y = w.gemm_fused(to_dev(x), packed, sp, 8, 8, bias=to_dev(b), activation="relu")
    torch.cuda.synchronize()
    want = np.maximum(np.array([-4.125, -3.75, -4.875, -5.5, -3.125, -5.75, -7.875, 22.5]) + np.arange(8) / 2.0, 0.0)
    assert np.array_equal(y.cpu().numpy().astype(np.float64)[0], want)


def test_fused_full_size_decode_layer_sampled(w, oracle_mod):
    M, K, N, G = 16, 4096, 22016, 128
    x, q, s = inputs.problem(M, K, N, G, 21)
    bias, resid = epilogue_inputs(M, N, 22)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    y = w.gemm_fused(to_dev(x), packed, sp, N, G, bias=to_dev(bias), residual=to_dev(resid), activation="silu")
    torch.cuda.synchronize()
    rows = np.arange(M)
    cols = np.random.default_rng(0).choice(N, 256, replace=False)
    z, absum = oracle_mod.gemm_sample(x, q, s, G, rows, cols)
    y_ref = oracle_mod.epilogue(z, bias=bias, residual=resid, activation="silu", rows=rows, cols=cols)
    check_within_fused(y.cpu().numpy()[np.ix_(rows, cols)], y_ref, z, absum,
                       np.abs(bias.astype(np.float64))[cols][None, :], np.abs(resid.astype(np.float64))[np.ix_(rows, cols)],
                       "decode layer 16x4096x22016 silu")


def test_fused_rejects_bad_activation(w):
    x = torch.zeros((1, 64), dtype=torch.float16, device="cuda")
    packed, sp = w.pack(torch.full((64, 64), 8, dtype=torch.uint8, device="cuda"),
                        torch.ones((1, 64), dtype=torch.float16, device="cuda"), 64)
    y = torch.empty((1, 64), dtype=torch.float16, device="cuda")
    st = w.lib().w4a16_gemm_fused(w._ptr(x), w._ptr(packed), w._ptr(sp), w._ptr(y), 1, 64, 64, 64, None, None, 7, None, 0,
                                  w._stream(None))
    assert st == w.ERR_INVALID_ARG

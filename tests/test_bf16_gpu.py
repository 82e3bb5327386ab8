"""GPU parity of BF16 activations (w4a16_bf16_gemm: 4-bit codes, zero-point 8, X,
scales, bias, residual and Y in bfloat16) against the oracle's BF16 GEMM, with the
bound derived for BF16 rounding (tests/parity.py: 2^-7 of sum |x*w| + 2^-8 |y|).

Shapes cover every tile height, the direct store and the split-K fix-up, groups
of 32 and one group per column, ragged M/N/K, the fused epilogue and a full-size
decode layer on sampled outputs."""
import numpy as np
import pytest

from tests.parity import REL_OUT_BF16, REL_SUM_BF16, check_within, check_within_fused
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


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def to_bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_problem(M, N, K, G, seed):
    return inputs.activations_bf16(M, K, seed), inputs.codes(K, N, seed), inputs.scales_bf16(K, N, G, seed)


def y_values(y):
    return y.float().cpu().numpy().astype(np.float64)


SHAPES = [
    (1, 256, 16384, 128),     # split-K, 16-row tile
    (3, 136, 200, 200),       # ragged, one group per column
    (17, 4096, 4000, 64),     # 32-row tile, ragged K
    (64, 512, 1024, 128),     # 64-row tile pair (cluster)
    (128, 1024, 2048, 32),    # 128-row tile pair, groups of 32
    (300, 264, 136, 32),      # 256-row tiles, two row tiles
    (1024, 1024, 1024, 128),  # 256-row tiles, four row tiles
    (300, 20000, 264, 264),   # 256-row tiles, split region first, then whole tiles
]


def test_bf16_scales_pack_as_bits(w):
    K, N, G = 256, 200, 128
    s = inputs.scales_bf16(K, N, G, 5)
    _, sp = w.pack(to_dev(inputs.codes(K, N, 5)), to_dev_bf16(s), G)
    torch.cuda.synchronize()
    assert sp.dtype == torch.bfloat16
    got = to_bits(sp).reshape(2, 2, 128)   # [tile][group][column]
    for nt in range(2):
        cols = min(128, N - nt * 128)
        assert np.array_equal(got[nt, :, :cols], s[:, nt * 128: nt * 128 + cols])


@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_bf16_parity(w, oracle_mod, M, N, K, G):
    x, q, s = bf16_problem(M, N, K, G, 35)
    packed, sp = w.pack(to_dev(q), to_dev_bf16(s), G)
    y = w.bf16_gemm(to_dev_bf16(x), packed, sp, N, G)
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    y_ref, absum = oracle_mod.gemm_bf16(x, q, s, G)
    check_within(y_values(y), y_ref, absum, "BF16 M=%d N=%d K=%d G=%d" % (M, N, K, G),
                 rel_sum=REL_SUM_BF16, rel_out=REL_OUT_BF16)


@pytest.mark.parametrize("M,N,K,G", [(1, 256, 16384, 128), (64, 512, 1024, 128), (300, 264, 136, 32)])
def test_bf16_parity_with_fused_epilogue(w, oracle_mod, M, N, K, G):
    x, q, s = bf16_problem(M, N, K, G, 45)
    r = np.random.default_rng(46)
    bias = inputs.to_bf16_bits(r.standard_normal(N).astype(np.float32))
    resid = inputs.to_bf16_bits((r.standard_normal((M, N)) * 0.5).astype(np.float32))
    packed, sp = w.pack(to_dev(q), to_dev_bf16(s), G)
    y = w.bf16_gemm(to_dev_bf16(x), packed, sp, N, G, bias=to_dev_bf16(bias), residual=to_dev_bf16(resid),
                    activation="silu")
    torch.cuda.synchronize()
    z, absum = oracle_mod.gemm_bf16(x, q, s, G)
    y_ref = oracle_mod.epilogue(z, bias=bias, residual=resid, activation="silu", dtype="bf16")
    b = oracle_mod.bf16_to_double(bias)
    rr = oracle_mod.bf16_to_double(resid)
    check_within_fused(y_values(y), y_ref, z, absum, np.abs(b)[None, :], np.abs(rr),
                       "BF16 + SiLU M=%d N=%d K=%d" % (M, N, K), rel_sum=REL_SUM_BF16, rel_out=REL_OUT_BF16)


def test_bf16_full_size_decode_layer_sampled(w, oracle_mod):
    M, K, N, G = 16, 4096, 22016, 128
    x, q, s = bf16_problem(M, N, K, G, 95)
    packed, sp = w.pack(to_dev(q), to_dev_bf16(s), G)
    y = w.bf16_gemm(to_dev_bf16(x), packed, sp, N, G)
    torch.cuda.synchronize()
    rows = np.arange(M)
    cols = np.random.default_rng(4).choice(N, 256, replace=False)
    y_ref, absum = oracle_mod.gemm_sample_bf16(x, q, s, G, rows, cols)
    check_within(y_values(y)[np.ix_(rows, cols)], y_ref, absum, "BF16 16x4096x22016",
                 rel_sum=REL_SUM_BF16, rel_out=REL_OUT_BF16)


def test_bf16_codes_8_give_zero(w):
    M, N, K, G = 8, 256, 512, 128
    x = inputs.activations_bf16(M, K, 75)
    s = inputs.scales_bf16(K, N, G, 75)
    packed, sp = w.pack(torch.full((K, N), 8, dtype=torch.uint8, device="cuda"), to_dev_bf16(s), G)
    y = w.bf16_gemm(to_dev_bf16(x), packed, sp, N, G)
    torch.cuda.synchronize()
    assert not torch.any(y.float() != 0)

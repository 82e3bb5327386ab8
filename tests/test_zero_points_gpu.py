"""GPU parity of the per-group zero-point format, dequant(W) = (q - z[g][n]) * s[g][n]
(w4a16_pack_zeros, w4a16_gemm_zp), against the oracle with the same zero-points.

Shapes cover the direct store and the split-K fix-up, 16- to 256-row tiles, groups
of 32 (several groups in one pipeline stage) and one group per column, ragged
M/N/K, the fused epilogue, the extreme zero-points 0 and 15 against the extreme
codes, and a full-size decode layer on sampled outputs. With every zero-point 8 the
result must equal the symmetric kernel's bit for bit."""
import numpy as np
import pytest

from tests.parity import forced_path
from tests.parity import check_within, check_within_fused
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


def packed_problem(w, M, N, K, G, seed):
    x, q, s = inputs.problem(M, K, N, G, seed)
    z = inputs.zeros(K, N, G, seed)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    zp = w.pack_zeros(to_dev(z), K, G)
    return x, q, s, z, packed, sp, zp


@pytest.mark.parametrize("K,N,G", [(4096, 200, 128), (200, 136, 200), (4000, 4096, 64), (96, 8, 32)])
def test_pack_zeros_round_trips(w, oracle_mod, K, N, G):
    z = inputs.zeros(K, N, G, seed=3)
    zp = w.pack_zeros(to_dev(z), K, G)
    torch.cuda.synchronize()
    assert zp.numel() == w.zeros_bytes(K, N, G)
    z2, bad = oracle_mod.unpack_zeros(zp.cpu().numpy(), z.shape[0], N)
    assert bad == 0 and np.array_equal(z2, z)


SHAPES = [
    (1, 256, 16384, 128),     # split-K, 16-row tile
    (3, 136, 200, 200),       # ragged, one group per column
    (17, 4096, 4000, 64),     # 32-row tile, ragged K
    (64, 512, 1024, 128),     # 64-row tile pair (cluster)
    (128, 1024, 2048, 32),    # 128-row tile pair, groups of 32
    (300, 264, 136, 32),      # 256-row tiles, two row tiles
    (1024, 1024, 1024, 128),  # 256-row tiles, four row tiles
]


@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_zero_point_parity(w, oracle_mod, M, N, K, G):
    x, q, s, z, packed, sp, zp = packed_problem(w, M, N, K, G, 31)
    y = w.gemm_zp(to_dev(x), packed, sp, zp, N, G)
    torch.cuda.synchronize()
    y_ref, absum = oracle_mod.gemm(x, q, s, G, z=z)
    check_within(y.cpu().numpy(), y_ref, absum, "zero-points M=%d N=%d K=%d G=%d" % (M, N, K, G))


@pytest.mark.parametrize("M,N,K,G", [(1, 256, 16384, 128), (64, 512, 1024, 128), (300, 264, 136, 32)])
def test_zero_point_parity_with_fused_epilogue(w, oracle_mod, M, N, K, G):
    x, q, s, z, packed, sp, zp = packed_problem(w, M, N, K, G, 41)
    rng = np.random.default_rng(42)
    bias = rng.standard_normal(N).astype(np.float16)
    resid = (rng.standard_normal((M, N)) * 0.5).astype(np.float16)
    y = w.gemm_zp(to_dev(x), packed, sp, zp, N, G, bias=to_dev(bias), residual=to_dev(resid), activation="silu")
    torch.cuda.synchronize()
    zz, absum = oracle_mod.gemm(x, q, s, G, z=z)
    y_ref = oracle_mod.epilogue(zz, bias=bias, residual=resid, activation="silu")
    check_within_fused(y.cpu().numpy(), y_ref, zz, absum, np.abs(bias.astype(np.float64))[None, :],
                       np.abs(resid.astype(np.float64)), "zero-points + SiLU M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K,G", [(1, 4096, 4096, 128), (16, 4096, 4096, 128), (32, 4096, 11008, 128),
                                     (64, 512, 1024, 128), (128, 1024, 2048, 32), (300, 264, 136, 32)])
def test_zero_points_of_eight_equal_the_symmetric_kernel(w, M, N, K, G):
    """Zero-points all 8 through the zero-point kernel give the symmetric tensor-core
    kernel's results bit for bit (the symmetric format is held on the tensor-core
    path here: with M <= 4 the dispatcher would otherwise take the CUDA-core kernel,
    whose sums run in another order)."""
    x, q, s = inputs.problem(M, K, N, G, 51)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    zp = w.pack_zeros(torch.full(((K + G - 1) // G, N), 8, dtype=torch.uint8, device="cuda"), K, G)
    xd = to_dev(x)
    bias = to_dev(np.random.default_rng(52).standard_normal(N).astype(np.float16))
    with forced_path(w, 2):
        a = w.gemm(xd, packed, sp, N, G)
        c = w.gemm_fused(xd, packed, sp, N, G, bias=bias, activation="relu")
    b = w.gemm_zp(xd, packed, sp, zp, N, G)
    d = w.gemm_zp(xd, packed, sp, zp, N, G, bias=bias, activation="relu")
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(c, d)


def test_extreme_zero_points_and_codes(w, oracle_mod):
    """Codes and zero-points drawn from {0, 15} only: q - z spans -15 .. 15."""
    M, N, K, G = 16, 384, 1024, 64
    rng = np.random.default_rng(61)
    x = inputs.activations(M, K, 61)
    q = (rng.integers(0, 2, size=(K, N)) * 15).astype(np.uint8)
    z = (rng.integers(0, 2, size=(K // G, N)) * 15).astype(np.uint8)
    s = inputs.scales(K, N, G, 61)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    zp = w.pack_zeros(to_dev(z), K, G)
    y = w.gemm_zp(to_dev(x), packed, sp, zp, N, G)
    torch.cuda.synchronize()
    y_ref, absum = oracle_mod.gemm(x, q, s, G, z=z)
    check_within(y.cpu().numpy(), y_ref, absum, "extreme zero-points")


def test_codes_equal_to_zero_points_give_zero(w):
    M, N, K, G = 8, 256, 512, 128
    z = inputs.zeros(K, N, G, 71)
    q = np.repeat(z, G, axis=0)
    x = inputs.activations(M, K, 71)
    s = inputs.scales(K, N, G, 71)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    zp = w.pack_zeros(to_dev(z), K, G)
    y = w.gemm_zp(to_dev(x), packed, sp, zp, N, G)
    torch.cuda.synchronize()
    assert not torch.any(y.float() != 0)


def test_zero_point_full_size_decode_layer_sampled(w, oracle_mod):
    M, K, N, G = 16, 4096, 22016, 128
    x, q, s, z, packed, sp, zp = packed_problem(w, M, N, K, G, 81)
    y = w.gemm_zp(to_dev(x), packed, sp, zp, N, G)
    torch.cuda.synchronize()
    rows = np.arange(M)
    cols = np.random.default_rng(1).choice(N, 256, replace=False)
    y_ref, absum = oracle_mod.gemm_sample(x, q, s, G, rows, cols, z=z)
    check_within(y.cpu().numpy()[np.ix_(rows, cols)], y_ref, absum, "zero-points 16x4096x22016")


def test_null_zero_points_are_rejected(w):
    x, q, s = inputs.problem(4, 256, 256, 128, 91)
    packed, sp = w.pack(to_dev(q), to_dev(s), 128)
    with pytest.raises(w.W4A16Error):
        w.gemm_zp(to_dev(x), packed, sp, None, 256, 128)

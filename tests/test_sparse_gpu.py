"""GPU parity of 2:4 sparse 4-bit codes (w4a16_sp_pack, w4a16_sp_gemm): the packed
bytes equal the oracle's restatement of the sparse layout bit for bit, and the GEMM
matches the oracle's dense GEMM on the same (2:4 sparse) codes within the FP16 bound.

Shapes cover 16- to 128-row tiles (M > 128 runs several 128-row tiles), the direct
store and the split-K fix-up, groups of 32 and one group per column, ragged M/N/K,
the fused epilogue, and a full-size decode layer on sampled outputs."""
import numpy as np
import pytest

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


def sp_problem(M, N, K, G, seed):
    return inputs.activations(M, K, seed), inputs.codes_2to4(K, N, seed), inputs.scales(K, N, G, seed)


@pytest.mark.parametrize("K,N,G", [(256, 128, 128), (4000, 200, 64), (200, 136, 200), (1024, 4096, 32)])
def test_sp_pack_matches_the_oracle_bit_for_bit(w, oracle_mod, K, N, G):
    q = inputs.codes_2to4(K, N, 3)
    s = inputs.scales(K, N, G, 3)
    viol = torch.zeros(1, dtype=torch.int64, device="cuda")
    packed, sp = w.sp_pack(to_dev(q), to_dev(s), G, violations=viol)
    torch.cuda.synchronize()
    want, want_viol = oracle_mod.sp_pack(q)
    assert packed.numel() == w.sp_packed_bytes(K, N, G) == want.size
    assert np.array_equal(packed.cpu().numpy(), want)
    assert int(viol.item()) == want_viol == 0
    s2, bad = oracle_mod.unpack_scales(sp.cpu().numpy(), s.shape[0], N)
    assert bad == 0 and np.array_equal(s2, s.view(np.uint16))


def test_sp_pack_counts_groups_that_are_not_2to4(w, oracle_mod):
    K, N, G = 256, 128, 128
    q = inputs.codes_2to4(K, N, 4)
    q[0:4, 0] = [1, 2, 3, 4]
    q[8:11, 7] = [5, 6, 7]
    viol = torch.zeros(1, dtype=torch.int64, device="cuda")
    packed, _ = w.sp_pack(to_dev(q), to_dev(inputs.scales(K, N, G, 4)), G, violations=viol)
    torch.cuda.synchronize()
    want, want_viol = oracle_mod.sp_pack(q)
    assert int(viol.item()) == want_viol == 2
    assert np.array_equal(packed.cpu().numpy(), want)


SHAPES = [
    (1, 256, 16384, 128),     # split-K, 16-row tile
    (3, 136, 200, 200),       # ragged, one group per column
    (17, 4096, 4000, 64),     # 32-row tile, ragged K
    (64, 512, 1024, 128),     # 64-row tile pair (cluster)
    (128, 1024, 2048, 32),    # 128-row tile pair, groups of 32
    (300, 264, 136, 32),      # three 128-row tiles
    (1024, 1024, 1024, 128),  # eight 128-row tiles
]


@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_sp_parity(w, oracle_mod, M, N, K, G):
    x, q, s = sp_problem(M, N, K, G, 37)
    packed, sp = w.sp_pack(to_dev(q), to_dev(s), G)
    y = w.sp_gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    y_ref, absum = oracle_mod.gemm(x, q, s, G)
    check_within(y.cpu().numpy(), y_ref, absum, "2:4 sparse M=%d N=%d K=%d G=%d" % (M, N, K, G))


@pytest.mark.parametrize("M,N,K,G", [(1, 256, 16384, 128), (64, 512, 1024, 128), (300, 264, 136, 32)])
def test_sp_parity_with_fused_epilogue(w, oracle_mod, M, N, K, G):
    x, q, s = sp_problem(M, N, K, G, 47)
    rng = np.random.default_rng(48)
    bias = rng.standard_normal(N).astype(np.float16)
    resid = (rng.standard_normal((M, N)) * 0.5).astype(np.float16)
    packed, sp = w.sp_pack(to_dev(q), to_dev(s), G)
    y = w.sp_gemm(to_dev(x), packed, sp, N, G, bias=to_dev(bias), residual=to_dev(resid), activation="silu")
    torch.cuda.synchronize()
    z, absum = oracle_mod.gemm(x, q, s, G)
    y_ref = oracle_mod.epilogue(z, bias=bias, residual=resid, activation="silu")
    check_within_fused(y.cpu().numpy(), y_ref, z, absum, np.abs(bias.astype(np.float64))[None, :],
                       np.abs(resid.astype(np.float64)), "2:4 sparse + SiLU M=%d N=%d K=%d" % (M, N, K))


def test_sp_and_dense_kernels_agree_on_2to4_codes(w):
    """The same 2:4 codes through the dense and the sparse kernel: the products are
    the same, only the order of summation differs."""
    M, N, K, G = 16, 4096, 4096, 128
    x, q, s = sp_problem(M, N, K, G, 57)
    xd = to_dev(x)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    dense = w.gemm(xd, packed, sp, N, G).float()
    spk, ssp = w.sp_pack(to_dev(q), to_dev(s), G)
    sparse = w.sp_gemm(xd, spk, ssp, N, G).float()
    torch.cuda.synchronize()
    tol = 2.0 ** -9 * dense.abs() + 1e-2
    assert bool(((sparse - dense).abs() <= tol).all())


def test_sp_full_size_decode_layer_sampled(w, oracle_mod):
    M, K, N, G = 16, 4096, 22016, 128
    x, q, s = sp_problem(M, N, K, G, 97)
    packed, sp = w.sp_pack(to_dev(q), to_dev(s), G)
    y = w.sp_gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    rows = np.arange(M)
    cols = np.random.default_rng(5).choice(N, 256, replace=False)
    y_ref, absum = oracle_mod.gemm_sample(x, q, s, G, rows, cols)
    check_within(y.cpu().numpy()[np.ix_(rows, cols)], y_ref, absum, "2:4 sparse 16x4096x22016")

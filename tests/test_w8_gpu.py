"""GPU parity of the W8A16 format, dequant(W) = (q - 128) * s with 8-bit codes
(w4a16_w8_pack, w4a16_w8_gemm), against the oracle's 8-bit GEMM.

Shapes cover every tile height (16 to 256 rows of X, 128-value stages), the direct
store and the split-K fix-up, groups of 32 and one group per column, ragged
M/N/K, the fused epilogue, the extreme codes 0 and 255, a caller workspace sized
by w4a16_workspace_bytes, and a full-size decode layer on sampled outputs."""
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


def codes8(K, N, seed):
    return inputs.rng(seed, inputs.CODE_STREAM).integers(0, 256, size=(K, N), dtype=np.uint8)


def problem8(M, N, K, G, seed):
    x = inputs.activations(M, K, seed)
    q = codes8(K, N, seed)
    # 8-bit codes span 16x the 4-bit range: scales 16x smaller keep |w| alike
    s = inputs.scales(K, N, G, seed, mult=0.02 / 16)
    return x, q, s


@pytest.mark.parametrize("K,N,G", [(4096, 200, 128), (200, 136, 200), (4000, 4096, 64), (8, 8, 8)])
def test_w8_pack_round_trips(w, oracle_mod, K, N, G):
    q = codes8(K, N, 3)
    s = inputs.scales(K, N, G, 3)
    packed, sp = w.w8_pack(to_dev(q), to_dev(s), G)
    torch.cuda.synchronize()
    assert packed.numel() == w.w8_packed_bytes(K, N, G) == oracle_mod.packed_bytes_w8(K, N)
    q2, bad = oracle_mod.unpack_w8(packed.cpu().numpy(), K, N)
    assert bad == 0 and np.array_equal(q2, q)
    s2, bad = oracle_mod.unpack_scales(sp.cpu().numpy(), s.shape[0], N)
    assert bad == 0 and np.array_equal(s2, s.view(np.uint16))


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
def test_w8_parity(w, oracle_mod, M, N, K, G):
    x, q, s = problem8(M, N, K, G, 33)
    packed, sp = w.w8_pack(to_dev(q), to_dev(s), G)
    y = w.w8_gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    y_ref, absum = oracle_mod.gemm_w8(x, q, s, G)
    check_within(y.cpu().numpy(), y_ref, absum, "W8 M=%d N=%d K=%d G=%d" % (M, N, K, G))


@pytest.mark.parametrize("M,N,K,G", [(1, 256, 16384, 128), (64, 512, 1024, 128), (300, 264, 136, 32)])
def test_w8_parity_with_fused_epilogue(w, oracle_mod, M, N, K, G):
    x, q, s = problem8(M, N, K, G, 43)
    rng = np.random.default_rng(44)
    bias = rng.standard_normal(N).astype(np.float16)
    resid = (rng.standard_normal((M, N)) * 0.5).astype(np.float16)
    packed, sp = w.w8_pack(to_dev(q), to_dev(s), G)
    y = w.w8_gemm(to_dev(x), packed, sp, N, G, bias=to_dev(bias), residual=to_dev(resid), activation="silu")
    torch.cuda.synchronize()
    z, absum = oracle_mod.gemm_w8(x, q, s, G)
    y_ref = oracle_mod.epilogue(z, bias=bias, residual=resid, activation="silu")
    check_within_fused(y.cpu().numpy(), y_ref, z, absum, np.abs(bias.astype(np.float64))[None, :],
                       np.abs(resid.astype(np.float64)), "W8 + SiLU M=%d N=%d K=%d" % (M, N, K))


def test_w8_extreme_codes(w, oracle_mod):
    M, N, K, G = 16, 384, 1024, 64
    x = inputs.activations(M, K, 63)
    q = (np.random.default_rng(63).integers(0, 2, size=(K, N)) * 255).astype(np.uint8)
    s = inputs.scales(K, N, G, 63, mult=0.02 / 16)
    packed, sp = w.w8_pack(to_dev(q), to_dev(s), G)
    y = w.w8_gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    y_ref, absum = oracle_mod.gemm_w8(x, q, s, G)
    check_within(y.cpu().numpy(), y_ref, absum, "W8 codes 0 / 255")


def test_w8_codes_128_give_zero(w):
    M, N, K, G = 8, 256, 512, 128
    x = inputs.activations(M, K, 73)
    s = inputs.scales(K, N, G, 73)
    packed, sp = w.w8_pack(torch.full((K, N), 128, dtype=torch.uint8, device="cuda"), to_dev(s), G)
    y = w.w8_gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    assert not torch.any(y.float() != 0)


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (32, 4096, 11008), (256, 5120, 5120)])
def test_w8_with_caller_workspace(w, oracle_mod, M, N, K):
    G = 128
    x, q, s = problem8(M, N, K, G, 83)
    packed, sp = w.w8_pack(to_dev(q), to_dev(s), G)
    ws = torch.zeros(w.workspace_bytes(M, N, K, G), dtype=torch.uint8, device="cuda")
    y = w.w8_gemm(to_dev(x), packed, sp, N, G, workspace=ws)
    y2 = w.w8_gemm(to_dev(x), packed, sp, N, G, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)   # the fix-up is deterministic and the workspace self-resetting
    rows = np.arange(M)
    cols = np.random.default_rng(2).choice(N, 128, replace=False)
    y_ref, absum = oracle_mod.gemm_sample_w8(x, q, s, G, rows, cols)
    check_within(y.cpu().numpy()[np.ix_(rows, cols)], y_ref, absum, "W8 caller workspace %dx%dx%d" % (M, N, K))


def test_w8_full_size_decode_layer_sampled(w, oracle_mod):
    M, K, N, G = 16, 4096, 22016, 128
    x, q, s = problem8(M, N, K, G, 93)
    packed, sp = w.w8_pack(to_dev(q), to_dev(s), G)
    y = w.w8_gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    rows = np.arange(M)
    cols = np.random.default_rng(3).choice(N, 256, replace=False)
    y_ref, absum = oracle_mod.gemm_sample_w8(x, q, s, G, rows, cols)
    check_within(y.cpu().numpy()[np.ix_(rows, cols)], y_ref, absum, "W8 16x4096x22016")

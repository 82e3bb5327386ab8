"""GPU parity of row-strided activations, outputs and residuals (w4a16_gemm_strided)
against the CPU oracle, on every kernel: the decode kernel (up to sixteen rows of X),
the tensor-core kernel (every tile height) and the CUDA-core kernel (forced).

X is the leading K columns of a wider tensor, Y a column slice of a wider buffer
whose other columns must stay untouched, the residual a slice of a third buffer; the
oracle sees the same values densely. Also: a decode-layer chain that reads the
leading columns of each previous output in place, equal bit for bit to the same chain
on dense copies.
"""
import numpy as np
import pytest

from tests.parity import check_within, check_within_fused
from tests.parity import forced_path as forced
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


CASES = [
    # (M, N, K, G, path, extra columns of X, of Y, of the residual)
    (1, 4096, 4096, 128, 3, 8192, 64, 24),
    (5, 1024, 2048, 64, 3, 40, 8, 8),
    (16, 768, 1024, 128, 3, 1024, 16, 0),
    (2, 4096, 4000, 4000, 3, 96, 24, 8),
    (16, 4096, 4096, 128, 2, 8192, 64, 24),
    (40, 1024, 2048, 32, 2, 8, 8, 16),
    (300, 1032, 520, 520, 2, 56, 8, 8),
    (3, 4104, 1000, 1000, 2, 24, 16, 8),
    # Y and residual rows that are not 16-byte aligned (row strides not a multiple of 8):
    # the tensor-core kernel's unsplit tiles then store and read element by element
    (300, 1032, 520, 520, 2, 56, 3, 5),
    (3, 4104, 1000, 1000, 2, 24, 1, 3),
    (128, 1024, 512, 128, 2, 8, 5, 7),
    (2, 1024, 2048, 128, 1, 64, 8, 8),
    (4, 264, 520, 32, 1, 8, 8, 8),
]


@pytest.mark.parametrize("M,N,K,G,path,ex_x,ex_y,ex_r", CASES)
def test_strided_against_the_oracle(w, oracle_mod, M, N, K, G, path, ex_x, ex_y, ex_r):
    x, q, s = inputs.problem(M, K, N, G, seed=M + K + path, scale_kind="halfnormal")
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    rng = np.random.default_rng(M + N)
    x_wide = rng.standard_normal((M, K + ex_x)).astype(np.float16)
    x_wide[:, :K] = x
    bias = rng.standard_normal(N).astype(np.float16)
    resid_wide = rng.standard_normal((M, N + ex_r)).astype(np.float16)
    y_wide = torch.full((M, N + ex_y), 7.0, dtype=torch.float16, device="cuda")
    xd = to_dev(x_wide)[:, :K]
    rd = to_dev(resid_wide)[:, :N]
    z, absum = oracle_mod.gemm(x, q, s, G)
    with forced(w, path):
        assert w.plan(M, N, K, G)[0] == path
        y = w.gemm_strided(xd, packed, sp, N, G, y=y_wide[:, :N])
        torch.cuda.synchronize()
        check_within(y.cpu().numpy(), z, absum, "strided path %d M=%d N=%d K=%d" % (path, M, N, K))
        y2 = w.gemm_strided(xd, packed, sp, N, G, bias=to_dev(bias), residual=rd, activation="silu",
                            y=y_wide[:, :N])
        torch.cuda.synchronize()
    resid = resid_wide[:, :N]
    ref = oracle_mod.epilogue(z, bias=bias, residual=np.ascontiguousarray(resid), activation="silu")
    check_within_fused(y2.cpu().numpy(), ref, z, absum, np.abs(bias.astype(np.float64)),
                       np.abs(resid.astype(np.float64)), "strided fused path %d M=%d" % (path, M))
    if ex_y:
        assert torch.all(y_wide[:, N:] == 7.0), "columns outside the slice of Y were written"
    assert w.check_device_status() == w.OK


@pytest.mark.parametrize("M", [1, 8, 16])
def test_chain_reading_leading_columns_in_place(w, M):
    """QKV -> O (+ the layer input) -> gate/up (SiLU) -> down (+ the O output), each GEMM
    reading the leading columns of the previous output in place: equal bit for bit to the
    same chain on dense copies of those columns."""
    G = 128
    dims = [(4096, 12288), (4096, 4096), (4096, 22016), (11008, 4096)]
    layers = []
    for i, (K, N) in enumerate(dims):
        q, s = inputs.codes(K, N, 70 + i), inputs.scales(K, N, G, 70 + i, "halfnormal", 0.01)
        layers.append(w.pack(to_dev(q), to_dev(s), G))
    x = to_dev(inputs.activations(M, 4096, 9))
    qkv = w.gemm(x, *layers[0], 12288, G)
    o = w.gemm_strided(qkv[:, :4096], *layers[1], 4096, G, residual=x)
    gu = w.gemm_strided(o, *layers[2], 22016, G, activation="silu")
    out = w.gemm_strided(gu[:, :11008], *layers[3], 4096, G, residual=o)
    o_ref = w.gemm_fused(qkv[:, :4096].contiguous(), *layers[1], 4096, G, residual=x.clone())
    gu_ref = w.gemm_fused(o_ref, *layers[2], 22016, G, activation="silu")
    out_ref = w.gemm_fused(gu_ref[:, :11008].contiguous(), *layers[3], 4096, G, residual=o_ref.clone())
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(gu, gu_ref) and torch.equal(out, out_ref)

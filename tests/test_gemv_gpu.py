"""GPU parity of the CUDA-core kernel for one to four rows of X (path 1) against the
CPU oracle, beside the tensor-core kernel (path 2) forced on the same inputs.

The dispatcher does not pick path 1 by itself (the decode kernel measured faster on
every decode layer); here both paths are forced in turn
on the same shapes, each against the oracle: small and ragged shapes spanning several column
blocks of both widths (16, 32), the edge sweep (group = K and group 32, N = 256
with K = 16384, K = 4000 and 4040), and the four full-size decode layers at
M = 1 .. 4 compared element by element. Also: the fused epilogue, bit-identical
repeats, chained launches that read the previous output, and a GEMM issued right
after its repack with no synchronisation in between.
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


@pytest.fixture
def w1(w):
    """The library with the CUDA-core kernel forced wherever it serves (M <= 4)."""
    prev = w.force_path(1)
    yield w
    w.force_path(prev)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


SHAPES = [
    # (M, N, K, G, scale kind): column blocks of 16 (N < 4864) and 32,
    # ragged N (not a multiple of the block), K not a multiple of 32, one group
    (1, 4096, 4096, 128, "halfnormal"),
    (2, 4096, 4096, 128, "halfnormal"),
    (3, 4096, 4096, 128, "halfnormal"),
    (4, 4096, 4096, 128, "halfnormal"),
    (1, 8192, 4096, 64, "halfnormal"),
    (2, 12288, 4096, 128, "halfnormal"),
    (4, 22016, 4096, 128, "loguniform"),
    (1, 8, 8, 8, "halfnormal"),
    (3, 136, 200, 200, "halfnormal"),
    (2, 264, 520, 32, "loguniform"),
    (1, 1032, 4040, 128, "halfnormal"),
    (4, 4104, 1000, 1000, "loguniform"),
    (3, 256, 16384, 128, "loguniform"),
    (1, 4096, 4000, 4000, "loguniform"),
    (4, 9736, 2056, 32, "halfnormal"),
]


@pytest.mark.parametrize("M,N,K,G,kind", SHAPES)
def test_both_paths_against_the_oracle(w, oracle_mod, M, N, K, G, kind):
    x, q, s = inputs.problem(M, K, N, G, seed=M * 11 + K, scale_kind=kind)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    y_ref, absum = oracle_mod.gemm(x, q, s, G)
    xd = to_dev(x)
    for path in (1, 2):
        with forced(w, path):
            assert w.plan(M, N, K, G)[0] == path
            y = w.gemm(xd, packed, sp, N, G)
        torch.cuda.synchronize()
        check_within(y.cpu().numpy(), y_ref, absum, "path %d M=%d N=%d K=%d G=%d" % (path, M, N, K, G))


def test_full_size_decode_layers_elementwise(w1, oracle_mod):
    w = w1
    """The four Llama-2-7B-like decode layers at M = 1, 2, 3, 4, every element."""
    G = 128
    for (K, N) in inputs.LLAMA2_7B_LAYERS:
        q = inputs.codes(K, N, 0)
        s = inputs.scales(K, N, G, 0)
        packed, sp = w.pack(to_dev(q), to_dev(s), G)
        for M in (1, 2, 3, 4):
            x = inputs.activations(M, K, M)
            y = w.gemm(to_dev(x), packed, sp, N, G)
            y_ref, absum = oracle_mod.gemm(x, q, s, G)
            check_within(y.cpu().numpy(), y_ref, absum, "decode M=%d K=%d N=%d" % (M, K, N))
        del packed, sp


def test_edge_sweep(w1, oracle_mod):
    w = w1
    for M in (1, 3):
        for (N, K, G) in [(4096, 4096, 4096), (4096, 4096, 32), (256, 16384, 128), (4096, 4000, 128),
                          (4096, 4040, 128)]:
            x, q, s = inputs.problem(M, K, N, G, seed=M + K, scale_kind="loguniform")
            packed, sp = w.pack(to_dev(q), to_dev(s), G)
            y = w.gemm(to_dev(x), packed, sp, N, G)
            y_ref, absum = oracle_mod.gemm(x, q, s, G)
            check_within(y.cpu().numpy(), y_ref, absum, "edge M=%d N=%d K=%d G=%d" % (M, N, K, G))


def test_subnormal_scales_and_invariants(w1, oracle_mod):
    w = w1
    M, N, K, G = 3, 256, 512, 128
    x, q, _ = inputs.problem(M, K, N, G, seed=4)
    s = (np.random.default_rng(0).integers(1, 1024, size=(K // G, N)) * 2.0 ** -24).astype(np.float16)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    y = w.gemm(to_dev(x), packed, sp, N, G).cpu().numpy()
    check_within(y, *oracle_mod.gemm(x, q, s, G), "subnormal scales")
    # zero scales and all codes 8 give zero; one nonzero code gives one scaled column
    y0 = w.gemm(to_dev(x), *w.pack(to_dev(q), to_dev(np.zeros_like(s)), G), N, G).cpu().numpy()
    assert np.all(y0 == 0)
    q1 = np.full_like(q, 8)
    q1[300, 77] = 1
    s1 = np.ones_like(s)
    y1 = w.gemm(to_dev(x), *w.pack(to_dev(q1), to_dev(s1), G), N, G).cpu().numpy()
    assert np.all(np.delete(y1, 77, axis=1) == 0)
    assert np.array_equal(y1[:, 77], (x[:, 300].astype(np.float64) * -7).astype(np.float16))


def test_fused_epilogue(w1, oracle_mod):
    w = w1
    M, N, K, G = 4, 4096, 2048, 128
    x, q, s = inputs.problem(M, K, N, G, seed=12)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    rng = np.random.default_rng(3)
    bias = rng.standard_normal(N).astype(np.float16)
    resid = rng.standard_normal((M, N)).astype(np.float16)
    z, absum = oracle_mod.gemm(x, q, s, G)
    for act in ("none", "silu", "relu"):
        y = w.gemm_fused(to_dev(x), packed, sp, N, G, bias=to_dev(bias), activation=act)
        ref = oracle_mod.epilogue(z, bias=bias, activation=act)
        check_within_fused(y.cpu().numpy(), ref, z, absum, np.abs(bias.astype(np.float64)), 0.0, "bias+" + act)
    r = to_dev(resid)
    y = w.gemm_fused(to_dev(x), packed, sp, N, G, residual=r, y=r)   # in place
    ref = oracle_mod.epilogue(z, residual=resid)
    check_within_fused(y.cpu().numpy(), ref, z, absum, 0.0, np.abs(resid.astype(np.float64)), "residual in place")


def test_deterministic(w1):
    w = w1
    for (M, N, K) in ((1, 4096, 11008), (4, 22016, 4096)):
        x, q, s = inputs.problem(M, K, N, 128, seed=7)
        packed, sp = w.pack(to_dev(q), to_dev(s), 128)
        xd = to_dev(x)
        ys = [w.gemm(xd, packed, sp, N, 128).cpu().numpy().view(np.uint16) for _ in range(3)]
        assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


def test_chained_launches_read_the_previous_output(w1):
    w = w1
    """Each launch may start before the previous one ends but reads X only after it
    completes: a chain of M = 1 GEMMs launched back to back, plain and from a CUDA
    Graph, equals the chain with a synchronisation after every launch."""
    G = 128
    dims = [(4096, 12288), (12288, 4096), (4096, 22016), (22016, 4096)]
    layers = []
    for i, (K, N) in enumerate(dims):
        q, s = inputs.codes(K, N, 60 + i), inputs.scales(K, N, G, 60 + i, "halfnormal", 0.01)
        layers.append((w.pack(to_dev(q), to_dev(s), G), N))
    x = to_dev(inputs.activations(1, 4096, 5))

    def chain(sync):
        h, outs = x, []
        for (packed, sp), N in layers:
            h = w.gemm(h, packed, sp, N, G)
            outs.append(h)
            if sync:
                torch.cuda.synchronize()
        return outs

    ref = [o.clone() for o in chain(True)]
    got = chain(False)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        outs = chain(False)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, ref):
        assert torch.equal(a, b)


def test_gemm_right_after_its_repack(w, oracle_mod):
    """A GEMM enqueued directly after the repack of its weights, with no
    synchronisation in between, reads the repacked weights (each repack ends with a
    kernel that writes nothing, which is all the GEMM may overlap). All three paths;
    the weight buffers are reused with new codes on every round."""
    N, K, G = 4096, 4096, 128
    packed = torch.empty(w.packed_words(K, N, G), dtype=torch.int32, device="cuda")
    sp = torch.empty(w.scales_elems(K, N, G), dtype=torch.float16, device="cuda")
    for rnd, (M, path) in enumerate(((1, 1), (4, 1), (16, 2), (1, 2), (1, 3), (8, 3), (16, 3))):
        x, q, s = inputs.problem(M, K, N, G, seed=90 + rnd)
        qd, sd, xd = to_dev(q), to_dev(s), to_dev(x)
        torch.cuda.synchronize()
        with forced(w, path):
            w.pack(qd, sd, G, out=(packed, sp))
            y = w.gemm(xd, packed, sp, N, G)
        torch.cuda.synchronize()
        check_within(y.cpu().numpy(), *oracle_mod.gemm(x, q, s, G), "round %d (M=%d, path %d)" % (rnd, M, path))

"""GPU parity of the decode kernel (path 3: register-level unpack feeding warp-level
MMAs, one to sixteen rows of X) against the CPU oracle.

The dispatcher picks it by itself for up to eight rows of X when K is a multiple of
32 (sixteen on layers of at most 4096 x 4096); here it is also forced for nine to
sixteen rows. Covered: small and ragged
shapes spanning several column blocks of every width (16, 32, 48, 64, 80) and every group
size (32, 64, 128, K, K not a power of two), beside the tensor-core kernel forced on
the same inputs; the four full-size decode layers at M = 1, 3, 8 and 16 compared
element by element; the 18432 x 73728 layer on sampled columns; the edge sweep;
subnormal scales and exact invariants; the fused epilogue; bit-identical repeats;
chained launches that read the previous output.
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
def w3(w):
    """The library with the decode kernel forced wherever it serves (M <= 16, K a multiple of 32)."""
    prev = w.force_path(3)
    yield w
    w.force_path(prev)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


SHAPES = [
    # (M, N, K, G, scale kind): blocks of 16 columns (N below 64 blocks of 64 per SM)
    # and of 64, ragged N, every group size, one group of K not a power of two
    (1, 4096, 4096, 128, "halfnormal"),
    (2, 4096, 4096, 128, "halfnormal"),
    (5, 4096, 4096, 64, "halfnormal"),
    (8, 4096, 4096, 128, "loguniform"),
    (9, 1024, 2048, 64, "halfnormal"),
    (16, 4096, 4096, 128, "halfnormal"),
    (1, 12288, 4096, 128, "halfnormal"),
    (7, 12288, 4096, 32, "loguniform"),
    (3, 22016, 4096, 128, "halfnormal"),
    (13, 4104, 1024, 128, "halfnormal"),
    (2, 264, 544, 32, "loguniform"),
    (1, 8, 32, 32, "halfnormal"),
    (4, 136, 224, 224, "halfnormal"),
    (16, 768, 1024, 1024, "loguniform"),
    (1, 4096, 4000, 4000, "loguniform"),
    (6, 9736, 2048, 32, "halfnormal"),
    (11, 256, 16384, 128, "loguniform"),
    # blocks of 48 and 80 columns (boxes of 16 columns, blocks straddling two 128-column
    # tiles, ragged last blocks past N) and of 32, with groups of 32, 64, 128 and K
    (1, 20008, 2048, 64, "halfnormal"),
    (8, 19464, 1024, 128, "loguniform"),
    (3, 12296, 1024, 32, "halfnormal"),
    (5, 24320, 512, 512, "loguniform"),
    (2, 7304, 2048, 128, "halfnormal"),
]


@pytest.mark.parametrize("M,N,K,G,kind", SHAPES)
def test_decode_and_tensor_core_against_the_oracle(w, oracle_mod, M, N, K, G, kind):
    x, q, s = inputs.problem(M, K, N, G, seed=M * 13 + K, scale_kind=kind)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    y_ref, absum = oracle_mod.gemm(x, q, s, G)
    xd = to_dev(x)
    for path in (3, 2):
        with forced(w, path):
            assert w.plan(M, N, K, G)[0] == path
            y = w.gemm(xd, packed, sp, N, G)
        torch.cuda.synchronize()
        check_within(y.cpu().numpy(), y_ref, absum, "path %d M=%d N=%d K=%d G=%d" % (path, M, N, K, G))


def random_shapes(n, seed):
    """Seeded random shapes: 1..16 rows of X, N a multiple of 8 up to 16000, K a
    multiple of 32 up to 4000, groups of 32, 64, 128 or K; every block width, ragged
    last blocks and stages, odd and even rings."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.integers(1, 17))
        N = 8 * int(rng.integers(1, 2001))
        K = 32 * int(rng.integers(1, 126))
        G = int(rng.choice([32, 64, 128, K]))
        out.append((M, N, K, G))
    return out


@pytest.mark.parametrize("M,N,K,G", random_shapes(24, 77))
def test_random_shapes_against_the_oracle(w3, oracle_mod, M, N, K, G):
    w = w3
    x, q, s = inputs.problem(M, K, N, G, seed=M + N + K, scale_kind="loguniform")
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    assert w.plan(M, N, K, G)[0] == 3
    y = w.gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    check_within(y.cpu().numpy(), *oracle_mod.gemm(x, q, s, G), "random M=%d N=%d K=%d G=%d" % (M, N, K, G))
    assert w.check_device_status() == w.OK


def test_full_size_decode_layers_elementwise(w, oracle_mod):
    """The four Llama-2-7B-like decode layers at M = 1, 3, 8 (the dispatcher's own
    choice) and 16 (forced), every element."""
    G = 128
    for (K, N) in inputs.LLAMA2_7B_LAYERS:
        q = inputs.codes(K, N, 0)
        s = inputs.scales(K, N, G, 0)
        packed, sp = w.pack(to_dev(q), to_dev(s), G)
        for M in (1, 3, 8, 16):
            x = inputs.activations(M, K, M)
            with forced(w, 3 if M > 8 else 0):
                assert w.plan(M, N, K, G)[0] == 3
                y = w.gemm(to_dev(x), packed, sp, N, G)
            y_ref, absum = oracle_mod.gemm(x, q, s, G)
            check_within(y.cpu().numpy(), y_ref, absum, "decode M=%d K=%d N=%d" % (M, K, N))
        del packed, sp


def test_large_layer_sampled(w, oracle_mod):
    """The 18432 x 73728 layer (blocks of 64 columns, 1152 CTAs) at M = 1 and 8, every
    row on 512 sampled columns."""
    K, N, G = 18432, 73728, 128
    q = inputs.codes(K, N, 3)
    s = inputs.scales(K, N, G, 3)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    cols = np.sort(np.random.default_rng(5).choice(N, 512, replace=False))
    for M in (1, 8):
        x = inputs.activations(M, K, 40 + M)
        assert w.plan(M, N, K, G)[0] == 3
        y = w.gemm(to_dev(x), packed, sp, N, G).cpu().numpy()
        y_ref, absum = oracle_mod.gemm_sample(x, q, s, G, np.arange(M), cols)
        check_within(y[:, cols], y_ref, absum, "large layer M=%d" % M)


def test_edge_sweep(w3, oracle_mod):
    w = w3
    for M in (1, 3, 9, 16):
        for (N, K, G) in [(4096, 4096, 4096), (4096, 4096, 32), (256, 16384, 128), (4096, 4000, 128),
                          (4096, 4000, 4000)]:
            x, q, s = inputs.problem(M, K, N, G, seed=M + K + G, scale_kind="loguniform")
            packed, sp = w.pack(to_dev(q), to_dev(s), G)
            assert w.plan(M, N, K, G)[0] == 3
            y = w.gemm(to_dev(x), packed, sp, N, G)
            y_ref, absum = oracle_mod.gemm(x, q, s, G)
            check_within(y.cpu().numpy(), y_ref, absum, "edge M=%d N=%d K=%d G=%d" % (M, N, K, G))


def test_subnormal_scales_and_invariants(w3, oracle_mod):
    w = w3
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


def test_fused_epilogue(w3, oracle_mod):
    w = w3
    for (M, N, K, G) in ((4, 4096, 2048, 128), (12, 12288, 1024, 64)):
        x, q, s = inputs.problem(M, K, N, G, seed=12 + M)
        packed, sp = w.pack(to_dev(q), to_dev(s), G)
        rng = np.random.default_rng(3)
        bias = rng.standard_normal(N).astype(np.float16)
        resid = rng.standard_normal((M, N)).astype(np.float16)
        z, absum = oracle_mod.gemm(x, q, s, G)
        for act in ("none", "silu", "relu"):
            y = w.gemm_fused(to_dev(x), packed, sp, N, G, bias=to_dev(bias), activation=act)
            ref = oracle_mod.epilogue(z, bias=bias, activation=act)
            check_within_fused(y.cpu().numpy(), ref, z, absum, np.abs(bias.astype(np.float64)), 0.0,
                               "M=%d bias+%s" % (M, act))
        r = to_dev(resid)
        y = w.gemm_fused(to_dev(x), packed, sp, N, G, residual=r, y=r)   # in place
        ref = oracle_mod.epilogue(z, residual=resid)
        check_within_fused(y.cpu().numpy(), ref, z, absum, 0.0, np.abs(resid.astype(np.float64)),
                           "M=%d residual in place" % M)


def test_deterministic(w3):
    w = w3
    for (M, N, K) in ((1, 4096, 11008), (8, 22016, 4096), (16, 4096, 4096)):
        x, q, s = inputs.problem(M, K, N, 128, seed=7)
        packed, sp = w.pack(to_dev(q), to_dev(s), 128)
        xd = to_dev(x)
        ys = [w.gemm(xd, packed, sp, N, 128).cpu().numpy().view(np.uint16) for _ in range(3)]
        assert np.array_equal(ys[0], ys[1]) and np.array_equal(ys[0], ys[2])


@pytest.mark.parametrize("M", [1, 8])
def test_chained_launches_read_the_previous_output(w, M):
    """Each launch may start before the previous one ends (its weight copies do) but
    reads X only after it completes: a chain of GEMMs launched back to back, plain
    and from a CUDA Graph, equals the chain with a synchronisation after every launch."""
    G = 128
    dims = [(4096, 12288), (12288, 4096), (4096, 22016), (22016, 4096)]
    layers = []
    for i, (K, N) in enumerate(dims):
        q, s = inputs.codes(K, N, 60 + i), inputs.scales(K, N, G, 60 + i, "halfnormal", 0.01)
        layers.append((w.pack(to_dev(q), to_dev(s), G), N))
    x = to_dev(inputs.activations(M, 4096, 5))
    assert w.plan(M, 12288, 4096, G)[0] == 3

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

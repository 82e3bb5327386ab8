"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small and ragged shapes are compared element by element; the full-size
workloads (in the launch configuration the benchmark times) on sampled
elements, which the oracle evaluates one by one. The acceptance bound is
|y - y_ref| <= 1e-3 * sum_k |x w| + 2^-10 |y_ref| per element.
"""
import numpy as np
import pytest

from tests.parity import check_within, forced_path
from tests.test_oracle import hand_inputs, read_golden
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


def run_gpu(w, x, q, s, G, N=None):
    K, N = q.shape
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    y = w.gemm(to_dev(x), packed, sp, N, G)
    torch.cuda.synchronize()
    return y.cpu().numpy(), packed, sp


def test_pack_round_trip(w, oracle_mod):
    for (K, N, G) in [(64, 128, 64), (200, 136, 200), (8, 8, 8), (4040, 256, 128), (4096, 384, 32), (520, 264, 32)]:
        q = inputs.codes(K, N, seed=K + N)
        s = inputs.scales(K, N, G, seed=3)
        packed, sp = w.pack(to_dev(q), to_dev(s), G)
        torch.cuda.synchronize()
        p = packed.cpu().numpy().view(np.uint32)
        q2, bad = oracle_mod.unpack(p, K, N)
        assert bad == 0 and np.array_equal(q2, q), (K, N, G)
        assert np.array_equal(p, oracle_mod.pack(q))
        s2, bad = oracle_mod.unpack_scales(sp.cpu().numpy().view(np.uint16), -(-K // G), N)
        assert bad == 0 and np.array_equal(s2, s.view(np.uint16))
    for pattern in (0, 15):
        q = np.full((256, 256), pattern, np.uint8)
        packed, _ = w.pack(to_dev(q), to_dev(np.ones((2, 256), np.float16)), 128)
        q2, bad = oracle_mod.unpack(packed.cpu().numpy().view(np.uint32), 256, 256)
        assert bad == 0 and np.array_equal(q2, q)


def test_pack_masks_codes_to_low_nibble(w, oracle_mod):
    q = inputs.codes(64, 128, seed=9)
    packed, _ = w.pack(to_dev(q | 0xF0), to_dev(np.ones((1, 128), np.float16)), 64)
    q2, bad = oracle_mod.unpack(packed.cpu().numpy().view(np.uint32), 64, 128)
    assert bad == 0 and np.array_equal(q2, q)


def test_hand_example_is_bit_exact(w):
    g = read_golden()
    x, q, s = hand_inputs(8)           # G = K = 8, one scale per column
    y, _, _ = run_gpu(w, x, q, s, 8)
    assert np.array_equal(y[0].astype(np.float64), g["G8_y"]), y


SMALL = [
    # (M, N, K, G, scale kind) spanning several tiles, ragged M/N/K tails
    (16, 4096, 4096, 128, "halfnormal"),      # single GEMM, M=16, K=N=4096
    (1, 8, 8, 8, "halfnormal"),
    (3, 136, 200, 200, "halfnormal"),
    (17, 264, 520, 32, "loguniform"),
    (1, 4096, 4096, 32, "loguniform"),
    (127, 384, 1024, 64, "halfnormal"),
    (33, 512, 2048, 128, "halfnormal"),
    (64, 640, 1024, 128, "halfnormal"),
    (100, 256, 640, 128, "halfnormal"),
    (130, 256, 640, 128, "halfnormal"),
    (300, 264, 136, 32, "halfnormal"),
    (517, 392, 776, 128, "halfnormal"),
    (5, 4096, 4040, 128, "halfnormal"),
    (17, 4096, 4000, 4000, "loguniform"),
    (3, 256, 16384, 128, "loguniform"),
]


@pytest.mark.parametrize("M,N,K,G,kind", SMALL)
def test_parity_small(w, oracle_mod, M, N, K, G, kind):
    x, q, s = inputs.problem(M, K, N, G, seed=M * 7 + K, scale_kind=kind)
    y, _, _ = run_gpu(w, x, q, s, G)
    y_ref, absum = oracle_mod.gemm(x, q, s, G)
    check_within(y, y_ref, absum, "M=%d N=%d K=%d G=%d" % (M, N, K, G))


def test_subnormal_scales(w, oracle_mod):
    M, N, K, G = 9, 256, 512, 128
    x, q, _ = inputs.problem(M, K, N, G, seed=4)
    s = (np.random.default_rng(0).integers(1, 1024, size=(K // G, N)) * 2.0 ** -24).astype(np.float16)
    y, _, _ = run_gpu(w, x, q, s, G)
    y_ref, absum = oracle_mod.gemm(x, q, s, G)
    check_within(y, y_ref, absum, "subnormal scales")


def test_invariants(w):
    M, N, K, G = 20, 256, 512, 64
    x, q, s = inputs.problem(M, K, N, G, seed=5)
    y0, _, _ = run_gpu(w, x, q, np.zeros_like(s), G)
    assert np.all(y0 == 0)
    y8, _, _ = run_gpu(w, x, np.full_like(q, 8), s, G)
    assert np.all(y8 == 0)
    q1 = np.full_like(q, 8)
    q1[77, 130] = 13
    y1, _, _ = run_gpu(w, x, q1, s, G)
    expect = (x[:, 77].astype(np.float64) * 5 * float(s[77 // G, 130])).astype(np.float16)
    others = np.delete(y1, 130, axis=1)
    assert np.all(others == 0)
    assert np.allclose(y1[:, 130].astype(np.float64), expect.astype(np.float64), rtol=2e-3, atol=0)
    # doubling the scales doubles the output exactly (products and sums scale by 2)
    y, _, _ = run_gpu(w, x, q, s, G)
    y2, _, _ = run_gpu(w, x, q, (s.astype(np.float32) * 2).astype(np.float16), G)
    assert np.array_equal(y2.astype(np.float32), 2 * y.astype(np.float32))


def test_deterministic(w):
    M, N, K, G = 16, 4096, 4096, 128
    x, q, s = inputs.problem(M, K, N, G, seed=0)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    xd = to_dev(x)
    ys = [w.gemm(xd, packed, sp, N, G).cpu().numpy() for _ in range(3)]
    assert np.array_equal(ys[0].view(np.uint16), ys[1].view(np.uint16))
    assert np.array_equal(ys[0].view(np.uint16), ys[2].view(np.uint16))
    assert w.check_device_status() == w.OK


def test_workspace_variant_and_graph_capture(w):
    M, N, K, G = 37, 1024, 2048, 128
    x, q, s = inputs.problem(M, K, N, G, seed=2)
    packed, sp = w.pack(to_dev(q), to_dev(s), G)
    xd = to_dev(x)
    y_ref = w.gemm(xd, packed, sp, N, G)
    nbytes = w.workspace_bytes(M, N, K, G)
    ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device="cuda")
    y = w.gemm_ws(xd, packed, sp, N, G, ws)
    assert torch.equal(y, y_ref)
    # w4a16_workspace_bytes covers every weight format's plan, so a workspace a little
    # short of it may still suffice here; one without room for the partials never does
    with pytest.raises(w.W4A16Error) as e:
        w.gemm_ws(xd, packed, sp, N, G, ws[:1024])
    assert e.value.status == w.ERR_WORKSPACE
    # capture into a CUDA graph and replay
    y_g = torch.empty_like(y_ref)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        w.gemm_ws(xd, packed, sp, N, G, ws, y=y_g)
    for _ in range(3):
        y_g.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_g, y_ref)
    assert w.check_device_status(ws) == w.OK


def test_invalid_arguments_on_device(w):
    x = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    packed, sp = w.pack(torch.zeros((64, 128), dtype=torch.uint8, device="cuda"),
                        torch.ones((1, 128), dtype=torch.float16, device="cuda"), 64)
    with pytest.raises(w.W4A16Error) as e:
        w.gemm(x, packed, sp, 128, 48)
    assert e.value.status == w.ERR_INVALID_ARG
    xo = torch.zeros(4 * 64 + 1, dtype=torch.float16, device="cuda")[1:].view(4, 64)
    with pytest.raises(w.W4A16Error) as e:
        w.gemm(xo, packed, sp, 128, 64)
    assert e.value.status == w.ERR_INVALID_ARG
    y = w.gemm(torch.zeros((0, 64), dtype=torch.float16, device="cuda"), packed, sp, 128, 64)
    assert y.shape == (0, 128)


def sampled_parity(w, oracle_mod, cases, G, scale_mult, outlier_frac=0.0, n_rows=8, n_cols=512, seed=0):
    """Full-size problems, compared at a seeded sample of rows x columns."""
    by_shape = {}
    for (M, K, N) in cases:
        by_shape.setdefault((K, N), []).append(M)
    rs = np.random.default_rng(seed)
    worst = 0.0
    for (K, N), Ms in by_shape.items():
        q = inputs.codes(K, N, seed)
        s = inputs.scales(K, N, G, seed, "halfnormal", scale_mult)
        packed, sp = w.pack(to_dev(q), to_dev(s), G)
        for M in Ms:
            x = inputs.activations(M, K, seed, outlier_frac)
            y = w.gemm(to_dev(x), packed, sp, N, G)
            rows = np.unique(np.concatenate([[0, M - 1], rs.integers(0, M, size=n_rows)]))
            cols = np.unique(np.concatenate([[0, N - 1], rs.integers(0, N, size=n_cols)]))
            y_s = y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
            y_ref, absum = oracle_mod.gemm_sample(x, q, s, G, rows, cols)
            worst = max(worst, check_within(y_s, y_ref, absum, "M=%d K=%d N=%d" % (M, K, N)))
        del packed, sp
    return worst


def test_full_size_decode_sweep(w, oracle_mod):
    wl = inputs.WORKLOADS["llama2_7b_decode_sweep"]
    sampled_parity(w, oracle_mod, wl["cases"], wl["group_size"], wl["scale_mult"])


def test_full_size_large_layer(w, oracle_mod):
    wl = inputs.WORKLOADS["large_layer_18432x73728"]
    sampled_parity(w, oracle_mod, wl["cases"], wl["group_size"], wl["scale_mult"], n_cols=256)


def test_full_size_prefill(w, oracle_mod):
    wl = inputs.WORKLOADS["llama2_13b_prefill"]
    sampled_parity(w, oracle_mod, wl["cases"], wl["group_size"], wl["scale_mult"], wl["outlier_frac"],
                   n_rows=6, n_cols=128)


def test_edge_sweep(w, oracle_mod):
    for M in inputs.EDGE_M:
        for (N, K, G) in [(4096, 4096, 4096), (4096, 4096, 32), (256, 16384, 128), (4096, 4000, 128),
                          (4096, 4040, 128)]:
            x, q, s = inputs.problem(M, K, N, G, seed=M + K, scale_kind="loguniform")
            y, _, _ = run_gpu(w, x, q, s, G)
            cols = np.arange(0, N, 7)
            y_ref, absum = oracle_mod.gemm_sample(x, q, s, G, np.arange(M), cols)
            check_within(y[:, cols], y_ref, absum, "edge M=%d N=%d K=%d G=%d" % (M, N, K, G))


def test_device_plan_matches_host_mirror(w):
    """The dispatcher on the device picks the grid that the schedule mirror (whose
    coverage and bounds the CPU tests check) computes for the same SM count."""
    from tests.test_schedule import dispatch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shapes = [(m, n, k) for (m, k, n) in inputs.WORKLOADS["llama2_7b_decode_sweep"]["cases"] if m <= 32]
    shapes += [(1, 256, 16384), (3, 136, 200), (17, 4096, 4000), (1, 73728, 18432), (16, 73728, 18432),
               (2, 8192, 4096), (64, 4096, 4096), (128, 4096, 4096), (128, 4096, 11008), (100, 392, 776)]
    for force in (0, 1, 2, 3):
        prev = w.force_path(force)
        try:
            for (M, N, K) in shapes:
                path, tm, grid = w.plan(M, N, K, 128)
                P = dispatch(M, N, K, 128, sms, force=force)
                assert (path, tm) == (P["path"], P["tm"]), (M, N, K, force, path, tm, grid)
                if path == 1:   # persistent grid: at most one CTA per block, at least one per SM or block
                    assert min(P["blocks"], sms) <= grid <= P["blocks"], (M, N, K, grid, P["blocks"])
                else:
                    assert grid == P["grid"], (M, N, K, force, grid, P["grid"])
        finally:
            w.force_path(prev)


def _chain(w, x_d, layers, G, stream_sync):
    """Back-to-back GEMMs where each one's X is the previous one's output (fused
    SiLU on the widest layer, an in-place residual on the last), all on one stream."""
    outs = []
    h = x_d
    for i, (packed, sp, N, epi) in enumerate(layers):
        if epi == "silu":
            h = w.gemm_fused(h, packed, sp, N, G, activation="silu")
        elif epi == "residual":
            r = outs[0][:, :N].clone()   # a fresh buffer, added to in place
            h = w.gemm_fused(h, packed, sp, N, G, residual=r, y=r)
        else:
            h = w.gemm(h, packed, sp, N, G)
        outs.append(h)
        if stream_sync:
            torch.cuda.synchronize()
    return outs


def test_chained_gemms_read_the_previous_output(w, oracle_mod):
    """Each launch may start before the previous one ends (programmatic dependent
    launch) but must read X only after it completes: a chain launched back to back,
    plain and captured in a CUDA Graph, equals the same chain with a synchronisation
    between launches bit for bit, and every stage matches the oracle applied to the
    GPU's own input of that stage."""
    G, M = 128, 16
    dims = [(4096, 4096, None), (4096, 11008, "silu"), (11008, 4096, None), (4096, 4096, "residual")]
    rng_seed = 40
    layers, host = [], []
    for i, (K, N, epi) in enumerate(dims):
        q = inputs.codes(K, N, rng_seed + i)
        s = inputs.scales(K, N, G, rng_seed + i, "halfnormal", 0.01)
        packed, sp = w.pack(to_dev(q), to_dev(s), G)
        layers.append((packed, sp, N, epi))
        host.append((q, s))
    x = inputs.activations(M, 4096, rng_seed)
    ref = _chain(w, to_dev(x), layers, G, stream_sync=True)
    ref = [o.clone() for o in ref]
    got = _chain(w, to_dev(x), layers, G, stream_sync=False)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    # the same chain captured in a CUDA graph (workspace allocated already)
    xg = to_dev(x)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        outs_g = _chain(w, xg, layers, G, stream_sync=False)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs_g, ref):
        assert torch.equal(a, b)
    # each stage against the oracle on its actual input
    cols = np.random.default_rng(1).choice(4096, 128, replace=False)
    prev = x
    for i, ((q, s), (_, _, N, epi)) in enumerate(zip(host, layers)):
        rows = np.arange(M)
        c = cols[cols < N]
        z, absum = oracle_mod.gemm_sample(prev, q, s, G, rows, c)
        y = ref[i].cpu().numpy()
        if epi is None:
            from tests.parity import check_within
            check_within(y[:, c], z, absum, "chain stage %d" % i)
        else:
            from tests.parity import check_within_fused
            resid = ref[0].cpu().numpy()[:, :N] if epi == "residual" else None
            y_ref = oracle_mod.epilogue(z, residual=resid, activation="silu" if epi == "silu" else "none",
                                        rows=rows if resid is not None else None, cols=c if resid is not None else None)
            check_within_fused(y[:, c], y_ref, z, absum, 0.0,
                               np.abs(resid[np.ix_(rows, c)].astype(np.float64)) if resid is not None else 0.0,
                               "chain stage %d" % i)
        prev = y


@pytest.mark.parametrize("M,N,K,G", [(16, 32768, 1024, 128), (100, 40000, 512, 64), (300, 20000, 264, 264)])
def test_split_region_then_whole_tiles(w, oracle_mod, M, N, K, G):
    """Shapes with more tiles than SMs: the tiles past the last whole wave are split
    among every CTA and run first, the rest go whole (one region of 104 tiles with 1
    whole tile per CTA, and regions grown by a wave with 1 whole tile per CTA, at 16,
    128 and 256 rows per tile). Every element against the oracle, bit-identical over
    three runs."""
    with forced_path(w, 2):
        assert w.plan(M, N, K, G)[0] == 2
        x, q, s = inputs.problem(M, K, N, G, seed=M + N)
        packed, sp = w.pack(to_dev(q), to_dev(s), G)
        xd = to_dev(x)
        ys = [w.gemm(xd, packed, sp, N, G).cpu().numpy() for _ in range(3)]
    z, absum = oracle_mod.gemm(x, q, s, G)
    check_within(ys[0], z, absum, "split region M=%d N=%d K=%d" % (M, N, K))
    assert np.array_equal(ys[0].view(np.uint16), ys[1].view(np.uint16))
    assert np.array_equal(ys[0].view(np.uint16), ys[2].view(np.uint16))
    assert w.check_device_status() == w.OK

"""Guard bands around Y: every GEMM entry point writes the M x N outputs and nothing
on either side of them.

Y is a view into a larger buffer whose 64 elements before and after it hold a NaN
bit pattern that no finite result has. After the call the pattern must be intact,
and Y must equal bit for bit what the same call writes into a fresh tensor (the
kernels are deterministic, and that result is checked against the oracle by the
parity tests). The shapes cover ragged M and N tails, split-K tiles, 2-CTA
clusters and 256-row tiles; every weight format and the fused epilogue take part.
"""
import numpy as np
import pytest

from weight_only_int4_02_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 64        # 16-bit elements on each side (128 bytes: Y stays 16-byte aligned)
CANARY = 0x7E55   # a quiet NaN in binary16 and a NaN in bfloat16 too


@pytest.fixture(scope="module")
def w():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from weight_only_int4_02_gb300 import w4a16
    w4a16.lib()
    return w4a16


def t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def guarded(M, N, dtype):
    """(base, y): base an int16 buffer of M*N + 2*GUARD canaries, y its middle M x N
    elements viewed as dtype."""
    base = torch.full((M * N + 2 * GUARD,), CANARY, dtype=torch.int16, device=DEV)
    y = base.view(dtype)[GUARD:GUARD + M * N].view(M, N)
    assert y.is_contiguous() and y.data_ptr() % 16 == 0
    return base, y


def check_guards(base, what):
    b = base.cpu().numpy()
    assert np.all(b[:GUARD] == CANARY), "%s: write before y" % what
    assert np.all(b[-GUARD:] == CANARY), "%s: write after y" % what


def bits(y):
    return y.contiguous().view(torch.int16).cpu().numpy()


def same_call_twice(fn, M, N, dtype, what):
    y_plain = fn(None)
    base, y = guarded(M, N, dtype)
    out = fn(y)
    torch.cuda.synchronize()
    assert out.data_ptr() == y.data_ptr()
    check_guards(base, what)
    assert np.array_equal(bits(y), bits(y_plain)), "%s: guarded result differs" % what


SHAPES = [
    (1, 256, 16384, 128),     # split-K, 16-row tile
    (3, 136, 200, 200),       # ragged N, one group per column
    (16, 4096, 4096, 128),    # the decode kernel, sixteen rows of X
    (32, 2048, 4096, 128),    # tile-aligned split of 32-row tiles
    (17, 264, 520, 32),       # 32-row tile, ragged M and N
    (100, 392, 776, 128),     # 128-row tile pair, odd tile count (phantom tile)
    (300, 264, 136, 32),      # 256-row tiles, ragged last row tile
]


@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_int4_writes_only_y(w, M, N, K, G):
    x, q, s = inputs.problem(M, K, N, G, seed=M + N)
    packed, sp = w.pack(t(q), t(s), G)
    xd = t(x)
    same_call_twice(lambda y: w.gemm(xd, packed, sp, N, G, y=y), M, N, torch.float16, "gemm")
    bias = t(inputs.rng(M + N, inputs.SCALE_STREAM).standard_normal(N).astype(np.float16))
    resid = t(inputs.activations(M, N, seed=M + 1))
    same_call_twice(lambda y: w.gemm_fused(xd, packed, sp, N, G, bias=bias, residual=resid, activation="silu", y=y),
                    M, N, torch.float16, "gemm_fused")
    zp = w.pack_zeros(t(inputs.zeros(K, N, G, seed=M)), K, G)
    same_call_twice(lambda y: w.gemm_zp(xd, packed, sp, zp, N, G, y=y), M, N, torch.float16, "gemm_zp")


@pytest.mark.parametrize("M,N,K,G", SHAPES)
def test_other_formats_write_only_y(w, M, N, K, G):
    x = t(inputs.activations(M, K, seed=M + N))
    q8 = inputs.rng(M + N, inputs.CODE_STREAM).integers(0, 256, size=(K, N), dtype=np.uint8)
    s8 = inputs.scales(K, N, G, M + N, mult=0.02 / 16)
    p8, sp8 = w.w8_pack(t(q8), t(s8), G)
    same_call_twice(lambda y: w.w8_gemm(x, p8, sp8, N, G, y=y), M, N, torch.float16, "w8_gemm")

    s = inputs.scales(K, N, G, M + N)
    psp, ssp = w.sp_pack(t(inputs.codes_2to4(K, N, seed=M + N)), t(s), G)
    same_call_twice(lambda y: w.sp_gemm(x, psp, ssp, N, G, y=y), M, N, torch.float16, "sp_gemm")

    to_bf16 = lambda a: t(a.view(np.int16)).view(torch.bfloat16)
    xb, sb = inputs.activations_bf16(M, K, M + N), inputs.scales_bf16(K, N, G, M + N)
    packed, spb = w.pack(t(inputs.codes(K, N, M + N)), to_bf16(sb), G)
    xbd = to_bf16(xb)
    same_call_twice(lambda y: w.bf16_gemm(xbd, packed, spb, N, G, y=y), M, N, torch.bfloat16, "bf16_gemm")
    assert w.check_device_status() == w.OK

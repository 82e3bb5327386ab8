"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects invalid arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from weight_only_int4_02_gb300 import build
    build.build()
    from weight_only_int4_02_gb300 import w4a16
    return w4a16.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "w4a16.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
    from weight_only_int4_02_gb300 import w4a16
    for name in w4a16.EXPORTS:
        assert name in names


def declared_arities():
    """{function: number of parameters} from the header's declarations."""
    text = open(os.path.join(ROOT, "include", "w4a16.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(w4a16_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", text):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(lib):
    from weight_only_int4_02_gb300 import w4a16
    arity = declared_arities()
    assert len(arity) >= 20
    for name in w4a16.EXPORTS:
        fn = getattr(lib, name)
        if fn.argtypes is None:
            assert arity[name] == 0, name
        else:
            assert len(fn.argtypes) == arity[name], (name, len(fn.argtypes), arity[name])


def test_sizes(lib):
    assert lib.w4a16_layout_version() == 2
    assert lib.w4a16_packed_words(4096, 4096, 128) == 32 * 64 * 1024
    assert lib.w4a16_packed_words(4040, 4096, 128) == 32 * 64 * 1024
    assert lib.w4a16_packed_words(8, 8, 8) == 4 * 1024
    assert lib.w4a16_packed_words(4000, 4096, 128) == 32 * 64 * 1024
    assert lib.w4a16_packed_words(11008, 4096, 128) == 32 * 172 * 1024
    assert lib.w4a16_scales_elems(4096, 4096, 128) == 32 * 32 * 128
    assert lib.w4a16_scales_elems(4000, 4096, 128) == 32 * 32 * 128
    assert lib.w4a16_scales_elems(4096, 4096, -1) == 32 * 1 * 128
    assert lib.w4a16_scales_elems(4096, 256, 32) == 2 * 128 * 128
    # packed bytes of the 72k x 18k layer
    assert lib.w4a16_packed_words(18432, 73728, 128) * 4 == 18432 * 73728 // 2
    # 4-bit zero-points: 64 bytes per (column tile, group)
    assert lib.w4a16_zeros_bytes(4096, 4096, 128) == 32 * 32 * 64
    assert lib.w4a16_zeros_bytes(4000, 4096, 128) == 32 * 32 * 64
    assert lib.w4a16_zeros_bytes(4096, 200, -1) == 2 * 1 * 64
    assert lib.w4a16_zeros_bytes(4096, 4096, 96) == 0
    # 2:4 sparse codes: 6144 bytes per (column tile, 128 values of k)
    assert lib.w4a16_sp_packed_bytes(4096, 4096, 128) == 32 * 32 * 6144
    assert lib.w4a16_sp_packed_bytes(4040, 4096, 128) == 32 * 32 * 6144
    assert lib.w4a16_sp_packed_bytes(4096, 4096, 96) == 0
    # 8-bit codes: one byte per weight, K padded to a multiple of 256
    assert lib.w4a16_w8_packed_bytes(4096, 4096, 128) == 4096 * 4096
    assert lib.w4a16_w8_packed_bytes(4040, 4096, 128) == 4096 * 4096
    assert lib.w4a16_w8_packed_bytes(8, 8, 8) == 256 * 128
    assert lib.w4a16_w8_packed_bytes(4096, 4096, 96) == 0


@pytest.mark.parametrize("K,N,G", [(0, 8, 8), (8, 0, 8), (12, 8, 12), (8, 12, 8), (4096, 4096, 16),
                                   (4096, 4096, 96), (4096, 4096, 256), (-8, 8, 32)])
def test_invalid_sizes(lib, K, N, G):
    assert lib.w4a16_packed_words(K, N, G) == 0
    assert lib.w4a16_scales_elems(K, N, G) == 0


def test_invalid_arguments_return_before_any_device_work(lib):
    from weight_only_int4_02_gb300 import w4a16 as w
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    # bad sizes, bad group, null pointers: INVALID_ARG without a device
    assert lib.w4a16_gemm(p, p, p, p, 4, 12, 64, 64, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm(p, p, p, p, 4, 64, 64, 48, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm(None, p, p, p, 4, 64, 64, 64, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm(p, p, p, p, -1, 64, 64, 64, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm(p, p, p, p, 0, 64, 64, 64, None) == w.OK   # M = 0 is a no-op
    assert lib.w4a16_pack(p, p, p, p, 64, 60, 64, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm_ws(p, p, p, p, 4, 64, 64, 64, None, 0, None) == w.ERR_INVALID_ARG
    odd = ctypes.c_void_p(ctypes.addressof(buf) + 8)
    assert lib.w4a16_gemm(odd, p, p, p, 4, 64, 64, 64, None) in (w.ERR_INVALID_ARG,)
    # zero-point GEMM: zero-points required, aligned; activation in range
    assert lib.w4a16_gemm_zp(p, p, p, None, p, 4, 64, 64, 64, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm_zp(p, p, p, odd, p, 4, 64, 64, 64, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm_zp(p, p, p, p, p, 4, 64, 64, 64, None, None, 3, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm_zp(p, p, p, p, p, 4, 64, 64, 48, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_gemm_zp(p, p, p, p, p, 0, 64, 64, 64, None, None, 0, None, 0, None) == w.OK
    assert lib.w4a16_pack_zeros(None, p, 64, 64, 64, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_pack_zeros(p, odd, 64, 64, 64, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_pack_zeros(p, p, 64, 60, 64, None) == w.ERR_INVALID_ARG
    # BF16 activations
    assert lib.w4a16_bf16_gemm(p, p, p, p, 4, 64, 64, 64, None, None, 3, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_bf16_gemm(p, p, p, p, 4, 64, 64, 48, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_bf16_gemm(odd, p, p, p, 4, 64, 64, 64, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_bf16_gemm(p, p, p, p, 0, 64, 64, 64, None, None, 0, None, 0, None) == w.OK
    # failure-detection self-test: the limit must be in 1 .. 10^10 ns, the workspace 256-byte aligned
    assert lib.w4a16_selftest_wait_timeout(None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_selftest_wait_timeout(None, 10 ** 11, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_selftest_wait_timeout(odd, 1000, None) == w.ERR_INVALID_ARG
    # 2:4 sparse codes
    assert lib.w4a16_sp_gemm(p, p, p, p, 4, 64, 64, 64, None, None, 3, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_sp_gemm(p, odd, p, p, 4, 64, 64, 64, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_sp_gemm(p, p, p, p, 0, 64, 64, 64, None, None, 0, None, 0, None) == w.OK
    assert lib.w4a16_sp_pack(None, p, p, p, 64, 64, 64, None, None) == w.ERR_INVALID_ARG
    four = ctypes.c_void_p(ctypes.addressof(buf) + 4)
    assert lib.w4a16_sp_pack(p, p, p, p, 64, 64, 64, four, None) == w.ERR_INVALID_ARG
    # row strides: ldx >= K and a multiple of 8, ldy >= N, ldr >= N with a residual
    sg = lib.w4a16_gemm_strided   # (x, ldx, packed, scales, y, ldy, M, N, K, G, bias, residual, ldr, act, ws, n, s)
    assert sg(p, 56, p, p, p, 64, 4, 64, 64, 64, None, None, 0, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert sg(p, 68, p, p, p, 64, 4, 64, 64, 64, None, None, 0, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert sg(p, 64, p, p, p, 60, 4, 64, 64, 64, None, None, 0, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert sg(p, 64, p, p, p, 64, 4, 64, 64, 64, None, p, 32, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert sg(p, 64, p, p, p, 64, 4, 64, 64, 64, None, p, 0, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert sg(p, 64, p, p, p, 64, 4, 64, 64, 64, None, None, 0, 3, None, 0, None) == w.ERR_INVALID_ARG
    assert sg(p, 72, p, p, p, 80, 0, 64, 64, 64, None, None, 0, 0, None, 0, None) == w.OK   # M = 0
    # 8-bit codes
    assert lib.w4a16_w8_gemm(p, p, p, p, 4, 64, 64, 64, None, None, 3, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_w8_gemm(p, p, p, p, 4, 64, 64, 48, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_w8_gemm(None, p, p, p, 4, 64, 64, 64, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_w8_gemm(p, odd, p, p, 4, 64, 64, 64, None, None, 0, None, 0, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_w8_gemm(p, p, p, p, 0, 64, 64, 64, None, None, 0, None, 0, None) == w.OK
    assert lib.w4a16_w8_pack(None, p, p, p, 64, 64, 64, None) == w.ERR_INVALID_ARG
    assert lib.w4a16_w8_pack(p, p, odd, p, 64, 64, 64, None) == w.ERR_INVALID_ARG
    for s in range(6):
        assert lib.w4a16_status_string(s)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "weight_only_int4_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f


def test_binding_rejects_short_or_strided_buffers_before_any_launch(lib):
    torch = pytest.importorskip("torch")
    from weight_only_int4_02_gb300 import w4a16 as w
    M, N, K, G = 4, 256, 512, 128
    x = torch.zeros((M, K), dtype=torch.float16)
    y = torch.zeros((M, N), dtype=torch.float16)
    packed = torch.zeros(w.packed_words(K, N, G), dtype=torch.int32)
    sp = torch.zeros(w.scales_elems(K, N, G), dtype=torch.float16)
    w.check_buffers(x, packed, sp, N, G, y)                                  # exact sizes pass
    for bad in [dict(packed=packed[:-1]), dict(scales_packed=sp[:-8]), dict(y=y[:, :-8]),
                dict(y=torch.zeros((N, M), dtype=torch.float16).t()), dict(y=torch.zeros((M, N), dtype=torch.float32))]:
        args = dict(packed=packed, scales_packed=sp, y=y)
        args.update(bad)
        with pytest.raises(w.W4A16Error) as e:
            w.check_buffers(x, args["packed"], args["scales_packed"], N, G, args["y"])
        assert e.value.status == w.ERR_INVALID_ARG
    # the other formats' weight sizes
    w.check_buffers(x, torch.zeros(w.w8_packed_bytes(K, N, G), dtype=torch.uint8), sp, N, G, y, "w8")
    with pytest.raises(w.W4A16Error):
        w.check_buffers(x, packed, sp, N, G, y, "w8")                       # 4-bit buffer for 8-bit codes
    w.check_buffers(x, torch.zeros(w.sp_packed_bytes(K, N, G), dtype=torch.uint8), sp, N, G, y, "sparse")
    zp = torch.zeros(w.zeros_bytes(K, N, G), dtype=torch.uint8)
    w.check_buffers(x, packed, sp, N, G, y, "int4", zp)
    with pytest.raises(w.W4A16Error):
        w.check_buffers(x, packed, sp, N, G, y, "int4", zp[:-16])
    # sizes the library rejects itself are left to it
    w.check_buffers(x, packed[:1], sp[:1], N, 48, y)

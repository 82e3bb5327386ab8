"""CPU oracle for the W4A16 matmul. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. The product library never loads it, and this package
imports nothing from the product package.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, FP64, k-ascending sums);
this module compiles it with gcc and marshals numpy arrays through ctypes.
Definitions and citations are in the C file's header.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_w4a16.so")
_lib = None


def build(force=False):
    """Compile the oracle library with gcc (no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.w4o_half_to_double.argtypes = [ctypes.c_uint16]
        lib.w4o_half_to_double.restype = ctypes.c_double
        lib.w4o_decode_halves.argtypes = [P, P, ctypes.c_size_t]
        lib.w4o_dequant_zp.argtypes = [P, P, P, I, I, I, P]
        lib.w4o_gemm_zp.argtypes = [P, P, P, P, I, I, I, I, P, P, I]
        lib.w4o_gemm_zp.restype = I
        lib.w4o_gemm_sample_zp.argtypes = [P, P, P, P, I, I, I, I, P, I, P, I, P, P, I]
        lib.w4o_gemm_sample_zp.restype = I
        lib.w4o_packed_words.argtypes = [I, I]
        lib.w4o_packed_words.restype = ctypes.c_size_t
        lib.w4o_locate.argtypes = [I, I, I, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(I)]
        lib.w4o_unpack.argtypes = [P, I, I, P]
        lib.w4o_unpack.restype = ctypes.c_longlong
        lib.w4o_pack.argtypes = [P, I, I, P]
        lib.w4o_unpack_scales.argtypes = [P, I, I, P]
        lib.w4o_unpack_scales.restype = ctypes.c_longlong
        lib.w4o_unpack_zeros.argtypes = [P, I, I, P]
        lib.w4o_unpack_zeros.restype = ctypes.c_longlong
        lib.w4o_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.w4o_bf16_to_double.restype = ctypes.c_double
        lib.w4o_decode_bf16.argtypes = [P, P, ctypes.c_size_t]
        lib.w4o_gemm_sample_bf16.argtypes = [P, P, P, I, I, I, I, P, I, P, I, P, P, I]
        lib.w4o_gemm_sample_bf16.restype = I
        lib.w4o_sp_packed_bytes.argtypes = [I, I]
        lib.w4o_sp_packed_bytes.restype = ctypes.c_size_t
        lib.w4o_sp_pack.argtypes = [P, I, I, P]
        lib.w4o_sp_pack.restype = ctypes.c_longlong
        lib.w4o_sp_unpack.argtypes = [P, I, I, P]
        lib.w4o_sp_unpack.restype = ctypes.c_longlong
        lib.w4o_gemm_sample_w8.argtypes = [P, P, P, I, I, I, I, P, I, P, I, P, P, I]
        lib.w4o_gemm_sample_w8.restype = I
        lib.w4o_dequant_w8.argtypes = [P, P, I, I, I, P]
        lib.w4o_packed_bytes_w8.argtypes = [I, I]
        lib.w4o_packed_bytes_w8.restype = ctypes.c_size_t
        lib.w4o_locate_w8.argtypes = [I, I, I]
        lib.w4o_locate_w8.restype = ctypes.c_size_t
        lib.w4o_unpack_w8.argtypes = [P, I, I, P]
        lib.w4o_unpack_w8.restype = ctypes.c_longlong
        lib.w4o_pack_w8.argtypes = [P, I, I, P]
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16
    return a


def n_groups(K, G):
    return -(-K // G)


def half_to_double(bits):
    """Decode binary16 bit patterns (uint16 array) to float64 with the oracle's decoder."""
    b = _bits16(np.asarray(bits))
    out = np.empty(b.shape, np.float64)
    _load().w4o_decode_halves(_ptr(b), _ptr(out), b.size)
    return out


def _zeros(z, K, N, G):
    """Zero-points as a contiguous uint8 [ceil(K/G)][N] array, or None for 8."""
    if z is None:
        return None
    z = np.ascontiguousarray(z, dtype=np.uint8)
    assert z.shape == (n_groups(K, G), N) and int(z.max(initial=0)) <= 15
    return z


def dequant(q, s, G, z=None):
    """w[k][n] = (q[k][n] - z[k // G][n]) * s[k // G][n] in float64 (z = 8 when None)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _bits16(s)
    K, N = q.shape
    assert s.shape == (n_groups(K, G), N)
    z = _zeros(z, K, N, G)
    w = np.empty((K, N), np.float64)
    _load().w4o_dequant_zp(_ptr(q), _ptr(s), _ptr(z) if z is not None else None, K, N, G, _ptr(w))
    return w


def _threads(threads):
    return threads if threads else (os.cpu_count() or 1)


def gemm(x, q, s, G, threads=None, z=None):
    """(y, absum): y = x @ dequant(q, s, z) in float64 (k ascending), absum = sum |x*w|."""
    x = _bits16(x)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _bits16(s)
    M, K = x.shape
    K2, N = q.shape
    assert K == K2 and s.shape == (n_groups(K, G), N)
    z = _zeros(z, K, N, G)
    y = np.empty((M, N), np.float64)
    a = np.empty((M, N), np.float64)
    rc = _load().w4o_gemm_zp(_ptr(x), _ptr(q), _ptr(s), _ptr(z) if z is not None else None, M, N, K, G,
                             _ptr(y), _ptr(a), _threads(threads))
    assert rc == 0
    return y, a


def gemm_sample(x, q, s, G, rows, cols, threads=None, z=None):
    """(y, absum) restricted to rows x cols: y[i][j] = y_ref[rows[i]][cols[j]]."""
    x = _bits16(x)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _bits16(s)
    M, K = x.shape
    N = q.shape[1]
    z = _zeros(z, K, N, G)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    cols = np.ascontiguousarray(cols, dtype=np.int32)
    y = np.empty((rows.size, cols.size), np.float64)
    a = np.empty((rows.size, cols.size), np.float64)
    rc = _load().w4o_gemm_sample_zp(_ptr(x), _ptr(q), _ptr(s), _ptr(z) if z is not None else None, M, N, K, G,
                                    _ptr(rows), rows.size, _ptr(cols), cols.size, _ptr(y), _ptr(a),
                                    _threads(threads))
    assert rc == 0
    return y, a


def packed_words(K, N):
    return int(_load().w4o_packed_words(K, N))


def locate(K, k, n):
    """(word index, nibble) of weight (k, n) in the packed layout."""
    w = ctypes.c_size_t()
    i = ctypes.c_int()
    _load().w4o_locate(K, k, n, ctypes.byref(w), ctypes.byref(i))
    return w.value, i.value


def unpack(packed, K, N):
    """(codes[K][N], number of padding nibbles that are not 8)."""
    p = np.ascontiguousarray(packed, dtype=np.uint32)
    assert p.size == packed_words(K, N)
    codes = np.empty((K, N), np.uint8)
    bad = _load().w4o_unpack(_ptr(p), K, N, _ptr(codes))
    return codes, int(bad)


def pack(codes):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    K, N = codes.shape
    out = np.empty(packed_words(K, N), np.uint32)
    _load().w4o_pack(_ptr(codes), K, N, _ptr(out))
    return out


def unpack_scales(sp, ng, N):
    """(s[ng][N] as uint16 bits, number of padding entries that are not 0)."""
    sp = _bits16(sp)
    s = np.empty((ng, N), np.uint16)
    bad = _load().w4o_unpack_scales(_ptr(sp), ng, N, _ptr(s))
    return s, int(bad)


# ------------------------------------------------------------------ 2:4 sparse 4-bit codes
# The GEMM of 2:4 sparse codes is the dense definition (gemm, gemm_sample) on the
# dense codes; these functions restate the sparse packed layout.
def sp_packed_bytes(K, N):
    return int(_load().w4o_sp_packed_bytes(K, N))


def sp_pack(codes):
    """(packed uint8 array, number of groups of four with more than two codes other than 8)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    K, N = codes.shape
    out = np.empty(sp_packed_bytes(K, N), np.uint8)
    v = _load().w4o_sp_pack(_ptr(codes), K, N, _ptr(out))
    return out, int(v)


def sp_unpack(packed, K, N):
    """(dense codes[K][N], number of malformed or non-empty padding groups)."""
    p = np.ascontiguousarray(packed).view(np.uint8).ravel()
    assert p.size == sp_packed_bytes(K, N)
    codes = np.empty((K, N), np.uint8)
    bad = _load().w4o_sp_unpack(_ptr(p), K, N, _ptr(codes))
    return codes, int(bad)


# ------------------------------------------------------------------ BF16 activations
def bf16_to_double(bits):
    """Decode bfloat16 bit patterns (uint16 array) to float64 with the oracle's decoder."""
    b = np.ascontiguousarray(np.asarray(bits), dtype=np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().w4o_decode_bf16(_ptr(b), _ptr(out), b.size)
    return out


def gemm_sample_bf16(x, q, s, G, rows, cols, threads=None):
    """(y, absum) restricted to rows x cols, x and s bfloat16 bit patterns (uint16)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    M, K = x.shape
    N = q.shape[1]
    assert q.shape[0] == K and s.shape == (n_groups(K, G), N)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    cols = np.ascontiguousarray(cols, dtype=np.int32)
    y = np.empty((rows.size, cols.size), np.float64)
    a = np.empty((rows.size, cols.size), np.float64)
    rc = _load().w4o_gemm_sample_bf16(_ptr(x), _ptr(q), _ptr(s), M, N, K, G, _ptr(rows), rows.size,
                                      _ptr(cols), cols.size, _ptr(y), _ptr(a), _threads(threads))
    assert rc == 0
    return y, a


def gemm_bf16(x, q, s, G, threads=None):
    """(y, absum) = x @ dequant(q, s) in float64 for bfloat16 x and s (bit patterns)."""
    return gemm_sample_bf16(x, q, s, G, np.arange(np.shape(x)[0]), np.arange(np.shape(q)[1]), threads)


# ------------------------------------------------------------------ W8A16 (8-bit codes, zero-point 128)
def dequant_w8(q, s, G):
    """w[k][n] = (q[k][n] - 128) * s[k // G][n] in float64, q 8-bit codes."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _bits16(s)
    K, N = q.shape
    assert s.shape == (n_groups(K, G), N)
    w = np.empty((K, N), np.float64)
    _load().w4o_dequant_w8(_ptr(q), _ptr(s), K, N, G, _ptr(w))
    return w


def gemm_sample_w8(x, q, s, G, rows, cols, threads=None):
    """(y, absum) of the W8A16 format restricted to rows x cols."""
    x = _bits16(x)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = _bits16(s)
    M, K = x.shape
    N = q.shape[1]
    assert q.shape[0] == K and s.shape == (n_groups(K, G), N)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    cols = np.ascontiguousarray(cols, dtype=np.int32)
    y = np.empty((rows.size, cols.size), np.float64)
    a = np.empty((rows.size, cols.size), np.float64)
    rc = _load().w4o_gemm_sample_w8(_ptr(x), _ptr(q), _ptr(s), M, N, K, G, _ptr(rows), rows.size,
                                    _ptr(cols), cols.size, _ptr(y), _ptr(a), _threads(threads))
    assert rc == 0
    return y, a


def gemm_w8(x, q, s, G, threads=None):
    """(y, absum) = x @ dequant_w8(q, s) in float64 (k ascending), all rows and columns."""
    M, N = np.shape(x)[0], np.shape(q)[1]
    return gemm_sample_w8(x, q, s, G, np.arange(M), np.arange(N), threads)


def packed_bytes_w8(K, N):
    return int(_load().w4o_packed_bytes_w8(K, N))


def locate_w8(K, k, n):
    """Byte index of weight (k, n) in the 8-bit packed layout."""
    return int(_load().w4o_locate_w8(K, k, n))


def unpack_w8(packed, K, N):
    """(codes[K][N], number of padding bytes that are not 128)."""
    p = np.ascontiguousarray(packed).view(np.uint8).ravel()
    assert p.size == packed_bytes_w8(K, N)
    codes = np.empty((K, N), np.uint8)
    bad = _load().w4o_unpack_w8(_ptr(p), K, N, _ptr(codes))
    return codes, int(bad)


def pack_w8(codes):
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    K, N = codes.shape
    out = np.empty(packed_bytes_w8(K, N), np.uint8)
    _load().w4o_pack_w8(_ptr(codes), K, N, _ptr(out))
    return out


def unpack_zeros(zp, ng, N):
    """(z[ng][N] as uint8, number of padding nibbles that are not 8) from the
    tile-ordered 4-bit zero-points."""
    zp = np.ascontiguousarray(zp, dtype=np.uint8)
    assert zp.size == -(-N // 128) * ng * 64
    z = np.empty((ng, N), np.uint8)
    bad = _load().w4o_unpack_zeros(_ptr(zp), ng, N, _ptr(z))
    return z, int(bad)


def epilogue(z, bias=None, residual=None, activation="none", rows=None, cols=None, dtype="f16"):
    """The fused epilogue in float64 on GEMM results z (float64 [M][N], or the
    sample rows x cols of it): act(z + bias[n]) + residual[m][n]. dtype "bf16":
    bias and residual are bfloat16 bit patterns (uint16).

    Follows "quant_marlin_kernel", "End-to-end flow" (the output tile flows into a
    bias add, then an activation); the residual add after the activation is the
    reading of a transformer block's skip connection. bias (float16 [N]) and
    residual (float16 [M][N]) are decoded with the oracle's own binary16 decoder;
    SiLU(z) = z / (1 + e^-z) with numpy's exp, ReLU(z) = max(z, 0)."""
    z = np.array(z, dtype=np.float64, copy=True)
    decode = bf16_to_double if dtype == "bf16" else half_to_double
    if bias is not None:
        b = decode(bias)
        z += b if cols is None else b[np.asarray(cols)]
    if activation == "silu":
        with np.errstate(over="ignore"):
            z = z / (1.0 + np.exp(-z))
    elif activation == "relu":
        z = np.maximum(z, 0.0)
    else:
        assert activation == "none", activation
    if residual is not None:
        r = decode(residual)
        z += r if rows is None else r[np.ix_(np.asarray(rows), np.asarray(cols))]
    return z

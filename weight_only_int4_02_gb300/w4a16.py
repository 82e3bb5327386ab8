"""Python binding of libw4a16.so (ctypes; argument marshalling only).

Every step of the matmul runs in the library's CUDA kernels. Tensors are torch
CUDA tensors used as plain device buffers; FP16 data crosses the ABI as binary16
bit patterns. There is no fallback: if the library is not built, or the device
is not an sm_103 GPU, the calls raise.
"""
import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libw4a16.so")
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(6)

EXPORTS = ["w4a16_layout_version", "w4a16_status_string", "w4a16_last_cuda_error", "w4a16_packed_words",
           "w4a16_scales_elems", "w4a16_pack", "w4a16_gemm", "w4a16_workspace_bytes", "w4a16_gemm_ws",
           "w4a16_check_device_status", "w4a16_plan", "w4a16_gemm_noalloc", "w4a16_gemm_fused",
           "w4a16_zeros_bytes", "w4a16_pack_zeros", "w4a16_gemm_zp", "w4a16_w8_packed_bytes", "w4a16_w8_pack",
           "w4a16_w8_gemm", "w4a16_bf16_gemm", "w4a16_sp_packed_bytes", "w4a16_sp_pack", "w4a16_sp_gemm",
           "w4a16_selftest_wait_timeout", "w4a16_force_path", "w4a16_set_wait_limit_ns", "w4a16_gemm_strided"]

ACTIVATIONS = {"none": 0, "silu": 1, "relu": 2}


class W4A16Error(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = "%s: %s" % (what, lib().w4a16_status_string(status).decode())
        if status == ERR_CUDA:
            msg += " (cudaError %d)" % lib().w4a16_last_cuda_error()
        super().__init__(msg)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libw4a16.so is not built (%s); run __graft_entry__.build()" % _LIB_PATH)
        L = ctypes.CDLL(_LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.w4a16_layout_version.restype = I
        L.w4a16_status_string.argtypes = [I]
        L.w4a16_status_string.restype = ctypes.c_char_p
        L.w4a16_last_cuda_error.restype = I
        L.w4a16_packed_words.argtypes = [I, I, I]
        L.w4a16_packed_words.restype = Z
        L.w4a16_scales_elems.argtypes = [I, I, I]
        L.w4a16_scales_elems.restype = Z
        L.w4a16_pack.argtypes = [P, P, P, P, I, I, I, P]
        L.w4a16_pack.restype = I
        L.w4a16_gemm.argtypes = [P, P, P, P, I, I, I, I, P]
        L.w4a16_gemm.restype = I
        L.w4a16_workspace_bytes.argtypes = [I, I, I, I]
        L.w4a16_workspace_bytes.restype = Z
        L.w4a16_gemm_ws.argtypes = [P, P, P, P, I, I, I, I, P, Z, P]
        L.w4a16_gemm_ws.restype = I
        L.w4a16_check_device_status.argtypes = [P, P]
        L.w4a16_check_device_status.restype = I
        L.w4a16_plan.argtypes = [I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)]
        L.w4a16_plan.restype = I
        L.w4a16_force_path.argtypes = [I]
        L.w4a16_force_path.restype = I
        L.w4a16_set_wait_limit_ns.argtypes = [ctypes.c_longlong]
        L.w4a16_set_wait_limit_ns.restype = ctypes.c_longlong
        L.w4a16_gemm_noalloc.argtypes = [P, P, P, P, I, I, I, I, P]
        L.w4a16_gemm_noalloc.restype = I
        L.w4a16_gemm_fused.argtypes = [P, P, P, P, I, I, I, I, P, P, I, P, Z, P]
        L.w4a16_gemm_fused.restype = I
        L.w4a16_gemm_strided.argtypes = [P, I, P, P, P, I, I, I, I, I, P, P, I, I, P, Z, P]
        L.w4a16_gemm_strided.restype = I
        L.w4a16_zeros_bytes.argtypes = [I, I, I]
        L.w4a16_zeros_bytes.restype = Z
        L.w4a16_pack_zeros.argtypes = [P, P, I, I, I, P]
        L.w4a16_pack_zeros.restype = I
        L.w4a16_gemm_zp.argtypes = [P, P, P, P, P, I, I, I, I, P, P, I, P, Z, P]
        L.w4a16_gemm_zp.restype = I
        L.w4a16_selftest_wait_timeout.argtypes = [P, ctypes.c_longlong, P]
        L.w4a16_selftest_wait_timeout.restype = I
        L.w4a16_sp_packed_bytes.argtypes = [I, I, I]
        L.w4a16_sp_packed_bytes.restype = Z
        L.w4a16_sp_pack.argtypes = [P, P, P, P, I, I, I, P, P]
        L.w4a16_sp_pack.restype = I
        L.w4a16_sp_gemm.argtypes = [P, P, P, P, I, I, I, I, P, P, I, P, Z, P]
        L.w4a16_sp_gemm.restype = I
        L.w4a16_bf16_gemm.argtypes = [P, P, P, P, I, I, I, I, P, P, I, P, Z, P]
        L.w4a16_bf16_gemm.restype = I
        L.w4a16_w8_packed_bytes.argtypes = [I, I, I]
        L.w4a16_w8_packed_bytes.restype = Z
        L.w4a16_w8_pack.argtypes = [P, P, P, P, I, I, I, P]
        L.w4a16_w8_pack.restype = I
        L.w4a16_w8_gemm.argtypes = [P, P, P, P, I, I, I, I, P, P, I, P, Z, P]
        L.w4a16_w8_gemm.restype = I
        _lib = L
    return _lib


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != OK:
        raise W4A16Error(status, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _nbytes(t):
    return t.numel() * t.element_size()


def check_buffers(x, packed, scales_packed, N, group_size, y, weight_format="int4", zeros_packed=None):
    """Raise W4A16Error(ERR_INVALID_ARG) before any launch when a buffer is smaller than
    its shape needs or not contiguous (the C ABI sees only pointers). Sizes the
    library rejects anyway (invalid K, N or group size) are left to it."""
    M, K = x.shape
    need_w = {"int4": packed_words(K, N, group_size) * 4, "w8": w8_packed_bytes(K, N, group_size),
              "sparse": sp_packed_bytes(K, N, group_size)}[weight_format]
    need_s = scales_elems(K, N, group_size) * 2
    if need_w == 0 or need_s == 0:
        return
    checks = [(packed, need_w, "packed weights"), (scales_packed, need_s, "packed scales"), (y, M * N * 2, "y")]
    if zeros_packed is not None:
        checks.append((zeros_packed, zeros_bytes(K, N, group_size), "packed zero-points"))
    for t, need, what in checks:
        if not t.is_contiguous():
            raise W4A16Error(ERR_INVALID_ARG, "%s is not contiguous" % what)
        if _nbytes(t) < need:
            raise W4A16Error(ERR_INVALID_ARG, "%s hold %d bytes, the shape needs %d" % (what, _nbytes(t), need))
    if tuple(y.shape) != (M, N) or y.element_size() != 2:
        raise W4A16Error(ERR_INVALID_ARG, "y must be a 16-bit [M][N] tensor")


def check_buffers_weights(packed, scales_packed, K, N, group_size):
    """check_buffers for the weights alone (the activations may be strided views)."""
    need_w, need_s = packed_words(K, N, group_size) * 4, scales_elems(K, N, group_size) * 2
    if need_w == 0 or need_s == 0:
        return
    for t, need, what in ((packed, need_w, "packed weights"), (scales_packed, need_s, "packed scales")):
        if not t.is_contiguous():
            raise W4A16Error(ERR_INVALID_ARG, "%s is not contiguous" % what)
        if _nbytes(t) < need:
            raise W4A16Error(ERR_INVALID_ARG, "%s hold %d bytes, the shape needs %d" % (what, _nbytes(t), need))


def layout_version():
    return lib().w4a16_layout_version()


def packed_words(K, N, group_size):
    return lib().w4a16_packed_words(K, N, group_size)


def scales_elems(K, N, group_size):
    return lib().w4a16_scales_elems(K, N, group_size)


def workspace_bytes(M, N, K, group_size):
    return lib().w4a16_workspace_bytes(M, N, K, group_size)


def pack(codes, scales, group_size, stream=None, out=None):
    """Repack codes (uint8 [K][N]) and scales (float16 or bfloat16 [ceil(K/G)][N]) on the GPU.

    Returns (packed int32 words, packed scales of the scales' dtype)."""
    K, N = codes.shape
    assert codes.dtype == torch.uint8 and scales.dtype in (torch.float16, torch.bfloat16)
    assert codes.is_cuda and scales.is_cuda and codes.is_contiguous() and scales.is_contiguous()
    nw, ns = packed_words(K, N, group_size), scales_elems(K, N, group_size)
    if nw == 0 or ns == 0:
        raise W4A16Error(ERR_INVALID_ARG, "pack")
    if out is None:
        packed = torch.empty(nw, dtype=torch.int32, device=codes.device)
        sp = torch.empty(ns, dtype=scales.dtype, device=codes.device)
    else:
        packed, sp = out
    _check(lib().w4a16_pack(_ptr(codes), _ptr(scales), _ptr(packed), _ptr(sp), K, N, group_size, _stream(stream)),
           "w4a16_pack")
    return packed, sp


def gemm(x, packed, scales_packed, N, group_size, y=None, stream=None):
    """y = x @ dequant(W) for x float16 [M][K]; returns y float16 [M][N]."""
    M, K = x.shape
    assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous()
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    check_buffers(x, packed, scales_packed, N, group_size, y, 'int4')
    _check(lib().w4a16_gemm(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(y), M, N, K, group_size,
                            _stream(stream)), "w4a16_gemm")
    return y


def gemm_ws(x, packed, scales_packed, N, group_size, workspace, y=None, stream=None):
    """As gemm, with a caller-owned workspace (uint8 CUDA tensor, zeroed once before first use)."""
    M, K = x.shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    check_buffers(x, packed, scales_packed, N, group_size, y, 'int4')
    _check(lib().w4a16_gemm_ws(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(y), M, N, K, group_size,
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "w4a16_gemm_ws")
    return y


def selftest_wait_timeout(limit_ns, workspace=None, stream=None):
    """Launch one warp whose bounded wait on a barrier that nothing completes gives up
    after limit_ns and sets the workspace's error word (see check_device_status)."""
    _check(lib().w4a16_selftest_wait_timeout(_ptr(workspace), int(limit_ns), _stream(stream)),
           "w4a16_selftest_wait_timeout")


def check_device_status(workspace=None, stream=None):
    """Synchronise and return the status of the kernels' bounded waits (OK or ERR_TIMEOUT)."""
    return lib().w4a16_check_device_status(_ptr(workspace), _stream(stream))


def plan(M, N, K, group_size):
    """(path, tile_m, grid) chosen for this shape on the current device."""
    p, t, g = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().w4a16_plan(M, N, K, group_size, ctypes.byref(p), ctypes.byref(t), ctypes.byref(g)), "w4a16_plan")
    return p.value, t.value, g.value


def set_wait_limit_ns(limit_ns):
    """Set the limit of the kernels' bounded waits (for tests of failure detection);
    returns the previous limit. limit_ns <= 0 only reads it."""
    return lib().w4a16_set_wait_limit_ns(int(limit_ns))


def force_path(path):
    """Force the dispatcher's choice for the 4-bit FP16 format: 0 automatic, 1 the
    CUDA-core kernel wherever it applies (M <= 4), 2 the tensor-core kernel, 3 the
    decode kernel wherever it applies (M <= 16, K a multiple of 32).
    Returns the previous setting."""
    prev = lib().w4a16_force_path(int(path))
    if prev < 0:
        raise W4A16Error(ERR_INVALID_ARG, "w4a16_force_path(%r)" % (path,))
    return prev


def gemm_noalloc(x, packed, scales_packed, N, group_size, y=None, stream=None):
    """As gemm, for callers that may not allocate device memory: the split-K
    scratch is a fixed array inside the library (see w4a16_gemm_noalloc)."""
    M, K = x.shape
    assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous()
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    check_buffers(x, packed, scales_packed, N, group_size, y, 'int4')
    _check(lib().w4a16_gemm_noalloc(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(y), M, N, K, group_size,
                                    _stream(stream)), "w4a16_gemm_noalloc")
    return y


def gemm_fused(x, packed, scales_packed, N, group_size, bias=None, residual=None, activation="none", y=None,
               workspace=None, stream=None):
    """y = act(x @ dequant(W) + bias) + residual, fused into the GEMM's epilogue.

    bias: float16 [N] or None; residual: float16 [M][N] or None (may be y itself);
    activation: "none", "silu" or "relu"; workspace: as gemm_ws, or None for the
    library's own."""
    M, K = x.shape
    assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous()
    for t, shape in ((bias, (N,)), (residual, (M, N))):
        if t is not None:
            assert t.dtype == torch.float16 and t.is_cuda and t.is_contiguous() and tuple(t.shape) == shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check_buffers(x, packed, scales_packed, N, group_size, y, 'int4')
    _check(lib().w4a16_gemm_fused(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(y), M, N, K, group_size,
                                  _ptr(bias), _ptr(residual), ACTIVATIONS[activation], _ptr(workspace), ws_bytes,
                                  _stream(stream)), "w4a16_gemm_fused")
    return y


def _row_stride(t, cols, name):
    """Elements between rows of a 2-D float16 CUDA view whose rows are contiguous."""
    assert t.dtype == torch.float16 and t.is_cuda and t.dim() == 2, name
    assert t.shape[1] == cols and (t.stride(1) == 1 or t.shape[1] == 1), name
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), cols)


def gemm_strided(x, packed, scales_packed, N, group_size, bias=None, residual=None, activation="none", y=None,
                 workspace=None, stream=None):
    """gemm_fused on row-strided 2-D views (rows contiguous, rows any distance apart):
    x may be the leading K columns of a wider tensor, y and residual slices of wider
    buffers; the strides are taken from the views."""
    M, K = x.shape
    ldx = _row_stride(x, K, "x")
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    ldy = _row_stride(y, N, "y")
    ldr = _row_stride(residual, N, "residual") if residual is not None else 0
    if bias is not None:
        assert bias.dtype == torch.float16 and bias.is_cuda and bias.is_contiguous() and tuple(bias.shape) == (N,)
    check_buffers_weights(packed, scales_packed, K, N, group_size)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().w4a16_gemm_strided(_ptr(x), ldx, _ptr(packed), _ptr(scales_packed), _ptr(y), ldy, M, N, K,
                                    group_size, _ptr(bias), _ptr(residual), ldr, ACTIVATIONS[activation],
                                    _ptr(workspace), ws_bytes, _stream(stream)), "w4a16_gemm_strided")
    return y


def zeros_bytes(K, N, group_size):
    return lib().w4a16_zeros_bytes(K, N, group_size)


def pack_zeros(zeros, K, group_size, stream=None, out=None):
    """Repack per-group zero-points (uint8 [ceil(K/G)][N], values 0..15) on the GPU
    into the tile-ordered 4-bit layout; returns a uint8 tensor."""
    ng, N = zeros.shape
    assert zeros.dtype == torch.uint8 and zeros.is_cuda and zeros.is_contiguous()
    nb = zeros_bytes(K, N, group_size)
    if nb == 0:
        raise W4A16Error(ERR_INVALID_ARG, "pack_zeros")
    zp = torch.empty(nb, dtype=torch.uint8, device=zeros.device) if out is None else out
    _check(lib().w4a16_pack_zeros(_ptr(zeros), _ptr(zp), K, N, group_size, _stream(stream)), "w4a16_pack_zeros")
    return zp


def gemm_zp(x, packed, scales_packed, zeros_packed, N, group_size, bias=None, residual=None, activation="none",
            y=None, workspace=None, stream=None):
    """y = act(x @ dequant(W) + bias) + residual with per-group zero-points:
    dequant(W)[k][n] = (q[k][n] - z[k // G][n]) * s[k // G][n]. Arguments as gemm_fused,
    plus zeros_packed from pack_zeros."""
    M, K = x.shape
    assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous()
    for t, shape in ((bias, (N,)), (residual, (M, N))):
        if t is not None:
            assert t.dtype == torch.float16 and t.is_cuda and t.is_contiguous() and tuple(t.shape) == shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check_buffers(x, packed, scales_packed, N, group_size, y, 'int4', zeros_packed)
    _check(lib().w4a16_gemm_zp(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(zeros_packed), _ptr(y), M, N, K,
                               group_size, _ptr(bias), _ptr(residual), ACTIVATIONS[activation], _ptr(workspace),
                               ws_bytes, _stream(stream)), "w4a16_gemm_zp")
    return y


def w8_packed_bytes(K, N, group_size):
    return lib().w4a16_w8_packed_bytes(K, N, group_size)


def w8_pack(codes, scales, group_size, stream=None):
    """Repack 8-bit codes (uint8 [K][N], 0..255) and scales (float16 [ceil(K/G)][N]).

    Returns (packed uint8 codes, packed float16 scales)."""
    K, N = codes.shape
    assert codes.dtype == torch.uint8 and scales.dtype == torch.float16
    assert codes.is_cuda and scales.is_cuda and codes.is_contiguous() and scales.is_contiguous()
    nb, ns = w8_packed_bytes(K, N, group_size), scales_elems(K, N, group_size)
    if nb == 0 or ns == 0:
        raise W4A16Error(ERR_INVALID_ARG, "w8_pack")
    packed = torch.empty(nb, dtype=torch.uint8, device=codes.device)
    sp = torch.empty(ns, dtype=torch.float16, device=codes.device)
    _check(lib().w4a16_w8_pack(_ptr(codes), _ptr(scales), _ptr(packed), _ptr(sp), K, N, group_size,
                               _stream(stream)), "w4a16_w8_pack")
    return packed, sp


def w8_gemm(x, packed, scales_packed, N, group_size, bias=None, residual=None, activation="none", y=None,
            workspace=None, stream=None):
    """y = act(x @ dequant8(W) + bias) + residual, dequant8(W) = (q - 128) * s. Arguments as gemm_fused,
    with packed from w8_pack."""
    M, K = x.shape
    assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous()
    for t, shape in ((bias, (N,)), (residual, (M, N))):
        if t is not None:
            assert t.dtype == torch.float16 and t.is_cuda and t.is_contiguous() and tuple(t.shape) == shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check_buffers(x, packed, scales_packed, N, group_size, y, 'w8')
    _check(lib().w4a16_w8_gemm(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(y), M, N, K, group_size,
                               _ptr(bias), _ptr(residual), ACTIVATIONS[activation], _ptr(workspace), ws_bytes,
                               _stream(stream)), "w4a16_w8_gemm")
    return y


def bf16_gemm(x, packed, scales_packed, N, group_size, bias=None, residual=None, activation="none", y=None,
              workspace=None, stream=None):
    """y = act(x @ dequant(W) + bias) + residual with bfloat16 x, scales, bias, residual and y
    (4-bit codes, zero-point 8; packed and scales_packed from pack with bfloat16 scales)."""
    M, K = x.shape
    assert x.dtype == torch.bfloat16 and x.is_cuda and x.is_contiguous()
    assert scales_packed.dtype == torch.bfloat16
    for t, shape in ((bias, (N,)), (residual, (M, N))):
        if t is not None:
            assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous() and tuple(t.shape) == shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check_buffers(x, packed, scales_packed, N, group_size, y, 'int4')
    _check(lib().w4a16_bf16_gemm(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(y), M, N, K, group_size,
                                 _ptr(bias), _ptr(residual), ACTIVATIONS[activation], _ptr(workspace), ws_bytes,
                                 _stream(stream)), "w4a16_bf16_gemm")
    return y


def sp_packed_bytes(K, N, group_size):
    return lib().w4a16_sp_packed_bytes(K, N, group_size)


def sp_pack(codes, scales, group_size, stream=None, violations=None):
    """Repack 2:4 sparse codes (uint8 [K][N]: at most two codes other than 8 in every
    aligned group of four k) and scales (float16 [ceil(K/G)][N]).

    Returns (packed uint8, packed float16 scales). violations: an int64 CUDA tensor
    of one element to which the number of groups that are not 2:4 is added, or None."""
    K, N = codes.shape
    assert codes.dtype == torch.uint8 and scales.dtype == torch.float16
    assert codes.is_cuda and scales.is_cuda and codes.is_contiguous() and scales.is_contiguous()
    nb, ns = sp_packed_bytes(K, N, group_size), scales_elems(K, N, group_size)
    if nb == 0 or ns == 0:
        raise W4A16Error(ERR_INVALID_ARG, "sp_pack")
    if violations is not None:
        assert violations.dtype == torch.int64 and violations.is_cuda and violations.numel() == 1
    packed = torch.empty(nb, dtype=torch.uint8, device=codes.device)
    sp = torch.empty(ns, dtype=torch.float16, device=codes.device)
    _check(lib().w4a16_sp_pack(_ptr(codes), _ptr(scales), _ptr(packed), _ptr(sp), K, N, group_size,
                               _ptr(violations), _stream(stream)), "w4a16_sp_pack")
    return packed, sp


def sp_gemm(x, packed, scales_packed, N, group_size, bias=None, residual=None, activation="none", y=None,
            workspace=None, stream=None):
    """y = act(x @ dequant(W) + bias) + residual for 2:4 sparse codes packed by sp_pack.
    Arguments as gemm_fused."""
    M, K = x.shape
    assert x.dtype == torch.float16 and x.is_cuda and x.is_contiguous()
    for t, shape in ((bias, (N,)), (residual, (M, N))):
        if t is not None:
            assert t.dtype == torch.float16 and t.is_cuda and t.is_contiguous() and tuple(t.shape) == shape
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check_buffers(x, packed, scales_packed, N, group_size, y, 'sparse')
    _check(lib().w4a16_sp_gemm(_ptr(x), _ptr(packed), _ptr(scales_packed), _ptr(y), M, N, K, group_size,
                               _ptr(bias), _ptr(residual), ACTIVATIONS[activation], _ptr(workspace), ws_bytes,
                               _stream(stream)), "w4a16_sp_gemm")
    return y

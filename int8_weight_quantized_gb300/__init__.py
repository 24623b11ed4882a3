"""INT8 quantized linear layer for one NVIDIA GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/ck_int8.h`` (library ``lib/libck_int8.so``,
built by ``build.py``).  The functions have the C names and only marshal arguments:
they check dtypes/shapes, allocate outputs with torch when the caller passes none,
and hand raw device pointers plus the current CUDA stream to the library.  Every step
of the computation runs in the library's CUDA kernels; if the library is missing or
the device is not a GB300 the call raises -- there is no other implementation.
"""
import ctypes
import os

import torch

from . import build as _build

TENSORWISE, PER_ROW, CONVROT = 0, 1, 2
OUT_BF16, OUT_F16, OUT_F32 = 0, 1, 2
# output element type of the dequant epilogue, by torch dtype
OUT_DTYPES = {torch.bfloat16: OUT_BF16, torch.float16: OUT_F16, torch.float32: OUT_F32}
CK_OK, CK_ERR_INVALID_ARG, CK_ERR_UNSUPPORTED_DEVICE, CK_ERR_CUDA, CK_ERR_TIMEOUT = range(5)
STATUS_NAMES = {0: "CK_OK", 1: "CK_ERR_INVALID_ARG", 2: "CK_ERR_UNSUPPORTED_DEVICE", 3: "CK_ERR_CUDA",
                4: "CK_ERR_TIMEOUT"}

LIB_PATH = _build.LIB
_lib = None


class CkError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


def load_library(path=None):
    """Load libck_int8.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("libck_int8.so is not built (expected at %s); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
    L = ctypes.CDLL(path)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sig = {
        "ck_quantize_int8_rowwise": ([P, I64, I64, I, P, P, P], I),
        "ck_quantize_tensorwise_workspace_size": ([], SZ),
        "ck_quantize_int8_tensorwise": ([P, I64, I64, P, P, P, SZ, P], I),
        "ck_quantize_int8_tensorwise_noalloc": ([P, I64, I64, P, P, P], I),
        "ck_int8_linear_workspace_size": ([I64, I64, I64, I], SZ),
        "ck_int8_linear_workspace_views": ([I64, I64, I64, I, ctypes.POINTER(SZ), ctypes.POINTER(SZ)], I),
        "ck_int8_linear": ([P, P, P, P, P, P, I64, I64, I64, I, I, P, SZ, P], I),
        "ck_convrot_prepare_weight": ([P, I64, I64, P, P, P], I),
        "ck_int8_weight_codes": ([P, I64, I64, P, P], I),
        "ck_int8_linear_codes_workspace_size": ([I64, I64, I64, I], SZ),
        "ck_int8_linear_codes": ([P, P, P, P, P, P, I64, I64, I64, I, I, P, SZ, P], I),
        "ck_int8_linear_host_workspace_size": ([I64, I64, I64, I, I, I64], SZ),
        "ck_int8_linear_host": ([P, P, P, P, P, I64, I64, I64, I, I, I64, P, SZ, P], I),
        "ck_int8_gemm_workspace_size": ([I64, I64, I64], SZ),
        "ck_w8a16_linear_workspace_size": ([I64, I64, I64, I], SZ),
        "ck_w8a16_linear": ([P, P, P, P, P, P, I64, I64, I64, I, I, P, SZ, P], I),
        "ck_int8_gemm_dequant": ([P, P, P, P, P, P, P, I64, I64, I64, I, I, P, SZ, P], I),
        "ck_int8_gemm_s32": ([P, P, P, I64, I64, I64, P, SZ, P], I),
        "ck_profile_begin": ([I], I),
        "ck_profile_end": ([ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), I], I),
        "ck_last_error": ([], ctypes.c_char_p),
        "ck_device_error": ([I], I),
        "ck_gemm_tile_config": ([I64, I64, I64, P, P, P, P], I),
        "ck_selftest_wait_timeout": ([ctypes.c_uint64, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(status):
    if status != CK_OK:
        msg = load_library().ck_last_error()
        raise CkError(status, msg.decode() if msg else "")


def _ptr(t):
    # a plain int: the c_void_p argument types convert it (0 / None is NULL)
    return None if t is None else t.data_ptr()


# The current stream's handle without building a torch Stream object (that costs ~3 us a
# call, as much as a kernel launch); the public route where the fast one is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream):
    if stream is None:
        if _raw_stream is not None and _cur_device is not None:
            return _raw_stream(_cur_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _req(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.shape != shape:
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)


_workspaces = {}


def workspace(nbytes, device=None):
    """A cached uint8 device buffer of at least nbytes (one per device)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    buf = _workspaces.get(device)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _workspaces[device] = buf
    return buf


def ck_quantize_int8_rowwise(x, rotate=False, q=None, x_scale=None, stream=None):
    """Per-row quantize of bf16 x [M,K]; returns (q int8 [M,K], x_scale fp32 [M])."""
    M, K = x.shape
    _req(x, torch.bfloat16, (M, K), "x")
    q = torch.empty((M, K), dtype=torch.int8, device=x.device) if q is None else q
    x_scale = torch.empty((M,), dtype=torch.float32, device=x.device) if x_scale is None else x_scale
    _req(q, torch.int8, (M, K), "q")
    _req(x_scale, torch.float32, (M,), "x_scale")
    _check(load_library().ck_quantize_int8_rowwise(_ptr(x), M, K, int(bool(rotate)), _ptr(q), _ptr(x_scale),
                                                   _stream(stream)))
    return q, x_scale


def ck_quantize_int8_tensorwise(x, q=None, x_scale=None, ws=None, stream=None):
    """Tensorwise quantize of bf16 x [M,K]; returns (q int8 [M,K], x_scale fp32 [1])."""
    M, K = x.shape
    _req(x, torch.bfloat16, (M, K), "x")
    q = torch.empty((M, K), dtype=torch.int8, device=x.device) if q is None else q
    x_scale = torch.empty((1,), dtype=torch.float32, device=x.device) if x_scale is None else x_scale
    _req(q, torch.int8, (M, K), "q")
    _req(x_scale, torch.float32, (1,), "x_scale")
    L = load_library()
    if ws is None:
        ws = workspace(L.ck_quantize_tensorwise_workspace_size(), x.device)
    _check(L.ck_quantize_int8_tensorwise(_ptr(x), M, K, _ptr(q), _ptr(x_scale), _ptr(ws), ws.numel(),
                                         _stream(stream)))
    return q, x_scale


def ck_quantize_int8_tensorwise_noalloc(x, q, x_scale, stream=None):
    """Tensorwise quantize into caller-provided q int8 [M,K] and x_scale fp32 [1]; the
    library allocates nothing (its partial maxima live in a fixed built-in array)."""
    M, K = x.shape
    _req(x, torch.bfloat16, (M, K), "x")
    _req(q, torch.int8, (M, K), "q")
    _req(x_scale, torch.float32, (1,), "x_scale")
    _check(load_library().ck_quantize_int8_tensorwise_noalloc(_ptr(x), M, K, _ptr(q), _ptr(x_scale),
                                                              _stream(stream)))
    return q, x_scale


def ck_int8_linear_workspace_size(M, N, K, mode):
    return load_library().ck_int8_linear_workspace_size(M, N, K, int(mode))


def ck_int8_linear_workspace_views(M, N, K, mode):
    """(codes_offset, x_scale_offset): byte offsets in ck_int8_linear's workspace of the
    activation codes (bf16 integers [M,K]) and x_scale (fp32 [M], or [1] in tensorwise
    mode) left by the last call."""
    codes, xs = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().ck_int8_linear_workspace_views(M, N, K, int(mode), ctypes.byref(codes), ctypes.byref(xs)))
    return codes.value, xs.value


def linear_workspace_codes(ws, M, N, K, mode):
    """Views into a ck_int8_linear workspace (a uint8 device tensor): the activation codes
    as bf16 [M,K] and x_scale fp32 [M] or [1], as the layer's last call left them."""
    co, xo = ck_int8_linear_workspace_views(M, N, K, mode)
    codes = ws[co:co + 2 * M * K].view(torch.bfloat16).view(M, K)
    n = 1 if mode == TENSORWISE else M
    x_scale = ws[xo:xo + 4 * n].view(torch.float32)
    return codes, x_scale


def _out_code(out_dtype):
    if out_dtype not in OUT_DTYPES:
        raise ValueError("out_dtype must be torch.bfloat16, torch.float16 or torch.float32, got %s" % (out_dtype,))
    return OUT_DTYPES[out_dtype]


def _residual(residual, out_dtype, M, N):
    if residual is not None:
        _req(residual, out_dtype, (M, N), "residual")
    return residual


def ck_int8_linear(x, w, w_scale, bias=None, mode=PER_ROW, y=None, ws=None, stream=None, out_dtype=torch.bfloat16,
                   residual=None):
    """y [M,N] of out_dtype = dequant(int32 GEMM(quantize(x [@ H]), w)) (+ bias) (+ residual);
    residual has y's type and shape and may be y itself."""
    code = _out_code(out_dtype)
    M, K = x.shape
    N = w.shape[0]
    _req(x, torch.bfloat16, (M, K), "x")
    _req(w, torch.int8, (N, K), "w")
    _req(w_scale, torch.float32, (1,) if mode == TENSORWISE else (N,), "w_scale")
    if bias is not None:
        _req(bias, torch.bfloat16, (N,), "bias")
    y = torch.empty((M, N), dtype=out_dtype, device=x.device) if y is None else y
    _req(y, out_dtype, (M, N), "y")
    L = load_library()
    if ws is None:  # a workspace the caller gives is checked for size by the library
        ws = workspace(L.ck_int8_linear_workspace_size(M, N, K, int(mode)), x.device)
    _residual(residual, out_dtype, M, N)
    _check(L.ck_int8_linear(_ptr(x), _ptr(w), _ptr(w_scale), _ptr(bias), _ptr(residual), _ptr(y), M, N, K, int(mode),
                            code, _ptr(ws), ws.numel(), _stream(stream)))
    return y


def ck_int8_weight_codes(w, w_codes=None, stream=None):
    """The weight's GEMM operand, once per layer: int8 w [N,K] -> bf16 codes [N,K]."""
    N, K = w.shape
    _req(w, torch.int8, (N, K), "w")
    w_codes = torch.empty((N, K), dtype=torch.bfloat16, device=w.device) if w_codes is None else w_codes
    _req(w_codes, torch.bfloat16, (N, K), "w_codes")
    _check(load_library().ck_int8_weight_codes(_ptr(w), N, K, _ptr(w_codes), _stream(stream)))
    return w_codes


def ck_int8_linear_codes(x, w_codes, w_scale, bias=None, mode=PER_ROW, y=None, ws=None, stream=None,
                         out_dtype=torch.bfloat16, residual=None):
    """ck_int8_linear with the weight given as its bf16 codes (from ck_int8_weight_codes)."""
    code = _out_code(out_dtype)
    M, K = x.shape
    N = w_codes.shape[0]
    _req(x, torch.bfloat16, (M, K), "x")
    _req(w_codes, torch.bfloat16, (N, K), "w_codes")
    _req(w_scale, torch.float32, (1,) if mode == TENSORWISE else (N,), "w_scale")
    if bias is not None:
        _req(bias, torch.bfloat16, (N,), "bias")
    y = torch.empty((M, N), dtype=out_dtype, device=x.device) if y is None else y
    _req(y, out_dtype, (M, N), "y")
    L = load_library()
    if ws is None:
        ws = workspace(L.ck_int8_linear_codes_workspace_size(M, N, K, int(mode)), x.device)
    _residual(residual, out_dtype, M, N)
    _check(L.ck_int8_linear_codes(_ptr(x), _ptr(w_codes), _ptr(w_scale), _ptr(bias), _ptr(residual), _ptr(y), M, N,
                                  K, int(mode), code, _ptr(ws), ws.numel(), _stream(stream)))
    return y


def ck_int8_linear_host(x, w, w_scale, bias=None, mode=PER_ROW, y=None, ws=None, stream=None,
                        out_dtype=torch.bfloat16, slab_rows=0):
    """The layer on a HOST activation x bf16 [M,K] (pinned for overlapped copies) into a
    host output y [M,N] of out_dtype; w, w_scale, bias on the device.  The copies and the
    kernels are pipelined over row slabs; y is complete when `stream` has completed."""
    code = _out_code(out_dtype)
    M, K = x.shape
    N = w.shape[0]
    if x.dtype != torch.bfloat16 or x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 host tensor")
    _req(w, torch.int8, (N, K), "w")
    _req(w_scale, torch.float32, (1,) if mode == TENSORWISE else (N,), "w_scale")
    if bias is not None:
        _req(bias, torch.bfloat16, (N,), "bias")
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, pin_memory=x.is_pinned())
    if y.dtype != out_dtype or tuple(y.shape) != (M, N) or y.is_cuda or not y.is_contiguous():
        raise ValueError("y must be a contiguous host tensor of shape %s and type %s" % ((M, N), out_dtype))
    L = load_library()
    if ws is None:
        ws = workspace(L.ck_int8_linear_host_workspace_size(M, N, K, int(mode), code, int(slab_rows)), w.device)
    _check(L.ck_int8_linear_host(_ptr(x), _ptr(w), _ptr(w_scale), _ptr(bias), _ptr(y), M, N, K, int(mode), code,
                                 int(slab_rows), _ptr(ws), ws.numel(), _stream(stream)))
    return y


def ck_w8a16_linear(x, w, w_scale, bias=None, mode=PER_ROW, y=None, ws=None, stream=None, out_dtype=torch.bfloat16,
                    residual=None):
    """y [M,N] of out_dtype = (bf16 x [@ H]) . (int8 w)^T summed in fp32, * w_scale (+ bias) (+ residual)."""
    code = _out_code(out_dtype)
    M, K = x.shape
    N = w.shape[0]
    _req(x, torch.bfloat16, (M, K), "x")
    _req(w, torch.int8, (N, K), "w")
    _req(w_scale, torch.float32, (1,) if mode == TENSORWISE else (N,), "w_scale")
    if bias is not None:
        _req(bias, torch.bfloat16, (N,), "bias")
    y = torch.empty((M, N), dtype=out_dtype, device=x.device) if y is None else y
    _req(y, out_dtype, (M, N), "y")
    L = load_library()
    if ws is None:
        ws = workspace(L.ck_w8a16_linear_workspace_size(M, N, K, int(mode)), x.device)
    _residual(residual, out_dtype, M, N)
    _check(L.ck_w8a16_linear(_ptr(x), _ptr(w), _ptr(w_scale), _ptr(bias), _ptr(residual), _ptr(y), M, N, K,
                             int(mode), code, _ptr(ws), ws.numel(), _stream(stream)))
    return y


def ck_convrot_prepare_weight(W, w=None, w_scale=None, stream=None):
    """ConvRot weight: fp32 W [N,K] -> (int8 codes of W @ H^T [N,K], fp32 row scales [N])."""
    N, K = W.shape
    _req(W, torch.float32, (N, K), "W")
    w = torch.empty((N, K), dtype=torch.int8, device=W.device) if w is None else w
    w_scale = torch.empty((N,), dtype=torch.float32, device=W.device) if w_scale is None else w_scale
    _req(w, torch.int8, (N, K), "w")
    _req(w_scale, torch.float32, (N,), "w_scale")
    _check(load_library().ck_convrot_prepare_weight(_ptr(W), N, K, _ptr(w), _ptr(w_scale), _stream(stream)))
    return w, w_scale


def ck_int8_gemm_dequant(q, x_scale, w, w_scale, bias=None, scalar_scales=False, y=None, ws=None, stream=None,
                         out_dtype=torch.bfloat16, residual=None):
    """GEMM + fused dequant on pre-quantized q int8 [M,K]; returns y [M,N] of out_dtype."""
    code = _out_code(out_dtype)
    M, K = q.shape
    N = w.shape[0]
    _req(q, torch.int8, (M, K), "q")
    _req(w, torch.int8, (N, K), "w")
    _req(x_scale, torch.float32, (1,) if scalar_scales else (M,), "x_scale")
    _req(w_scale, torch.float32, (1,) if scalar_scales else (N,), "w_scale")
    if bias is not None:
        _req(bias, torch.bfloat16, (N,), "bias")
    y = torch.empty((M, N), dtype=out_dtype, device=q.device) if y is None else y
    _req(y, out_dtype, (M, N), "y")
    L = load_library()
    if ws is None:
        ws = workspace(L.ck_int8_gemm_workspace_size(M, N, K), q.device)
    _residual(residual, out_dtype, M, N)
    _check(L.ck_int8_gemm_dequant(_ptr(q), _ptr(x_scale), _ptr(w), _ptr(w_scale), _ptr(bias), _ptr(residual), _ptr(y),
                                  M, N, K, int(bool(scalar_scales)), code, _ptr(ws), ws.numel(), _stream(stream)))
    return y


def ck_int8_gemm_s32(q, w, acc=None, ws=None, stream=None):
    """Raw exact int32 accumulators acc [M,N] = q [M,K] . w [N,K]^T."""
    M, K = q.shape
    N = w.shape[0]
    _req(q, torch.int8, (M, K), "q")
    _req(w, torch.int8, (N, K), "w")
    acc = torch.empty((M, N), dtype=torch.int32, device=q.device) if acc is None else acc
    _req(acc, torch.int32, (M, N), "acc")
    L = load_library()
    if ws is None:
        ws = workspace(L.ck_int8_gemm_workspace_size(M, N, K), q.device)
    _check(L.ck_int8_gemm_s32(_ptr(q), _ptr(w), _ptr(acc), M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    return acc


def ck_last_error():
    msg = load_library().ck_last_error()
    return msg.decode() if msg else ""


def ck_gemm_tile_config(M, N, K):
    """(bn, cta_pair, resident_units, k_split) of the GEMM launch for an M x N x K problem."""
    bn, pair, res, split = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64(), ctypes.c_int()
    _check(load_library().ck_gemm_tile_config(M, N, K, ctypes.byref(bn), ctypes.byref(pair), ctypes.byref(res),
                                              ctypes.byref(split)))
    return bn.value, bool(pair.value), res.value, split.value


def ck_device_error(clear=True):
    return load_library().ck_device_error(int(bool(clear)))


def ck_selftest_wait_timeout(timeout_ns=1_000_000, stream=None):
    """Returns the status code of the bounded-wait self-test (CK_ERR_TIMEOUT expected)."""
    return load_library().ck_selftest_wait_timeout(int(timeout_ns), _stream(stream))


PROFILE_KINDS = ("quantize", "widen", "gemm")


def ck_profile_begin(with_events=True):
    _check(load_library().ck_profile_begin(int(bool(with_events))))


def ck_profile_end():
    """Returns {kind: (device_ms, launches)} for the launches since ck_profile_begin()."""
    n = len(PROFILE_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _check(load_library().ck_profile_end(ms, cnt, n))
    return {k: (ms[i], cnt[i]) for i, k in enumerate(PROFILE_KINDS)}

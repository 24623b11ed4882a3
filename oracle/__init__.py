"""CPU oracle for the INT8 quantized linear layer -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and the cpu_baseline / reference leg of
bench.py may import this package.  The product path (the CUDA library and its
Python binding) never does; it shares no code with it.

The arithmetic lives in ``ck_oracle.c`` (plain C); this module only marshals numpy
arrays into it.  bf16 tensors travel as ``uint16`` bit patterns.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.ck_oracle_quantize_rowwise.argtypes = [P, I64, I64, ctypes.c_int, P, P]
        L.ck_oracle_quantize_rowwise.restype = ctypes.c_int
        L.ck_oracle_quantize_tensorwise.argtypes = [P, I64, I64, P, P]
        L.ck_oracle_quantize_tensorwise.restype = ctypes.c_int
        L.ck_oracle_gemm_s32.argtypes = [P, P, P, I64, I64, I64]
        L.ck_oracle_gemm_s32.restype = ctypes.c_int
        L.ck_oracle_dequant.argtypes = [P, P, P, P, ctypes.c_int, I64, I64, P]
        L.ck_oracle_dequant.restype = None
        L.ck_oracle_dequant_typed.argtypes = [P, P, P, P, ctypes.c_int, I64, I64, ctypes.c_int, P]
        L.ck_oracle_dequant_typed.restype = None
        L.ck_oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.ck_oracle_f32_to_f16.restype = ctypes.c_uint16
        L.ck_oracle_int8_linear.argtypes = [P, P, P, P, I64, I64, I64, ctypes.c_int, P, P, P, P]
        L.ck_oracle_int8_linear.restype = ctypes.c_int
        L.ck_oracle_fwht128.argtypes = [P]
        L.ck_oracle_fwht128.restype = None
        L.ck_oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.ck_oracle_bf16_to_f32.restype = ctypes.c_float
        L.ck_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.ck_oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.ck_oracle_prepare_convrot_weight.argtypes = [P, I64, I64, P, P]
        L.ck_oracle_prepare_convrot_weight.restype = ctypes.c_int
        L.ck_oracle_w8a16_linear.argtypes = [P, P, P, P, I64, I64, I64, ctypes.c_int, P, P]
        L.ck_oracle_w8a16_linear.restype = ctypes.c_int
        L.ck_oracle_dequant_residual.argtypes = [P, P, P, P, P, ctypes.c_int, I64, I64, ctypes.c_int, P]
        L.ck_oracle_dequant_residual.restype = None
        L.ck_oracle_num_threads.argtypes = []
        L.ck_oracle_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s, got %s" % (dtype, a.dtype))
    return a


TENSORWISE, PER_ROW, CONVROT = 0, 1, 2


def num_threads():
    return lib().ck_oracle_num_threads()


def bf16_to_f32(bits):
    """bf16 bit patterns (uint16) -> float32, via the oracle's own conversion."""
    bits = _c(bits, np.uint16)
    f = np.empty(bits.shape, np.float32)
    flat, out = bits.reshape(-1), f.reshape(-1)
    L = lib()
    for i in range(flat.size):
        out[i] = L.ck_oracle_bf16_to_f32(int(flat[i]))
    return f


def f32_to_bf16(vals):
    """float32 -> bf16 bits with the oracle's round-to-nearest-even."""
    vals = _c(vals, np.float32)
    out = np.empty(vals.shape, np.uint16)
    L = lib()
    for i, v in enumerate(vals.reshape(-1)):
        out.reshape(-1)[i] = L.ck_oracle_f32_to_bf16(float(v))
    return out


def fwht128(v):
    """x @ H for one 128-block (fp32), H the normalized Sylvester Hadamard matrix."""
    v = np.array(v, dtype=np.float32, copy=True)
    if v.shape != (128,):
        raise ValueError("fwht128 takes a 128-vector")
    lib().ck_oracle_fwht128(_p(v))
    return v


def quantize_rowwise(x_bits, rotate=False):
    """Per-row quantize: returns (q int8 [M,K], x_scale fp32 [M])."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    xs = np.empty((M,), np.float32)
    rc = lib().ck_oracle_quantize_rowwise(_p(x), M, K, int(bool(rotate)), _p(q), _p(xs))
    if rc != 0:
        raise ValueError("oracle quantize_rowwise rejected the arguments (rc=%d)" % rc)
    return q, xs


def quantize_tensorwise(x_bits):
    """Tensorwise quantize: returns (q int8 [M,K], x_scale fp32 [1])."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    xs = np.empty((1,), np.float32)
    rc = lib().ck_oracle_quantize_tensorwise(_p(x), M, K, _p(q), _p(xs))
    if rc != 0:
        raise ValueError("oracle quantize_tensorwise rejected the arguments (rc=%d)" % rc)
    return q, xs


def gemm_s32(q, w):
    """Exact int32 accumulators acc[m,n] = sum_k q[m,k] w[n,k]."""
    q = _c(q, np.int8)
    w = _c(w, np.int8)
    M, K = q.shape
    N, K2 = w.shape
    if K != K2:
        raise ValueError("K mismatch")
    acc = np.empty((M, N), np.int32)
    rc = lib().ck_oracle_gemm_s32(_p(q), _p(w), _p(acc), M, N, K)
    if rc != 0:
        raise ValueError("oracle gemm_s32 failed (rc=%d)" % rc)
    return acc


def dequant(acc, xs, ws, bias_bits=None, scalar_scales=False):
    """fp32 epilogue -> bf16 bits [M,N]."""
    acc = _c(acc, np.int32)
    xs = _c(xs, np.float32)
    ws = _c(ws, np.float32)
    b = None if bias_bits is None else _c(bias_bits, np.uint16)
    M, N = acc.shape
    y = np.empty((M, N), np.uint16)
    lib().ck_oracle_dequant(_p(acc), _p(xs), _p(ws), _p(b), int(bool(scalar_scales)), M, N, _p(y))
    return y


OUT_BF16, OUT_F16, OUT_F32 = 0, 1, 2


def f32_to_f16(vals):
    """float32 -> IEEE half bits with the oracle's round-to-nearest-even."""
    vals = _c(vals, np.float32)
    out = np.empty(vals.shape, np.uint16)
    L = lib()
    for i, v in enumerate(vals.reshape(-1)):
        out.reshape(-1)[i] = L.ck_oracle_f32_to_f16(float(v))
    return out


def dequant_typed(acc, xs, ws, bias_bits=None, scalar_scales=False, out_dtype=OUT_BF16):
    """fp32 epilogue -> bf16 bits / fp16 bits (uint16) or fp32 values [M,N]."""
    acc = _c(acc, np.int32)
    xs = _c(xs, np.float32)
    ws = _c(ws, np.float32)
    b = None if bias_bits is None else _c(bias_bits, np.uint16)
    M, N = acc.shape
    y = np.empty((M, N), np.float32 if out_dtype == OUT_F32 else np.uint16)
    lib().ck_oracle_dequant_typed(_p(acc), _p(xs), _p(ws), _p(b), int(bool(scalar_scales)), M, N, int(out_dtype),
                                  _p(y))
    return y


def dequant_residual(acc, xs, ws, residual, bias_bits=None, scalar_scales=False, out_dtype=OUT_BF16):
    """Epilogue with a residual: residual is float32 [M,N] (values of the output-type
    tensor, converted exactly); returns bf16 / fp16 bits or fp32 values [M,N]."""
    acc = _c(acc, np.int32)
    xs = _c(xs, np.float32)
    ws = _c(ws, np.float32)
    r = _c(residual, np.float32)
    b = None if bias_bits is None else _c(bias_bits, np.uint16)
    M, N = acc.shape
    y = np.empty((M, N), np.float32 if out_dtype == OUT_F32 else np.uint16)
    lib().ck_oracle_dequant_residual(_p(acc), _p(xs), _p(ws), _p(b), _p(r), int(bool(scalar_scales)), M, N,
                                     int(out_dtype), _p(y))
    return y


def int8_linear(x_bits, w, ws, bias_bits=None, mode=PER_ROW, out_dtype=OUT_BF16):
    """Whole layer; returns dict(y=bf16 bits [M,N], q, xs, acc)."""
    x = _c(x_bits, np.uint16)
    w = _c(w, np.int8)
    ws = _c(ws, np.float32)
    b = None if bias_bits is None else _c(bias_bits, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    y = np.empty((M, N), np.uint16)
    q = np.empty((M, K), np.int8)
    xs = np.empty((1 if mode == TENSORWISE else M,), np.float32)
    acc = np.empty((M, N), np.int32)
    rc = lib().ck_oracle_int8_linear(_p(x), _p(w), _p(ws), _p(b), M, N, K, int(mode),
                                     _p(y), _p(q), _p(xs), _p(acc))
    if rc != 0:
        raise ValueError("oracle int8_linear failed (rc=%d)" % rc)
    if out_dtype != OUT_BF16:
        y = dequant_typed(acc, xs, ws, b, scalar_scales=(mode == TENSORWISE), out_dtype=out_dtype)
    return {"y": y, "q": q, "xs": xs, "acc": acc}


def prepare_convrot_weight(W):
    """ConvRot weight: W fp32 [N,K] -> (w int8 [N,K] of W @ H^T, w_scale fp32 [N])."""
    W = _c(W, np.float32)
    N, K = W.shape
    w = np.empty((N, K), np.int8)
    ws = np.empty((N,), np.float32)
    rc = lib().ck_oracle_prepare_convrot_weight(_p(W), N, K, _p(w), _p(ws))
    if rc != 0:
        raise ValueError("oracle prepare_convrot_weight rejected the arguments (rc=%d)" % rc)
    return w, ws


def w8a16_linear(x_bits, w, ws, bias_bits=None, mode=PER_ROW):
    """16-bit-activation path: (y, mag), both float64 [M,N]; y before output rounding,
    mag = |w_scale| * sum |a * w| (bounds any fp32 evaluation's rounding error)."""
    x = _c(x_bits, np.uint16)
    w = _c(w, np.int8)
    ws = _c(ws, np.float32)
    b = None if bias_bits is None else _c(bias_bits, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    y = np.empty((M, N), np.float64)
    mag = np.empty((M, N), np.float64)
    rc = lib().ck_oracle_w8a16_linear(_p(x), _p(w), _p(ws), _p(b), M, N, K, int(mode), _p(y), _p(mag))
    if rc != 0:
        raise ValueError("oracle w8a16_linear rejected the arguments (rc=%d)" % rc)
    return y, mag

"""The tensorwise quantize entry point that allocates nothing.

It serves callers that cannot allocate device memory (for example code running under
CUDA graph capture, or a real-time loop with a fixed memory budget): they pass inputs
and outputs only, and the library keeps its partial maxima in a fixed array built into
the module.  These tests call it through the C ABI and compare it with the allocating
entry point, ck_quantize_int8_tensorwise, which must give the identical int8 codes and
scale (the tolerance of every quantize test here: bit-exact).  The file is collected
last so that a failure here cannot hide any other test's result.
"""
import ctypes

import pytest
import torch

import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda"


def call_noalloc(x, q, x_scale):
    L = ck.load_library()
    M, K = x.shape
    P = ctypes.c_void_p
    return L.ck_quantize_int8_tensorwise_noalloc(P(x.data_ptr()), M, K, P(q.data_ptr()), P(x_scale.data_ptr()),
                                                 P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_the_allocating_entry_point_on_two_calls_in_a_row():
    # the first call fills 512 partial maxima, the second only 17: stale slots of the
    # shared array must not leak into the second result
    for (M, K), seed in (((4096, 4096), 41), ((333, 1040), 42)):
        x = synthetic.normal_bf16((M, K), seed, device=DEV)
        q_ref, s_ref = ck.ck_quantize_int8_tensorwise(x)
        q = torch.empty((M, K), dtype=torch.int8, device=DEV)
        s = torch.empty((1,), dtype=torch.float32, device=DEV)
        st = call_noalloc(x, q, s)
        assert st == ck.CK_OK, ck.ck_last_error()
        torch.cuda.synchronize()
        assert torch.equal(s, s_ref)
        assert torch.equal(q, q_ref)
    assert ck.ck_device_error(clear=False) == 0


def test_noalloc_rejects_tensors_beyond_its_fixed_scratch():
    x = torch.zeros((16, 4096), dtype=torch.bfloat16, device=DEV)
    q = torch.zeros((16, 4096), dtype=torch.int8, device=DEV)
    s = torch.zeros((1,), dtype=torch.float32, device=DEV)
    L = ck.load_library()
    P = ctypes.c_void_p
    # 32769 x 4096 = 134,221,824 values > 134,217,728: rejected before any launch
    st = L.ck_quantize_int8_tensorwise_noalloc(P(x.data_ptr()), 32769, 4096, P(q.data_ptr()), P(s.data_ptr()),
                                               P(torch.cuda.current_stream().cuda_stream))
    assert st == ck.CK_ERR_INVALID_ARG
    assert "no-allocation limit" in ck.ck_last_error()
    # the same buffers at their real size (well inside the limit) are accepted
    assert call_noalloc(x, q, s) == ck.CK_OK
    torch.cuda.synchronize()

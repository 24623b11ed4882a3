"""The tensorwise quantize entry point that allocates nothing.

Some callers may not touch an allocator while they run: real-time loops that reserve
their whole device-memory budget up front, hosts whose own memory manager must account
for every byte on the GPU, and plugins inside such hosts, which see only the buffers they
are handed.  ck_quantize_int8_tensorwise_noalloc serves them: they pass inputs and
outputs only, and the library keeps its partial maxima in a fixed array built into the
module.  These tests call it through the C ABI on two calls in a row and compare its
int8 codes and scale with the allocating entry point, ck_quantize_int8_tensorwise, and
with the CPU oracle: bit-exact, the tolerance of every quantize test here.  The file is
collected last so that a failure here cannot hide any other test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
from helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
VALUES_PER_PARTIAL = 4096 * 8  # input values behind one partial maximum of the built-in array


def call_noalloc(x, q, x_scale):
    L = ck.load_library()
    M, K = x.shape
    P = ctypes.c_void_p
    return L.ck_quantize_int8_tensorwise_noalloc(P(x.data_ptr()), M, K, P(q.data_ptr()), P(x_scale.data_ptr()),
                                                 P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_the_allocating_entry_point_on_two_calls_in_a_row():
    # the first call fills 512 partial maxima of the shared array, the second only
    # ceil(333 * 1040 / 32768) = 11 of them, with a smaller maximum: the first call's
    # slots left behind must not leak into the second result
    shapes = [((4096, 4096), 41, 4.0), ((333, 1040), 42, 0.5)]
    parts = [-(-M * K // VALUES_PER_PARTIAL) for (M, K), _, _ in shapes]
    assert parts == [512, 11]
    for (M, K), seed, gain in shapes:
        x = (synthetic.normal_bf16((M, K), seed).float() * gain).to(torch.bfloat16)
        q_ora, s_ora = oracle.quantize_tensorwise(bits(x))
        xd = x.to(DEV)
        q_ref, s_ref = ck.ck_quantize_int8_tensorwise(xd)
        q = torch.full((M, K), -128, dtype=torch.int8, device=DEV)  # a code the clamp never writes
        s = torch.full((1,), float("nan"), dtype=torch.float32, device=DEV)
        st = call_noalloc(xd, q, s)
        assert st == ck.CK_OK, ck.ck_last_error()
        torch.cuda.synchronize()
        assert torch.equal(s, s_ref)
        assert torch.equal(q, q_ref)
        assert s.cpu().numpy().view(np.uint32)[0] == s_ora.view(np.uint32)[0]
        assert np.array_equal(q.cpu().numpy(), q_ora)
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
    assert float(s[0]) == 0.0 and int(q.abs().max()) == 0

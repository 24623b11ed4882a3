"""Failure detection on the GPU without faulting it: a bounded wait that nothing will
complete gives up and reports CK_ERR_TIMEOUT, the context stays usable, and bad
arguments on real buffers come back as statuses, not faults."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_wait_timeout_is_reported_and_context_survives():
    assert ck.ck_device_error(clear=True) == 0
    st = ck.ck_selftest_wait_timeout(timeout_ns=2_000_000)  # 2 ms
    assert st == ck.CK_ERR_TIMEOUT, ck.ck_last_error()
    assert ck.ck_device_error(clear=True) == 0  # the self-test cleared its own bit
    # the context is still usable: a normal GEMM afterwards is exact
    q = synthetic.int8_uniform((128, 64), seed=1)
    w = synthetic.int8_uniform((256, 64), seed=2)
    acc = ck.ck_int8_gemm_s32(q.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), oracle.gemm_s32(q.numpy(), w.numpy()))
    assert ck.ck_device_error(clear=False) == 0


def test_bad_arguments_on_real_buffers():
    L = ck.load_library()
    x = torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((16, 64), dtype=torch.int8, device=DEV)
    ws = torch.zeros((16,), dtype=torch.float32, device=DEV)
    y = torch.zeros((16, 16), dtype=torch.bfloat16, device=DEV)
    work = torch.zeros((1 << 20,), dtype=torch.uint8, device=DEV)
    P = ctypes.c_void_p
    stream = P(torch.cuda.current_stream().cuda_stream)
    # misaligned activation pointer
    st = L.ck_int8_linear(P(x.data_ptr() + 2), P(w.data_ptr()), P(ws.data_ptr()), None, None, P(y.data_ptr()), 16, 16, 64,
                          1, 0, P(work.data_ptr()), work.numel(), stream)
    assert st == ck.CK_ERR_INVALID_ARG and "aligned" in ck.ck_last_error()
    # workspace too small
    st = L.ck_int8_linear(P(x.data_ptr()), P(w.data_ptr()), P(ws.data_ptr()), None, None, P(y.data_ptr()), 16, 16, 64,
                          1, 0, P(work.data_ptr()), 64, stream)
    assert st == ck.CK_ERR_INVALID_ARG and "workspace" in ck.ck_last_error()
    torch.cuda.synchronize()
    assert ck.ck_device_error(clear=False) == 0


def test_device_is_a_gb300():
    major, minor = torch.cuda.get_device_capability()
    assert (major, minor) == (10, 3)

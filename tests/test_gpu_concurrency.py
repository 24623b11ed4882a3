"""Layers on several streams at once: each call's result equals the same call run alone.
The tensorwise layer's single preparation launch has its blocks exchange maxima, so all of
its blocks must be resident together; it is launched cooperatively, which the runtime
only starts when they can be, also while another stream's kernels hold part of the GPU."""
import numpy as np
import pytest
import torch

import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic

from helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("modes", [(ck.TENSORWISE, ck.TENSORWISE), (ck.TENSORWISE, ck.PER_ROW)])
def test_layers_on_concurrent_streams(modes):
    M, N, K = 2048, 2048, 2048
    calls = []
    for j, mode in enumerate(modes):
        x = synthetic.normal_bf16((M, K), 90 + j).to(DEV)
        w = synthetic.int8_uniform((N, K), 92 + j).to(DEV)
        ws = synthetic.scale_uniform(1 if mode == ck.TENSORWISE else N, 94 + j, mul=0.01).to(DEV)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
        work = ck.workspace(ck.ck_int8_linear_workspace_size(M, N, K, mode))
        ref = bits(ck.ck_int8_linear(x, w, ws, None, mode=mode))
        calls.append((x, w, ws, y, work, mode, ref, torch.cuda.Stream()))
    torch.cuda.synchronize()
    for rep in range(20):
        for x, w, ws, y, work, mode, ref, s in calls:
            with torch.cuda.stream(s):
                ck.ck_int8_linear(x, w, ws, None, mode=mode, y=y, ws=work)
        torch.cuda.synchronize()
        for x, w, ws, y, work, mode, ref, s in calls:
            assert np.array_equal(bits(y), ref), "rep %d mode %d differs from the call run alone" % (rep, mode)
    assert ck.ck_device_error(clear=True) == 0

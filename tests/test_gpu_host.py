"""ck_int8_linear_host: the layer on host memory, pipelined over row slabs (the copy of
the next slab in, the kernels of this one, the copy of the previous one out, on three
streams).  Its output must equal the device-memory layer's bit for bit, whatever the
slab size, mode, output type or kind of host memory, and the oracle's (0 ulp)."""
import numpy as np
import pytest
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
from helpers import bits, out_bits, ulp_distance, MAX_ULP

pytestmark = pytest.mark.gpu
DEV = "cuda"


def layer_inputs(M, N, K, mode, seed):
    x = synthetic.normal_bf16((M, K), seed)
    if mode == synthetic.CONVROT:
        w, ws = oracle.prepare_convrot_weight(synthetic.normal_f32((N, K), seed + 1, std=0.02).numpy())
        w, ws = torch.from_numpy(w), torch.from_numpy(ws)
    else:
        w = synthetic.int8_uniform((N, K), seed + 1)
        ws = synthetic.scale_uniform(1 if mode == synthetic.TENSORWISE else N, seed + 2)
    b = synthetic.normal_bf16((1, N), seed + 3, std=0.5).reshape(N)
    return x, w, ws, b


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("slab_rows", [0, 128, 300])
@pytest.mark.parametrize("mode", [synthetic.TENSORWISE, synthetic.PER_ROW, synthetic.CONVROT])
def test_host_layer_equals_device_layer(mode, slab_rows, pinned):
    M, N, K = 1000, 264, 1152  # 8, 4 or 1 slabs, a ragged last one
    x, w, ws, b = layer_inputs(M, N, K, mode, seed=500 + mode)
    wd, wsd, bd = w.to(DEV), ws.to(DEV), b.to(DEV)
    ref = bits(ck.ck_int8_linear(x.to(DEV), wd, wsd, bd, mode=mode))
    xh = x.pin_memory() if pinned else x.clone()
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, pin_memory=pinned)
    ck.ck_int8_linear_host(xh, wd, wsd, bd, mode=mode, y=y, slab_rows=slab_rows)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y), ref)
    want = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=mode)["y"]
    assert ulp_distance(bits(y), want).max() <= MAX_ULP


@pytest.mark.parametrize("out_dtype,code", [(torch.float32, oracle.OUT_F32), (torch.float16, oracle.OUT_F16)])
def test_host_layer_output_types(out_dtype, code):
    M, N, K = 700, 520, 1024
    x, w, ws, b = layer_inputs(M, N, K, synthetic.PER_ROW, seed=520)
    y = ck.ck_int8_linear_host(x.pin_memory(), w.to(DEV), ws.to(DEV), b.to(DEV), mode=synthetic.PER_ROW,
                               out_dtype=out_dtype, slab_rows=256)
    torch.cuda.synchronize()
    want = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=synthetic.PER_ROW, out_dtype=code)["y"]
    if code == oracle.OUT_F32:
        want = want.view(np.uint32)
    assert ulp_distance(out_bits(y), want).max() <= MAX_ULP


def test_host_layer_many_slabs_and_calls_in_a_row():
    """20 slabs of a 4096-wide layer, two calls in a row into the same output (the second
    with other inputs): each equals the device layer."""
    M, N, K = 10000, 4096, 2048
    wd = synthetic.int8_uniform((N, K), 531).to(DEV)
    wsd = synthetic.scale_uniform(N, 532).to(DEV)
    y = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    for seed in (533, 534):
        x = synthetic.normal_bf16((M, K), seed)
        ref = ck.ck_int8_linear(x.to(DEV), wd, wsd, None, mode=synthetic.PER_ROW)
        ck.ck_int8_linear_host(x.pin_memory(), wd, wsd, None, mode=synthetic.PER_ROW, y=y, slab_rows=512)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref.cpu().view(torch.int16))
    assert ck.ck_device_error(clear=False) == 0

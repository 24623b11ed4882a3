"""CUDA graph capture of the layer: a captured call replayed with new data in the same
buffers gives exactly what uncaptured calls give.  The single-launch tensorwise
preparation and the GEMM's K-split tail tag their cross-block exchanges per call; under
capture the library uses the untagged forms instead (a replay repeats its arguments), and
these tests replay the same graph with different inputs to check that no state leaks from
one replay into the next."""
import numpy as np
import pytest
import torch

import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
import oracle

from helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(M, N, K, mode, seed):
    x0 = synthetic.normal_bf16((M, K), seed).to(DEV)
    x1 = (synthetic.normal_bf16((M, K), seed + 1) * 3).to(DEV)  # a different maximum
    w = synthetic.int8_uniform((N, K), seed + 2).to(DEV)
    ws = synthetic.scale_uniform(1 if mode == ck.TENSORWISE else N, seed + 3, mul=0.01).to(DEV)
    b = synthetic.normal_bf16((1, N), seed + 4).reshape(N).to(DEV)
    return x0, x1, w, ws, b


@pytest.mark.parametrize("mode", [ck.TENSORWISE, ck.PER_ROW, ck.CONVROT])
def test_linear_graph_replays_match_eager(mode):
    M, N, K = 512, 768, 1024
    x0, x1, w, ws, b = _inputs(M, N, K, mode, 40 + mode)
    ref0 = bits(ck.ck_int8_linear(x0, w, ws, b, mode=mode))
    ref1 = bits(ck.ck_int8_linear(x1, w, ws, b, mode=mode))
    assert not np.array_equal(ref0, ref1)
    x = x0.clone()
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    work = ck.workspace(ck.ck_int8_linear_workspace_size(M, N, K, mode))
    ck.ck_int8_linear(x, w, ws, b, mode=mode, y=y, ws=work)  # the uncaptured first call
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ck.ck_int8_linear(x, w, ws, b, mode=mode, y=y, ws=work)
    for src, ref in ((x1, ref1), (x0, ref0), (x1, ref1), (x1, ref1)):
        x.copy_(src)
        y.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), ref), "replay differs from the uncaptured call"
    assert ck.ck_device_error(clear=True) == 0


def test_split_gemm_graph_replays_exact(monkeypatch):
    """A shape whose last wave is split along K when uncaptured: captured, it runs
    unsplit, and every replay gives the exact accumulators."""
    monkeypatch.setenv("CK_GEMM_PAIR", "1")
    monkeypatch.setenv("CK_GEMM_SPLIT", "2")
    M, N, K = 512, 1024, 2048
    assert ck.ck_gemm_tile_config(M, N, K)[3] == 2
    qs = [synthetic.int8_uniform((M, K), 70 + i) for i in range(2)]
    w = synthetic.int8_uniform((N, K), 72)
    refs = [oracle.gemm_s32(q.numpy(), w.numpy()) for q in qs]
    q = qs[0].to(DEV)
    wd = w.to(DEV)
    acc = torch.empty((M, N), dtype=torch.int32, device=DEV)
    work = ck.workspace(ck.load_library().ck_int8_gemm_workspace_size(M, N, K))
    ck.ck_int8_gemm_s32(q, wd, acc=acc, ws=work)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), refs[0])  # uncaptured: split
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ck.ck_int8_gemm_s32(q, wd, acc=acc, ws=work)
    for i in (1, 0, 1):
        q.copy_(qs[i].to(DEV))
        acc.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(acc.cpu().numpy(), refs[i])
    assert ck.ck_device_error(clear=True) == 0


@pytest.mark.parametrize("mode", [ck.TENSORWISE, ck.PER_ROW, ck.CONVROT])
def test_w8a16_graph_replays_match_eager(mode):
    """The 16-bit-activation layer (widening or rotation launch + GEMM) under capture."""
    M, N, K = 384, 512, 1024
    x0, x1, w, ws, b = _inputs(M, N, K, mode, 60 + mode)
    ref0 = bits(ck.ck_w8a16_linear(x0, w, ws, b, mode=mode))
    ref1 = bits(ck.ck_w8a16_linear(x1, w, ws, b, mode=mode))
    x = x0.clone()
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    work = ck.workspace(max(16, ck.load_library().ck_w8a16_linear_workspace_size(M, N, K, mode)))
    ck.ck_w8a16_linear(x, w, ws, b, mode=mode, y=y, ws=work)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ck.ck_w8a16_linear(x, w, ws, b, mode=mode, y=y, ws=work)
    for src, ref in ((x1, ref1), (x0, ref0), (x1, ref1)):
        x.copy_(src)
        y.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(y), ref)
    assert ck.ck_device_error(clear=True) == 0

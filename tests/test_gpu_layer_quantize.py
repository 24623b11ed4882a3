"""The activation quantize that ck_int8_linear runs itself, bit for bit against the oracle.

The layer's preparation kernel writes the activation codes (as bf16 integers, the tensor
cores' operand format) and x_scale into the caller's workspace; the GEMM reads them from
there.  ck_int8_linear_workspace_views tells where, so these tests read what the layer's
own kernels computed -- the row kernels of per-row and ConvRot mode, and the tensorwise
preparation whose blocks exchange their maxima -- and compare every code and every scale
with the oracle's q and x_scale (issue #278, section "2. quantize_int8_rowwise raises
instead of falling back"; issue #280, "Exactness": bit-identical results), next to the
layer's output y (0 ulp).  The workspace starts full of random bytes between guard bands.
"""
import numpy as np
import pytest
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
from helpers import (bits, bf16_ulp_distance, guarded_workspace, assert_workspace_guards_intact, MAX_ULP)

pytestmark = pytest.mark.gpu
DEV = "cuda"
TW, PR, CR = synthetic.TENSORWISE, synthetic.PER_ROW, synthetic.CONVROT

# (M, N, K, mode).  Tensorwise preparation on GB300: at most 608 blocks of 256 threads
# (four per SM, all resident), each thread keeping the first 13 of its 16-byte vectors in
# shared memory for the quantize pass.
CASES = [
    (4096, 4096, 4096, TW),   # 608 blocks (the largest grid), 14 vectors per thread: 13 kept, 1 re-read
    (8192, 256, 8192, TW),    # 54 vectors per thread: 41 re-read from memory
    (2048, 256, 4096, TW),    # 7 vectors per thread, all kept on chip
    (333, 264, 1040, TW),     # 170 blocks, ragged last block
    (300, 264, 1152, TW),
    (1, 8, 16, TW),           # one block, two vectors
    (4096, 4096, 4096, PR),
    (300, 264, 1152, PR),     # ragged rows and columns
    (333, 264, 1040, PR),
    (5, 64, 5376, PR),        # the 80666x28672x5376 row length (128 threads x 6 vectors per row)
    (3, 64, 20000, PR),       # rows too long for registers: two passes per row
    (300, 264, 1152, CR),
    (4, 64, 16384, CR),       # the longest register-resident ConvRot row
    (3, 64, 32768, CR),       # two passes per row with the rotation
]


def case_inputs(M, N, K, mode, seed):
    oc = synthetic.outlier_columns(K, 0.01, seed + 404) if mode == CR else None
    x = synthetic.normal_bf16((M, K), seed, outlier_channels=oc)
    if mode == CR:
        w, ws = oracle.prepare_convrot_weight(synthetic.normal_f32((N, K), seed + 505, std=0.02).numpy())
        w, ws = torch.from_numpy(w), torch.from_numpy(ws)
    else:
        w = synthetic.int8_uniform((N, K), seed + 101)
        ws = synthetic.scale_uniform(1 if mode == TW else N, seed + 202)
    b = synthetic.normal_bf16((1, N), seed + 303, std=0.02).reshape(N)
    return x, w, ws, b


def layer_and_codes(x, w, ws, b, mode, work):
    M, K = x.shape
    N = w.shape[0]
    y = ck.ck_int8_linear(x.to(DEV), w.to(DEV), ws.to(DEV), b.to(DEV), mode=mode, ws=work)
    codes, xs = ck.linear_workspace_codes(work, M, N, K, mode)
    torch.cuda.synchronize()
    return y, codes.float().cpu(), xs.cpu()


def check_codes(codes, xs, ref, mode):
    # every code an integer in [-127, 127] (a zero may carry either sign)
    assert bool((codes == codes.round()).all()) and float(codes.abs().max()) <= 127.0
    q = codes.to(torch.int8).numpy()
    bad = np.argwhere(q != ref["q"])
    assert bad.size == 0, "%d codes differ, first at %s: layer %d oracle %d" % (
        len(bad), bad[0], q[tuple(bad[0])], ref["q"][tuple(bad[0])])
    got = xs.numpy().view(np.uint32)
    want = ref["xs"].view(np.uint32)
    assert got.shape == want.shape and np.array_equal(got, want), "x_scale differs"


@pytest.mark.parametrize("M,N,K,mode", CASES,
                         ids=["%s_%dx%dx%d" % (synthetic.MODE_NAMES[c[3]], c[0], c[1], c[2]) for c in CASES])
def test_layer_codes_and_scales_match_the_oracle(M, N, K, mode):
    x, w, ws, b = case_inputs(M, N, K, mode, seed=M + 3 * K + mode)
    ref = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=mode)
    wbuf, work, before = guarded_workspace(ck.ck_int8_linear_workspace_size(M, N, K, mode), seed=K + mode)
    y, codes, xs = layer_and_codes(x, w, ws, b, mode, work)
    assert_workspace_guards_intact(wbuf, before)
    check_codes(codes, xs, ref, mode)
    d = bf16_ulp_distance(bits(y), ref["y"])
    assert d.max() <= MAX_ULP, "max ulp %d" % d.max()
    assert ck.ck_device_error(clear=False) == 0


def test_convrot_workload_layer_codes():
    """The ConvRot workload (4096x12288x3072, 1% outlier channels x20, bias): the layer's
    rotated-and-quantized activation equals the oracle's."""
    case = synthetic.case_from_spec(synthetic.CONVROT_4096)
    w, ws = oracle.prepare_convrot_weight(case.w_float.numpy())
    w, ws = torch.from_numpy(w), torch.from_numpy(ws)
    ref = oracle.int8_linear(bits(case.x), w.numpy(), ws.numpy(), bits(case.bias), mode=CR)
    work = torch.empty(ck.ck_int8_linear_workspace_size(case.M, case.N, case.K, CR), dtype=torch.uint8, device=DEV)
    y, codes, xs = layer_and_codes(case.x, w, ws, case.bias, CR, work)
    check_codes(codes, xs, ref, CR)
    assert bf16_ulp_distance(bits(y), ref["y"]).max() <= MAX_ULP


@pytest.mark.parametrize("mode", [TW, PR, CR])
def test_consecutive_calls_leave_nothing_behind(mode):
    """Two calls in a row on one workspace, the second with a smaller maximum: its codes
    and scales are its own (the tensorwise exchange slots still hold the first call's
    maxima, under another tag)."""
    M, N, K = 1024, 256, 2048
    work = torch.empty(ck.ck_int8_linear_workspace_size(M, N, K, mode), dtype=torch.uint8, device=DEV)
    for i, gain in enumerate((8.0, 0.25)):
        x, w, ws, b = case_inputs(M, N, K, mode, seed=900 + i)
        x = (x.float() * gain).to(torch.bfloat16)
        ref = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=mode)
        y, codes, xs = layer_and_codes(x, w, ws, b, mode, work)
        check_codes(codes, xs, ref, mode)
        assert bf16_ulp_distance(bits(y), ref["y"]).max() <= MAX_ULP


@pytest.mark.parametrize("K", [1152, 3072])
def test_convrot_layer_codes_at_half_integer_quotients(K):
    """The layer's ConvRot preparation (bf16 codes) on rows whose rotated values all sit
    within fp32 rounding of half-integer multiples of the scale (the construction of
    test_gpu_quantize._half_integer_rows): every code is decided by the quotient's last
    bits and must equal the oracle's."""
    from test_gpu_quantize import _half_integer_rows
    M, N = 200, 128
    x = _half_integer_rows(M, K, seed=K)
    _, w, ws, b = case_inputs(M, N, K, CR, seed=K + 1)
    ref = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=CR)
    work = torch.empty(ck.ck_int8_linear_workspace_size(M, N, K, CR), dtype=torch.uint8, device=DEV)
    y, codes, xs = layer_and_codes(x, w, ws, b, CR, work)
    check_codes(codes, xs, ref, CR)
    assert bf16_ulp_distance(bits(y), ref["y"]).max() <= MAX_ULP

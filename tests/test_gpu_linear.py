"""The whole layer, ck_int8_linear, on the workloads of the comfy-kitchen pages, against
the CPU oracle, bit for bit: full outputs where the oracle finishes in seconds, seeded row
samples (plus the first and last 16 rows) on the multi-GB shapes, including the
M*N >= 2^31 boundary of issue #136.  Every output is written into a buffer pre-filled with
NaN between two guard bands: after the call no element may still be NaN (every tile was
written, at its own address) and the bands must be untouched."""
import numpy as np
import pytest
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
from helpers import (bits, bf16_ulp_distance, out_bits, ulp_distance, MAX_ULP, guarded, assert_guards_intact,
                     assert_all_written, NAN16, NAN32)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def convrot_weight(case):
    w, ws = oracle.prepare_convrot_weight(case.w_float.cpu().numpy())
    return torch.from_numpy(w), torch.from_numpy(ws)


def run_full(spec):
    case = synthetic.case_from_spec(spec)
    if case.mode == synthetic.CONVROT:
        w, ws = convrot_weight(case)
    else:
        w, ws = case.w, case.w_scale
    b = case.bias
    ref = oracle.int8_linear(bits(case.x), w.numpy(), ws.numpy(), None if b is None else bits(b), mode=case.mode)
    ybuf, y = guarded((case.M, case.N), torch.bfloat16, NAN16)
    ck.ck_int8_linear(case.x.to(DEV), w.to(DEV), ws.to(DEV), None if b is None else b.to(DEV), mode=case.mode, y=y)
    torch.cuda.synchronize()
    assert_guards_intact(ybuf, NAN16)
    assert_all_written(ybuf, NAN16)
    d = bf16_ulp_distance(bits(y), ref["y"])
    assert d.max() <= MAX_ULP, "%s: max ulp %d at %s" % (spec[0], d.max(), np.unravel_index(d.argmax(), d.shape))
    return case, y


def test_per_row_256x512x512():
    run_full(synthetic.PER_ROW_SMALL)


@pytest.mark.parametrize("out_dtype,code", [(torch.float16, oracle.OUT_F16), (torch.float32, oracle.OUT_F32)])
@pytest.mark.parametrize("mode", [synthetic.TENSORWISE, synthetic.PER_ROW, synthetic.CONVROT])
def test_output_types(mode, out_dtype, code):
    """int8_linear(x, w, ws, out_dtype): the same layer with fp16 and fp32 outputs."""
    M, N, K = 300, 264, 1152
    x = synthetic.normal_bf16((M, K), seed=61 + mode)
    if mode == synthetic.CONVROT:
        w, ws = oracle.prepare_convrot_weight(synthetic.normal_f32((N, K), seed=62, std=0.02).numpy())
        w, ws = torch.from_numpy(w), torch.from_numpy(ws)
    else:
        w = synthetic.int8_uniform((N, K), seed=62)
        ws = synthetic.scale_uniform(1 if mode == synthetic.TENSORWISE else N, seed=63)
    b = synthetic.normal_bf16((1, N), seed=64, std=0.5).reshape(N)
    ref = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=mode, out_dtype=code)["y"]
    if code == oracle.OUT_F32:
        ref = ref.view(np.uint32)
    pattern = NAN32 if code == oracle.OUT_F32 else NAN16
    ybuf, y = guarded((M, N), out_dtype, pattern)
    ck.ck_int8_linear(x.to(DEV), w.to(DEV), ws.to(DEV), b.to(DEV), mode=mode, out_dtype=out_dtype, y=y)
    torch.cuda.synchronize()
    assert_guards_intact(ybuf, pattern)
    assert_all_written(ybuf, pattern)
    assert y.dtype == out_dtype
    d = ulp_distance(out_bits(y), ref)
    assert d.max() <= MAX_ULP, "max ulp %d at %s" % (d.max(), np.unravel_index(d.argmax(), d.shape))


def test_tensorwise_4096_cubed_with_bias():
    run_full(synthetic.TENSORWISE_4096)


def test_convrot_4096x12288x3072_with_bias():
    case, y = run_full(synthetic.CONVROT_4096)
    # the rotated layer stays close to the float layer it approximates
    ref = case.x.float() @ case.w_float.T + case.bias.float()
    rel = (y.float().cpu() - ref).norm() / ref.norm()
    assert rel < 0.02


@pytest.mark.parametrize("spec", synthetic.SWEEP[:2], ids=lambda s: s[0])
def test_sweep_small_shapes_full(spec):
    run_full(spec)


def boundary_rows(M, N):
    """The rows around the int32 element-offset limit: row r holds elements r*N ..
    r*N + N - 1, so the row that crosses 2^31 and its neighbours (issue #136, "Summary")."""
    r = (2 ** 31) // N
    return [i for i in (r - 1, r, r + 1) if 0 <= i < M]


def run_sampled(spec):
    name, M, N, K, mode, bias, frac, seed = spec
    # the activation is drawn on the GPU (multi-GB); the weight on the CPU, as the oracle needs all of it
    x = synthetic.normal_bf16((M, K), seed, device=DEV)
    w = synthetic.int8_uniform((N, K), seed + 101)
    ws = synthetic.scale_uniform(N, seed + 202)
    # y inside a NaN-filled buffer with guard bands: every one of the M*N outputs must be
    # overwritten with a finite value, nothing written outside
    ybuf, y = guarded((M, N), torch.bfloat16, NAN16)
    ck.ck_int8_linear(x, w.to(DEV), ws.to(DEV), None, mode=mode, y=y)
    torch.cuda.synchronize()
    assert_guards_intact(ybuf, NAN16)
    for r0 in range(0, M, 8192):
        assert bool(torch.isfinite(y[r0:r0 + 8192]).all()), "%s: a non-finite output in rows %d.." % (name, r0)
    rows = sorted(set(synthetic.sample_rows(M, seed=1000 + seed)) | set(boundary_rows(M, N)))
    idx = torch.tensor(rows, device=DEV)
    xr = bits(x.index_select(0, idx))
    ref = oracle.int8_linear(xr, w.numpy(), ws.numpy(), None, mode=mode)
    got = bits(y.index_select(0, idx))
    d = bf16_ulp_distance(got, ref["y"])
    assert d.max() <= MAX_ULP, "%s: max ulp %d at sample row %d" % (name, d.max(), rows[int(d.max(axis=1).argmax())])
    del x, y, ybuf
    torch.cuda.empty_cache()


@pytest.mark.slow
@pytest.mark.parametrize("spec", synthetic.SWEEP[2:], ids=lambda s: s[0])
def test_sweep_large_shapes_sampled(spec):
    run_sampled(spec)


@pytest.mark.slow
@pytest.mark.parametrize("spec", synthetic.LARGE_INDEX, ids=lambda s: s[0])
def test_large_index_boundary_sampled(spec):
    assert spec[1] * spec[2] >= 2 ** 31 - 21504  # straddles the int32 element-offset limit
    M, N = spec[1], spec[2]
    assert boundary_rows(M, N)[-1] == min(M - 1, 2 ** 31 // N + 1)  # the sample includes the crossing row
    run_sampled(spec)


@pytest.mark.parametrize("mode", [synthetic.TENSORWISE, synthetic.PER_ROW, synthetic.CONVROT])
def test_linear_residual_in_place(mode):
    """A residual-stream update y += layer(x), in place, through the whole layer."""
    M, N, K = 300, 264, 1152
    x = synthetic.normal_bf16((M, K), seed=71 + mode)
    if mode == synthetic.CONVROT:
        w, ws = oracle.prepare_convrot_weight(synthetic.normal_f32((N, K), seed=72, std=0.02).numpy())
        w, ws = torch.from_numpy(w), torch.from_numpy(ws)
    else:
        w = synthetic.int8_uniform((N, K), seed=72)
        ws = synthetic.scale_uniform(1 if mode == synthetic.TENSORWISE else N, seed=73)
    b = synthetic.normal_bf16((1, N), seed=74, std=0.5).reshape(N)
    r = synthetic.normal_bf16((M, N), seed=75, std=3.0)
    ref8 = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=mode)
    ref = oracle.dequant_residual(ref8["acc"], ref8["xs"], ws.numpy(), r.float().numpy(), bits(b),
                                  scalar_scales=(mode == synthetic.TENSORWISE))
    ybuf, y = guarded((M, N), torch.bfloat16, NAN16)
    y.copy_(r.to(DEV))
    ck.ck_int8_linear(x.to(DEV), w.to(DEV), ws.to(DEV), b.to(DEV), mode=mode, y=y, residual=y)
    torch.cuda.synchronize()
    assert_guards_intact(ybuf, NAN16)
    d = bf16_ulp_distance(bits(y), ref)
    assert d.max() <= MAX_ULP, "max ulp %d" % d.max()


@pytest.mark.parametrize("mode", [synthetic.TENSORWISE, synthetic.PER_ROW, synthetic.CONVROT])
def test_linear_with_prepared_weight_codes(mode):
    """The weight's codes prepared once (ck_int8_weight_codes) and the layer run on them
    (ck_int8_linear_codes): the codes equal the int8 weight, and every output equals
    ck_int8_linear's and the oracle's, two calls in a row."""
    M, N, K = 1000, 776, 1152
    x = synthetic.normal_bf16((M, K), seed=81 + mode)
    if mode == synthetic.CONVROT:
        w, ws = oracle.prepare_convrot_weight(synthetic.normal_f32((N, K), seed=82, std=0.02).numpy())
        w, ws = torch.from_numpy(w), torch.from_numpy(ws)
    else:
        w = synthetic.int8_uniform((N, K), seed=82)
        ws = synthetic.scale_uniform(1 if mode == synthetic.TENSORWISE else N, seed=83)
    b = synthetic.normal_bf16((1, N), seed=84, std=0.5).reshape(N)
    wd, wsd, bd = w.to(DEV), ws.to(DEV), b.to(DEV)
    cbuf, codes = guarded((N, K), torch.bfloat16, NAN16)
    ck.ck_int8_weight_codes(wd, w_codes=codes)
    torch.cuda.synchronize()
    assert_guards_intact(cbuf, NAN16)
    assert torch.equal(codes.float().cpu(), w.float())
    want = oracle.int8_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=mode)["y"]
    xd = x.to(DEV)
    ref = bits(ck.ck_int8_linear(xd, wd, wsd, bd, mode=mode))
    for _ in range(2):
        ybuf, y = guarded((M, N), torch.bfloat16, NAN16)
        ck.ck_int8_linear_codes(xd, codes, wsd, bd, mode=mode, y=y)
        torch.cuda.synchronize()
        assert_guards_intact(ybuf, NAN16)
        assert np.array_equal(bits(y), ref)
        assert bf16_ulp_distance(bits(y), want).max() <= MAX_ULP

"""GPU parity of the 16-bit-activation path (ck_w8a16_linear) against the oracle's
double-precision value.  The tolerance follows from the arithmetic: products of bf16
activations and int8 codes are exact in fp32, the tensor cores sum K of them in fp32 (at
most about K * 2^-24 * sum|a w| of error in any order), then one fp32 multiply, one fp32
add and the rounding to the output type:
    |y - y_ref| <= ulp_out(y_ref) + 2^-24 * (K + 8) * (mag + |bias|)
with mag = |w_scale| * sum_k |a w| from the oracle.  The rotated ConvRot operand is a
rounding decision and is checked bit for bit (identity weights, fp32 output)."""
import numpy as np
import pytest
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
from helpers import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"
SIG_BITS = {torch.bfloat16: 8, torch.float16: 11, torch.float32: 24}


def ulp(v, p):
    """One unit in the last place of |v| for a p-bit significand (at least the smallest normal's)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - (p - 1))


def check(x, w, ws, b, mode, out_dtype):
    M, K = x.shape
    y_ref, mag = oracle.w8a16_linear(bits(x), w.numpy(), ws.numpy(), None if b is None else bits(b), mode=mode)
    y = ck.ck_w8a16_linear(x.to(DEV), w.to(DEV), ws.to(DEV), None if b is None else b.to(DEV), mode=mode,
                           out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ck.ck_device_error(clear=False) == 0
    got = y.float().cpu().numpy().astype(np.float64)
    babs = 0.0 if b is None else np.abs(b.float().numpy().astype(np.float64))[None, :]
    tol = ulp(y_ref, SIG_BITS[out_dtype]) + 2.0 ** -24 * (K + 8) * (mag + babs)
    err = np.abs(got - y_ref)
    worst = np.unravel_index(np.argmax(err / tol), err.shape)
    assert np.all(err <= tol), "err %g > tol %g at %s (ref %g)" % (err[worst], tol[worst], worst, y_ref[worst])
    return err, tol


def make(M, N, K, mode, seed, with_bias=True):
    x = synthetic.normal_bf16((M, K), seed=seed)
    if mode == synthetic.CONVROT:
        w, ws = oracle.prepare_convrot_weight(synthetic.normal_f32((N, K), seed=seed + 1, std=0.02).numpy())
        w, ws = torch.from_numpy(w), torch.from_numpy(ws)
    else:
        w = synthetic.int8_uniform((N, K), seed=seed + 1)
        ws = synthetic.scale_uniform(1 if mode == synthetic.TENSORWISE else N, seed=seed + 2, mul=0.01)
    b = synthetic.normal_bf16((1, N), seed=seed + 3, std=0.5).reshape(N) if with_bias else None
    return x, w, ws, b


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32, torch.float16])
@pytest.mark.parametrize("mode", [synthetic.TENSORWISE, synthetic.PER_ROW, synthetic.CONVROT])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (129, 264, 1152), (1, 8, 128), (300, 712, 2048), (3, 264, 384)])
def test_w8a16_parity(M, N, K, mode, out_dtype):
    x, w, ws, b = make(M, N, K, mode, seed=M + N + K)
    check(x, w, ws, b, mode, out_dtype)


def test_w8a16_long_k_without_bias():
    """K = 8192 summed in one fp32 TMEM accumulation."""
    x, w, ws, _ = make(512, 1024, 8192, synthetic.PER_ROW, seed=5, with_bias=False)
    check(x, w, ws, None, synthetic.PER_ROW, torch.bfloat16)


@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("bn", [256, 160, 96, 32])
def test_w8a16_every_tile_width(monkeypatch, bn, pair):
    monkeypatch.setenv("CK_GEMM_BN", str(bn))
    monkeypatch.setenv("CK_GEMM_PAIR", pair)
    x, w, ws, b = make(300, 712, 1104, synthetic.PER_ROW, seed=bn)
    check(x, w, ws, b, synthetic.PER_ROW, torch.float32)


@pytest.mark.parametrize("mode", [synthetic.PER_ROW, synthetic.CONVROT])
@pytest.mark.parametrize("M,K", [(64, 256), (3, 384), (33, 1024)])
def test_w8a16_operand_bit_exact(M, K, mode):
    """Identity weights, unit scales, fp32 output: y = a exactly, so the activation
    operand (x itself, or the once-rounded bf16(x @ H)) is compared bit for bit."""
    oc = synthetic.outlier_columns(K, 0.01, seed=M)
    x = synthetic.normal_bf16((M, K), seed=K + M, outlier_channels=oc)
    w = torch.eye(K, dtype=torch.int8)
    ws = torch.ones(K, dtype=torch.float32)
    y_ref, _ = oracle.w8a16_linear(bits(x), w.numpy(), ws.numpy(), None, mode=mode)
    y = ck.ck_w8a16_linear(x.to(DEV), w.to(DEV), ws.to(DEV), None, mode=mode, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().astype(np.float64), y_ref)


def test_w8a16_matches_the_int8_path_on_lossless_inputs():
    """Activations whose per-row quantization is lossless: both paths compute the same
    real number, and their bf16 outputs agree to one step."""
    M, N, K = 128, 256, 1024
    g = np.random.default_rng(77)
    q = g.integers(-127, 128, size=(M, K))
    q[:, 0] = 127
    e = g.integers(-6, 4, size=(M, 1))
    x = torch.tensor((q * (2.0 ** e)).astype(np.float32)).to(torch.bfloat16)
    w = synthetic.int8_uniform((N, K), seed=78)
    ws = synthetic.scale_uniform(N, seed=79, mul=0.01)
    y8 = ck.ck_int8_linear(x.to(DEV), w.to(DEV), ws.to(DEV), None, mode=ck.PER_ROW).float().cpu()
    y16 = ck.ck_w8a16_linear(x.to(DEV), w.to(DEV), ws.to(DEV), None, mode=ck.PER_ROW).float().cpu()
    torch.cuda.synchronize()
    assert torch.all((y8 - y16).abs() <= y8.abs() * 2.0 ** -7 + 1e-30)


def test_w8a16_rejects_bad_arguments():
    x = torch.zeros((4, 200), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((8, 200), dtype=torch.int8, device=DEV)
    with pytest.raises(ck.CkError):
        ck.ck_w8a16_linear(x, w, torch.ones(8, device=DEV), mode=ck.PER_ROW)  # K % 16
    x = torch.zeros((4, 144), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((8, 144), dtype=torch.int8, device=DEV)
    with pytest.raises(ck.CkError) as e:
        ck.ck_w8a16_linear(x, w, torch.ones(8, device=DEV), mode=ck.CONVROT)  # K % 128
    assert "128" in str(e.value)


@pytest.mark.parametrize("mode", [synthetic.PER_ROW, synthetic.CONVROT])
def test_w8a16_residual(mode):
    """The residual is one more fp32 add: the bound gains 2^-24 * |residual|."""
    M, N, K = 129, 264, 1152
    x, w, ws, b = make(M, N, K, mode, seed=11)
    r = synthetic.normal_bf16((M, N), seed=12, std=2.0)
    y_ref, mag = oracle.w8a16_linear(bits(x), w.numpy(), ws.numpy(), bits(b), mode=mode)
    rf = r.float().numpy().astype(np.float64)
    y = ck.ck_w8a16_linear(x.to(DEV), w.to(DEV), ws.to(DEV), b.to(DEV), mode=mode, residual=r.to(DEV))
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    ref = y_ref + rf
    babs = np.abs(b.float().numpy().astype(np.float64))[None, :]
    tol = ulp(ref, 8) + 2.0 ** -24 * (K + 8) * (mag + babs + np.abs(rf))
    assert np.all(np.abs(got - ref) <= tol)

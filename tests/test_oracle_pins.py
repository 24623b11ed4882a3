"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not share code with: worked
examples derived by hand from the definition (tests/golden/), closed forms, brute
force in pure Python, library routines (numpy integer matmul, torch's bf16 rounding,
Python's round-half-even), exact rational arithmetic, and the algebra of the Hadamard
matrix.  A dropped term, a wrong sign, a swapped index or a transposed operand in the
oracle makes at least one of them fail.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from int8_weight_quantized_gb300 import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(t):
    """bf16 torch tensor -> uint16 numpy bit patterns."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_bf16_bits(vals):
    return bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def sylvester(n):
    """Unnormalized Sylvester Hadamard matrix by the recursive block construction."""
    H = np.array([[1.0]])
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


# ---------------------------------------------------------------- quantize
def load_worked_examples():
    rows = []
    with open(os.path.join(GOLDEN, "quantize_worked_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            xs, s, q = [p.strip() for p in line.split("|")]
            rows.append(([float(v) for v in xs.split()], float(s), [int(v) for v in q.split()]))
    return rows


@pytest.mark.parametrize("example", load_worked_examples())
def test_quantize_worked_examples(example):
    x, s_expect, q_expect = example
    xb = to_bf16_bits([x])
    assert np.array_equal(oracle.bf16_to_f32(xb)[0], np.array(x, np.float32)), "fixture value not bf16-exact"
    q, xs = oracle.quantize_rowwise(xb)
    assert xs[0] == np.float32(s_expect)
    assert q[0].tolist() == q_expect


def test_quantize_round_half_even_on_every_tie():
    # amax = 127 * 2^e  ->  x_scale = 2^e exactly; x = (n + 1/2) * 2^e lands exactly on a tie.
    for e in (-6, 0, 3):
        n = np.arange(0, 127)
        ties = (n + 0.5) * 2.0 ** e
        row = np.concatenate([[127 * 2.0 ** e], ties, -ties])
        xb = to_bf16_bits([row.tolist()])
        assert np.array_equal(oracle.bf16_to_f32(xb)[0].astype(np.float64), row)
        q, xs = oracle.quantize_rowwise(xb)
        assert xs[0] == np.float32(2.0 ** e)
        expect = [127] + [round(v + 0.5) for v in n] + [-round(v + 0.5) for v in n]  # Python rounds half to even
        assert q[0].tolist() == expect


def test_quantize_invariants_random_rows():
    x = synthetic.normal_bf16((64, 384), seed=11)
    xb = bits(x)
    q, xs = oracle.quantize_rowwise(xb)
    xf = x.float().numpy().astype(np.float64)
    amax = np.abs(xf).max(axis=1)
    # the scale is the row maximum over 127, correctly rounded to fp32
    for m in range(64):
        exact = Fraction(float(amax[m])) / 127
        assert abs(Fraction(float(xs[m])) - exact) <= exact * Fraction(1, 2 ** 24)
    # every non-zero row reaches the full code range, and every code is within half a step
    assert np.all(np.abs(q).max(axis=1) == 127)
    assert np.all(np.sign(q) * np.sign(xf) >= 0)
    err = np.abs(xf / xs.astype(np.float64)[:, None] - q)
    assert err.max() <= 0.5 + 1e-5


def test_quantize_zero_and_subnormal_rows():
    tiny = np.array([0x0001, 0x8003, 0x0040, 0x0000] * 4, np.uint16)  # bf16 subnormals
    zero = np.zeros(16, np.uint16)
    q, xs = oracle.quantize_rowwise(np.stack([zero, tiny]))
    assert xs[0] == 0.0 and np.all(q[0] == 0)
    assert xs[1] > 0
    xf = oracle.bf16_to_f32(tiny).astype(np.float64)
    assert np.abs(q[1]).max() == 127
    assert np.all(np.abs(xf / float(xs[1]) - q[1]) <= 0.5 + 1e-3)


def test_tensorwise_equals_rowwise_when_rows_share_the_maximum():
    x = synthetic.normal_bf16((32, 256), seed=12).float()
    g = x.abs().max()
    x[:, 7] = g  # every row now holds the global maximum
    xb = bits(x.to(torch.bfloat16))
    qt, st = oracle.quantize_tensorwise(xb)
    qr, sr = oracle.quantize_rowwise(xb)
    assert np.all(sr == st[0])
    assert np.array_equal(qt, qr)
    assert st[0] == np.float32(np.float32(g.item()) / np.float32(127.0))


def test_tensorwise_scale_is_global():
    x = synthetic.normal_bf16((16, 64), seed=13)
    xb = bits(x)
    q, s = oracle.quantize_tensorwise(xb)
    xf = x.float().numpy().astype(np.float64)
    assert np.abs(q).max() == 127
    assert np.all(np.abs(xf / float(s[0]) - q) <= 0.5 + 1e-5)
    # rows with a small maximum use fewer codes than in per-row mode
    qr, _ = oracle.quantize_rowwise(xb)
    assert np.abs(q).max(axis=1).min() < 127 == np.abs(qr).max(axis=1).min()


# ---------------------------------------------------------------- GEMM
def test_gemm_brute_force_tiny():
    rng = np.random.default_rng(5)
    q = rng.integers(-127, 128, size=(2, 16), dtype=np.int8)
    w = rng.integers(-127, 128, size=(3, 16), dtype=np.int8)
    acc = oracle.gemm_s32(q, w)
    for m in range(2):
        for n in range(3):
            s = 0
            for k in range(16):
                s += int(q[m, k]) * int(w[n, k])
            assert acc[m, n] == s


def test_gemm_matches_numpy_integer_matmul():
    rng = np.random.default_rng(6)
    q = rng.integers(-127, 128, size=(37, 96), dtype=np.int8)
    w = rng.integers(-127, 128, size=(40, 96), dtype=np.int8)
    ref = q.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(oracle.gemm_s32(q, w), ref.astype(np.int32))


def test_gemm_one_hot_weights_select_columns():
    rng = np.random.default_rng(7)
    q = rng.integers(-127, 128, size=(9, 32), dtype=np.int8)
    cols = [3, 0, 31, 17, 17, 5, 8, 30]
    w = np.zeros((len(cols), 32), np.int8)
    for n, k in enumerate(cols):
        w[n, k] = -1 if n % 2 else 1
    acc = oracle.gemm_s32(q, w)
    for n, k in enumerate(cols):
        assert np.array_equal(acc[:, n], q[:, k].astype(np.int32) * (-1 if n % 2 else 1))


@pytest.mark.parametrize("K", [16, 1024, 65536, 131072])
def test_gemm_extreme_magnitudes(K):
    q = np.full((2, K), 127, np.int8)
    q[1, ::2] = -127
    w = np.full((2, K), 127, np.int8)
    w[1] = -127
    acc = oracle.gemm_s32(q, w)
    assert acc[0, 0] == 127 * 127 * K and acc[0, 1] == -127 * 127 * K
    assert acc[1, 0] == 0 and acc[1, 1] == 0


# ---------------------------------------------------------------- epilogue
def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(8)
    v = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 3000),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130, 3.0e38], np.float32)])
    v = v.astype(np.float32)
    mine = oracle.f32_to_bf16(v)
    ref = bits(torch.from_numpy(v).to(torch.bfloat16))
    assert np.array_equal(mine, ref)


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(18)
    v = np.concatenate([
        (rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 6, 4000)).astype(np.float32),
        np.array([65504.0, 65519.9, 65520.0, 70000.0, -65520.0, 2.0 ** -14, 2.0 ** -24, 2.0 ** -25,
                  2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 0.0, -0.0,
                  5.960464477539063e-08, 6.097555160522461e-05, 1e-8], np.float32)]).astype(np.float32)
    mine = oracle.f32_to_f16(v)
    ref = v.astype(np.float16).view(np.uint16)
    bad = np.nonzero(mine != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(mine[i]), hex(ref[i])) for i in bad[:5]]


@pytest.mark.parametrize("out_dtype", [oracle.OUT_F16, oracle.OUT_F32])
def test_dequant_typed_outputs_share_the_fp32_value(out_dtype):
    rng = np.random.default_rng(19)
    acc = rng.integers(-10 ** 6, 10 ** 6, size=(6, 16), dtype=np.int64).astype(np.int32)
    xs = (rng.random(6) * 1e-3).astype(np.float32)
    ws = (rng.random(16) * 1e-2).astype(np.float32)
    b = to_bf16_bits(rng.standard_normal(16) * 0.1)
    f32 = oracle.dequant_typed(acc, xs, ws, b, out_dtype=oracle.OUT_F32)
    # the fp32 output is the epilogue value itself: bf16 and fp16 are its roundings
    assert np.array_equal(oracle.dequant_typed(acc, xs, ws, b, out_dtype=oracle.OUT_BF16),
                          bits(torch.from_numpy(f32).to(torch.bfloat16)))
    if out_dtype == oracle.OUT_F16:
        assert np.array_equal(oracle.dequant_typed(acc, xs, ws, b, out_dtype=out_dtype),
                              f32.astype(np.float16).view(np.uint16))
    # and it is within its rounding bound of the exact value
    for m in range(6):
        for n in range(16):
            prod = Fraction(int(acc[m, n])) * Fraction(float(xs[m])) * Fraction(float(ws[n]))
            bias = Fraction(float(oracle.bf16_to_f32(b[n:n + 1])[0]))
            # three fp32 roundings, each at most half an ulp of an intermediate bounded by
            # the operands' magnitudes (the sum may cancel)
            bound = (abs(prod) + abs(bias)) * Fraction(4, 2 ** 24)
            assert abs(Fraction(float(f32[m, n])) - (prod + bias)) <= bound


def test_dequant_hand_example():
    acc = np.array([[1000, -3, 0, 7]], np.int32)
    xs = np.array([0.5], np.float32)
    ws = np.array([0.25, 2.0, 8.0, 0.125], np.float32)
    b = to_bf16_bits([1.0, -0.5, 3.0, 0.0])
    y = oracle.bf16_to_f32(oracle.dequant(acc, xs, ws, b))
    # 1000*0.5*0.25 + 1 = 126;  -3*0.5*2 - 0.5 = -3.5;  0 + 3 = 3;  7*0.5*0.125 = 0.4375
    assert y[0].tolist() == [126.0, -3.5, 3.0, 0.4375]


def test_dequant_within_rounding_of_exact_value():
    rng = np.random.default_rng(9)
    M, N = 12, 24
    acc = rng.integers(-2 ** 30, 2 ** 30, size=(M, N), dtype=np.int64).astype(np.int32)
    xs = (rng.random(M).astype(np.float32) * np.float32(2e-3)).astype(np.float32)
    ws = (rng.random(N).astype(np.float32) * np.float32(1e-2)).astype(np.float32)
    prod_scale = np.abs(acc).astype(np.float64) * xs[:, None] * ws[None, :]
    bias_f = (rng.standard_normal(N) * np.median(prod_scale)).astype(np.float32)
    b = to_bf16_bits(bias_f)
    bf = oracle.bf16_to_f32(b)
    y = oracle.bf16_to_f32(oracle.dequant(acc, xs, ws, b))
    for m in range(M):
        for n in range(N):
            exact = Fraction(int(acc[m, n])) * Fraction(float(xs[m])) * Fraction(float(ws[n])) + Fraction(float(bf[n]))
            # three fp32 roundings (<= 3 * 2^-24 relative to the operands' magnitude) then one bf16 rounding
            mag = abs(Fraction(int(acc[m, n])) * Fraction(float(xs[m])) * Fraction(float(ws[n]))) + abs(Fraction(float(bf[n])))
            bound = abs(exact) * Fraction(1, 2 ** 8) + mag * Fraction(4, 2 ** 24)
            assert abs(Fraction(float(y[m, n])) - exact) <= bound, (m, n)


def test_dequant_scalar_scales_equal_broadcast_vectors():
    rng = np.random.default_rng(10)
    acc = rng.integers(-10 ** 6, 10 ** 6, size=(5, 16), dtype=np.int64).astype(np.int32)
    xs1, ws1 = np.array([3.1e-3], np.float32), np.array([7.7e-3], np.float32)
    b = to_bf16_bits(rng.standard_normal(16))
    a = oracle.dequant(acc, xs1, ws1, b, scalar_scales=True)
    v = oracle.dequant(acc, np.repeat(xs1, 5), np.repeat(ws1, 16), b, scalar_scales=False)
    assert np.array_equal(a, v)
    nob = oracle.dequant(acc, xs1, ws1, None, scalar_scales=True)
    assert not np.array_equal(a, nob)


# ---------------------------------------------------------------- Hadamard / ConvRot
def test_sylvester_construction_is_orthogonal():
    H = sylvester(128)
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    assert np.array_equal(H, H.T)


def test_fwht_constant_bits():
    c = oracle.fwht128(np.eye(128, dtype=np.float32)[0])[0]
    assert np.float32(c).view(np.uint32) == 0x3DB504F3


def test_fwht_unit_vectors_are_rows_of_H():
    H = sylvester(128) / np.sqrt(128.0)
    for i in (0, 1, 2, 5, 64, 77, 127):
        out = oracle.fwht128(np.eye(128, dtype=np.float32)[i]).astype(np.float64)
        assert np.allclose(out, H[i], rtol=0, atol=1e-7)


def test_fwht_matches_dense_product():
    H = sylvester(128) / np.sqrt(128.0)
    rng = np.random.default_rng(12)
    for _ in range(8):
        v = rng.standard_normal(128).astype(np.float32)
        dense = v.astype(np.float64) @ H
        out = oracle.fwht128(v).astype(np.float64)
        assert np.max(np.abs(out - dense)) <= 1e-6 * np.max(np.abs(dense))


def test_fwht_is_an_involution_and_isometry():
    rng = np.random.default_rng(13)
    v = rng.standard_normal(128).astype(np.float32)
    once = oracle.fwht128(v)
    twice = oracle.fwht128(once)
    assert np.allclose(twice, v, rtol=0, atol=1e-5)
    assert abs(np.linalg.norm(once.astype(np.float64)) - np.linalg.norm(v.astype(np.float64))) < 1e-5


def test_rotated_basis_equivalence_in_double():
    # (x H)(W H^T)^T = x H H^T W^T = x W^T: the GEMM may run entirely in the rotated basis
    rng = np.random.default_rng(14)
    K = 256
    Hb = sylvester(128) / np.sqrt(128.0)
    H = np.kron(np.eye(K // 128), Hb)
    x = rng.standard_normal((6, K))
    W = rng.standard_normal((5, K))
    lhs = (x @ H) @ (W @ H.T).T
    assert np.allclose(lhs, x @ W.T, rtol=1e-9, atol=1e-9)


def test_rowwise_rotation_uses_the_block_transform():
    # quantizing with rotate=1 equals quantizing the pre-rotated row with rotate=0 whenever
    # the rotated values are themselves bf16-exact: rows of +-c at single positions rotate
    # into +-c/sqrt(128) patterns; take c = sqrt(128) * 2^-3 so every rotated value is +-2^-3
    # (exact in bf16 and fp32 whichever butterfly order is used).
    K = 256
    c = np.float32(np.sqrt(128.0) * 0.125)
    row = np.zeros(K, np.float32)
    row[0] = 1.0
    row[128 + 5] = -1.0
    xr = to_bf16_bits([row.tolist()])
    q, xs = oracle.quantize_rowwise(xr, rotate=True)
    H = sylvester(128)
    v = np.concatenate([H[0], -H[5]]) / np.sqrt(128.0)
    assert xs[0] == np.float32(np.float32(1 / np.sqrt(128.0)) / np.float32(127))
    assert np.array_equal(q[0], np.round(v / np.abs(v).max() * 127).astype(np.int8))
    del c


def test_convrot_weight_preparation():
    rng = np.random.default_rng(15)
    W = (rng.standard_normal((6, 256)) * 0.02).astype(np.float32)
    w, ws = oracle.prepare_convrot_weight(W)
    H = np.kron(np.eye(2), sylvester(128) / np.sqrt(128.0))
    Wr = W.astype(np.float64) @ H.T
    assert np.allclose(ws, np.abs(Wr).max(axis=1) / 127, rtol=1e-6)
    assert np.all(np.abs(w).max(axis=1) == 127)
    assert np.all(np.abs(Wr / ws[:, None].astype(np.float64) - w) <= 0.5 + 1e-4)


def test_convrot_linear_approximates_float_layer_and_beats_per_row_on_outliers():
    M, N, K = 64, 96, 512
    case = synthetic.make_case("t", M, N, K, synthetic.CONVROT, bias=True, seed=21, outlier_frac=0.01)
    xb = bits(case.x)
    W = case.w_float.numpy()
    bb = bits(case.bias)
    w_rot, ws_rot = oracle.prepare_convrot_weight(W)
    y_rot = oracle.bf16_to_f32(oracle.int8_linear(xb, w_rot, ws_rot, bb, mode=oracle.CONVROT)["y"])
    # per-row baseline on the same layer: weight quantized without the rotation
    amax = np.abs(W).max(axis=1)
    ws_pl = (amax / np.float32(127)).astype(np.float32)
    w_pl = np.clip(np.round(W / ws_pl[:, None]), -127, 127).astype(np.int8)
    y_pl = oracle.bf16_to_f32(oracle.int8_linear(xb, w_pl, ws_pl, bb, mode=oracle.PER_ROW)["y"])
    ref = case.x.float().numpy().astype(np.float64) @ W.T.astype(np.float64) + oracle.bf16_to_f32(bb)
    e_rot = np.linalg.norm(y_rot - ref) / np.linalg.norm(ref)
    e_pl = np.linalg.norm(y_pl - ref) / np.linalg.norm(ref)
    assert e_rot < 0.02
    assert e_rot < e_pl


# ---------------------------------------------------------------- whole layer
@pytest.mark.parametrize("mode", [synthetic.TENSORWISE, synthetic.PER_ROW])
def test_linear_is_close_to_the_float_layer(mode):
    M, N, K = 48, 80, 256
    case = synthetic.make_case("t", M, N, K, mode, bias=True, seed=31)
    out = oracle.int8_linear(bits(case.x), case.w.numpy(), case.w_scale.numpy(), bits(case.bias), mode=mode)
    wf = case.w.numpy().astype(np.float64) * (case.w_scale.numpy().astype(np.float64)[:, None]
                                              if mode == synthetic.PER_ROW else float(case.w_scale[0]))
    ref = case.x.float().numpy().astype(np.float64) @ wf.T + oracle.bf16_to_f32(bits(case.bias))
    y = oracle.bf16_to_f32(out["y"]).astype(np.float64)
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 0.02  # the quantization error the pages call "~1 % against a bf16 reference"
    # and the composition is the GEMM of the quantized codes
    assert np.array_equal(out["acc"], out["q"].astype(np.int64) @ case.w.numpy().astype(np.int64).T)


# ---- the 16-bit-activation path (issue #278, "Suggested fix") -----------------------

def test_w8a16_brute_force_in_rationals():
    """Tiny case summed in exact rational arithmetic from the definition
    y = w_scale[n] * sum_k a[m,k] * w[n,k] + bias[n]."""
    M, N, K = 3, 4, 32
    x = synthetic.normal_bf16((M, K), seed=901)
    w = synthetic.int8_uniform((N, K), seed=902).numpy()
    ws = synthetic.scale_uniform(N, seed=903).numpy()
    b = synthetic.normal_bf16((1, N), seed=904).reshape(N)
    y, mag = oracle.w8a16_linear(bits(x), w, ws, bits(b), mode=oracle.PER_ROW)
    xf = x.float().numpy()
    bf = b.float().numpy()
    for m in range(M):
        for n in range(N):
            s = sum(Fraction(float(xf[m, k])) * int(w[n, k]) for k in range(K))
            exact = Fraction(float(ws[n])) * s + Fraction(float(bf[n]))
            assert abs(Fraction(y[m, n]) - exact) <= Fraction(1, 2 ** 50) * (abs(exact) + 1)
            ref_mag = Fraction(float(ws[n])) * sum(abs(Fraction(float(xf[m, k])) * int(w[n, k])) for k in range(K))
            assert abs(Fraction(mag[m, n]) - ref_mag) <= Fraction(1, 2 ** 50) * (ref_mag + 1)


def test_w8a16_one_hot_weights_select_activations():
    """w[n] = c * e_{k_n}: y[m,n] = w_scale[n] * c * x[m,k_n] + bias[n], exactly."""
    M, N, K = 5, 6, 48
    x = synthetic.normal_bf16((M, K), seed=911)
    ks = [3, 0, 47, 20, 11, 33]
    cs = [1, -127, 127, 5, -2, 64]
    w = np.zeros((N, K), np.int8)
    for n, (k, c) in enumerate(zip(ks, cs)):
        w[n, k] = c
    ws = np.array([0.5, 0.25, 2.0, 1.0, 0.125, 4.0], np.float32)  # powers of two: exact
    y, _ = oracle.w8a16_linear(bits(x), w, ws, None, mode=oracle.PER_ROW)
    xf = x.float().numpy().astype(np.float64)
    for n, (k, c) in enumerate(zip(ks, cs)):
        assert np.array_equal(y[:, n], float(ws[n]) * c * xf[:, k])


def test_w8a16_tensorwise_uses_the_single_scale():
    M, N, K = 4, 8, 64
    x = synthetic.normal_bf16((M, K), seed=921)
    w = synthetic.int8_uniform((N, K), seed=922).numpy()
    y1, m1 = oracle.w8a16_linear(bits(x), w, np.array([0.01], np.float32), None, mode=oracle.TENSORWISE)
    y2, m2 = oracle.w8a16_linear(bits(x), w, np.full((N,), 0.01, np.float32), None, mode=oracle.PER_ROW)
    assert np.array_equal(y1, y2) and np.array_equal(m1, m2)


def test_w8a16_agrees_with_the_int8_path_when_quantization_is_lossless():
    """Rows that are integers times 2^e with |max| = 127 * 2^e quantize without loss
    (x_scale = 2^e, q = x / 2^e), so the INT8 layer and the 16-bit path compute the
    same real number: the INT8 epilogue rounds it in fp32 and then to bf16, the
    16-bit value rounded to bf16 must be within one bf16 step of it."""
    M, N, K = 8, 16, 256
    g = np.random.default_rng(931)
    q = g.integers(-127, 128, size=(M, K))
    q[:, 0] = 127
    e = g.integers(-6, 4, size=(M, 1))
    xv = (q * (2.0 ** e)).astype(np.float32)
    x = torch.tensor(xv).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.tensor(xv))  # all exact in bf16
    w = synthetic.int8_uniform((N, K), seed=932).numpy()
    ws = synthetic.scale_uniform(N, seed=933).numpy()
    b = synthetic.normal_bf16((1, N), seed=934).reshape(N)
    r8 = oracle.int8_linear(bits(x), w, ws, bits(b), mode=oracle.PER_ROW)
    assert np.array_equal(r8["xs"], (2.0 ** e[:, 0]).astype(np.float32))
    y16, _ = oracle.w8a16_linear(bits(x), w, ws, bits(b), mode=oracle.PER_ROW)
    y16_bits = oracle.f32_to_bf16(y16.astype(np.float32))
    d = np.abs(oracle.bf16_to_f32(y16_bits).astype(np.float64) - oracle.bf16_to_f32(r8["y"]).astype(np.float64))
    step = np.abs(oracle.bf16_to_f32(r8["y"]).astype(np.float64)) * 2.0 ** -7 + 1e-30
    assert np.all(d <= step)


def test_w8a16_convrot_rounds_the_rotated_activation_once():
    """x rows = c * e_j (c a power of two): x @ H = c * H[j] / sqrt(128), whose fp32
    values are +-c * 0x3DB504F3, rounded to bf16 0x3DB5.  With an all-ones weight row,
    y = w_scale * c * bf16(1/sqrt(128)) * sum_k H[j,k] = 128 * (...) for j = 0, else 0."""
    K = 128
    rows = [0, 1, 5, 127]
    c = 4.0
    xv = np.zeros((len(rows), K), np.float32)
    for i, j in enumerate(rows):
        xv[i, j] = c
    x = torch.tensor(xv).to(torch.bfloat16)
    w = np.ones((2, K), np.int8)
    ws = np.array([1.0, 0.5], np.float32)
    y, mag = oracle.w8a16_linear(bits(x), w, ws, None, mode=oracle.CONVROT)
    h = float(oracle.bf16_to_f32(np.array([0x3DB5], np.uint16))[0])
    for i, j in enumerate(rows):
        expect = c * h * (128 if j == 0 else 0)
        assert y[i, 0] == expect and y[i, 1] == 0.5 * expect
        assert mag[i, 0] == c * h * 128


def test_w8a16_convrot_approximates_the_float_layer():
    """The rotated-basis layer with an INT8 weight approximates x @ W^T (the only loss
    is the weight's quantization and one bf16 rounding of x @ H)."""
    M, N, K = 16, 64, 512
    x = synthetic.normal_bf16((M, K), seed=941)
    W = synthetic.normal_f32((N, K), seed=942, std=0.02).numpy()
    w, ws = oracle.prepare_convrot_weight(W)
    y, _ = oracle.w8a16_linear(bits(x), w, ws, None, mode=oracle.CONVROT)
    ref = x.float().numpy().astype(np.float64) @ W.astype(np.float64).T
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) < 0.01


# ---- residual-fused epilogue ---------------------------------------------------------

@pytest.mark.parametrize("out_dtype", [oracle.OUT_BF16, oracle.OUT_F16, oracle.OUT_F32])
def test_residual_zero_is_the_plain_epilogue(out_dtype):
    M, N = 16, 24
    g = np.random.default_rng(951)
    acc = g.integers(-2 ** 20, 2 ** 20, size=(M, N)).astype(np.int32)
    xs = synthetic.scale_uniform(M, seed=952, mul=0.02).numpy()
    ws = synthetic.scale_uniform(N, seed=953, mul=0.01).numpy()
    b = bits(synthetic.normal_bf16((1, N), seed=954).reshape(N))
    plain = oracle.dequant_typed(acc, xs, ws, b, out_dtype=out_dtype)
    with_r = oracle.dequant_residual(acc, xs, ws, np.zeros((M, N), np.float32), b, out_dtype=out_dtype)
    assert np.array_equal(plain.view(np.uint8), with_r.view(np.uint8))


def test_residual_cancelling_the_layer_gives_zero():
    """r = -(the fp32 layer value): the last addition is exact and gives 0."""
    M, N = 8, 16
    g = np.random.default_rng(961)
    acc = g.integers(-2 ** 20, 2 ** 20, size=(M, N)).astype(np.int32)
    xs = synthetic.scale_uniform(M, seed=962).numpy()
    ws = synthetic.scale_uniform(N, seed=963).numpy()
    t = oracle.dequant_typed(acc, xs, ws, None, out_dtype=oracle.OUT_F32)
    y = oracle.dequant_residual(acc, xs, ws, -t, None, out_dtype=oracle.OUT_F32)
    assert np.all(y == 0.0)


def test_residual_hand_example():
    """acc = 12, xs = 0.5, ws = 0.25, bias = 1, r = 0.5: ((12 * 0.5) * 0.25 + 1) + 0.5 = 3."""
    acc = np.array([[12]], np.int32)
    y = oracle.dequant_residual(acc, np.array([0.5], np.float32), np.array([0.25], np.float32),
                                np.array([[0.5]], np.float32), to_bf16_bits([1.0]), out_dtype=oracle.OUT_F32)
    assert y[0, 0] == 3.0


def test_residual_within_rounding_of_the_exact_value():
    """Every fp32 step rounds once: the result is within 4 * 2^-24 * (|acc xs ws| +
    |bias| + |r|) of the exact rational value (fp32 output)."""
    M, N = 12, 20
    g = np.random.default_rng(971)
    acc = g.integers(-2 ** 22, 2 ** 22, size=(M, N)).astype(np.int32)
    xs = synthetic.scale_uniform(M, seed=972).numpy()
    ws = synthetic.scale_uniform(N, seed=973).numpy()
    b = synthetic.normal_bf16((1, N), seed=974).reshape(N)
    r = g.standard_normal((M, N)).astype(np.float32)
    y = oracle.dequant_residual(acc, xs, ws, r, bits(b), out_dtype=oracle.OUT_F32)
    bf = b.float().numpy()
    for m in range(M):
        for n in range(N):
            prod = Fraction(int(acc[m, n])) * Fraction(float(xs[m])) * Fraction(float(ws[n]))
            exact = prod + Fraction(float(bf[n])) + Fraction(float(r[m, n]))
            bound = (abs(prod) + abs(Fraction(float(bf[n]))) + abs(Fraction(float(r[m, n])))) * Fraction(4, 2 ** 24)
            assert abs(Fraction(float(y[m, n])) - exact) <= bound


# ---------------------------------------------------------------- epilogue operation order
def _rne_f32_bits(v):
    """Exact rational -> fp32 bits, round to nearest even (normal numbers only), written
    out from the format's definition: 24 significant bits, exponent bias 127."""
    if v == 0:
        return 0
    sign = 0x80000000 if v < 0 else 0
    a = abs(Fraction(v))
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    m = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if fl == 1 << 24:
        fl >>= 1
        e += 1
    assert -126 <= e <= 127
    return sign | ((e + 127) << 23) | (fl - (1 << 23))


def _f32_value(b):
    """fp32 bits -> exact rational (normal numbers)."""
    e = ((b >> 23) & 0xFF) - 127
    m = (b & 0x7FFFFF) | (1 << 23)
    v = Fraction(m) * Fraction(2) ** (e - 23)
    return -v if b & 0x80000000 else v


def _bf16_value(b):
    return _f32_value(b << 16)


def _read_epilogue_examples():
    rows = []
    with open(os.path.join(GOLDEN, "epilogue_order_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            acc, xs, ws, bias, want, other = [p.strip() for p in line.split("|")]
            rows.append((int(acc), int(xs, 16), int(ws, 16), None if bias == "-" else int(bias, 16), int(want, 16),
                         int(other, 16)))
    return rows


def test_epilogue_order_worked_examples():
    """The hand-derived examples of tests/golden/epilogue_order_examples.txt: the oracle's
    epilogue gives the left-to-right bits, which exact rational arithmetic confirms step by
    step; the contrasting evaluation (another multiplication order, or an FMA for the bias
    add) gives the other bits, so a change of order in the oracle would fail here."""
    rows = _read_epilogue_examples()
    assert len(rows) == 2
    for acc, xs_b, ws_b, bias_b, want, other in rows:
        xs, ws = _f32_value(xs_b), _f32_value(ws_b)
        t1 = _rne_f32_bits(acc * xs)
        t2 = _rne_f32_bits(_f32_value(t1) * ws)
        if bias_b is None:
            left = t2
            alt = _rne_f32_bits(acc * _f32_value(_rne_f32_bits(xs * ws)))          # acc * (xs * ws)
            alt2 = _rne_f32_bits(_f32_value(_rne_f32_bits(acc * ws)) * xs)         # (acc * ws) * xs
            assert alt == alt2 == other
        else:
            left = _rne_f32_bits(_f32_value(t2) + _bf16_value(bias_b))
            alt = _rne_f32_bits(_f32_value(t1) * ws + _bf16_value(bias_b))        # fused multiply-add
            assert alt == other
        assert left == want and want != other
        got = oracle.dequant_typed(np.array([[acc]], np.int32), np.array([xs_b], np.uint32).view(np.float32),
                                   np.array([ws_b], np.uint32).view(np.float32),
                                   None if bias_b is None else np.array([bias_b], np.uint16),
                                   out_dtype=oracle.OUT_F32)
        assert int(got.view(np.uint32)[0, 0]) == want, "oracle epilogue gave %#x, expected %#x" % (
            int(got.view(np.uint32)[0, 0]), want)
        # the same value through the tensorwise (scalar-scale) form of the epilogue
        got_s = oracle.dequant_typed(np.array([[acc]], np.int32), np.array([xs_b], np.uint32).view(np.float32),
                                     np.array([ws_b], np.uint32).view(np.float32),
                                     None if bias_b is None else np.array([bias_b], np.uint16),
                                     scalar_scales=True, out_dtype=oracle.OUT_F32)
        assert int(got_s.view(np.uint32)[0, 0]) == want

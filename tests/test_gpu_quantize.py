"""GPU parity of the activation quantize kernels against the CPU oracle: int8 codes and
fp32 scales must be bit-identical (integer decisions taken in fp32 on both sides)."""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
from helpers import (bits, from_bits, guarded, assert_guards_intact, assert_all_written, CODE_NEVER, NAN32)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def check_rowwise(x_cpu, rotate):
    """Codes and scales written into guard-banded buffers pre-filled with values the
    quantize never produces (code -128, NaN scales): every element must be written, none
    outside, and all of them equal to the oracle's."""
    q_ref, s_ref = oracle.quantize_rowwise(bits(x_cpu), rotate=rotate)
    M, K = x_cpu.shape
    qbuf, q = guarded((M, K), torch.int8, CODE_NEVER)
    sbuf, s = guarded((M,), torch.float32, NAN32)
    ck.ck_quantize_int8_rowwise(x_cpu.to(DEV), rotate=rotate, q=q, x_scale=s)
    torch.cuda.synchronize()
    assert_guards_intact(qbuf, CODE_NEVER)
    assert_guards_intact(sbuf, NAN32)
    assert_all_written(qbuf, CODE_NEVER)
    assert_all_written(sbuf, NAN32)
    s_np = s.cpu().numpy()
    assert np.array_equal(s_np.view(np.uint32), s_ref.view(np.uint32)), "x_scale differs"
    qn = q.cpu().numpy()
    bad = np.argwhere(qn != q_ref)
    assert bad.size == 0, "q differs at %d places, first %s: gpu %d oracle %d" % (
        len(bad), bad[0], qn[tuple(bad[0])], q_ref[tuple(bad[0])])


# register-resident paths for every threads-per-row choice of the plain rows (32 x 2/4/8,
# 64 x 6/8, 128 x 6/8, 256 x 6/8: K up to 16384), ragged row tails, and the two-pass path
# for longer rows
@pytest.mark.parametrize("M,K", [(256, 512), (37, 16), (9, 48), (21, 1024), (100, 2048), (11, 3072), (3, 6144),
                                 (5, 5376), (7, 6160), (13, 4096), (9, 8192), (3, 12288), (2, 16384), (2, 16400),
                                 (2, 65536)])
def test_rowwise_parity(M, K):
    check_rowwise(synthetic.normal_bf16((M, K), seed=100 + K), rotate=False)


@pytest.mark.parametrize("M,K", [(64, 128), (33, 384), (16, 4096), (3, 8192), (2, 4224), (3, 12288),
                                 (2, 16384), (2, 16512)])
def test_rowwise_convrot_parity(M, K):
    oc = synthetic.outlier_columns(K, 0.01, seed=7)
    check_rowwise(synthetic.normal_bf16((M, K), seed=200 + K, outlier_channels=oc), rotate=True)


def test_convrot_workload_quantize_parity():
    M, K = 4096, 3072
    oc = synthetic.outlier_columns(K, 0.01, seed=5 + 404)
    check_rowwise(synthetic.normal_bf16((M, K), seed=5, outlier_channels=oc), rotate=True)


def test_exhaustive_bf16_significands():
    """Every bf16 row maximum significand x every bf16 value below it (13 binades, both
    signs): the reciprocal-and-correction quotient must round exactly like IEEE division."""
    vals = []
    for e in range(0, 13):
        for m in range(128):
            v = (1.0 + m / 128.0) * 2.0 ** (-e)
            vals += [v, -v]
    vals = np.array(vals, np.float64)
    rows = []
    for e_top in (0, 40, -60):
        for m in range(128):
            amax = (1.0 + m / 128.0) * 2.0 ** e_top
            r = vals * 2.0 ** e_top
            r = r[np.abs(r) <= amax]
            row = np.zeros(3344, np.float64)
            row[0] = amax
            row[1:1 + len(r)] = r
            rows.append(row)
    x = torch.tensor(np.array(rows), dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(x.float().double(), torch.tensor(np.array(rows)))  # all bf16-exact
    check_rowwise(x, rotate=False)


def test_zero_and_subnormal_rows():
    x = synthetic.normal_bf16((6, 256), seed=3)
    xb = bits(x).copy()
    xb[0] = 0
    xb[1] = 0x8000  # -0
    xb[2] = np.array([0x0001, 0x8003, 0x0040, 0x0000] * 64, np.uint16)
    xb[3, 1:] = 0
    check_rowwise(from_bits(xb), rotate=False)
    check_rowwise(from_bits(xb), rotate=True)


@pytest.mark.parametrize("M,K", [(4096, 4096), (7, 48), (1, 16), (333, 1040)])
def test_tensorwise_parity(M, K):
    x = synthetic.normal_bf16((M, K), seed=300 + K)
    q_ref, s_ref = oracle.quantize_tensorwise(bits(x))
    qbuf, q = guarded((M, K), torch.int8, CODE_NEVER)
    sbuf, s = guarded((1,), torch.float32, NAN32)
    ck.ck_quantize_int8_tensorwise(x.to(DEV), q=q, x_scale=s)
    torch.cuda.synchronize()
    assert_guards_intact(qbuf, CODE_NEVER)
    assert_guards_intact(sbuf, NAN32)
    assert_all_written(qbuf, CODE_NEVER)
    assert s.cpu().numpy().view(np.uint32)[0] == s_ref.view(np.uint32)[0]
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_empty_batch_is_a_no_op():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    q, s = ck.ck_quantize_int8_rowwise(x)
    torch.cuda.synchronize()
    assert q.shape == (0, 64) and s.shape == (0,)


@pytest.mark.parametrize("N,K", [(12288, 3072), (5, 128), (33, 16384), (3, 16512), (7, 4224), (256, 512)])
def test_convrot_weight_preparation_parity(N, K):
    """W fp32 -> int8 codes of W @ H^T and fp32 row scales, bit-exact with the oracle's
    preparation (the ConvRot workload's weight is the first shape)."""
    W = synthetic.normal_f32((N, K), seed=N + K, std=0.02)
    w_ref, s_ref = oracle.prepare_convrot_weight(W.numpy())
    w, s = ck.ck_convrot_prepare_weight(W.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    wn = w.cpu().numpy()
    bad = np.argwhere(wn != w_ref)
    assert bad.size == 0, "%d codes differ, first %s" % (len(bad), bad[0])


def test_convrot_weight_preparation_rejects_unaligned_k():
    W = torch.zeros((4, 200), dtype=torch.float32, device=DEV)
    with pytest.raises(ck.CkError) as e:
        ck.ck_convrot_prepare_weight(W)
    assert "128" in str(e.value)


def test_every_bf16_row_maximum():
    """x_scale = fl(max|x| / 127) for every finite non-negative bf16 row maximum (32640
    of them, subnormals and zero included), and the codes of a row holding its maximum,
    its negative, a third of it and zeros: bit-exact with the oracle's IEEE division."""
    amax = np.arange(0, 0x7F80, dtype=np.uint16)
    K = 16
    xb = np.zeros((amax.size, K), np.uint16)
    xb[:, 0] = amax
    xb[:, 1] = amax | 0x8000
    third = (torch.from_numpy(amax.view(np.int16)).view(torch.bfloat16).float() / 3).to(torch.bfloat16)
    xb[:, 2] = bits(third)
    check_rowwise(from_bits(xb), rotate=False)


def _half_integer_rows(M, K, seed):
    """bf16 rows whose rotated values all sit within fp32 rounding of a half-integer
    multiple of the row's scale: block 0 holds 254 at one position (its transform is
    +-254/sqrt(128) everywhere, the row maximum, so x_scale is about 2/sqrt(128)); every
    other 128-block holds two integers a, b with a + b odd, whose transform is
    +-(a + b)/sqrt(128) or +-(a - b)/sqrt(128), i.e. (a +- b)/2 in units of the scale."""
    rng = np.random.default_rng(seed)
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        x[m, rng.integers(0, 128)] = 254.0 * (1 if m % 2 else -1)
        for blk in range(1, K // 128):
            p1, p2 = rng.choice(128, 2, replace=False)
            a = int(rng.integers(-127, 128))
            b = int(rng.integers(-127, 127))
            if (a + b) % 2 == 0:
                b += 1
            x[m, blk * 128 + p1], x[m, blk * 128 + p2] = a, b
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(64, 1024), (48, 3072), (16, 4096), (8, 16384)])
def test_convrot_half_integer_quotients(M, K):
    """Nearly every code of these rows is decided by the last bits of the quotient (the
    near-tie branch of the ConvRot rounding, packed and scalar slots alike): the GPU codes
    and scales must still equal the oracle's IEEE division."""
    x = _half_integer_rows(M, K, seed=K + M)
    _, s_ref = oracle.quantize_rowwise(bits(x), rotate=True)
    # the quotients in exact arithmetic (float64 transform): within 2^-12 of a half-integer
    H = scipy.linalg.hadamard(128) / np.sqrt(128.0)
    v = (x.double().numpy().reshape(M, K // 128, 128) @ H).reshape(M, K)[:, 128:]
    t = np.abs(v / s_ref.astype(np.float64)[:, None])
    assert (np.abs(t - np.floor(t) - 0.5) < 2.0 ** -12).mean() > 0.95
    check_rowwise(x, rotate=True)


def test_convrot_weight_half_integer_quotients():
    """The same construction through the ConvRot weight preparation (fp32 rows)."""
    W = _half_integer_rows(96, 1024, seed=3).float()
    w_ref, s_ref = oracle.prepare_convrot_weight(W.numpy())
    w, s = ck.ck_convrot_prepare_weight(W.to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(w.cpu().numpy(), w_ref)

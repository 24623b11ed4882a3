"""GPU parity of the tensor-core GEMM: raw int32 accumulators bit-exact against the
oracle (including adversarial inputs that stress the exact-fp32-chunk argument), and
the fused dequant epilogue bit-identical to the oracle's (0 ulp in every output type).
Outputs and workspaces sit between guard bands pre-filled with values the kernels never
write, so a skipped tile or a stray write fails the test."""
import numpy as np
import pytest
import torch

import oracle
import int8_weight_quantized_gb300 as ck
from int8_weight_quantized_gb300 import synthetic
from helpers import (bits, bf16_ulp_distance, out_bits, ulp_distance, MAX_ULP, guarded, assert_guards_intact,
                     assert_all_written, guarded_workspace, assert_workspace_guards_intact, NAN16, NAN32, ACC_NEVER)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_acc(q, w):
    """The raw accumulators, written between guard bands of a value no exact accumulator
    can take (INT32_MIN), with a guard-banded workspace of random bytes."""
    M, K = q.shape
    N = w.shape[0]
    abuf, acc = guarded((M, N), torch.int32, ACC_NEVER)
    wbuf, ws, before = guarded_workspace(ck.load_library().ck_int8_gemm_workspace_size(M, N, K), seed=M + N)
    ck.ck_int8_gemm_s32(q.to(DEV), w.to(DEV), acc=acc, ws=ws)
    torch.cuda.synchronize()
    assert_guards_intact(abuf, ACC_NEVER)
    assert_all_written(abuf, ACC_NEVER)
    assert_workspace_guards_intact(wbuf, before)
    return acc.cpu().numpy()


# several tiles, ragged M/N/K tails, one and several 1024-wide K chunks; single tile rows
# (unpaired CTAs) and odd numbers of tile rows (the last CTA pair's second tile lies
# wholly below M)
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (1, 8, 16), (129, 264, 80), (300, 520, 1040),
                                   (128, 256, 2048), (1000, 776, 3088), (77, 1032, 5376), (384, 256, 256),
                                   (640, 1280, 1024), (2304, 512, 160)])
def test_s32_parity(M, N, K):
    q = synthetic.int8_uniform((M, K), seed=M + K)
    w = synthetic.int8_uniform((N, K), seed=N + 7 * K)
    ref = oracle.gemm_s32(q.numpy(), w.numpy())
    got = gpu_acc(q, w)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, "%d mismatches, first at %s: %d vs %d" % (len(bad), bad[0], got[tuple(bad[0])],
                                                                     ref[tuple(bad[0])])


@pytest.mark.parametrize("K", [1024, 1040, 2048, 4096, 65536])
def test_s32_extreme_magnitudes(K):
    """All +127 x +127 reaches the largest chunk partial (16,516,096 < 2^24 per 1024);
    [127]*1023 + [1] keeps an odd total near 2^24 (low-bit retention); alternating signs
    cancel exactly."""
    M, N = 130, 264
    q = torch.full((M, K), 127, dtype=torch.int8)
    q[1::4] = -127
    q[2::4, ::2] = -127
    q[3::4, 1023::1024] = 1
    w = torch.full((N, K), 127, dtype=torch.int8)
    w[1::2] = -127
    w[2::8, 1023::1024] = 1
    ref = oracle.gemm_s32(q.numpy(), w.numpy())
    got = gpu_acc(q, w)
    assert np.array_equal(got, ref)
    assert got[0, 0] == 127 * 127 * K


def test_s32_int32_range_end():
    """K = 131072 (the largest accepted): |acc| = 2,114,060,288, near the int32 limit."""
    M, N, K = 128, 256, 131072
    q = torch.full((M, K), 127, dtype=torch.int8)
    q[1::2] = -127
    w = torch.full((N, K), 127, dtype=torch.int8)
    got = gpu_acc(q, w)
    assert got[0, 0] == 127 * 127 * K and got[1, 0] == -127 * 127 * K
    assert np.all(got[0::2] == 127 * 127 * K) and np.all(got[1::2] == -127 * 127 * K)


@pytest.mark.parametrize("scalar", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (129, 264, 1040), (1, 8, 16), (385, 520, 192)])
def test_dequant_parity(M, N, K, scalar, with_bias):
    q = synthetic.int8_uniform((M, K), seed=11 + M)
    w = synthetic.int8_uniform((N, K), seed=12 + N)
    xs = synthetic.scale_uniform(1 if scalar else M, seed=13, mul=0.02)
    ws = synthetic.scale_uniform(1 if scalar else N, seed=14, mul=0.01)
    b = synthetic.normal_bf16((1, N), seed=15, std=0.5).reshape(N) if with_bias else None
    acc = oracle.gemm_s32(q.numpy(), w.numpy())
    ref = oracle.dequant(acc, xs.numpy(), ws.numpy(), None if b is None else bits(b), scalar_scales=scalar)
    ybuf, y = guarded((M, N), torch.bfloat16, NAN16)
    ck.ck_int8_gemm_dequant(q.to(DEV), xs.to(DEV), w.to(DEV), ws.to(DEV), None if b is None else b.to(DEV),
                            scalar_scales=scalar, y=y)
    torch.cuda.synchronize()
    assert_guards_intact(ybuf, NAN16)
    assert_all_written(ybuf, NAN16)
    d = bf16_ulp_distance(bits(y), ref)
    assert d.max() <= MAX_ULP, "max ulp %d at %s" % (d.max(), np.unravel_index(d.argmax(), d.shape))


@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("bn", [256, 224, 192, 160, 128, 96, 64, 32])
def test_s32_every_tile_width(monkeypatch, bn, pair):
    """The tile width is chosen per launch (multiples of 32 up to 256); every width, with
    CTA pairs and with single CTAs, gives the exact accumulators (ragged M, N and K)."""
    monkeypatch.setenv("CK_GEMM_BN", str(bn))
    monkeypatch.setenv("CK_GEMM_PAIR", pair)
    assert ck.ck_gemm_tile_config(300, 712, 1104)[:2] == (bn, pair == "1")
    M, N, K = 300, 712, 1104
    q = synthetic.int8_uniform((M, K), seed=bn + 1)
    w = synthetic.int8_uniform((N, K), seed=bn + 2)
    assert np.array_equal(gpu_acc(q, w), oracle.gemm_s32(q.numpy(), w.numpy()))


@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("K", [16, 64, 80, 128, 144, 192, 1040])
def test_s32_k_inside_and_across_stages(monkeypatch, K, pair):
    """CTA pairs stage 128-deep k-blocks (two 64-deep boxes per operand), single CTAs
    64-deep ones: K shorter than one box, than one stage, and ending inside a stage's first
    or second box all give the exact accumulators (the boxes past K are zero-filled)."""
    monkeypatch.setenv("CK_GEMM_PAIR", pair)
    M, N = 300, 264
    assert ck.ck_gemm_tile_config(M, N, K)[1] == (pair == "1")
    q = synthetic.int8_uniform((M, K), seed=K + 11)
    w = synthetic.int8_uniform((N, K), seed=K + 12)
    assert np.array_equal(gpu_acc(q, w), oracle.gemm_s32(q.numpy(), w.numpy()))


TYPED = [(torch.float16, oracle.OUT_F16), (torch.float32, oracle.OUT_F32), (torch.bfloat16, oracle.OUT_BF16)]


def typed_reference(q, w, xs, ws, b, scalar, code):
    acc = oracle.gemm_s32(q.numpy(), w.numpy())
    ref = oracle.dequant_typed(acc, xs.numpy(), ws.numpy(), None if b is None else bits(b), scalar_scales=scalar,
                               out_dtype=code)
    return ref.view(np.uint32) if code == oracle.OUT_F32 else ref


@pytest.mark.parametrize("out_dtype,code", TYPED)
@pytest.mark.parametrize("scalar,with_bias", [(False, True), (True, False), (False, False)])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (129, 264, 1040), (1, 8, 16), (385, 520, 192)])
def test_dequant_output_types(M, N, K, scalar, with_bias, out_dtype, code):
    """The epilogue's fp32 value rounded to fp16 / stored as fp32 (the out_dtype of
    int8_linear): bit-identical to the oracle in that type."""
    q = synthetic.int8_uniform((M, K), seed=21 + M)
    w = synthetic.int8_uniform((N, K), seed=22 + N)
    xs = synthetic.scale_uniform(1 if scalar else M, seed=23, mul=0.02)
    ws = synthetic.scale_uniform(1 if scalar else N, seed=24, mul=0.01)
    b = synthetic.normal_bf16((1, N), seed=25, std=0.5).reshape(N) if with_bias else None
    ref = typed_reference(q, w, xs, ws, b, scalar, code)
    pattern = NAN32 if out_dtype == torch.float32 else NAN16
    ybuf, y = guarded((M, N), out_dtype, pattern)
    ck.ck_int8_gemm_dequant(q.to(DEV), xs.to(DEV), w.to(DEV), ws.to(DEV), None if b is None else b.to(DEV),
                            scalar_scales=scalar, out_dtype=out_dtype, y=y)
    torch.cuda.synchronize()
    assert_guards_intact(ybuf, pattern)
    assert_all_written(ybuf, pattern)
    assert y.dtype == out_dtype
    d = ulp_distance(out_bits(y), ref)
    assert d.max() <= MAX_ULP, "max ulp %d at %s" % (d.max(), np.unravel_index(d.argmax(), d.shape))


def test_f16_output_overflow_and_subnormals():
    """Scales that push outputs past fp16's range (-> +-inf) and into its subnormals."""
    M, N, K = 130, 264, 256
    q = synthetic.int8_uniform((M, K), seed=31)
    w = synthetic.int8_uniform((N, K), seed=32)
    xs = synthetic.scale_uniform(M, seed=33, mul=1.0)
    xs[::3] *= 1e-9   # |y| ~ 1e-9 * 1e4 * ws: fp16 subnormals
    xs[1::3] *= 1e3   # |y| beyond 65504
    ws = synthetic.scale_uniform(N, seed=34, mul=0.01)
    ref = typed_reference(q, w, xs, ws, None, False, oracle.OUT_F16)
    y = ck.ck_int8_gemm_dequant(q.to(DEV), xs.to(DEV), w.to(DEV), ws.to(DEV), None, out_dtype=torch.float16)
    torch.cuda.synchronize()
    got = out_bits(y)
    assert np.any((ref & 0x7FFF) == 0x7C00) and np.any(((ref & 0x7C00) == 0) & ((ref & 0x3FF) != 0))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("bn", [256, 160, 96, 32])
def test_f32_output_every_tile_width(monkeypatch, bn):
    """fp32 outputs leave the tile in 16-column boxes: every tile width, ragged M and N."""
    monkeypatch.setenv("CK_GEMM_BN", str(bn))
    M, N, K = 300, 712, 272
    q = synthetic.int8_uniform((M, K), seed=bn + 41)
    w = synthetic.int8_uniform((N, K), seed=bn + 42)
    xs = synthetic.scale_uniform(M, seed=43, mul=0.02)
    ws = synthetic.scale_uniform(N, seed=44, mul=0.01)
    b = synthetic.normal_bf16((1, N), seed=45, std=0.5).reshape(N)
    ref = typed_reference(q, w, xs, ws, b, False, oracle.OUT_F32)
    ybuf, y = guarded((M, N), torch.float32, NAN32)
    ck.ck_int8_gemm_dequant(q.to(DEV), xs.to(DEV), w.to(DEV), ws.to(DEV), b.to(DEV), out_dtype=torch.float32, y=y)
    torch.cuda.synchronize()
    assert_guards_intact(ybuf, NAN32)
    assert_all_written(ybuf, NAN32)
    assert ulp_distance(out_bits(y), ref).max() <= MAX_ULP


def test_tile_config_query(monkeypatch):
    """The planner's choice is a valid configuration, follows the A/B overrides, and the
    GEMM stays exact when launched with whatever it picked."""
    for M, N, K in [(4096, 4096, 4096), (128, 4096, 4096), (80666, 28672, 5376), (1, 8, 16)]:
        bn, pair, resident, split = ck.ck_gemm_tile_config(M, N, K)
        assert bn % 32 == 0 and 32 <= bn <= 256 and resident >= 1 and 1 <= split <= 8
        assert not pair or (M + 127) // 128 >= 2
    monkeypatch.setenv("CK_GEMM_BN", "96")
    monkeypatch.setenv("CK_GEMM_PAIR", "0")
    assert ck.ck_gemm_tile_config(4096, 4096, 4096)[:2] == (96, False)
    monkeypatch.setenv("CK_GEMM_PAIR", "1")
    assert ck.ck_gemm_tile_config(4096, 4096, 4096)[:2] == (96, True)
    assert ck.ck_gemm_tile_config(128, 4096, 4096)[:2] == (96, False)  # one tile row: no pair


def run_s32(q, w, ws=None):
    M, K = q.shape
    N = w.shape[0]
    abuf, acc = guarded((M, N), torch.int32, ACC_NEVER)
    ck.ck_int8_gemm_s32(q.to(DEV), w.to(DEV), acc=acc, ws=ws)
    torch.cuda.synchronize()
    assert ck.ck_device_error(clear=False) == 0
    assert_guards_intact(abuf, ACC_NEVER)
    assert_all_written(abuf, ACC_NEVER)
    return acc.cpu().numpy()


# shapes whose last partial wave is split along K: CTA pairs and single CTAs, K ranges
# that do not divide evenly among the slices, one-slice-per-1024-K chunk boundaries
@pytest.mark.parametrize("M,N,K,pair,split", [
    (512, 1024, 2048, "1", "8"), (512, 1024, 2048, "1", "3"), (300, 712, 1104, "0", "4"), (300, 712, 1104, "1", "2"),
    (4096, 2560, 1040, "1", "2"), (130, 264, 4160, "0", "7"), (1000, 520, 3088, "1", "5"),
])
def test_split_tail_exact(monkeypatch, M, N, K, pair, split):
    """Units of the last partial wave computed as K-slices by different pairs / CTAs and
    summed by the slice that arrives last: the int32 accumulators stay exact."""
    monkeypatch.setenv("CK_GEMM_PAIR", pair)
    monkeypatch.setenv("CK_GEMM_SPLIT", split)
    assert ck.ck_gemm_tile_config(M, N, K)[3] == int(split)
    q = synthetic.int8_uniform((M, K), seed=M + 3)
    w = synthetic.int8_uniform((N, K), seed=N + 4)
    ref = oracle.gemm_s32(q.numpy(), w.numpy())
    # the slices' int32 partial sums and arrival slots live in the workspace: guard-banded
    wbuf, ws, before = guarded_workspace(ck.load_library().ck_int8_gemm_workspace_size(M, N, K), seed=M + K)
    for _ in range(2):  # the second launch finds the first one's arrival slots
        got = run_s32(q, w, ws=ws)
        bad = np.argwhere(got != ref)
        assert bad.size == 0, "%d mismatches, first at %s" % (len(bad), bad[0])
        assert_workspace_guards_intact(wbuf, before)


def test_split_tail_after_full_waves(monkeypatch):
    """4096^3 with 256x256 pair tiles: three full waves, the last 28 tiles split in two
    along K.  Exact on a row sample that includes the split tiles' rows (the last tile
    rows of the grouped order)."""
    monkeypatch.setenv("CK_GEMM_PAIR", "1")
    monkeypatch.setenv("CK_GEMM_BN", "256")
    monkeypatch.setenv("CK_GEMM_SPLIT", "2")
    M, N, K = 4096, 4096, 4096
    bn, pair, resident, split = ck.ck_gemm_tile_config(M, N, K)
    assert (bn, pair) == (256, True) and (resident != 76 or split == 2)
    q = synthetic.int8_uniform((M, K), seed=71)
    w = synthetic.int8_uniform((N, K), seed=72)
    got = run_s32(q, w)
    rows = synthetic.sample_rows(M, n_random=48, seed=73)
    ref = oracle.gemm_s32(q[rows].numpy(), w.numpy())
    assert np.array_equal(got[rows], ref)


def test_split_tail_ignores_stale_workspace(monkeypatch):
    """The arrival slots are tagged per launch: a workspace full of random bytes (or of
    an earlier launch's slots) changes nothing."""
    monkeypatch.setenv("CK_GEMM_SPLIT", "4")
    M, N, K = 512, 1024, 2048
    assert ck.ck_gemm_tile_config(M, N, K)[3] == 4
    q = synthetic.int8_uniform((M, K), seed=51)
    w = synthetic.int8_uniform((N, K), seed=52)
    ref = oracle.gemm_s32(q.numpy(), w.numpy())
    nbytes = ck.load_library().ck_int8_gemm_workspace_size(M, N, K)
    g = torch.Generator(device=DEV)
    g.manual_seed(53)
    ws = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=DEV, generator=g)
    assert np.array_equal(run_s32(q, w, ws=ws), ref)
    assert np.array_equal(run_s32(q, w, ws=ws), ref)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_split_tail_dequant(monkeypatch, out_dtype):
    """The fused epilogue after a K-split: bit-identical to the oracle, as without it."""
    monkeypatch.setenv("CK_GEMM_SPLIT", "3")
    M, N, K = 512, 1024, 2048
    q = synthetic.int8_uniform((M, K), seed=61)
    w = synthetic.int8_uniform((N, K), seed=62)
    xs = synthetic.scale_uniform(M, seed=63, mul=0.02)
    ws = synthetic.scale_uniform(N, seed=64, mul=0.01)
    b = synthetic.normal_bf16((1, N), seed=65, std=0.5).reshape(N)
    code = oracle.OUT_F32 if out_dtype == torch.float32 else oracle.OUT_BF16
    ref = typed_reference(q, w, xs, ws, b, False, code)
    y = ck.ck_int8_gemm_dequant(q.to(DEV), xs.to(DEV), w.to(DEV), ws.to(DEV), b.to(DEV), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ulp_distance(out_bits(y), ref).max() <= MAX_ULP


def residual_case(M, N, out_dtype, seed):
    r = synthetic.normal_bf16((M, N), seed=seed, std=2.0).to(out_dtype)
    return r, r.float().numpy()


@pytest.mark.parametrize("out_dtype,code", TYPED)
@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (129, 264, 1040), (1, 8, 16)])
def test_dequant_residual(M, N, K, inplace, out_dtype, code):
    """y = out(((acc * xs) * ws + bias) + residual), the residual in y's type; in place
    (residual is y) as well."""
    q = synthetic.int8_uniform((M, K), seed=81 + M)
    w = synthetic.int8_uniform((N, K), seed=82 + N)
    xs = synthetic.scale_uniform(M, seed=83, mul=0.02)
    ws = synthetic.scale_uniform(N, seed=84, mul=0.01)
    b = synthetic.normal_bf16((1, N), seed=85, std=0.5).reshape(N)
    r, r_np = residual_case(M, N, out_dtype, seed=86)
    acc = oracle.gemm_s32(q.numpy(), w.numpy())
    ref = oracle.dequant_residual(acc, xs.numpy(), ws.numpy(), r_np, bits(b), out_dtype=code)
    ref = ref.view(np.uint32) if code == oracle.OUT_F32 else ref
    r_dev = r.to(DEV)
    y = ck.ck_int8_gemm_dequant(q.to(DEV), xs.to(DEV), w.to(DEV), ws.to(DEV), b.to(DEV), out_dtype=out_dtype,
                                residual=r_dev, y=r_dev if inplace else None)
    torch.cuda.synchronize()
    d = ulp_distance(out_bits(y), ref)
    assert d.max() <= MAX_ULP, "max ulp %d" % d.max()


def test_residual_after_a_split_tail(monkeypatch):
    monkeypatch.setenv("CK_GEMM_SPLIT", "3")
    M, N, K = 512, 1024, 2048
    q = synthetic.int8_uniform((M, K), seed=91)
    w = synthetic.int8_uniform((N, K), seed=92)
    xs = synthetic.scale_uniform(M, seed=93, mul=0.02)
    ws = synthetic.scale_uniform(N, seed=94, mul=0.01)
    r, r_np = residual_case(M, N, torch.bfloat16, seed=95)
    ref = oracle.dequant_residual(oracle.gemm_s32(q.numpy(), w.numpy()), xs.numpy(), ws.numpy(), r_np, None)
    y = ck.ck_int8_gemm_dequant(q.to(DEV), xs.to(DEV), w.to(DEV), ws.to(DEV), None, residual=r.to(DEV))
    torch.cuda.synchronize()
    assert bf16_ulp_distance(bits(y), ref).max() <= MAX_ULP

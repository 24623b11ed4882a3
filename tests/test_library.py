"""The C-ABI library builds for sm_103a, loads on the host, and exports every entry
point include/ck_int8.h declares; the binding and the library reject bad arguments
before touching a GPU.  No compute call is made here."""
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ck_int8.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ck_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from int8_weight_quantized_gb300 import build
    build.build()
    import int8_weight_quantized_gb300 as ck
    return ck.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ck_quantize_int8_rowwise", "ck_int8_linear", "ck_int8_linear_workspace_size",
                     "ck_quantize_int8_tensorwise", "ck_int8_gemm_dequant", "ck_int8_gemm_s32",
                     "ck_last_error", "ck_device_error", "ck_selftest_wait_timeout"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_workspace_sizes(lib):
    import int8_weight_quantized_gb300 as ck
    M, N, K = 4096, 4096, 4096
    ws = lib.ck_int8_linear_workspace_size(M, N, K, ck.PER_ROW)
    assert ws >= 2 * M * K + 2 * N * K + 4 * M
    # 64-bit sizes: a workspace above 2^31 bytes is reported without wrapping
    big = lib.ck_int8_linear_workspace_size(200000, 21504, 8192, ck.PER_ROW)
    assert big >= 2 * 200000 * 8192 + 2 * 21504 * 8192 > 2 ** 31
    assert lib.ck_int8_gemm_workspace_size(M, N, K) >= 2 * (M + N) * K


def _call_linear(lib, M, N, K, mode, **kw):
    import ctypes
    P = ctypes.c_void_p
    ptr = P(4096)  # never dereferenced: validation fails first
    args = dict(x=ptr, w=ptr, ws=ptr, bias=None, y=ptr, work=ptr, nbytes=1 << 40, out_dtype=0)
    args.update(kw)
    return lib.ck_int8_linear(args["x"], args["w"], args["ws"], args["bias"], args.get("residual"), args["y"], M, N, K,
                              mode, args["out_dtype"], args["work"], args["nbytes"], None)


@pytest.mark.parametrize("M,N,K,mode,what", [
    (16, 16, 24, 1, "multiple of 16"),        # K % 16
    (16, 12, 32, 1, "multiple of 8"),         # N % 8
    (16, 16, 64, 2, "ConvRot"),               # ConvRot K % 128
    (16, 16, 32, 7, "mode"),                  # bad mode
    (-1, 16, 32, 1, ">= 0"),                  # negative M
    (16, 16, 262144, 1, "overflow"),          # K too large for int32
    (2 ** 31, 16, 32, 1, "2^31"),             # coordinate range
])
def test_invalid_shapes_are_rejected_without_a_gpu(lib, M, N, K, mode, what):
    import int8_weight_quantized_gb300 as ck
    st = _call_linear(lib, M, N, K, mode)
    assert st == ck.CK_ERR_INVALID_ARG
    assert what in ck.ck_last_error()


def test_unknown_output_type_is_rejected(lib):
    import int8_weight_quantized_gb300 as ck
    assert _call_linear(lib, 16, 16, 32, 1, out_dtype=3) == ck.CK_ERR_INVALID_ARG
    assert "out_dtype" in ck.ck_last_error()
    import ctypes
    P = ctypes.c_void_p(4096)
    st = lib.ck_int8_gemm_dequant(P, P, P, P, None, None, P, 16, 16, 32, 0, -1, P, 1 << 40, None)
    assert st == ck.CK_ERR_INVALID_ARG and "out_dtype" in ck.ck_last_error()
    with pytest.raises(ValueError):
        ck.ck_int8_linear(torch.zeros((16, 32), dtype=torch.bfloat16), torch.zeros((16, 32), dtype=torch.int8),
                          torch.ones(16), out_dtype=torch.int32)


def test_null_and_misaligned_pointers_are_rejected(lib):
    import ctypes
    import int8_weight_quantized_gb300 as ck
    assert _call_linear(lib, 16, 16, 32, 1, x=None) == ck.CK_ERR_INVALID_ARG
    assert "x must not be NULL" in ck.ck_last_error()
    assert _call_linear(lib, 16, 16, 32, 1, w=ctypes.c_void_p(4097)) == ck.CK_ERR_INVALID_ARG
    assert "16-byte aligned" in ck.ck_last_error()
    assert _call_linear(lib, 16, 16, 32, 1, nbytes=10) == ck.CK_ERR_INVALID_ARG
    assert "workspace too small" in ck.ck_last_error()
    assert _call_linear(lib, 16, 16, 32, 1, residual=ctypes.c_void_p(4104)) == ck.CK_ERR_INVALID_ARG
    assert "residual must be 16-byte aligned" in ck.ck_last_error()


def test_no_device_is_reported_not_faked(lib):
    """With valid arguments and no GPU the call fails with a CUDA/device status: there
    is no CPU fallback behind the ABI."""
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import int8_weight_quantized_gb300 as ck
    st = _call_linear(lib, 16, 16, 32, 1)
    assert st in (ck.CK_ERR_CUDA, ck.CK_ERR_UNSUPPORTED_DEVICE)


def test_binding_type_checks():
    import int8_weight_quantized_gb300 as ck
    x = torch.zeros((4, 32), dtype=torch.float32)
    with pytest.raises(TypeError):
        ck.ck_quantize_int8_rowwise(x)


def test_product_package_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "int8_weight_quantized_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ck_oracle" not in text, f


def test_tile_config_query_validates_without_a_gpu(lib):
    import ctypes
    import int8_weight_quantized_gb300 as ck
    bn, pair = ctypes.c_int(), ctypes.c_int()
    assert lib.ck_gemm_tile_config(16, 12, 32, ctypes.byref(bn), ctypes.byref(pair), None, None) == \
        ck.CK_ERR_INVALID_ARG
    st = lib.ck_gemm_tile_config(16, 16, 32, ctypes.byref(bn), ctypes.byref(pair), None, None)
    if not torch.cuda.is_available():
        assert st in (ck.CK_ERR_CUDA, ck.CK_ERR_UNSUPPORTED_DEVICE)


def test_workspace_views(lib):
    """Where the layer leaves its activation codes and scales: the codes first, x_scale
    after the bf16 activation and weight operands, both inside the workspace and aligned;
    bad arguments are rejected."""
    import ctypes
    import int8_weight_quantized_gb300 as ck
    for M, N, K, mode in [(4096, 4096, 4096, ck.TENSORWISE), (300, 264, 1152, ck.PER_ROW),
                          (4096, 12288, 3072, ck.CONVROT), (1, 8, 16, ck.TENSORWISE)]:
        co, xo = ck.ck_int8_linear_workspace_views(M, N, K, mode)
        size = lib.ck_int8_linear_workspace_size(M, N, K, mode)
        n_scales = 1 if mode == ck.TENSORWISE else M
        assert co == 0 and co + 2 * M * K <= xo
        assert xo >= 2 * M * K + 2 * N * K and xo % 256 == 0
        assert xo + 4 * n_scales <= size
    sz = ctypes.c_size_t()
    assert lib.ck_int8_linear_workspace_views(16, 8, 16, 7, ctypes.byref(sz), ctypes.byref(sz)) == ck.CK_ERR_INVALID_ARG
    assert lib.ck_int8_linear_workspace_views(16, 8, 16, 1, None, ctypes.byref(sz)) == ck.CK_ERR_INVALID_ARG


def test_host_layer_arguments(lib):
    """The host-memory layer: workspace sizes grow with the slab, bad arguments are
    rejected before any device work."""
    import ctypes
    import int8_weight_quantized_gb300 as ck
    a = lib.ck_int8_linear_host_workspace_size(10000, 4096, 2048, ck.PER_ROW, 0, 512)
    b = lib.ck_int8_linear_host_workspace_size(10000, 4096, 2048, ck.PER_ROW, 0, 1024)
    assert 2 * 512 * 4096 * 2 <= a < b
    # tensorwise keeps all of x on the device
    assert lib.ck_int8_linear_host_workspace_size(10000, 4096, 2048, ck.TENSORWISE, 0, 512) > a
    P = ctypes.c_void_p
    ptr = P(4096)
    st = lib.ck_int8_linear_host(ptr, ptr, ptr, None, ptr, 64, 64, 64, ck.PER_ROW, 0, -1, ptr, 1 << 40, None)
    assert st == ck.CK_ERR_INVALID_ARG and "slab_rows" in ck.ck_last_error()
    st = lib.ck_int8_linear_host(ptr, ptr, ptr, None, ptr, 64, 64, 60, ck.PER_ROW, 0, 0, ptr, 1 << 40, None)
    assert st == ck.CK_ERR_INVALID_ARG


def test_prepared_weight_entry_points_without_a_gpu(lib):
    """The layer on prepared weight codes: its workspace holds no widened weight, and bad
    arguments are rejected before any device work."""
    import ctypes
    import int8_weight_quantized_gb300 as ck
    M, N, K = 1000, 4096, 2048
    for mode in (ck.TENSORWISE, ck.PER_ROW, ck.CONVROT):
        full = lib.ck_int8_linear_workspace_size(M, N, K, mode)
        codes = lib.ck_int8_linear_codes_workspace_size(M, N, K, mode)
        assert codes > 0 and full - codes >= 2 * N * K  # the bf16 weight codes are the caller's
    P = ctypes.c_void_p
    ptr = P(4096)
    st = lib.ck_int8_linear_codes(ptr, None, ptr, None, None, ptr, 64, 64, 64, ck.PER_ROW, 0, ptr, 1 << 40, None)
    assert st == ck.CK_ERR_INVALID_ARG and "w_codes" in ck.ck_last_error()
    st = lib.ck_int8_linear_codes(ptr, P(4100), ptr, None, None, ptr, 64, 64, 64, ck.PER_ROW, 0, ptr, 1 << 40, None)
    assert st == ck.CK_ERR_INVALID_ARG and "aligned" in ck.ck_last_error()
    st = lib.ck_int8_linear_codes(ptr, ptr, ptr, None, None, ptr, 64, 64, 64, ck.PER_ROW, 0, ptr, 16, None)
    assert st == ck.CK_ERR_INVALID_ARG and "workspace" in ck.ck_last_error()
    st = lib.ck_int8_weight_codes(ptr, 64, 60, ptr, None)
    assert st == ck.CK_ERR_INVALID_ARG and "16" in ck.ck_last_error()
    assert lib.ck_int8_weight_codes(ptr, 0, 64, ptr, None) == ck.CK_OK  # no rows: nothing to do

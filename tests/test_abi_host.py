"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/dwconv.h declares, computes output
sizes, and rejects bad arguments before it touches the CUDA runtime."""
import ctypes
import os
import re

import pytest

import oracle
from depthwise_convolution_gb300 import _lib, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dwconv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dwconv_\w+)\s*\(", src)))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("dwconv_fwd", "dwconv_bwd_data", "dwconv_bwd_filter",
                     "dwconv_bwd_filter_workspace_size", "dwconv_output_size",
                     "dwconv_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libdwconv.so does not export {name}"
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


@pytest.mark.parametrize("H,W,F,S,D,P", [(56, 56, 7, 1, 1, 3), (112, 112, 5, 2, 2, 4), (56, 56, 31, 1, 1, 15),
                                         (8, 8, 3, 1, 1, 1), (7, 9, 3, 2, 1, 0), (10, 10, 3, 3, 2, 2),
                                         (5, 5, 4, 1, 1, 0), (17, 13, 5, 2, 3, 6)])
def test_output_size_matches_the_oracle(lib, H, W, F, S, D, P):
    assert ops.dwconv_output_size(H, W, F, F, S, D, P) == (oracle.out_extent(H, F, S, D, P),
                                                          oracle.out_extent(W, F, S, D, P))


@pytest.mark.parametrize("args", [(0, 4, 3, 3, 1, 1, 0), (4, 4, 5, 5, 1, 1, 0), (4, 4, 3, 3, 0, 1, 0),
                                  (4, 4, 3, 3, 1, 0, 0), (4, 4, 3, 3, 1, 1, -1)])
def test_output_size_rejects_bad_sizes(lib, args):
    oh = ctypes.c_int(-7)
    assert lib.dwconv_output_size(*args, ctypes.byref(oh), None) == _lib.ERR_INVALID_ARG
    assert oh.value == -7


@pytest.mark.parametrize("H,W,FH,FW,axes", [(9, 40, 1, 31, (1, 1, 1, 1, 0, 15)), (21, 30, 3, 5, (2, 1, 1, 1, 1, 2)),
                                             (17, 33, 5, 5, (1, 2, 2, 2, 4, 3)), (8, 8, 3, 3, (1, 3, 2, 1, 2, 0))])
def test_per_axis_output_size_matches_the_oracle(lib, H, W, FH, FW, axes):
    sh, sw, dh, dw, ph, pw = axes
    got = ops.dwconv_output_size(H, W, FH, FW, (sh, sw), (dh, dw), (ph, pw))
    assert got == (oracle.out_extent(H, FH, sh, dh, ph), oracle.out_extent(W, FW, sw, dw, pw))


def test_symmetric_forms_equal_the_per_axis_forms(lib):
    oh1, ow1, oh2, ow2 = (ctypes.c_int(0) for _ in range(4))
    assert lib.dwconv_output_size(17, 13, 5, 5, 2, 3, 6, ctypes.byref(oh1), ctypes.byref(ow1)) == 0
    assert lib.dwconv_output_size_2d(17, 13, 5, 5, 2, 2, 3, 3, 6, 6, ctypes.byref(oh2), ctypes.byref(ow2)) == 0
    assert (oh1.value, ow1.value) == (oh2.value, ow2.value)
    assert lib.dwconv_bwd_filter_workspace_size(4, 56, 56, 96, 7, 7, 1, 1, 3, _lib.FP16) == \
        lib.dwconv_bwd_filter_workspace_size_2d(4, 56, 56, 96, 7, 7, 1, 1, 1, 1, 3, 3, _lib.FP16)


def test_per_axis_validation_before_any_launch(lib):
    before = lib.dwconv_launch_count()
    A_ = 0x7F0000000000
    args = (2, 8, 8, 16, 3, 3)
    assert lib.dwconv_fwd_2d(*args, 1, 0, 1, 1, 1, 1, _lib.FP16, A_, A_, None, A_, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_fwd_2d(*args, 1, 1, 1, 1, 1, -1, _lib.FP16, A_, A_, None, A_, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_bwd_data_2d(*args, 1, 1, 1, 1, 1, 1, _lib.INT8, A_, A_, A_, None) == _lib.ERR_UNSUPPORTED
    assert lib.dwconv_bwd_filter_2d(*args, 1, 1, 1, 1, 1, 1, _lib.FP16, A_, A_, A_, None, 0, None) == \
        _lib.ERR_INVALID_ARG                                           # workspace too small
    assert lib.dwconv_launch_count() == before


def test_status_strings(lib):
    for code in range(6):
        assert lib.dwconv_status_string(code).decode().startswith("DWCONV_")
    assert b"unknown" in lib.dwconv_status_string(99)


# Fake device addresses: never dereferenced, because validation fails first.
A = 0x7F0000000000


def fwd(lib, *, N=2, H=8, W=8, C=16, F=3, S=1, D=1, P=1, dt=_lib.FP16, x=A, w=A, b=None, y=A):
    return lib.dwconv_fwd(N, H, W, C, F, F, S, D, P, dt, x, w, b, y, None)


def test_fwd_validation_before_any_launch(lib):
    before = lib.dwconv_launch_count()
    assert fwd(lib, N=0) == _lib.ERR_INVALID_ARG
    assert fwd(lib, C=-1) == _lib.ERR_INVALID_ARG
    assert fwd(lib, H=2, F=5, P=0) == _lib.ERR_INVALID_ARG        # empty output
    assert fwd(lib, S=0) == _lib.ERR_INVALID_ARG
    assert fwd(lib, P=-1) == _lib.ERR_INVALID_ARG
    assert fwd(lib, dt=7) == _lib.ERR_INVALID_ARG
    assert fwd(lib, x=None) == _lib.ERR_INVALID_ARG
    assert fwd(lib, y=None) == _lib.ERR_INVALID_ARG
    assert fwd(lib, x=A + 1) == _lib.ERR_MISALIGNED                 # fp16 needs 2-byte alignment
    assert fwd(lib, dt=_lib.FP32, w=A + 2) == _lib.ERR_MISALIGNED
    assert fwd(lib, dt=_lib.INT8, y=A + 2) == _lib.ERR_MISALIGNED  # int32 output
    assert fwd(lib, b=A + 2) == _lib.ERR_MISALIGNED                 # fp32 bias
    assert fwd(lib, N=1 << 20, H=1 << 12, W=1 << 12, C=1 << 10) == _lib.ERR_INVALID_ARG  # too large
    assert lib.dwconv_launch_count() == before


def test_backward_validation(lib):
    args = (2, 8, 8, 16, 3, 3, 1, 1, 1)
    assert lib.dwconv_bwd_data(*args, _lib.INT8, A, A, A, None) == _lib.ERR_UNSUPPORTED
    assert lib.dwconv_bwd_data(*args, _lib.BF16, None, A, A, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_bwd_data(*args, _lib.BF16, A, A, A + 1, None) == _lib.ERR_MISALIGNED
    need = lib.dwconv_bwd_filter_workspace_size(*args, _lib.BF16)
    assert need > 0
    assert lib.dwconv_bwd_filter(*args, _lib.INT8, A, A, A, A, need, None) == _lib.ERR_UNSUPPORTED
    assert lib.dwconv_bwd_filter(*args, _lib.BF16, A, A, A, A, need - 4, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_bwd_filter(*args, _lib.BF16, A, A, A, None, need, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_bwd_filter(*args, _lib.BF16, A, A, A + 2, A, need, None) == _lib.ERR_MISALIGNED


def fused(lib, *, dt=_lib.FP16, x=A, isc=None, ish=None, iact=0, b=None, osc=None, osh=None, oact=0, y=A):
    return lib.dwconv_fwd_fused_2d(2, 8, 8, 16, 3, 3, 1, 1, 1, 1, 1, 1, dt, x, isc, ish, iact, A, b,
                                   osc, osh, oact, y, None)


def test_fused_validation_before_any_launch(lib):
    before = lib.dwconv_launch_count()
    assert fused(lib, iact=5) == _lib.ERR_INVALID_ARG                  # activation outside the enum
    assert fused(lib, oact=-1) == _lib.ERR_INVALID_ARG
    assert fused(lib, dt=_lib.INT8, iact=_lib.ACT_RELU) == _lib.ERR_UNSUPPORTED
    assert fused(lib, dt=_lib.INT8, osh=A) == _lib.ERR_UNSUPPORTED
    assert fused(lib, isc=A + 2) == _lib.ERR_MISALIGNED                 # float vectors
    assert fused(lib, osh=A + 1) == _lib.ERR_MISALIGNED
    assert fused(lib, x=None, iact=_lib.ACT_GELU) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_launch_count() == before
    # the symmetric form validates the same way
    assert lib.dwconv_fwd_fused(2, 8, 8, 16, 3, 3, 1, 1, 1, _lib.FP16, A, None, None, 9, A, None, None, None, 0,
                                A, None) == _lib.ERR_INVALID_ARG


def test_python_fused_binding_checks_arguments():
    import torch
    x = torch.zeros(1, 4, 4, 8, dtype=torch.float16)
    w = torch.zeros(3, 3, 8, dtype=torch.float16)
    with pytest.raises(ValueError, match="unknown activation"):
        ops.dwconv_fwd_fused(x, w, in_act="tanh")
    with pytest.raises(ValueError, match="out_scale"):
        ops.dwconv_fwd_fused(x, w, out_scale=torch.ones(8, dtype=torch.float16))
    with pytest.raises(ValueError, match="CUDA"):
        ops.dwconv_fwd_fused(x, w, in_act="relu")


def test_half_accumulate_wgrad_validation(lib):
    args = (2, 8, 8, 16, 3, 3, 1, 1, 1)
    need = lib.dwconv_bwd_filter_workspace_size(*args, _lib.FP16)
    before = lib.dwconv_launch_count()
    for dt in (_lib.BF16, _lib.FP32, _lib.INT8):     # fp16 data only
        assert lib.dwconv_bwd_filter_ha(*args, dt, A, A, A, A, need, None) == _lib.ERR_UNSUPPORTED
    assert lib.dwconv_bwd_filter_ha(*args, _lib.FP16, A, A, A, A, need - 4, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_bwd_filter_ha(*args, _lib.FP16, None, A, A, A, need, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_bwd_filter_ha_2d(2, 8, 8, 16, 3, 3, 1, 1, 1, 1, 1, 1, _lib.FP16, A, A, A + 2, A, need,
                                       None) == _lib.ERR_MISALIGNED
    assert lib.dwconv_launch_count() == before


def test_fp8_is_forward_only(lib):
    args = (2, 8, 8, 16, 3, 3, 1, 1, 1)
    before = lib.dwconv_launch_count()
    F8 = _lib.FP8_E4M3
    assert lib.dwconv_bwd_data(*args, F8, A, A, A, None) == _lib.ERR_UNSUPPORTED
    assert lib.dwconv_bwd_filter_workspace_size(*args, F8) == 0
    assert lib.dwconv_bwd_filter(*args, F8, A, A, A, A, 1 << 20, None) == _lib.ERR_UNSUPPORTED
    assert lib.dwconv_bwd_filter_ha(*args, F8, A, A, A, A, 1 << 20, None) == _lib.ERR_UNSUPPORTED
    assert lib.dwconv_bwd_bias(2, 8, 8, 16, F8, A, A, A, 1 << 20, None) == _lib.ERR_UNSUPPORTED
    assert fused(lib, dt=F8, iact=_lib.ACT_RELU) == _lib.ERR_UNSUPPORTED   # no prologue for FP8
    assert fused(lib, dt=F8, y=A + 1) == _lib.ERR_MISALIGNED                 # bf16 output
    assert lib.dwconv_fwd(2, 8, 8, 16, 3, 3, 1, 1, 1, 5, A, A, None, A, None) == _lib.ERR_INVALID_ARG
    assert lib.dwconv_launch_count() == before


def test_workspace_size_is_a_pure_function_of_the_shape(lib):
    args = (128, 56, 56, 96, 7, 7, 1, 1, 3)
    a = lib.dwconv_bwd_filter_workspace_size(*args, _lib.FP16)
    assert a == lib.dwconv_bwd_filter_workspace_size(*args, _lib.BF16) > 0
    assert a % (7 * 7 * 96 * 4) == 0                       # whole slices of [FH][FW][C] floats
    assert lib.dwconv_bwd_filter_workspace_size(*args, _lib.INT8) == 0
    assert lib.dwconv_bwd_filter_workspace_size(0, 56, 56, 96, 7, 7, 1, 1, 3, _lib.FP16) == 0
    # a single output position cannot be split: one slice
    assert lib.dwconv_bwd_filter_workspace_size(1, 3, 3, 8, 3, 3, 1, 1, 0, _lib.FP32) == 3 * 3 * 8 * 4


def test_python_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(1, 4, 4, 8, dtype=torch.float16)
    w = torch.zeros(3, 3, 8, dtype=torch.float16)
    with pytest.raises(ValueError):
        ops.dwconv_fwd(x, w, pad=1)


def test_device_entry_points_report_a_missing_gpu_as_a_cuda_error(lib):
    # Without a GPU the failure-detection entry points return a status (nothing is launched).
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover these calls")
    assert lib.dwconv_selftest_timeout(None) == _lib.ERR_CUDA
    assert lib.dwconv_check_device_errors(None) == _lib.ERR_CUDA

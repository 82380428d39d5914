"""dwconv_bwd_filter_static, the weight gradient for callers that cannot
allocate device memory (for instance an operator living under a framework
whose allocator owns the device memory, or a deployment that forbids
allocation after start-up).  It uses scratch compiled into the library instead
of a caller workspace.

Called here straight through the C ABI (ctypes, raw device pointers) and
checked against the workspace entry point dwconv_bwd_filter on consecutive
calls, so that whatever one call leaves in the shared scratch cannot leak into
the next.  Both run the same kernels with the same split of the accumulation
axis and reduce it in a fixed order, so the two results must agree bit for
bit; each is also checked against the oracle within the usual tolerance.  This
file is named to be collected last.
"""
import pytest
import torch

import oracle
from depthwise_convolution_gb300 import _lib, ops
from parity import compare, random_inputs, to64

pytestmark = pytest.mark.gpu

CODE = {"fp32": _lib.FP32, "fp16": _lib.FP16, "bf16": _lib.BF16}


def static_call(lib, d, dtype, S, D, P, dw):
    x, dy = d["x"], d["dy"]
    N, H, W, C = x.shape
    FH, FW = d["w"].shape[:2]
    return lib.dwconv_bwd_filter_static(N, H, W, C, FH, FW, S, D, P, CODE[dtype], x.data_ptr(),
                                        dy.data_ptr(), dw.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)


# Consecutive calls: same shape with new data, then other shapes and dtypes.
CALLS = [
    ("bf16", (4, 28, 28, 96, 7, 7, 1, 1, 3), 11),
    ("bf16", (4, 28, 28, 96, 7, 7, 1, 1, 3), 12),
    ("fp16", (2, 20, 22, 64, 5, 5, 2, 2, 4), 13),
    ("fp32", (3, 13, 11, 40, 3, 3, 1, 1, 1), 14),
]


def check_one(lib, dtype, shape, seed):
    """One static call against the workspace entry point (bit for bit) and the
    oracle (within the tolerance of the other wgrad parity tests)."""
    N, H, W, C, FH, FW, S, D, P = shape
    host = random_inputs(dtype, N, H, W, C, FH, FW, S, D, P, seed=seed)
    d = {k: (None if v is None else v.cuda()) for k, v in host.items()}
    expect = ops.dwconv_bwd_filter(d["x"], d["dy"], FH, FW, S, D, P)
    got = torch.full((FH, FW, C), float("nan"), dtype=torch.float32, device="cuda")
    assert static_call(lib, d, dtype, S, D, P, got) == _lib.OK
    torch.cuda.synchronize()
    assert torch.equal(got, expect), f"static scratch {dtype} seed {seed}: differs from dwconv_bwd_filter"
    ref, mag = oracle.wgrad(to64(host["x"]), to64(host["dy"]), FH, FW, S, D, P)
    compare(to64(got), ref, mag, dtype, False, f"static scratch {dtype} seed {seed} vs oracle")


def test_static_scratch_matches_the_workspace_entry_point():
    lib = _lib.load()
    for dtype, shape, seed in CALLS:
        check_one(lib, dtype, shape, seed)


def test_static_scratch_rejects_shapes_beyond_its_size():
    lib = _lib.load()
    args = (1, 64, 64, 4096, 31, 31, 1, 1, 15)
    need = lib.dwconv_bwd_filter_workspace_size(*args, _lib.BF16)
    assert need > 8 << 20
    x = torch.zeros(1, 64, 64, 4096, dtype=torch.bfloat16, device="cuda")
    dw = torch.zeros(31, 31, 4096, dtype=torch.float32, device="cuda")
    before = lib.dwconv_launch_count()
    st = lib.dwconv_bwd_filter_static(*args, _lib.BF16, x.data_ptr(), x.data_ptr(), dw.data_ptr(), None)
    assert st == _lib.ERR_INVALID_ARG
    assert lib.dwconv_launch_count() == before
    assert lib.dwconv_bwd_filter_static(*args[:9], _lib.INT8, x.data_ptr(), x.data_ptr(),
                                        dw.data_ptr(), None) == _lib.ERR_UNSUPPORTED
    # A rejected call enqueues nothing and leaves the shared array usable: the
    # next valid call still matches the workspace entry point.
    check_one(lib, *CALLS[0][:2], seed=21)

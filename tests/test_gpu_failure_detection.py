"""Failure detection without a GPU fault: the library's bounded-wait path.

dwconv_selftest_timeout enqueues a wait that runs out on a shared-memory
barrier nothing completes (the kind of wait every tiled kernel makes for its
copies).  The next dwconv_check_device_errors must report DWCONV_ERR_TIMEOUT
once, the record must be cleared by that check, and the context must keep
working: a forward pass afterwards still matches the oracle.
"""
from __future__ import annotations

import pytest
import torch

from depthwise_convolution_gb300 import _lib, ops
from parity import check_fwd, random_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_once_and_context_stays_usable():
    ops.dwconv_check_device_errors()  # nothing pending
    ops.dwconv_selftest_timeout()
    with pytest.raises(_lib.DwconvError) as e:
        ops.dwconv_check_device_errors()
    assert e.value.status == _lib.ERR_TIMEOUT
    ops.dwconv_check_device_errors()  # the check cleared the record
    d = random_inputs("fp16", 2, 20, 40, 32, 7, 7, 1, 1, 3, seed=97)
    check_fwd(d, "fp16", 1, 1, 3, what="fwd after a reported timeout")


def test_timeout_on_a_side_stream_is_seen_by_that_stream_check():
    s = torch.cuda.Stream()
    ops.dwconv_selftest_timeout(stream=s)
    with pytest.raises(_lib.DwconvError) as e:
        ops.dwconv_check_device_errors(stream=s)
    assert e.value.status == _lib.ERR_TIMEOUT
    ops.dwconv_check_device_errors(stream=s)

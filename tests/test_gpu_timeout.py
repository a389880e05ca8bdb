"""Failure detection without a GPU fault: a host switch makes the GEMM's first
pipeline stage never arrive, every bounded wait in the kernel runs out after a
short limit, the kernel releases its tensor memory and returns, and the host
reads LYNX_ERR_TIMEOUT from the device error word.  The context stays usable:
the next call with the switch off gives the right answer."""
import numpy as np
import pytest

from oracle import cpp as O
import synth
from helpers import assert_y_close, to_bits, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(lynx):
    M, N, K = 256, 512, 512
    X = synth.act_bf16((1,), M, K, 0.05, 8.0)
    W = synth.gaussian_bf16((2,), (N, K), 1.0 / np.sqrt(K))
    LA = synth.gaussian_bf16((3,), (N, 64), 0.02)
    LB = synth.gaussian_bf16((4,), (64, K), 0.02)
    args = [to_dev(a) for a in (X, W, LA, LB)]
    assert lynx.lynx_sync_status() == lynx.LYNX_OK
    try:
        lynx.lynx_debug_set_fault(1, 50_000_000)  # 50 ms bound
        lynx.lynx_linear(*args)
        assert lynx.lynx_sync_status() == lynx.LYNX_ERR_TIMEOUT
    finally:
        lynx.lynx_debug_set_fault(0, 0)
    assert lynx.lynx_sync_status() == lynx.LYNX_OK  # the error word was cleared
    Y = lynx.lynx_linear(*args)
    assert lynx.lynx_sync_status() == lynx.LYNX_OK
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))

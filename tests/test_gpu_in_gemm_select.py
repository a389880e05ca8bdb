"""lynx_linear_fused: the 2:4 selection inside the GEMM (no sparsify pass).  Parity with the oracle at the stated
tolerance on ragged and structured inputs, agreement with the two-pass lynx_linear, and the full QKV size on
sampled rows."""
import numpy as np
import pytest

from oracle import cpp as O
import synth
from helpers import assert_y_close, to_bits, to_dev, widen

pytestmark = pytest.mark.gpu

CASES = [(256, 512, 512), (300, 520, 528), (1, 8, 16), (129, 136, 144), (200, 1000, 1024), (128, 256, 64),
         (384, 768, 3072), (200, 1003, 256), (600, 1160, 384), (777, 392, 1040)]


def _layer(M, N, K, seed, kind="act"):
    if kind == "act":
        X = synth.act_bf16((M, K, seed), M, K, 0.05, 8.0)
    elif kind == "gelu":
        X = synth.gelu_bf16((M, K, seed), M, K, 3.97, 0.0, 1.0)
    else:
        X = synth.structured_x(kind, M, K, seed)
    W = synth.gaussian_bf16((seed, 1), (N, K), 1.0 / np.sqrt(K))
    LA = synth.gaussian_bf16((seed, 2), (N, 64), 0.02)
    LB = synth.gaussian_bf16((seed, 3), (64, K), 0.02)
    return X, W, LA, LB


@pytest.mark.parametrize("M,N,K", CASES)
def test_in_gemm_select_matches_oracle(lynx, M, N, K):
    X, W, LA, LB = _layer(M, N, K, 41)
    Y = lynx.lynx_linear_fused(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


@pytest.mark.parametrize("kind", ["mixed", "equal", "two4", "ties", "zero", "gelu"])
def test_in_gemm_select_structured_inputs(lynx, kind):
    X, W, LA, LB = _layer(160, 384, 256, 43, kind)
    Y = to_bits(lynx.lynx_linear_fused(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB)))
    assert lynx.lynx_sync_status() == 0
    ref = O.linear(X, W, LA, LB)
    if kind == "zero":  # X = 0: both branches vanish
        assert np.all(Y == 0) and np.all(ref == 0)
    else:
        assert_y_close(Y, ref)


def test_in_gemm_select_agrees_with_two_pass(lynx):
    M, N, K = 512, 768, 3072
    X, W, LA, LB = _layer(M, N, K, 45)
    args = [to_dev(a) for a in (X, W, LA, LB)]
    y1 = to_bits(lynx.lynx_linear_fused(*args))
    y2 = to_bits(lynx.lynx_linear(*args))
    assert lynx.lynx_sync_status() == 0
    ref = O.linear(X, W, LA, LB)
    assert_y_close(y1, ref, "in-GEMM selection")
    assert_y_close(y2, ref, "two-pass")
    # the same selection and MMAs; s (summation order) and T' (T rounded to bf16 before the division by s: about
    # 2^-8 of the LoRA term, a tenth of an output unit) move the last bit of about one output in five
    assert np.mean(y1 == y2) > 0.7
    w1, w2 = widen(y1), widen(y2)
    assert np.linalg.norm(w1 - w2) <= 2.5e-3 * np.linalg.norm(w2)  # last-bit flips: about 2^-9 of |y|
    y3 = to_bits(lynx.lynx_linear_fused(*args))
    assert np.array_equal(y1, y3)


def test_in_gemm_select_full_size_qkv_sampled_rows(lynx):
    M, N, K = 4608, 9216, 3072
    X, W, LA, LB = _layer(M, N, K, 47)
    Y = to_bits(lynx.lynx_linear_fused(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB)))
    assert lynx.lynx_sync_status() == 0
    rows = np.r_[0:3, 255:258, 2047, 4600:4608]
    assert_y_close(Y[rows], O.linear(X[rows], W, LA, LB))


def test_in_gemm_select_argument_errors(lynx):
    import torch
    X, W, LA, LB = (to_dev(a) for a in _layer(64, 128, 256, 49))
    Y = torch.empty((64, 128), dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()
    lib = lynx.lib
    ws = torch.empty(lynx.lynx_dense_workspace_bytes(64, 64), dtype=torch.uint8, device="cuda")
    assert lib.lynx_linear_fused(p(X), p(W), None, p(LB), p(Y), 64, 128, 256, 64, p(ws), ws.numel(), None) == -1
    assert lib.lynx_linear_fused(p(X), p(W), p(LA), p(LB), p(Y), 64, 128, 256, 64, None, 0, None) == -1
    assert lib.lynx_linear_fused(p(X), p(W), p(LA), p(LB), p(Y), 64, 128, 256, 32, p(ws), ws.numel(), None) == -7
    assert lib.lynx_linear_fused(p(X), p(W), p(LA), p(LB), p(Y), 64, 128, 256, 64, p(ws), 16, None) == -4
    assert lib.lynx_linear_fused(p(X), p(W), p(LA), p(LB), p(Y), 64, 128, 250, 64, p(ws), ws.numel(), None) == -2

"""The largest sizes the C-ABI accepts (include/lynx.h: K <= 2^20, M <= 65535 * 128) and the smallest output
(N = 1), against the oracle: every row at the largest K, sampled rows (rows are independent) at the largest M."""
import numpy as np
import pytest

from oracle import cpp as O
import synth
from helpers import S_RTOL, assert_y_close, pack_meta_reference, to_bits, to_dev

pytestmark = pytest.mark.gpu


def _lora(seed, N, K):
    return (synth.gaussian_bf16((seed, 2), (N, 64), 0.02), synth.gaussian_bf16((seed, 3), (64, K), 0.02))


def test_linear_largest_k(lynx):
    """K = 2^20: 8192 channel blocks per row (one CTA pair walks all of them for the single output tile);
    the fp32 norm sums run over 2^20 terms per row."""
    M, N, K = 8, 40, 1 << 20
    X = synth.act_bf16((41, M, K), M, K, 0.03, 10.0)
    W = synth.gaussian_bf16((41, 1), (N, K), 1.0 / np.sqrt(K))
    LA, LB = _lora(41, N, K)
    vals, meta, s, T = lynx.lynx_sparsify_lora(to_dev(X), to_dev(LB))
    Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
    assert lynx.lynx_sync_status() == 0
    ref = O.sparsify(X)
    assert np.array_equal(to_bits(vals), ref["vals"])
    assert np.array_equal(meta.cpu().numpy(), pack_meta_reference(ref["meta"], M, K))
    np.testing.assert_allclose(s.cpu().numpy(), ref["s"], rtol=S_RTOL, atol=0)
    assert_y_close(to_bits(T), O.lora_down(X, LB, ref["s"]), "T")
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))


def test_linear_largest_m_sampled_rows(lynx):
    """M = 65535 * 128 = 8388480 rows (65536 row blocks of the pre-pass, 16384 pair tiles), K = 16, N = 8;
    the first and last rows (the ragged end) and 2000 random rows are compared with the oracle."""
    import torch
    M, N, K = 65535 * 128, 8, 16
    g = torch.Generator(device="cuda")
    g.manual_seed(43)
    Xd = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    W = synth.gaussian_bf16((43, 1), (N, K), 0.25)
    LA, LB = _lora(43, N, K)
    Y = lynx.lynx_linear(Xd, to_dev(W), to_dev(LA), to_dev(LB))
    vals, meta, s = lynx.lynx_sparsify(Xd)
    assert lynx.lynx_sync_status() == 0
    rng = np.random.default_rng(43)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(M - 200, M), rng.integers(0, M, 2000)]))
    idx = torch.from_numpy(rows).cuda()
    Xs = to_bits(Xd[idx])
    ref = O.sparsify(Xs)
    assert np.array_equal(to_bits(vals[idx]), ref["vals"])
    canon = lynx.lynx_meta_to_canonical(meta.cpu().numpy(), M, K)
    assert np.array_equal(canon[rows], ref["meta"])
    np.testing.assert_allclose(s[idx].cpu().numpy(), ref["s"], rtol=S_RTOL, atol=0)
    assert_y_close(to_bits(Y[idx]), O.linear(Xs, W, LA, LB))
    del Xd, Y, vals, meta, s
    torch.cuda.empty_cache()


@pytest.mark.parametrize("M,K", [(1, 16), (300, 3072)])
def test_linear_single_output_column(lynx, M, K):
    """N = 1: one W row, every pair tile almost entirely out of range; per-lane stores (N % 8 != 0)."""
    X = synth.act_bf16((44, M, K), M, K, 0.05, 8.0)
    W = synth.gaussian_bf16((44, 1), (1, K), 1.0 / np.sqrt(K))
    LA, LB = _lora(44, 1, K)
    Y = lynx.lynx_linear(to_dev(X), to_dev(W), to_dev(LA), to_dev(LB))
    assert lynx.lynx_sync_status() == 0
    assert_y_close(to_bits(Y), O.linear(X, W, LA, LB))

"""Pins of the CPU oracles against things other than themselves.

Two oracles compute the layer: the plain C++ one (``oracle/lynx_oracle.cpp``
through ``oracle/cpp.py``, the reference of the GPU tests) and the float64
numpy one (``oracle/lynx_oracle.py``).  Every pin below runs against both.

The RT-Lynx page prints no worked numeric example, so the oracles are pinned by
(a) hand-derived cases in tests/golden/hand_cases.json, (b) brute force over
every 4-tuple of a small alphabet with an independent formulation of the
selection, (c) closed-form invariants of the norm compensation, (d) pure-Python
loop evaluations of the layer on tiny inputs and (e) special cases that reduce
to a plain GEMM.  The two oracles are also compared with each other element by
element.  The last blocks plant mistakes in each oracle (on the CPU: a patched
numpy function, or a mutated copy of the C++ source compiled into a temporary
library) and check that some pin catches each one.
"""
import itertools
import json
import math
import os
import shutil
import tempfile

import numpy as np
import pytest

import oracle.cpp as CPP
import oracle.lynx_oracle as NP
import synth

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "hand_cases.json")))
SQRT2 = math.sqrt(2.0)


def bits(a):
    return synth.bf16_bits(np.asarray(a, dtype=np.float32))


@pytest.fixture(scope="module", params=["cpp", "numpy"])
def O(request):
    """Each oracle in turn: the C++ one (default build) and the numpy one."""
    return CPP.default() if request.param == "cpp" else NP


# ----------------------------------------------------------------------------- independent helpers
def brute_pair(group):
    """Lexicographically smallest index pair i < j maximising |x_i| + |x_j|.

    For "keep the two largest magnitudes, ties to the lower index" this is the
    same pair, reached without sorting.
    """
    best, arg = None, None
    for i, j in itertools.combinations(range(4), 2):
        v = abs(group[i]) + abs(group[j])
        if best is None or v > best:
            best, arg = v, (i, j)
    return arg


def exact_widen(b):
    """bf16 bits -> float64 through float32 (independent of both oracles' own conversions)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def loop_layer(x, w, la, lb):
    """Y = s*(X~ W^T) + (X LB^T) LA^T with Python loops and brute-force selection."""
    M, K = len(x), len(x[0])
    N, R = len(w), len(lb)
    y = [[0.0] * N for _ in range(M)]
    for m in range(M):
        row = x[m]
        kept = [0.0] * K
        for g in range(K // 4):
            i, j = brute_pair(row[4 * g:4 * g + 4])
            kept[4 * g + i] = row[4 * g + i]
            kept[4 * g + j] = row[4 * g + j]
        nx = math.sqrt(sum(v * v for v in row))
        nt = math.sqrt(sum(v * v for v in kept))
        s = nx / nt if nt > 0 else 1.0
        t = [sum(row[k] * lb[r][k] for k in range(K)) for r in range(R)]
        for n in range(N):
            ys = sum(kept[k] * w[n][k] for k in range(K))
            yr = sum(t[r] * la[n][r] for r in range(R))
            y[m][n] = s * ys + yr
    return np.array(y)


# ----------------------------------------------------------------------------- pins (reusable, any oracle)
ALPHABET = [-2.0, -1.0, -0.0, 0.0, 1.0, 2.0, 3.0]


def pin_widen(O):
    b = bits([0.0, -0.0, 1.0, -3.5, 1e-30, 65504.0, 3.0e38])
    assert np.array_equal(O.widen(b), exact_widen(b))
    assert np.signbit(O.widen(b)[1])


def pin_selection_exhaustive(O):
    tuples = np.array(list(itertools.product(ALPHABET, repeat=4)), dtype=np.float32)
    x = exact_widen(bits(tuples))
    i0, i1 = O.select_2of4(x)
    for t, a, b in zip(tuples.tolist(), i0[:, 0], i1[:, 0]):
        assert (a, b) == brute_pair(t), (t, a, b)


def pin_hand_sparsify(O):
    for case in GOLD["sparsify"]:
        xb = bits([case["x"]])
        out = O.sparsify(xb)
        m = out["mask"].reshape(-1, 4)
        kept = [tuple(np.nonzero(r)[0].tolist()) for r in m]
        assert kept == [tuple(p) for p in case["kept"]], case["name"]
        assert np.array_equal(out["vals"][0], bits(case["vals"])), case["name"]
        if case["meta"] is not None:
            assert out["meta"][0].tolist() == case["meta"], case["name"]
        assert abs(out["s"][0] - case["s"]) <= 1e-15 * case["s"], case["name"]


def pin_hand_linear(O):
    for case in GOLD["linear"]:
        y = O.linear(bits(case["X"]), bits(case["W"]), bits(case["LA"]), bits(case["LB"]))
        assert np.allclose(y, np.array(case["Y"]), rtol=1e-14, atol=0), (case["name"], y)


def pin_hand_lora_down(O):
    case = GOLD["linear"][0]
    X, LB = bits(case["X"]), bits(case["LB"])
    s = O.sparsify(X)["s"]
    # X LB^T = 1 - 3 + 2 + 0.5 + 4 = 4.5 (hand); divided by s = 5.5/sqrt(29)
    assert O.lora_down(X, LB)[0, 0] == 4.5
    assert abs(O.lora_down(X, LB, s)[0, 0] - 4.5 / (5.5 / math.sqrt(29.0))) < 1e-14


def pin_norm_restoration(O, X):
    x = exact_widen(X)
    out = O.sparsify(X)
    xt = np.where(out["mask"], x, 0.0)
    lhs = np.linalg.norm(out["s"][:, None] * xt, axis=1)
    rhs = np.linalg.norm(x, axis=1)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=0)
    assert np.all(out["s"] >= 1.0 - 1e-15) and np.all(out["s"] <= SQRT2 * (1 + 1e-15))


def pin_loops(O, seed, M=3, N=5, K=12, R=2):
    g = np.random.default_rng(seed)
    X = bits(g.standard_normal((M, K)))
    W = bits(g.standard_normal((N, K)))
    LA = bits(g.standard_normal((N, R)))
    LB = bits(g.standard_normal((R, K)))
    want = loop_layer(exact_widen(X).tolist(), exact_widen(W).tolist(), exact_widen(LA).tolist(),
                      exact_widen(LB).tolist())
    got = O.linear(X, W, LA, LB)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def pin_wsparse_loops(O, seed, M=3, N=4, K=12, R=2):
    """The weight-2:4 layer with Python loops: brute-force pair per group of each W row, no rescale."""
    g = np.random.default_rng(100 + seed)
    X, W, LA, LB = (bits(g.standard_normal(sh)) for sh in [(M, K), (N, K), (N, R), (R, K)])
    x, w, la, lb = (exact_widen(a).tolist() for a in (X, W, LA, LB))
    wk = []
    for n in range(N):
        kept = [0.0] * K
        for gi in range(K // 4):
            i, j = brute_pair(w[n][4 * gi:4 * gi + 4])
            kept[4 * gi + i] = w[n][4 * gi + i]
            kept[4 * gi + j] = w[n][4 * gi + j]
        wk.append(kept)
    want = [[sum(x[m][k] * wk[n][k] for k in range(K)) +
             sum(sum(x[m][k] * lb[r][k] for k in range(K)) * la[n][r] for r in range(R))
             for n in range(N)] for m in range(M)]
    assert np.allclose(O.linear_wsparse(X, W, LA, LB), want, rtol=1e-13, atol=1e-13)
    want_plain = [[sum(x[m][k] * wk[n][k] for k in range(K)) for n in range(N)] for m in range(M)]
    assert np.allclose(O.linear_wsparse(X, W), want_plain, rtol=1e-13, atol=1e-13)


def pin_dense_loops(O):
    g = np.random.default_rng(21)
    M, N, K, R = 3, 4, 8, 2
    X, W, LA, LB = (bits(g.standard_normal(sh)) for sh in [(M, K), (N, K), (N, R), (R, K)])
    x, w, la, lb = (exact_widen(a).tolist() for a in (X, W, LA, LB))
    want = [[sum(x[m][k] * w[n][k] for k in range(K)) +
             sum(sum(x[m][k] * lb[r][k] for k in range(K)) * la[n][r] for r in range(R))
             for n in range(N)] for m in range(M)]
    assert np.allclose(O.linear_dense(X, W, LA, LB), want, rtol=1e-13, atol=1e-13)
    want_plain = [[sum(x[m][k] * w[n][k] for k in range(K)) for n in range(N)] for m in range(M)]
    assert np.allclose(O.linear_dense(X, W), want_plain, rtol=1e-13, atol=1e-13)


def pin_meta_decodes_to_mask(O, kind="act"):
    M, K = 33, 64
    X = (synth.act_bf16((1, 2), M, K, 0.05, 8.0) if kind == "act" else synth.structured_x(kind, M, K, 3))
    out = O.sparsify(X)
    m = out["mask"].reshape(M, K // 4, 4)
    assert np.all(m.sum(-1) == 2)
    # vals are the kept entries, lower index first
    assert np.array_equal(out["vals"], X.reshape(M, K // 4, 4)[m].reshape(M, K // 2))
    # metadata decodes back to the mask
    meta = out["meta"]
    nib = np.stack([meta & 0xF, meta >> 4], axis=-1).reshape(M, K // 4)
    dec = np.zeros((M, K // 4, 4), dtype=bool)
    for g in range(K // 4):
        for r in range(M):
            n = int(nib[r, g])
            dec[r, g, n & 3] = True
            dec[r, g, n >> 2] = True
            assert (n & 3) < (n >> 2)
    assert np.array_equal(dec, m)


# ----------------------------------------------------------------------------- tests: pins hold (both oracles)
def test_widen_is_exact(O):
    pin_widen(O)


def test_selection_exhaustive_bruteforce(O):
    pin_selection_exhaustive(O)


def test_hand_cases_sparsify(O):
    pin_hand_sparsify(O)


def test_hand_case_linear(O):
    pin_hand_linear(O)


def test_lora_down_hand_case(O):
    pin_hand_lora_down(O)


@pytest.mark.parametrize("kind", ["act", "equal", "two4", "ties", "mixed"])
def test_exactly_two_per_group_and_packing(O, kind):
    pin_meta_decodes_to_mask(O, kind)


def test_norm_restoration_random(O):
    pin_norm_restoration(O, synth.act_bf16((5, 6), 64, 256, 0.03, 10.0))


def test_scale_special_cases(O):
    s = O.sparsify(synth.structured_x("equal", 16, 64, 1))["s"]
    assert np.allclose(s, SQRT2, rtol=1e-15, atol=0)
    s = O.sparsify(synth.structured_x("two4", 16, 64, 2))["s"]
    assert np.array_equal(s, np.ones(16))
    s = O.sparsify(synth.structured_x("zero", 4, 64, 3))["s"]
    assert np.array_equal(s, np.ones(4))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_linear_against_python_loops(O, seed):
    pin_loops(O, seed)


def test_linear_against_materialised_dense_reference(O):
    """S(X) as a dense M x K matrix and (LA LB) as a dense N x K matrix, a different association."""
    g = np.random.default_rng(11)
    M, N, K, R = 7, 10, 24, 3
    X = bits(g.standard_normal((M, K)) * 2)
    W, LA, LB = (bits(g.standard_normal(sh)) for sh in [(N, K), (N, R), (R, K)])
    x = exact_widen(X)
    sx = O.sparsify(X)
    S = sx["s"][:, None] * np.where(sx["mask"], x, 0.0)
    want = S @ exact_widen(W).T + x @ (exact_widen(LA) @ exact_widen(LB)).T
    assert np.allclose(O.linear(X, W, LA, LB), want, rtol=1e-12, atol=1e-12)


def test_already_24_and_zero_lora_is_plain_gemm(O):
    M, N, K, R = 5, 6, 16, 2
    X = synth.structured_x("two4", M, K, 4)
    g = np.random.default_rng(4)
    W = bits(g.standard_normal((N, K)))
    LA = np.zeros((N, R), dtype=np.uint16)
    LB = bits(g.standard_normal((R, K)))
    x, w = exact_widen(X).tolist(), exact_widen(W).tolist()
    gemm = np.array([[sum(x[m][k] * w[n][k] for k in range(K)) for n in range(N)] for m in range(M)])
    assert np.allclose(O.linear(X, W, LA, LB), gemm, rtol=1e-13, atol=1e-13)
    assert np.allclose(O.linear_dense(X, W), gemm, rtol=1e-13, atol=1e-13)


def test_zero_lb_leaves_scaled_sparse_branch(O):
    M, N, K, R = 4, 8, 32, 4
    X = synth.act_bf16((9,), M, K, 0.1, 8.0)
    g = np.random.default_rng(9)
    W, LA = bits(g.standard_normal((N, K))), bits(g.standard_normal((N, R)))
    LB = np.zeros((R, K), dtype=np.uint16)
    want = loop_layer(exact_widen(X).tolist(), exact_widen(W).tolist(), exact_widen(LA).tolist(),
                      exact_widen(LB).tolist())
    assert np.allclose(O.linear(X, W, LA, LB), want, rtol=1e-12, atol=1e-12)


def test_row_subset_equals_full_rows(O):
    t = synth.layer_tensors("tiny", "linear")
    rows = np.array([0, 3, 100, 255])
    full = O.linear(t["X"], t["W"], t["LA"], t["LB"])
    assert np.array_equal(O.linear(t["X"], t["W"], t["LA"], t["LB"], rows=rows), full[rows])


def test_dense_layer_against_loops(O):
    pin_dense_loops(O)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_weight_sparse_layer_against_python_loops(O, seed):
    pin_wsparse_loops(O, seed)


def test_weight_sparse_on_24_weights_is_the_dense_layer(O):
    """W that is already 2:4 (two zeros per group) is left unchanged: the dense layer's result."""
    W = synth.structured_x("two4", 24, 64, seed=3)
    X = synth.act_bf16((8, 1), 10, 64, 0.05, 8.0)
    LA, LB = synth.gaussian_bf16((8, 2), (24, 2), 0.1), synth.gaussian_bf16((8, 3), (2, 64), 0.1)
    assert np.array_equal(O.linear_wsparse(X, W, LA, LB), O.linear_dense(X, W, LA, LB))


def test_weight_sparse_is_the_transposed_activation_product(O):
    """X W~^T = (W~ X^T)^T, and W~ X^T is the activation path on W without its row scale: the same
    selection reached through the sparsified-activation functions."""
    X = synth.act_bf16((9, 1), 7, 32, 0.05, 8.0)
    W = synth.act_bf16((9, 2), 5, 32, 0.05, 8.0)
    zero_la, zero_lb = np.zeros((7, 2), np.uint16), np.zeros((2, 32), np.uint16)
    s_w = O.sparsify(W)["s"]
    via_activation = O.linear(W, X, zero_la, zero_lb) / s_w[:, None]
    assert np.allclose(O.linear_wsparse(X, W), via_activation.T, rtol=1e-12, atol=1e-12)


def test_lora_down_recombination(O):
    case = GOLD["linear"][0]
    X, LB, LA, W = (bits(case[k]) for k in ("X", "LB", "LA", "W"))
    s = O.sparsify(X)["s"]
    t = O.lora_down(X, LB, s)
    # s * (X~ W^T + T' LA^T) recombines to the layer output
    x = exact_widen(X)
    acc = np.where(O.sparsify(X)["mask"], x, 0.0) @ exact_widen(W).T + t @ exact_widen(LA).T
    assert np.allclose(s[:, None] * acc, O.linear(X, W, LA, LB), rtol=1e-14, atol=0)


# ----------------------------------------------------------------------------- the MLP activation (GELU of the up output)
def pin_gelu(O):
    """Closed forms: GELU(x) = x Phi(x); Phi(1) = 0.8413447460685429, Phi(-1) = 1 - Phi(1); GELU(0) = 0;
    GELU(x) - GELU(-x) = x (Phi(x) + Phi(-x) = 1); GELU(x) -> x and GELU(-x) -> 0 for large x."""
    g = O.gelu(np.array([1.0, -1.0, 0.0, 10.0, -10.0, 2.5, -2.5]))
    assert abs(g[0] - 0.8413447460685429) < 1e-15
    assert abs(g[1] + 0.15865525393145707) < 1e-15
    assert g[2] == 0.0
    assert abs(g[3] - 10.0) < 1e-14 and abs(g[4]) < 1e-14
    assert abs((g[5] - g[6]) - 2.5) < 1e-14


def pin_round_bf16(O):
    """Ties go to even on the 2^-7 grid of [1, 2); exactly representable values are kept; the grid of [2^k, 2^k+1)
    scales; every float32 rounds as torch rounds float32 to bf16."""
    ulp = 2.0 ** -7
    cases = [(1.0, 0x3F80), (1.0 + ulp / 2, 0x3F80), (1.0 + 1.5 * ulp, 0x3F82), (1.0 + ulp / 2 + 1e-12, 0x3F81),
             (-1.0 - ulp / 2, 0xBF80), (3.0, 0x4040), (0.0, 0x0000), (-0.0, 0x8000), (1e39, 0x7F80)]
    got = O.round_bf16(np.array([c[0] for c in cases]))
    assert got.tolist() == [c[1] for c in cases], [hex(v) for v in got]
    import torch
    f = np.random.default_rng(3).standard_normal(20000).astype(np.float32) * np.float32(7.0)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.round_bf16(f.astype(np.float64)), want)


def test_gelu_closed_forms(O):
    pin_gelu(O)


def test_round_bf16(O):
    pin_round_bf16(O)


def test_gelu_bf16_is_round_of_gelu(O):
    Y = synth.gaussian_bf16((4, 5), (16, 64), 2.0)
    assert np.array_equal(O.gelu_bf16(Y), O.round_bf16(O.gelu(exact_widen(Y))))


def test_mlp_input_chains_the_up_layer(O):
    """H = bf16(GELU(bf16(Y_up))) row by row, with Y_up the up layer (sparse or dense)."""
    g = np.random.default_rng(17)
    M, N, K, R = 6, 16, 24, 2
    X, W, LA, LB = (bits(g.standard_normal(sh)) for sh in [(M, K), (N, K), (N, R), (R, K)])
    for sparse in (True, False):
        y = O.linear(X, W, LA, LB) if sparse else O.linear_dense(X, W, LA, LB)
        want = O.gelu_bf16(O.round_bf16(y))
        assert np.array_equal(O.mlp_input(X, W, LA, LB, sparse=sparse), want)
        assert np.array_equal(O.mlp_input(X, W, LA, LB, sparse=sparse, rows=[4, 1]), want[[4, 1]])


# ----------------------------------------------------------------------------- the two oracles agree
@pytest.mark.parametrize("M,K,kind", [(33, 64, "act"), (40, 256, "mixed"), (16, 512, "ties"), (64, 3072, "gelu")])
def test_cpp_and_numpy_oracles_agree(M, K, kind):
    """Same selection, values and metadata bit for bit; s and Y to double rounding (summation orders differ)."""
    if kind == "act":
        X = synth.act_bf16((M, K, 1), M, K, 0.03, 10.0)
    elif kind == "gelu":
        X = synth.gelu_bf16((M, K, 1), M, K, 3.97, 0.0, 1.0)
    else:
        X = synth.structured_x(kind, M, K, 2)
    N, R = 40, 64
    W = synth.gaussian_bf16((M, K, 2), (N, K), 1.0 / math.sqrt(K))
    LA = synth.gaussian_bf16((M, K, 3), (N, R), 0.02)
    LB = synth.gaussian_bf16((M, K, 4), (R, K), 0.02)
    C = CPP.default()
    a, b = C.sparsify(X), NP.sparsify(X)
    for k in ("mask", "vals", "meta"):
        assert np.array_equal(a[k], b[k]), k
    np.testing.assert_allclose(a["s"], b["s"], rtol=1e-14, atol=0)
    for fa, fb in ((C.linear(X, W, LA, LB), NP.linear(X, W, LA, LB)),
                   (C.linear_dense(X, W, LA, LB), NP.linear_dense(X, W, LA, LB)),
                   (C.linear_wsparse(X, W, LA, LB), NP.linear_wsparse(X, W, LA, LB)),
                   (C.lora_down(X, LB, a["s"]), NP.lora_down(X, LB, b["s"]))):
        scale = np.max(np.abs(fb))
        assert np.max(np.abs(fa - fb)) <= 1e-12 * scale


def test_cpp_oracle_result_is_independent_of_thread_count():
    t = synth.layer_tensors("tiny", "linear")
    C = CPP.default()
    saved = C.threads
    try:
        C.threads = 1
        y1 = C.linear(t["X"], t["W"], t["LA"], t["LB"], rows=np.arange(0, 256, 3))
        C.threads = 7
        y7 = C.linear(t["X"], t["W"], t["LA"], t["LB"], rows=np.arange(0, 256, 3))
    finally:
        C.threads = saved
    assert np.array_equal(y1, y7)


# ----------------------------------------------------------------------------- input generator
def test_bf16_rounding_matches_torch():
    import torch
    a = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 37.0
    a[:4] = [0.0, -0.0, 1.00390625, 1.01171875]  # exact ties in bf16: round to even
    want = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.bf16_bits(a), want)


def test_inputs_are_deterministic():
    a = synth.layer_tensors("tiny", "linear")
    b = synth.layer_tensors("tiny", "linear")
    for k in ("X", "W", "LA", "LB"):
        assert np.array_equal(a[k], b[k])
    assert a["X"].shape == (256, 512) and a["W"].shape == (512, 512)
    assert a["LA"].shape == (512, 64) and a["LB"].shape == (64, 512)


# ----------------------------------------------------------------------------- planted mistakes: numpy oracle
def _ties_to_higher(x):
    M, K = x.shape
    mag = np.abs(x).reshape(M, K // 4, 4)[..., ::-1]
    order = 3 - np.argsort(-mag, axis=-1, kind="stable")
    top = np.sort(order[..., :2], axis=-1)
    return top[..., 0], top[..., 1]


def _smallest_two(x):
    M, K = x.shape
    order = np.argsort(np.abs(x).reshape(M, K // 4, 4), axis=-1, kind="stable")
    top = np.sort(order[..., :2], axis=-1)
    return top[..., 0], top[..., 1]


def _inverted_scale(x, mask):
    return 1.0 / _REAL["norm_scale"](x, mask)


def _no_lora(X, W, LA, LB, rows=None):
    return _REAL["linear"](X, W, np.zeros_like(LA), LB, rows)


def _reversed_lora_rows(X, W, LA, LB, rows=None):
    """LoRA-up with the rows of LA taken in reverse order: a wrong output index."""
    x = NP.widen(X)
    mask = NP.keep_mask(x)
    s = NP.norm_scale(x, mask)
    return s[:, None] * (np.where(mask, x, 0.0) @ NP.widen(W).T) + (x @ NP.widen(LB).T) @ NP.widen(LA)[::-1].T


def _unscaled_sparse(X, W, LA, LB, rows=None):
    x = NP.widen(X)
    mask = NP.keep_mask(x)
    return np.where(mask, x, 0.0) @ NP.widen(W).T + (x @ NP.widen(LB).T) @ NP.widen(LA).T


def _wsparse_keeps_all(X, W, LA=None, LB=None, rows=None):
    return NP.linear_dense(X, W, LA, LB, rows=rows)


_REAL = {"norm_scale": NP.norm_scale, "linear": NP.linear}

PINS = {
    "exhaustive": pin_selection_exhaustive,
    "hand_sparsify": pin_hand_sparsify,
    "hand_linear": pin_hand_linear,
    "hand_lora_down": pin_hand_lora_down,
    "norm": lambda O: pin_norm_restoration(O, synth.act_bf16((5, 6), 16, 64, 0.03, 10.0)),
    "loops": lambda O: pin_loops(O, 0),
    "wsparse_loops": lambda O: pin_wsparse_loops(O, 0),
    "dense_loops": pin_dense_loops,
    "meta_decode": pin_meta_decodes_to_mask,
    "gelu": pin_gelu,
    "round_bf16": pin_round_bf16,
}


@pytest.mark.parametrize("attr,fake,pins", [
    ("select_2of4", _ties_to_higher, ["exhaustive", "hand_sparsify"]),
    ("select_2of4", _smallest_two, ["exhaustive", "hand_sparsify", "loops"]),
    ("norm_scale", _inverted_scale, ["norm", "hand_sparsify", "loops"]),
    ("linear", _no_lora, ["hand_linear", "loops"]),
    ("linear", _reversed_lora_rows, ["loops"]),
    ("linear", _unscaled_sparse, ["hand_linear", "loops"]),
    ("select_2of4", _smallest_two, ["wsparse_loops"]),
    ("linear_wsparse", _wsparse_keeps_all, ["wsparse_loops"]),
])
def test_planted_mistake_is_caught_numpy(monkeypatch, attr, fake, pins):
    monkeypatch.setattr(NP, attr, fake)
    for p in pins:
        with pytest.raises(AssertionError):
            PINS[p](NP)


# ----------------------------------------------------------------------------- planted mistakes: C++ oracle
# Each mutation replaces one snippet of the C++ source (which must occur exactly once) and names the pins that
# must fail on the mutated build.
CPP_MUTATIONS = [
    ("ties to the higher index", "int order[4] = {0, 1, 2, 3};", "int order[4] = {3, 2, 1, 0};",
     ["exhaustive", "hand_sparsify"]),
    ("keeps the two smallest", "return std::fabs(g[a]) > std::fabs(g[b]);", "return std::fabs(g[a]) < std::fabs(g[b]);",
     ["exhaustive", "hand_sparsify", "loops", "wsparse_loops"]),
    ("inverted scale", "std::sqrt(nx / nt)", "std::sqrt(nt / nx)", ["norm", "hand_sparsify", "loops"]),
    ("norm over kept entries only", "nx += x[k] * x[k];", "if (keep[k]) nx += x[k] * x[k];",
     ["norm", "hand_sparsify", "loops"]),
    ("no LoRA branch", "Y[i * N + n] = s * ys[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];",
     "Y[i * N + n] = s * ys[static_cast<size_t>(n)];", ["hand_linear", "loops"]),
    ("unscaled sparse branch", "Y[i * N + n] = s * ys[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];",
     "Y[i * N + n] = ys[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];", ["hand_linear", "loops"]),
    ("LoRA-up rows reversed", "acc += t[static_cast<size_t>(r)] * la[n * R + r];",
     "acc += t[static_cast<size_t>(r)] * la[(N - 1 - n) * R + r];", ["loops", "dense_loops", "wsparse_loops"]),
    ("LoRA-down transposed index", "acc += x[k] * lb[r * K + k];", "acc += x[k] * lb[k * R + r];",
     ["loops", "dense_loops", "wsparse_loops"]),
    ("metadata nibble reversed", "byte |= static_cast<uint32_t>(first | (second << 2)) << (4 * h);",
     "byte |= static_cast<uint32_t>(second | (first << 2)) << (4 * h);", ["hand_sparsify", "meta_decode"]),
    ("lora_down multiplies by s", "T[m * R + r] = s ? acc / s[m] : acc;", "T[m * R + r] = s ? acc * s[m] : acc;",
     ["hand_lora_down"]),
    ("weight pruning skipped", "if (!keep[static_cast<size_t>(k)]) wt[static_cast<size_t>(n * K + k)] = 0.0;",
     "(void)keep;", ["wsparse_loops"]),
    ("GELU with tanh argument", "0.5 * x[i] * (1.0 + std::erf(x[i] / std::sqrt(2.0)))",
     "0.5 * x[i] * (1.0 + std::tanh(x[i] / std::sqrt(2.0)))", ["gelu"]),
    ("bf16 rounding truncates", "r = std::nearbyint(std::ldexp(m, 8));", "r = std::trunc(std::ldexp(m, 8));",
     ["round_bf16"]),
    ("dense layer drops its LoRA", "if (LA) lora_row(x.data(), la.data(), lb.data(), N, K, R, yr.data());\n"
     "    for (int64_t n = 0; n < N; ++n) Y[i * N + n] = y[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];\n"
     "  });\n  return 0;\n}\n\n// The weight-2:4",
     "for (int64_t n = 0; n < N; ++n) Y[i * N + n] = y[static_cast<size_t>(n)] + yr[static_cast<size_t>(n)];\n"
     "  });\n  return 0;\n}\n\n// The weight-2:4", ["dense_loops"]),
]


@pytest.fixture(scope="module")
def mutation_dir():
    d = tempfile.mkdtemp(prefix="lynx_oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,old,new,pins", CPP_MUTATIONS, ids=[m[0] for m in CPP_MUTATIONS])
def test_planted_mistake_is_caught_cpp(mutation_dir, name, old, new, pins):
    src = open(CPP.SOURCE).read()
    assert src.count(old) == 1, f"mutation site of '{name}' must occur exactly once"
    tag = "".join(c if c.isalnum() else "_" for c in name)
    path = os.path.join(mutation_dir, f"mut_{tag}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = CPP.build(source=path, out=os.path.join(mutation_dir, f"libmut_{tag}.so"), force=True)
    mutant = CPP.CppOracle(lib)
    PINS_OK = [p for p in PINS if p not in pins]
    for p in pins:
        with pytest.raises(AssertionError):
            PINS[p](mutant)
    # the pins that do not target this mistake keep passing on the unmutated parts (sanity of the harness)
    assert PINS_OK


def test_unmutated_cpp_build_passes_every_pin():
    C = CPP.default()
    for p, fn in PINS.items():
        fn(C)

"""Pins of the CPU oracle against things other than itself.

The RT-Lynx page prints no worked numeric example, so the oracle is pinned by
(a) hand-derived cases in tests/golden/hand_cases.json, (b) brute force over
every 4-tuple of a small alphabet with an independent formulation of the
selection, (c) closed-form invariants of the norm compensation, (d) pure-Python
loop evaluations of the layer on tiny inputs and (e) special cases that reduce
to a plain GEMM.  The last block plants mistakes in the oracle (on the CPU) and
checks that some pin catches each one.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle.lynx_oracle as O
import synth

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "hand_cases.json")))
SQRT2 = math.sqrt(2.0)


def bits(a):
    return synth.bf16_bits(np.asarray(a, dtype=np.float32))


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


# ----------------------------------------------------------------------------- pins (reusable)
ALPHABET = [-2.0, -1.0, -0.0, 0.0, 1.0, 2.0, 3.0]


def pin_selection_exhaustive():
    tuples = np.array(list(itertools.product(ALPHABET, repeat=4)), dtype=np.float32)
    x = O.widen(bits(tuples))
    i0, i1 = O.select_2of4(x)
    for t, a, b in zip(tuples.tolist(), i0[:, 0], i1[:, 0]):
        assert (a, b) == brute_pair(t), (t, a, b)


def pin_hand_sparsify():
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


def pin_hand_linear():
    for case in GOLD["linear"]:
        y = O.linear(bits(case["X"]), bits(case["W"]), bits(case["LA"]), bits(case["LB"]))
        assert np.allclose(y, np.array(case["Y"]), rtol=1e-14, atol=0), (case["name"], y)


def pin_norm_restoration(X):
    x = O.widen(X)
    out = O.sparsify(X)
    xt = np.where(out["mask"], x, 0.0)
    lhs = np.linalg.norm(out["s"][:, None] * xt, axis=1)
    rhs = np.linalg.norm(x, axis=1)
    assert np.allclose(lhs, rhs, rtol=1e-12, atol=0)
    assert np.all(out["s"] >= 1.0 - 1e-15) and np.all(out["s"] <= SQRT2 * (1 + 1e-15))


def pin_loops(seed, M=3, N=5, K=12, R=2):
    g = np.random.default_rng(seed)
    X = bits(g.standard_normal((M, K)))
    W = bits(g.standard_normal((N, K)))
    LA = bits(g.standard_normal((N, R)))
    LB = bits(g.standard_normal((R, K)))
    want = loop_layer(O.widen(X).tolist(), O.widen(W).tolist(), O.widen(LA).tolist(), O.widen(LB).tolist())
    got = O.linear(X, W, LA, LB)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- tests: pins hold
def test_selection_exhaustive_bruteforce():
    pin_selection_exhaustive()


def test_hand_cases_sparsify():
    pin_hand_sparsify()


def test_hand_case_linear():
    pin_hand_linear()


@pytest.mark.parametrize("kind", ["act", "equal", "two4", "ties", "mixed"])
def test_exactly_two_per_group_and_packing(kind):
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


def test_norm_restoration_random():
    pin_norm_restoration(synth.act_bf16((5, 6), 64, 256, 0.03, 10.0))


def test_scale_special_cases():
    s = O.sparsify(synth.structured_x("equal", 16, 64, 1))["s"]
    assert np.allclose(s, SQRT2, rtol=1e-15, atol=0)
    s = O.sparsify(synth.structured_x("two4", 16, 64, 2))["s"]
    assert np.array_equal(s, np.ones(16))
    s = O.sparsify(synth.structured_x("zero", 4, 64, 3))["s"]
    assert np.array_equal(s, np.ones(4))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_linear_against_python_loops(seed):
    pin_loops(seed)


def test_linear_against_materialised_dense_reference():
    """S(X) as a dense M x K matrix and (LA LB) as a dense N x K matrix, a different association."""
    g = np.random.default_rng(11)
    M, N, K, R = 7, 10, 24, 3
    X = bits(g.standard_normal((M, K)) * 2)
    W, LA, LB = (bits(g.standard_normal(sh)) for sh in [(N, K), (N, R), (R, K)])
    x = O.widen(X)
    sx = O.sparsify(X)
    S = sx["s"][:, None] * np.where(sx["mask"], x, 0.0)
    want = S @ O.widen(W).T + x @ (O.widen(LA) @ O.widen(LB)).T
    assert np.allclose(O.linear(X, W, LA, LB), want, rtol=1e-12, atol=1e-12)


def test_already_24_and_zero_lora_is_plain_gemm():
    M, N, K, R = 5, 6, 16, 2
    X = synth.structured_x("two4", M, K, 4)
    g = np.random.default_rng(4)
    W = bits(g.standard_normal((N, K)))
    LA = np.zeros((N, R), dtype=np.uint16)
    LB = bits(g.standard_normal((R, K)))
    x, w = O.widen(X).tolist(), O.widen(W).tolist()
    gemm = np.array([[sum(x[m][k] * w[n][k] for k in range(K)) for n in range(N)] for m in range(M)])
    assert np.allclose(O.linear(X, W, LA, LB), gemm, rtol=1e-13, atol=1e-13)
    assert np.allclose(O.linear_dense(X, W), gemm, rtol=1e-13, atol=1e-13)


def test_zero_lb_leaves_scaled_sparse_branch():
    M, N, K, R = 4, 8, 32, 4
    X = synth.act_bf16((9,), M, K, 0.1, 8.0)
    g = np.random.default_rng(9)
    W, LA = bits(g.standard_normal((N, K))), bits(g.standard_normal((N, R)))
    LB = np.zeros((R, K), dtype=np.uint16)
    want = loop_layer(O.widen(X).tolist(), O.widen(W).tolist(), O.widen(LA).tolist(), O.widen(LB).tolist())
    assert np.allclose(O.linear(X, W, LA, LB), want, rtol=1e-12, atol=1e-12)


def test_row_subset_equals_full_rows():
    t = synth.layer_tensors("tiny", "linear")
    rows = np.array([0, 3, 100, 255])
    full = O.linear(t["X"], t["W"], t["LA"], t["LB"])
    assert np.array_equal(O.linear(t["X"], t["W"], t["LA"], t["LB"], rows=rows), full[rows])


def test_dense_layer_with_lora_against_loops():
    g = np.random.default_rng(21)
    M, N, K, R = 3, 4, 8, 2
    X, W, LA, LB = (bits(g.standard_normal(sh)) for sh in [(M, K), (N, K), (N, R), (R, K)])
    x, w, la, lb = (O.widen(a).tolist() for a in (X, W, LA, LB))
    want = [[sum(x[m][k] * w[n][k] for k in range(K)) +
             sum(sum(x[m][k] * lb[r][k] for k in range(K)) * la[n][r] for r in range(R))
             for n in range(N)] for m in range(M)]
    assert np.allclose(O.linear_dense(X, W, LA, LB), want, rtol=1e-13, atol=1e-13)


def pin_wsparse_loops(seed, M=3, N=4, K=12, R=2):
    """The weight-2:4 layer with Python loops: brute-force pair per group of each W row, no rescale."""
    g = np.random.default_rng(100 + seed)
    X, W, LA, LB = (bits(g.standard_normal(sh)) for sh in [(M, K), (N, K), (N, R), (R, K)])
    x, w, la, lb = (O.widen(a).tolist() for a in (X, W, LA, LB))
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


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_weight_sparse_layer_against_python_loops(seed):
    pin_wsparse_loops(seed)


def test_weight_sparse_on_24_weights_is_the_dense_layer():
    """W that is already 2:4 (two zeros per group) is left unchanged: the dense layer's result."""
    W = synth.structured_x("two4", 24, 64, seed=3)
    X = synth.act_bf16((8, 1), 10, 64, 0.05, 8.0)
    LA, LB = synth.gaussian_bf16((8, 2), (24, 2), 0.1), synth.gaussian_bf16((8, 3), (2, 64), 0.1)
    assert np.array_equal(O.linear_wsparse(X, W, LA, LB), O.linear_dense(X, W, LA, LB))


def test_weight_sparse_is_the_transposed_activation_product():
    """X W~^T = (W~ X^T)^T, and W~ X^T is the activation path on W without its row scale: the same
    selection reached through the sparsified-activation functions."""
    X = synth.act_bf16((9, 1), 7, 32, 0.05, 8.0)
    W = synth.act_bf16((9, 2), 5, 32, 0.05, 8.0)
    zero_la, zero_lb = np.zeros((7, 2), np.uint16), np.zeros((2, 32), np.uint16)
    s_w = O.sparsify(W)["s"]
    via_activation = O.linear(W, X, zero_la, zero_lb) / s_w[:, None]
    assert np.allclose(O.linear_wsparse(X, W), via_activation.T, rtol=1e-12, atol=1e-12)


def test_lora_down_hand_case_and_recombination():
    case = GOLD["linear"][0]
    X, LB, LA, W = (bits(case[k]) for k in ("X", "LB", "LA", "W"))
    s = O.sparsify(X)["s"]
    t = O.lora_down(X, LB, s)
    # hand case: X LB^T = 1 - 3 + 2 + 0.5 + 4 = 4.5, s = 5.5/sqrt(29)
    assert abs(t[0, 0] - 4.5 / (5.5 / math.sqrt(29.0))) < 1e-14
    assert O.lora_down(X, LB)[0, 0] == 4.5
    # s * (X~ W^T + T' LA^T) recombines to the layer output
    x = O.widen(X)
    acc = np.where(O.sparsify(X)["mask"], x, 0.0) @ O.widen(W).T + t @ O.widen(LA).T
    assert np.allclose(s[:, None] * acc, O.linear(X, W, LA, LB), rtol=1e-14, atol=0)


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


# ----------------------------------------------------------------------------- planted mistakes
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
    x = O.widen(X)
    mask = O.keep_mask(x)
    s = O.norm_scale(x, mask)
    return s[:, None] * (np.where(mask, x, 0.0) @ O.widen(W).T) + (x @ O.widen(LB).T) @ O.widen(LA)[::-1].T


def _unscaled_sparse(X, W, LA, LB, rows=None):
    x = O.widen(X)
    mask = O.keep_mask(x)
    return np.where(mask, x, 0.0) @ O.widen(W).T + (x @ O.widen(LB).T) @ O.widen(LA).T


def _wsparse_keeps_all(X, W, LA=None, LB=None, rows=None):
    return O.linear_dense(X, W, LA, LB, rows=rows)


_REAL = {"norm_scale": O.norm_scale, "linear": O.linear}


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
def test_planted_mistake_is_caught(monkeypatch, attr, fake, pins):
    monkeypatch.setattr(O, attr, fake)
    run = {
        "exhaustive": pin_selection_exhaustive,
        "hand_sparsify": pin_hand_sparsify,
        "hand_linear": pin_hand_linear,
        "norm": lambda: pin_norm_restoration(synth.act_bf16((5, 6), 16, 64, 0.03, 10.0)),
        "loops": lambda: pin_loops(0),
        "wsparse_loops": lambda: pin_wsparse_loops(0),
    }
    for p in pins:
        with pytest.raises(AssertionError):
            run[p]()

"""Plain CPU oracle of the RT-Lynx activation-sparse linear layer.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
arms of ``bench.py`` (the timed CPU baseline and ``--impl reference``) may
import or run this module.  The library never does: it has no CPU fallback.

What is computed follows the RT-Lynx page (aitrends.kr article 60737):

* Method, "key mechanism": a Top-K based 2:4 selection of the activations gives
  X~; the sparse activation is S(X) = s * X~; the output is
  Y = Ys + Yr with Ys = S(X) W^T and Yr = X (LA LB)^T.
* Code examples, first formula: s = ||X||_2 / (||X~||_2 + eps), which restores
  the dense activation's L2 norm (Glossary, "Norm Compensation").
* Technical details: LoRA rank R = 64; QKV and Up/Down linears are sparsified;
  some single-stream layers are left dense (Selective Layer Skipping).

Readings taken where the page is silent:

* groups are 4 consecutive input channels (the K axis) of one token (row);
* "top-K" means the two largest |x| of each group; ties go to the lower index;
  a group with fewer than two nonzeros still keeps exactly two positions;
* the norm is taken per token over all K channels; eps = 0, and a row whose
  kept entries are all zero gets s = 1;
* the LoRA branch takes the dense, unscaled X; (LA LB)^T is applied as
  (X LB^T) LA^T, which is the same product;
* no bias; Y is reported in float64 here (the CUDA path rounds it to bf16).

Everything is float64 numpy from the bf16 inputs.  Matrix products use
numpy's matmul as a library primitive; there is no blocking or fusion.
Inputs are uint16 arrays of bf16 bit patterns, row-major:
X (M x K), W (N x K), LA (N x R), LB (R x K).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "widen", "select_2of4", "keep_mask", "norm_scale", "sparsify", "canonical_meta",
    "linear", "linear_dense", "linear_wsparse", "lora_down", "round_bf16", "gelu", "gelu_bf16", "mlp_input",
    "NIBBLE_OF_PAIR",
]

#: 4-bit metadata of a kept index pair (i0 < i1): i0 in bits 0-1, i1 in bits 2-3.
NIBBLE_OF_PAIR = {(i0, i1): i0 | (i1 << 2) for i0 in range(4) for i1 in range(i0 + 1, 4)}


def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (a bf16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def select_2of4(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Kept index pair (i0 < i1) of every group of 4 consecutive channels of every row.

    RT-Lynx page, Method: Top-K based 2:4 activation selection.  Within a
    group the entries are ranked by |x|, largest first, with a stable sort,
    so that of two equal magnitudes the lower channel index ranks first; the
    two first-ranked positions are kept.  Returns two int arrays of shape
    (M, K/4).
    """
    M, K = x.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    mag = np.abs(x).reshape(M, K // 4, 4)
    order = np.argsort(-mag, axis=-1, kind="stable")
    top = np.sort(order[..., :2], axis=-1)
    return top[..., 0], top[..., 1]


def keep_mask(x: np.ndarray) -> np.ndarray:
    """Boolean M x K mask of the kept entries (exactly two per group)."""
    M, K = x.shape
    i0, i1 = select_2of4(x)
    m = np.zeros((M, K // 4, 4), dtype=bool)
    np.put_along_axis(m, i0[..., None], True, axis=-1)
    np.put_along_axis(m, i1[..., None], True, axis=-1)
    return m.reshape(M, K)


def norm_scale(x: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """Per-row s = ||X||_2 / ||X~||_2 (RT-Lynx page, Code examples, first formula).

    eps is read as 0; a row whose kept entries are all zero has s = 1.
    """
    xt = np.where(mask, x, 0.0)
    nx = np.sqrt(np.sum(x * x, axis=1))
    nt = np.sqrt(np.sum(xt * xt, axis=1))
    s = np.ones_like(nx)
    nz = nt > 0
    s[nz] = nx[nz] / nt[nz]
    return s


def canonical_meta(i0: np.ndarray, i1: np.ndarray) -> np.ndarray:
    """Pack index pairs into bytes: group 2j in the low nibble of byte j, group 2j+1 in the high one."""
    nib = (i0 | (i1 << 2)).astype(np.uint8)
    M, G = nib.shape
    if G % 2:
        raise ValueError("K must be a multiple of 8 for byte-packed metadata")
    nib = nib.reshape(M, G // 2, 2)
    return (nib[..., 0] | (nib[..., 1] << 4)).astype(np.uint8)


def sparsify(X: np.ndarray) -> dict:
    """S(X) in compressed form: what the sparsification step hands to the sparse GEMM.

    Returns ``mask`` (M x K bool), ``vals`` (M x K/2 uint16: the kept bf16
    entries of each group, lower index first), ``meta`` (M x K/8 uint8,
    canonical packing of the kept index pairs; None
    unless K is a multiple of 8) and ``s`` (M float64).
    """
    Xb = np.asarray(X, dtype=np.uint16)
    x = widen(Xb)
    M, K = x.shape
    i0, i1 = select_2of4(x)
    g = Xb.reshape(M, K // 4, 4)
    v0 = np.take_along_axis(g, i0[..., None], axis=-1)
    v1 = np.take_along_axis(g, i1[..., None], axis=-1)
    vals = np.concatenate([v0, v1], axis=-1).reshape(M, K // 2)
    mask = keep_mask(x)
    meta = canonical_meta(i0, i1) if K % 8 == 0 else None
    return {"mask": mask, "vals": vals, "meta": meta, "s": norm_scale(x, mask)}


def linear(X, W, LA, LB, rows=None) -> np.ndarray:
    """Y = S(X) W^T + X (LA LB)^T in float64 (RT-Lynx page, Method; Code examples).

    ``rows`` selects a subset of the M rows; rows are independent, so the result
    equals the corresponding rows of the full product.
    """
    Xb = np.asarray(X, dtype=np.uint16)
    if rows is not None:
        Xb = Xb[np.asarray(rows)]
    x = widen(Xb)
    w = widen(W)
    mask = keep_mask(x)
    s = norm_scale(x, mask)
    xt = np.where(mask, x, 0.0)
    ys = s[:, None] * (xt @ w.T)
    yr = (x @ widen(LB).T) @ widen(LA).T
    return ys + yr


def lora_down(X, LB, s=None) -> np.ndarray:
    """First factor of the LoRA branch Yr = X (LA LB)^T = (X LB^T) LA^T, divided by s when given.

    RT-Lynx page, Method.  Dividing by the row scale s of the sparse branch
    lets Ys and Yr share one accumulator that is scaled by s at the end:
    s * (X~ W^T + (X LB^T / s) LA^T) = Ys + Yr.
    """
    t = widen(X) @ widen(LB).T
    if s is not None:
        t = t / np.asarray(s, dtype=np.float64)[:, None]
    return t


def linear_dense(X, W, LA=None, LB=None, rows=None) -> np.ndarray:
    """Y = X W^T (+ X (LA LB)^T when LoRA factors are given): a selectively skipped layer."""
    Xb = np.asarray(X, dtype=np.uint16)
    if rows is not None:
        Xb = Xb[np.asarray(rows)]
    x = widen(Xb)
    y = x @ widen(W).T
    if LA is not None and LB is not None:
        y = y + (x @ widen(LB).T) @ widen(LA).T
    return y


def linear_wsparse(X, W, LA=None, LB=None, rows=None) -> np.ndarray:
    """Y = X W~^T (+ X (LA LB)^T when LoRA factors are given): the weight-2:4 comparator.

    The RT-Lynx page compares its activation sparsity with 2:4 weight sparsity ("Sparse Weight" in Main
    results; Key idea: weight sparsity degrades DiT outputs more than activation sparsity).  Reading: W~ keeps
    the two largest |w| of every 4 consecutive input channels of each output row, ties to the lower index
    (the activation rule applied to the rows of W, along K as the sparse tensor core requires), with no norm
    compensation; the optional LoRA branch is the dense layer's.
    """
    Xb = np.asarray(X, dtype=np.uint16)
    if rows is not None:
        Xb = Xb[np.asarray(rows)]
    x = widen(Xb)
    w = widen(W)
    wt = np.where(keep_mask(w), w, 0.0)
    y = x @ wt.T
    if LA is not None and LB is not None:
        y = y + (x @ widen(LB).T) @ widen(LA).T
    return y


def round_bf16(x) -> np.ndarray:
    """Nearest bf16 value (8 significant bits, ties to even) of float64 values, as uint16 bit patterns.

    Magnitudes below 2^-126 round on the subnormal grid of 2^-133; values beyond the largest bf16 become
    infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    m, e = np.frexp(a)                                   # a = m 2^e, m in [0.5, 1)
    normal = e >= -125
    r = np.where(normal, np.rint(np.ldexp(m, 8)), np.rint(np.ldexp(a, 133)))  # rint: ties to even
    v = np.where(normal, np.ldexp(r, e - 8), np.ldexp(r, -133))
    v = np.where(v > 3.3895313892515355e38, np.inf, v)
    f = np.copysign(v, x).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def gelu(x) -> np.ndarray:
    """GELU with the exact error function, 0.5 x (1 + erf(x / sqrt 2)), in float64 (scipy's erf)."""
    from scipy.special import erf
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def gelu_bf16(Y) -> np.ndarray:
    """H = bf16(GELU(Y)) of a bf16 tensor Y (the MLP activation applied to the up layer's bf16 output)."""
    return round_bf16(gelu(widen(Y)))


def mlp_input(X, W, LA=None, LB=None, sparse=True, rows=None) -> np.ndarray:
    """The MLP down layer's input for the given rows: H = bf16(GELU(bf16(Y_up))), with Y_up the up layer
    (sparse: ``linear``, else ``linear_dense``) in float64, rounded to the up layer's bf16 output first."""
    y = linear(X, W, LA, LB, rows) if sparse else linear_dense(X, W, LA, LB, rows)
    return gelu_bf16(round_bf16(y))

"""Seeded synthetic DiT-linear inputs.

Every tensor is drawn from numpy's PCG64 generator, seeded from a tuple
(workload seed, tensor id, ...) through ``numpy.random.SeedSequence``, drawn in
float32 and rounded to bf16 (round to nearest even).  Arrays are returned as
``uint16`` bf16 bit patterns in row-major order, so that the oracle and the
CUDA path both start from the very same bits.

Shapes follow the diffusion-transformer layers that the RT-Lynx page applies
2:4 activation sparsity to (QKV projection and the MLP up/down maps, hidden
size 3072, MLP width 12288; "RT-Lynx" page, Technical details).  The value
distributions stand in for real DiT activations, which the page describes as
a few strongly active channels per token (Key idea):

* ``act``  -- N(0, 1) with a fixed random subset of channels (columns) scaled
  by a constant: the same outlier channels for every token;
* ``gelu`` -- exact-erf GELU applied to N(0, v): the element distribution of
  GELU(up-projection output), the nonnegative-leaning input of the MLP down
  projection.  v = 1 + f*(a*a - 1) is the variance that each entry of X·W_upᵀ
  has when W_up ~ N(0, 1/K) and X follows ``act``; the weights mix every input
  channel into every output, so the pre-activations carry no outlier channels;
* weights ``W ~ N(0, 1/K)`` (variance 1/K), LoRA factors ``N(0, 0.02)`` (std
  0.02), seeded per tensor.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "bf16_bits", "bf16_to_f32", "rng", "gaussian_bf16", "act_bf16", "gelu_bf16",
    "Layer", "Workload", "WORKLOADS", "layer_tensors", "layer_x", "sample_rows",
    "STACK_M", "structured_x",
]


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round a float32 array to bf16 (nearest, ties to even); return uint16 bits.

    Inputs are finite by construction, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF)  # finite values stay below 2^32 (the largest finite pattern is 0xFF7FFFFF)
    r += (u >> np.uint32(16)) & np.uint32(1)
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen uint16 bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def gaussian_bf16(key: tuple, shape: tuple, std: float) -> np.ndarray:
    g = rng(*key)
    a = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return bf16_bits(a)


def _outlier_channels(key: tuple, K: int, frac: float) -> np.ndarray:
    n = int(round(frac * K))
    return np.sort(rng(*key).permutation(K)[:n])


def act_bf16(key: tuple, M: int, K: int, frac: float, scale: float,
             chan_key: tuple | None = None) -> np.ndarray:
    """N(0,1) activations with round(frac*K) outlier channels scaled by ``scale``."""
    a = rng(*key).standard_normal((M, K), dtype=np.float32)
    ch = _outlier_channels(chan_key or key + (99,), K, frac)
    a[:, ch] *= np.float32(scale)
    return bf16_bits(a)


def _gelu(z: np.ndarray) -> np.ndarray:
    """Exact-erf GELU in float32 (the result is rounded to bf16 afterwards)."""
    from scipy.special import erf
    z = z.astype(np.float32, copy=False)
    return np.float32(0.5) * z * (np.float32(1.0) + erf(z * np.float32(1.0 / math.sqrt(2.0))))


def gelu_bf16(key: tuple, M: int, K: int, pre_var: float, frac: float, scale: float,
              chan_key: tuple | None = None) -> np.ndarray:
    """GELU(N(0, pre_var)), with round(frac*K) channels scaled by ``scale`` before the GELU (none for frac = 0)."""
    z = rng(*key).standard_normal((M, K), dtype=np.float32)
    z *= np.float32(math.sqrt(pre_var))
    ch = _outlier_channels(chan_key or key + (99,), K, frac)
    z[:, ch] *= np.float32(scale)
    out = np.empty_like(z)
    step = 1 << 20
    flat_in, flat_out = z.reshape(-1), out.reshape(-1)
    for i in range(0, flat_in.size, step):  # chunked to bound temporaries
        flat_out[i:i + step] = _gelu(flat_in[i:i + step])
    return bf16_bits(out)


@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    K: int          # input channels
    N: int          # output channels
    sparse: bool    # 2:4 activation sparsity (False: a selectively skipped dense layer)
    x: str          # "act" or "gelu"
    lid: int        # tensor-id base


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    M: int
    layers: tuple
    frac: float
    scale: float
    halves: int = 1     # >1: M rows stacked from independently seeded halves (CFG batch)
    blocks: int = 1     # repeated blocks with independent weights (block stack)
    rank: int = 64
    desc: str = ""

    def layer(self, name: str) -> Layer:
        for l in self.layers:
            if l.name == name:
                return l
        raise KeyError(name)


HIDDEN, MLP = 3072, 12288
_QKV = Layer("qkv", HIDDEN, 3 * HIDDEN, True, "act", 0)
_OUT = Layer("out", HIDDEN, HIDDEN, True, "act", 10)
_UP = Layer("up", HIDDEN, MLP, True, "act", 20)
_DOWN = Layer("down", MLP, HIDDEN, True, "gelu", 30)

#: M values of the block-stack sweep.
STACK_M = (1024, 4608, 9216, 16384)

WORKLOADS = {
    "tiny": Workload("tiny", 0, 256, (Layer("linear", 512, 512, True, "act", 0),), 0.05, 8.0,
                     desc="single linear 256x512 -> 512"),
    "qkv": Workload("qkv", 2, 4608, (_QKV,), 0.03, 10.0,
                    desc="attention QKV projection, 4096 image + 512 text tokens, hidden 3072"),
    "mlp": Workload("mlp", 3, 4608, (_UP, _DOWN), 0.03, 10.0,
                    desc="MLP up 3072->12288 then down 12288->3072"),
    "cfg2": Workload("cfg2", 4, 9216, (_QKV, _OUT, _UP, _DOWN), 0.03, 10.0, halves=2,
                     desc="CFG batch 2: cond + uncond sequences stacked, all four linears sparse"),
    "stack": Workload("stack", 5, 4608,
                      (_QKV, dataclasses.replace(_OUT, sparse=False), dataclasses.replace(_UP, sparse=False), _DOWN),
                      0.03, 10.0, blocks=8,
                      desc="8 single-stream blocks x (QKV sparse, out dense, up dense, down sparse)"),
}


def _x(wl: Workload, layer: Layer, M: int, block: int, batch: int = 0) -> np.ndarray:
    base = (wl.seed, M, block, layer.lid) + ((batch,) if batch else ())
    chan = (wl.seed, block, layer.lid, 99)
    parts = []
    rows = [M // wl.halves + (1 if h < M % wl.halves else 0) for h in range(wl.halves)]
    for h, mh in enumerate(rows):
        key = base + (0, h)
        if layer.x == "act":
            parts.append(act_bf16(key, mh, layer.K, wl.frac, wl.scale, chan_key=chan))
        else:
            pre_var = 1.0 + wl.frac * (wl.scale * wl.scale - 1.0)
            parts.append(gelu_bf16(key, mh, layer.K, pre_var, 0.0, 1.0, chan_key=chan))
    return parts[0] if len(parts) == 1 else np.concatenate(parts, axis=0)


def layer_tensors(workload: str, layer: str, M: int | None = None, block: int = 0,
                  with_x: bool = True, batch: int = 0) -> dict:
    """Seeded tensors of one linear: X (M x K), W (N x K), LA (N x R), LB (R x K), bf16 bits.

    ``batch`` > 0 draws another independent batch of activations for the same weights
    (one per data-parallel replica)."""
    wl = WORKLOADS[workload]
    ly = wl.layer(layer)
    M = wl.M if M is None else M
    wkey = (wl.seed, block, ly.lid)
    out = {
        "W": gaussian_bf16(wkey + (1,), (ly.N, ly.K), 1.0 / math.sqrt(ly.K)),
        "LA": gaussian_bf16(wkey + (2,), (ly.N, wl.rank), 0.02),
        "LB": gaussian_bf16(wkey + (3,), (wl.rank, ly.K), 0.02),
        "M": M, "N": ly.N, "K": ly.K, "R": wl.rank, "sparse": ly.sparse,
    }
    if with_x:
        out["X"] = _x(wl, ly, M, block, batch)
    return out


def layer_x(workload: str, layer: str, M: int | None = None, block: int = 0, batch: int = 0) -> np.ndarray:
    """The seeded activation X (M x K bf16 bits) of one linear alone: the same bits as layer_tensors()["X"]."""
    wl = WORKLOADS[workload]
    return _x(wl, wl.layer(layer), wl.M if M is None else M, block, batch)


def sample_rows(key: tuple, M: int, n: int = 512, edge: int = 64) -> np.ndarray:
    """Sorted row indices: ``n`` seeded random rows plus the first and last ``edge`` rows."""
    r = rng(*key).choice(M, size=min(n, M), replace=False)
    e = np.concatenate([np.arange(min(edge, M)), np.arange(max(0, M - edge), M)])
    return np.unique(np.concatenate([r, e]))


def structured_x(kind: str, M: int, K: int, seed: int = 0) -> np.ndarray:
    """Special-case activations (bf16 bits) for edge-case tests.

    ``equal``   every group of 4 holds four entries of one magnitude (random signs);
    ``two4``    already 2:4: two random positions of each group are zero;
    ``zero``    all zeros;
    ``ties``    entries drawn from {-2,-1,-0,+0,1,2} so that ties and signed zeros abound;
    ``mixed``   rows cycling through the kinds above plus plain Gaussian rows.
    """
    g = rng(seed, M, K, 7)
    if kind == "equal":
        mag = np.abs(g.standard_normal((M, K // 4, 1), dtype=np.float32)) + 0.5
        sgn = np.where(g.random((M, K // 4, 4)) < 0.5, -1.0, 1.0).astype(np.float32)
        return bf16_bits((mag * sgn).reshape(M, K))
    if kind == "two4":
        a = g.standard_normal((M, K // 4, 4), dtype=np.float32)
        order = np.argsort(g.random((M, K // 4, 4)), axis=-1)
        np.put_along_axis(a, order[..., :2], 0.0, axis=-1)
        return bf16_bits(a.reshape(M, K))
    if kind == "zero":
        return np.zeros((M, K), dtype=np.uint16)
    if kind == "ties":
        vals = np.array([-2.0, -1.0, -0.0, 0.0, 1.0, 2.0], dtype=np.float32)
        return bf16_bits(vals[g.integers(0, len(vals), size=(M, K))])
    if kind == "mixed":
        kinds = ["equal", "two4", "zero", "ties", None]
        out = np.empty((M, K), dtype=np.uint16)
        for i in range(M):
            k = kinds[i % len(kinds)]
            out[i] = (structured_x(k, 1, K, seed + i) if k else
                      bf16_bits(g.standard_normal((1, K), dtype=np.float32)))[0]
        return out
    raise ValueError(kind)

"""Shared test helpers: moving bf16 bit arrays between numpy and torch, and the
floating-point acceptance check for Y.

Tolerances for Y: relative Frobenius error <= 5e-3 and, per element,
|error| <= 2e-2 * rms(Y_ref) + half a bf16 unit in the last place of y_ref.
The max-abs bound is the arithmetic's; the second term is the rounding of the
bf16 output itself.  bf16 keeps 8 significant bits, so storing y moves it by
up to 2^-8 |y| (an element just above a power of two); at the largest |y| of
a multi-million-entry Gaussian-like output (~6 rms) that is up to 0.023 rms,
more than 2e-2 rms: the exact result rounded to bf16 could fail the bound
alone.  fp32 accumulation over K <= 12288 and the bf16 rounding of the M x 64
LoRA intermediate add far less than 5e-3 to the Frobenius error.
"""
from __future__ import annotations

import numpy as np

REL_FRO = 5e-3
MAX_ABS_RMS = 2e-2
S_RTOL = 1e-5


def to_dev(bits: np.ndarray, device="cuda"):
    import torch
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(device)


def to_bits(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def widen(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def half_ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |v|: the largest change storing v in bf16 makes (8 significant
    bits: 2^(floor(log2 |v|) - 8)); normal range."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 8)


def y_stats(y: np.ndarray, ref: np.ndarray) -> dict:
    err = y - ref
    rms = float(np.sqrt(np.mean(ref * ref)))
    fro = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(err))) if err.size else 0.0
    bound = MAX_ABS_RMS * rms + half_ulp_bf16(ref)
    worst = float(np.max(np.abs(err) / bound)) if err.size else 0.0
    cos = float(np.sum(y * ref) / max(np.linalg.norm(y) * np.linalg.norm(ref), 1e-300))
    return {"rel_fro": fro, "max_abs_over_rms": mx / max(rms, 1e-300), "max_abs_over_bound": worst, "cosine": cos,
            "nonfinite": int(np.count_nonzero(~np.isfinite(y)))}


def assert_y_close(y_bits: np.ndarray, ref: np.ndarray, what: str = "Y") -> dict:
    """Relative Frobenius error <= 5e-3 and, per element, |err| <= 2e-2 rms(Y_ref) + half a bf16 ulp of y_ref."""
    y = widen(y_bits)
    st = y_stats(y, ref)
    assert st["nonfinite"] == 0, (what, st)
    assert st["rel_fro"] <= REL_FRO, (what, st)
    assert st["max_abs_over_bound"] <= 1.0, (what, st)
    return st


def pack_meta_reference(canon: np.ndarray, M: int, K: int) -> np.ndarray:
    """The whole tensor-core metadata buffer described in include/lynx.h, built
    from canonical M x K/8 bytes: uint8 array of lynx_meta_bytes(M, K) bytes."""
    Mp, Kp = -(-M // 256) * 256, -(-K // 128) * 128
    C = Kp // 32                                   # 32-channel chunks per row
    nib = np.full((Mp, Kp // 4), 4, dtype=np.uint32)
    nib[:M, :K // 4] = np.stack([canon & 0xF, canon >> 4], axis=-1).reshape(M, K // 4)
    words = np.zeros((Mp, C), dtype=np.uint32)      # row word of every chunk
    for g in range(8):
        words |= nib[:, g::8] << np.uint32(4 * g)
    lo, hi = words & np.uint32(0xFFFF), words >> np.uint32(16)
    # TMEM order inside each 16-row block: lane 16b+i <- low halves of rows 16b+i, 16b+8+i;
    # lane 16b+8+i <- their high halves
    r = lo.reshape(Mp // 16, 2, 8, C)               # [16-row block, half (rows i / 8+i), i, chunk]
    h = hi.reshape(Mp // 16, 2, 8, C)
    lane_lo = r[:, 0] | (r[:, 1] << np.uint32(16))  # lanes 16b+i
    lane_hi = h[:, 0] | (h[:, 1] << np.uint32(16))  # lanes 16b+8+i
    lanes = np.stack([lane_lo, lane_hi], axis=1).reshape(Mp, C)   # lane-major within each 128-row block
    # [row block, lane, channel block, word] -> [row block, channel block, lane, word]
    out = lanes.reshape(Mp // 128, 128, Kp // 128, 4).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(out).reshape(-1).view(np.uint8)

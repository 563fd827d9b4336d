"""Oracle: rotate, clip, quantize to INT2 per group, pack 4 codes per byte (test infrastructure only).

[Article, "OSCAR 的设计"]: the oldest recent token is rotated, clipped,
quantized and packed and then demoted into the INT2 history; INT2 has only 4
levels; each 4 two-bit values are packed into 1 byte; the INT2 kernel
dequantizes with a scale and a zero point.

Readings (the pages fix none of the arithmetic below):
* Rotated value: x_hat[j] = the float32 nearest (ties to even) to the exact
  real number sum_i x[i] * R32[i][j], x in bf16, R32 the float32 copy of R.
* Per group of g consecutive rotated channels, with the clip ratio c of the
  (head, K/V), all in IEEE float32 with round-to-nearest-even:
      mn, mx = min, max of the group's x_hat
      lo = c * mn ; hi = c * mx
      s32 = (hi - lo) / 3                       (a true division)
      scale = bf16(s32) ; zero = bf16(lo)       (round to nearest even)
      code = clamp(rint((x_hat - zero) / scale), 0, 3)   (rint: ties to even)
  using the stored bf16 scale and zero as float32 values; when the stored
  scale is zero or not finite every code is 0.
* Packing: channel 4b+i of a head vector goes to byte b, bits 2i and 2i+1.
* Dequantization: code * scale + zero, evaluated in float64.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32


# ---- bf16 storage format -------------------------------------------------

def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); finite inputs only."""
    u = np.asarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(F32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


# ---- exactly rounded rotation -------------------------------------------

def round_sum_to_f32(terms) -> np.float32:
    """The float32 nearest (ties to even) to the exact sum of float64 `terms`.

    math.fsum returns the float64 nearest to the exact sum; that float64 rounds
    to the same float32 unless it sits exactly on a float32 midpoint, in which
    case the sign of the exact residual (again by fsum) picks the side.
    """
    terms = list(terms)
    s = math.fsum(terms)
    f = F32(s)
    if float(f) == s or not np.isfinite(f):
        return f
    if float(f) < s:
        lo, hi = f, np.nextafter(f, F32(np.inf))
    else:
        lo, hi = np.nextafter(f, F32(-np.inf)), f
    mid = (float(lo) + float(hi)) / 2.0          # exact: neighbours have 24-bit significands
    if s != mid:
        return f
    res = math.fsum(terms + [-s])
    if res > 0:
        return hi
    if res < 0:
        return lo
    return f                                      # exact tie: numpy rounded half to even


def rotate_exact(x_bits: np.ndarray, R32: np.ndarray) -> np.ndarray:
    """x_hat = round_f32(x @ R32) row by row; x_bits bf16 [n][d], R32 float32 [d][d] -> float32 [n][d]."""
    X = bf16_bits_to_f64(np.atleast_2d(x_bits))
    R = np.asarray(R32, dtype=F32).astype(np.float64)
    n, d = X.shape
    out = np.empty((n, d), F32)
    for r in range(n):
        prods = (X[r][:, None] * R).T.tolist()     # row j: the d exact products feeding channel j
        for j in range(d):
            out[r, j] = round_sum_to_f32(prods[j])
    return out


def rotate_exact_many(x_bits: np.ndarray, R32: np.ndarray) -> np.ndarray:
    """Same result as rotate_exact, for many rows: a float64 product y = x @ R32 has error at most
    gamma_128 * (|x| @ |R32|) (gamma_n = n u / (1 - n u), u = 2^-53, any summation order); where the
    interval y -/+ that bound rounds to one float32 at both ends, that float32 is the correctly rounded
    value; every other element is recomputed by rotate_exact's fsum path."""
    X = bf16_bits_to_f64(np.atleast_2d(x_bits))
    R = np.asarray(R32, dtype=F32).astype(np.float64)
    y = X @ R
    bound = (np.abs(X) @ np.abs(R)) * (1.5e-14 * (1 + 1e-10)) + 1e-300
    lo, hi = (y - bound).astype(F32), (y + bound).astype(F32)
    out = hi.copy()
    for r, j in zip(*np.nonzero(lo != hi)):
        out[r, j] = round_sum_to_f32((X[r] * R[:, j]).tolist())
    return out


# ---- clip + asymmetric INT2 quantizer ------------------------------------

def quantize_group(xh: np.ndarray, clip: float) -> tuple[np.ndarray, np.uint16, np.uint16]:
    """One group of float32 rotated values -> (codes uint8, scale bf16 bits, zero bf16 bits)."""
    xh = np.asarray(xh, dtype=F32)
    c = F32(clip)
    mn = F32(xh.min())
    mx = F32(xh.max())
    lo = F32(c * mn)
    hi = F32(c * mx)
    s32 = F32(F32(hi - lo) / F32(3.0))
    scale_bits = f32_to_bf16_bits(s32)
    zero_bits = f32_to_bf16_bits(lo)
    scale = bf16_bits_to_f32(scale_bits)[()]
    zero = bf16_bits_to_f32(zero_bits)[()]
    if scale == 0 or not np.isfinite(scale):
        codes = np.zeros(xh.shape, np.uint8)
    else:
        t = (xh - zero).astype(F32) / scale
        t = t.astype(F32)
        codes = np.clip(np.rint(t), 0, 3).astype(np.uint8)
    return codes, np.uint16(scale_bits), np.uint16(zero_bits)


def quantize_rotated(xh: np.ndarray, clip: float, group: int):
    """float32 [n][d] rotated rows -> codes [n][d] uint8, scale/zero bf16 bits [n][d/group]."""
    xh = np.atleast_2d(np.asarray(xh, F32))
    n, d = xh.shape
    assert d % group == 0
    ng = d // group
    codes = np.empty((n, d), np.uint8)
    scale = np.empty((n, ng), np.uint16)
    zero = np.empty((n, ng), np.uint16)
    for r in range(n):
        for gi in range(ng):
            sl = slice(gi * group, (gi + 1) * group)
            codes[r, sl], scale[r, gi], zero[r, gi] = quantize_group(xh[r, sl], clip)
    return codes, scale, zero


def quantize_rotated_many(xh: np.ndarray, clip: float, group: int):
    """quantize_rotated with the same float32 operations applied to all groups at once."""
    xh = np.atleast_2d(np.asarray(xh, F32))
    n, d = xh.shape
    ng = d // group
    xg = xh.reshape(n, ng, group)
    c = F32(clip)
    mn, mx = xg.min(axis=2), xg.max(axis=2)
    lo = (c * mn).astype(F32)
    hi = (c * mx).astype(F32)
    s32 = ((hi - lo).astype(F32) / F32(3.0)).astype(F32)
    scale_bits, zero_bits = f32_to_bf16_bits(s32), f32_to_bf16_bits(lo)
    scale, zero = bf16_bits_to_f32(scale_bits), bf16_bits_to_f32(zero_bits)
    valid = (scale != 0) & np.isfinite(scale)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((xg - zero[:, :, None]).astype(F32) / scale[:, :, None]).astype(F32)
        codes = np.clip(np.rint(t), 0, 3)
    codes = np.where(valid[:, :, None], codes, 0).astype(np.uint8).reshape(n, d)
    return codes, scale_bits.reshape(n, ng), zero_bits.reshape(n, ng)


def quantize_vectors_many(x_bits: np.ndarray, R32: np.ndarray, clip: float, group: int):
    codes, scale, zero = quantize_rotated_many(rotate_exact_many(x_bits, R32), clip, group)
    return pack_codes(codes), scale, zero


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[..., d] codes in 0..3 -> [..., d/4] bytes; channel 4b+i at bits 2i..2i+1 of byte b."""
    c = np.asarray(codes, np.uint8)
    assert c.shape[-1] % 4 == 0
    c = c.reshape(c.shape[:-1] + (c.shape[-1] // 4, 4))
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    parts = [(p >> (2 * i)) & 3 for i in range(4)]
    return np.stack(parts, axis=-1).reshape(p.shape[:-1] + (p.shape[-1] * 4,)).astype(np.uint8)


def quantize_vectors(x_bits: np.ndarray, R32: np.ndarray, clip: float, group: int):
    """bf16 rows [n][d] -> (packed codes [n][d/4], scale bits [n][ng], zero bits [n][ng])."""
    codes, scale, zero = quantize_rotated(rotate_exact(x_bits, R32), clip, group)
    return pack_codes(codes), scale, zero


def dequantize(packed: np.ndarray, scale_bits: np.ndarray, zero_bits: np.ndarray, group: int) -> np.ndarray:
    """code * scale + zero in float64; packed [..., d/4], scale/zero [..., d/group]."""
    codes = unpack_codes(packed).astype(np.float64)
    s = np.repeat(bf16_bits_to_f64(scale_bits), group, axis=-1)
    z = np.repeat(bf16_bits_to_f64(zero_bits), group, axis=-1)
    return codes * s + z


def pre_round_value(xh: np.ndarray, scale_bits, zero_bits, group: int) -> np.ndarray:
    """t = (x_hat - zero) / scale in float64 (used to judge how near a code lies to a rounding boundary)."""
    xh = np.asarray(xh, np.float64)
    s = np.repeat(bf16_bits_to_f64(scale_bits), group, axis=-1)
    z = np.repeat(bf16_bits_to_f64(zero_bits), group, axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        return (xh - z) / s

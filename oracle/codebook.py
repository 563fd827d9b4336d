"""Oracle: a 4-level Lloyd-Max codebook in place of the uniform INT2 levels (test infrastructure only).

[Article, the closing comparison with TurboQuant (after "评估结果")]: OSCAR's newest codebase adds a
stronger Lloyd-Max codebook on top of the attention-aware rotation.  The pages give no more; this
module is the plainest reading that keeps the rest of the pipeline:

* the scale and zero point of a group are those of the uniform quantizer (clip c, lo = c*min,
  hi = c*max, scale = bf16((hi - lo)/3), zero = bf16(lo)), and t = (x_hat - zero) / scale in float32 as
  there;
* a codebook is four float32 levels l_0 < l_1 < l_2 < l_3 in that coordinate, one per (KV head, K or V);
  the uniform quantizer is the codebook (0, 1, 2, 3);
* an element's code is the level nearest to t, ties to the even code: with midpoints
  m_i = (l_i + l_{i+1}) / 2 in float32, code = #{i : t > m_i} + #{i : t == m_i and i odd};
* the stored value dequantizes to zero + scale * l_code;
* Lloyd-Max calibration (Lloyd's method on the calibration values t of every element): from
  (0, 1, 2, 3), alternate the midpoints and the cell means (an empty cell keeps its level) until no
  level moves by more than 1e-12 or 200 iterations; the levels are returned rounded to float32.
"""
from __future__ import annotations

import numpy as np

from . import quant

F32 = np.float32
UNIFORM = np.array([0.0, 1.0, 2.0, 3.0], F32)


def midpoints(levels) -> np.ndarray:
    lv = np.asarray(levels, F32)
    return ((lv[:-1] + lv[1:]).astype(F32) * F32(0.5)).astype(F32)


def code_of_levels(t, levels) -> np.ndarray:
    """Nearest level to each float32 t, ties to the even code."""
    t = np.asarray(t, F32)
    m = midpoints(levels)
    above = (t[..., None] > m).sum(-1)
    tie_odd = ((t[..., None] == m) & (np.arange(3) % 2 == 1)).sum(-1)
    return (above + tie_odd).astype(np.uint8)


def quantize_rotated_cb(xh: np.ndarray, clip: float, group: int, levels):
    """float32 [n][d] rotated rows -> (codes [n][d], scale bits [n][ng], zero bits [n][ng]) with the
    uniform quantizer's scale and zero and the codebook's nearest-level codes."""
    xh = np.atleast_2d(np.asarray(xh, F32))
    n, d = xh.shape
    ng = d // group
    xg = xh.reshape(n, ng, group)
    c = F32(clip)
    lo = (c * xg.min(axis=2)).astype(F32)
    hi = (c * xg.max(axis=2)).astype(F32)
    s32 = ((hi - lo).astype(F32) / F32(3.0)).astype(F32)
    scale_bits, zero_bits = quant.f32_to_bf16_bits(s32), quant.f32_to_bf16_bits(lo)
    scale, zero = quant.bf16_bits_to_f32(scale_bits), quant.bf16_bits_to_f32(zero_bits)
    valid = (scale != 0) & np.isfinite(scale)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((xg - zero[:, :, None]).astype(F32) / scale[:, :, None]).astype(F32)
        codes = code_of_levels(t, levels)
    codes = np.where(valid[:, :, None], codes, 0).astype(np.uint8).reshape(n, d)
    return codes, scale_bits.reshape(n, ng), zero_bits.reshape(n, ng)


def quantize_vectors_cb(x_bits: np.ndarray, R32: np.ndarray, clip: float, group: int, levels):
    """bf16 rows [n][d] -> (packed codes, scale bits, zero bits) through the exactly rounded rotation."""
    codes, scale, zero = quantize_rotated_cb(quant.rotate_exact_many(x_bits, R32), clip, group, levels)
    return quant.pack_codes(codes), scale, zero


def dequantize_cb(packed: np.ndarray, scale_bits: np.ndarray, zero_bits: np.ndarray, group: int, levels):
    """zero + scale * level[code] in float64."""
    lv = np.asarray(levels, F32).astype(np.float64)
    codes = quant.unpack_codes(packed)
    s = np.repeat(quant.bf16_bits_to_f64(scale_bits), group, axis=-1)
    z = np.repeat(quant.bf16_bits_to_f64(zero_bits), group, axis=-1)
    return lv[codes] * s + z


def calibration_values(x_bits: np.ndarray, R32: np.ndarray, clip: float, group: int) -> np.ndarray:
    """All float32 t = (x_hat - zero) / scale of the rows x_bits [n][d] (groups with a zero scale left out)."""
    xh = quant.rotate_exact_many(x_bits, R32)
    n, d = xh.shape
    ng = d // group
    xg = xh.reshape(n, ng, group)
    c = F32(clip)
    lo = (c * xg.min(axis=2)).astype(F32)
    hi = (c * xg.max(axis=2)).astype(F32)
    scale = quant.bf16_bits_to_f32(quant.f32_to_bf16_bits(((hi - lo).astype(F32) / F32(3.0)).astype(F32)))
    zero = quant.bf16_bits_to_f32(quant.f32_to_bf16_bits(lo))
    valid = (scale != 0) & np.isfinite(scale)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((xg - zero[:, :, None]).astype(F32) / scale[:, :, None]).astype(F32)
    return t[valid].ravel()


def lloyd_max(t, iters: int = 200, tol: float = 1e-12) -> np.ndarray:
    """Four float32 levels by Lloyd's method on the values t (float64 cell means), from (0, 1, 2, 3)."""
    t = np.asarray(t, np.float64).ravel()
    lv = UNIFORM.astype(np.float64)
    for _ in range(iters):
        m = (lv[:-1] + lv[1:]) / 2
        cell = (t[:, None] > m).sum(-1) + ((t[:, None] == m) & (np.arange(3) % 2 == 1)).sum(-1)
        new = lv.copy()
        for i in range(4):
            sel = t[cell == i]
            if len(sel):
                new[i] = sel.mean()
        moved = np.max(np.abs(new - lv))
        lv = new
        if moved <= tol:
            break
    return lv.astype(F32)

"""Pins for oracle.quant: exact rounding, the INT2 quantizer, packing, bf16 storage.

Rotate, clip, quantize, pack 4 two-bit values per byte, dequantize with scale/zero point
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计").
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import quant
from oracle import rotation as rot
import synth

F32 = np.float32


def _exact_round_to_f32(fr: Fraction) -> np.float32:
    """Nearest float32 (ties to even) to an exact rational, by exact comparison with neighbours."""
    c = F32(float(fr))
    best = None
    for cand in (np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))):
        dist = abs(Fraction(float(cand)) - fr)
        key = (dist, int(np.array(cand, F32).view(np.uint32)) & 1)   # tie -> even significand
        if best is None or key < best[0]:
            best = (key, cand)
    return F32(best[1])


def test_round_sum_matches_exact_rationals():
    g = np.random.default_rng(0)
    for _ in range(300):
        n = int(g.integers(1, 40))
        terms = (g.standard_normal(n) * 2.0 ** g.integers(-30, 30, n)).tolist()
        exact = sum((Fraction(t) for t in terms), Fraction(0))
        assert quant.round_sum_to_f32(terms) == _exact_round_to_f32(exact)


def test_round_sum_midpoint_ties_and_residuals():
    one = 1.0
    mid = one + 2.0 ** -24                        # exactly halfway between 1 and 1 + 2^-23
    assert quant.round_sum_to_f32([mid]) == F32(1.0)                    # tie -> even
    assert quant.round_sum_to_f32([mid, 2.0 ** -80]) == F32(1.0 + 2.0 ** -23)
    assert quant.round_sum_to_f32([mid, -(2.0 ** -80)]) == F32(1.0)
    mid_odd = 1.0 + 3 * 2.0 ** -24                # between 1+2^-23 (odd) and 1+2^-22 (even)
    assert quant.round_sum_to_f32([mid_odd]) == F32(1.0 + 2.0 ** -22)
    # float64 sum lands on the midpoint only after rounding: residual decides
    assert quant.round_sum_to_f32([mid, 2.0 ** -60, -(2.0 ** -61)]) == F32(1.0 + 2.0 ** -23)


def test_rotate_exact_against_rationals():
    g = np.random.default_rng(1)
    d = 128
    R32 = rot.to_f32(rot.rotation_from_gaussian(synth.gaussian_matrix(3, d)))
    xb = synth.to_bf16_bits(g.standard_normal((3, d)) * 7)
    xh = quant.rotate_exact(xb, R32)
    X = quant.bf16_bits_to_f64(xb)
    for r in range(3):
        for j in range(0, d, 9):
            exact = sum((Fraction(float(X[r, i])) * Fraction(float(R32[i, j])) for i in range(d)), Fraction(0))
            assert xh[r, j] == _exact_round_to_f32(exact)


def test_rotate_signed_permutation_orientation():
    # R[0][1] = 1, R[1][0] = -1, R[2][3] = 1, R[3][2] = 1: x_hat = x @ R = [-x1, x0, x3, x2]
    R = np.zeros((4, 4), F32)
    R[0, 1], R[1, 0], R[2, 3], R[3, 2] = 1, -1, 1, 1
    xb = synth.to_bf16_bits(np.array([[1.5, -2.0, 3.25, 0.5]]))
    assert np.array_equal(quant.rotate_exact(xb, R)[0], np.array([2.0, 1.5, 0.5, 3.25], F32))


def test_quantize_group_hand_examples():
    x = np.array([-1.5, -0.5, 0.5, 1.5], F32)
    codes, s, z = quant.quantize_group(x, 1.0)
    assert list(codes) == [0, 1, 2, 3] and s == 0x3F80 and z == 0xBFC0        # scale 1.0, zero -1.5
    codes, s, z = quant.quantize_group(x, 0.5)
    # lo = -0.75, hi = 0.75, scale 0.5: t = -1.5, 0.5, 2.5, 4.5 -> clamp/ties-to-even -> 0, 0, 2, 3
    assert list(codes) == [0, 0, 2, 3] and s == 0x3F00 and z == 0xBF40


def test_scale_is_true_division_then_bf16():
    x = np.array([0.0, 0.25, 0.75, 1.0], F32)       # hi - lo = 1 -> s32 = fp32(1/3) = 0x3EAAAAAB
    _, s, z = quant.quantize_group(x, 1.0)
    assert s == 0x3EAB and z == 0x0000
    assert F32(F32(1.0) / F32(3.0)).view(np.uint32) == 0x3EAAAAAB


def test_constant_group_gives_zero_scale_and_zero_codes():
    codes, s, z = quant.quantize_group(np.full(32, 2.5, F32), 0.9)
    assert s == 0 and np.all(codes == 0)
    assert quant.bf16_bits_to_f32(z) == F32(2.25)


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(2)
    x = (g.standard_normal(20000) * 10.0 ** g.uniform(-6, 6, 20000)).astype(F32)
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(F32)        # exact bf16 midpoints
    x = np.concatenate([x, ties, -ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(quant.f32_to_bf16_bits(x), ref)


def test_pack_layout_and_round_trip():
    assert quant.pack_codes(np.array([1, 2, 3, 0], np.uint8))[0] == 0b00111001
    allb = np.arange(256, dtype=np.uint8)
    assert np.array_equal(quant.pack_codes(quant.unpack_codes(allb[:, None]))[:, 0], allb)
    c = np.random.default_rng(3).integers(0, 4, (17, 128)).astype(np.uint8)
    assert np.array_equal(quant.unpack_codes(quant.pack_codes(c)), c)


@pytest.mark.parametrize("group", [32, 64, 128])
def test_four_levels_and_error_bound(group):
    g = np.random.default_rng(group)
    xh = (g.standard_normal((64, 128)) * 3).astype(F32)
    codes, s, z = quant.quantize_rotated(xh, 1.0, group)
    for r in range(64):
        for gi in range(128 // group):
            cg = codes[r, gi * group:(gi + 1) * group]
            assert len(set(cg.tolist())) <= 4
            assert cg.min() == 0 and cg.max() == 3          # symmetric data spans the range at c = 1
    deq = quant.dequantize(quant.pack_codes(codes), s, z, group)
    sc = np.repeat(quant.bf16_bits_to_f64(s), group, axis=1)
    # inside the clip range the reconstruction error is at most half a step (plus bf16 rounding of zero/scale)
    assert np.all(np.abs(deq - xh) <= 0.5 * sc + 0.02 * sc + 1e-6)


def test_clip_saturates_outside_range():
    xh = np.array([-4.0, -1.0, 0.0, 1.0, 4.0] + [0.5] * 27, F32)
    codes, s, z = quant.quantize_group(xh, 0.5)       # lo = -2, hi = 2
    assert codes[0] == 0 and codes[4] == 3


def test_dequantize_closed_form():
    packed = quant.pack_codes(np.array([[0, 1, 2, 3] * 32], np.uint8))
    s = quant.f32_to_bf16_bits(np.array([[0.5]], F32))
    z = quant.f32_to_bf16_bits(np.array([[-1.0]], F32))
    assert np.array_equal(quant.dequantize(packed, s, z, 128)[0], np.array([-1.0, -0.5, 0.0, 0.5] * 32))


@pytest.mark.parametrize("group", [32, 128])
def test_many_row_paths_equal_plain_paths(group):
    g = np.random.default_rng(9)
    d = 128
    R32 = rot.to_f32(rot.rotation_from_gaussian(synth.gaussian_matrix(9, d)))
    ch = synth.outlier_channels(9, 1, d, 4)
    xb = synth.outlier_kv(9, 40, 1, d, ch)[:, 0]
    assert np.array_equal(quant.rotate_exact_many(xb, R32), quant.rotate_exact(xb, R32))
    xh = quant.rotate_exact(xb, R32)
    a = quant.quantize_rotated(xh, 0.9, group)
    b = quant.quantize_rotated_many(xh, 0.9, group)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    # degenerate groups (constant) agree too
    const = np.full((3, d), 1.5, np.float32)
    for u, v in zip(quant.quantize_rotated(const, 0.9, group), quant.quantize_rotated_many(const, 0.9, group)):
        assert np.array_equal(u, v)


def test_rotate_many_resolves_midpoints_exactly():
    # y = 1 + 2^-24 (an exact float32 midpoint) plus/minus tiny residuals: the bound interval
    # straddles the midpoint, so the exact path must decide.
    R = np.zeros((128, 128), np.float32)
    R[0, 0], R[1, 0], R[2, 0] = 1.0, 2.0 ** -24, 2.0 ** -60
    for third, want in ((1.0, F32(1.0 + 2.0 ** -23)), (-1.0, F32(1.0)), (0.0, F32(1.0))):
        x = np.zeros((1, 128), np.float32)
        x[0, :3] = [1.0, 1.0, third]
        xb = synth.to_bf16_bits(x)
        assert quant.rotate_exact_many(xb, R)[0, 0] == want == quant.rotate_exact(xb, R)[0, 0]

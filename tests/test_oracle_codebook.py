"""Pins for oracle.codebook: the 4-level codebook quantizer and Lloyd-Max calibration (the Lloyd-Max
codebook that OSCAR's newest codebase adds, "超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化",
closing comparison with TurboQuant)."""
import numpy as np
import pytest
from scipy.stats import norm

from oracle import codebook, pool as opool, quant
from oracle import rotation as rot
import synth


def test_uniform_levels_are_the_uniform_quantizer():
    """Every float32 t (including exact halves and out-of-range values) gets clamp(rint(t), 0, 3)."""
    g = np.random.default_rng(0)
    t = np.concatenate([g.uniform(-2, 5, 20000), np.arange(-2, 5.01, 0.25), [np.float32(0.5), np.float32(2.5)]])
    t = t.astype(np.float32)
    np.testing.assert_array_equal(codebook.code_of_levels(t, codebook.UNIFORM),
                                  np.clip(np.rint(t), 0, 3).astype(np.uint8))


def test_uniform_codebook_reproduces_the_pool_quantizer():
    R = rot.to_f32(rot.rotation_from_gaussian(synth.gaussian_matrix(5, 128)))
    x = synth.outlier_kv(6, 300, 1, 128, np.array([[3, 40, 77, 100]]))[:, 0]
    for g in (32, 128):
        a = quant.quantize_vectors_many(x, R, 0.9, g)
        b = codebook.quantize_vectors_cb(x, R, 0.9, g, codebook.UNIFORM)
        for u, v in zip(a, b):
            np.testing.assert_array_equal(u, v)


def test_nearest_level_with_ties_to_even():
    lv = np.array([0.25, 1.0, 2.25, 2.75], np.float32)
    m = codebook.midpoints(lv)                      # 0.625, 1.625, 2.5
    t = np.array([-1, 0.6, 0.625, 0.7, 1.625, 1.7, 2.5, 2.6, 9], np.float32)
    np.testing.assert_array_equal(codebook.code_of_levels(t, lv), [0, 0, 0, 1, 2, 2, 2, 3, 3])
    # brute force: nearest level, ties to the even index
    for v in np.linspace(-1, 4, 401).astype(np.float32):
        d = np.abs(lv.astype(np.float64) - float(v))
        cand = np.flatnonzero(d == d.min())
        want = cand[0] if len(cand) == 1 else [c for c in cand if c % 2 == 0][0]
        assert codebook.code_of_levels(np.float32(v), lv) == want, v
    assert np.all(np.diff(m) > 0)


def test_lloyd_max_uniform_distribution_closed_form():
    """For t uniform on [0, 3] the optimal four levels are the centres of four equal cells."""
    t = (np.arange(300000) + 0.5) / 100000.0
    np.testing.assert_allclose(codebook.lloyd_max(t), [0.375, 1.125, 1.875, 2.625], atol=1e-5)


def test_lloyd_max_gaussian_textbook_levels():
    """The 4-level Lloyd-Max quantizer of N(0, 1) has levels +-0.4528 and +-1.5104 (Max, 1960)."""
    z = norm.ppf((np.arange(400000) + 0.5) / 400000)
    lv = codebook.lloyd_max(1.5 + 0.5 * z)
    np.testing.assert_allclose((lv - 1.5) / 0.5, [-1.5104, -0.4528, 0.4528, 1.5104], atol=2e-3)


def test_lloyd_max_levels_are_their_cells_centroids():
    t = np.random.default_rng(3).gamma(2.0, 0.6, 50000).clip(0, 3)
    lv = codebook.lloyd_max(t).astype(np.float64)
    m = (lv[:-1] + lv[1:]) / 2
    cell = (t[:, None] > m).sum(-1)
    for i in range(4):
        assert lv[i] == pytest.approx(t[cell == i].mean(), abs=1e-6)


def test_codebook_pool_round_trip_and_distortion():
    """A pool with a calibrated codebook stores the codes of nearest levels; its dequantized history
    is closer to the rotated vectors than the uniform levels' on the calibration distribution."""
    d, L = 128, 320 + 640
    ch = synth.outlier_channels(7, 1, d, 4)
    K = synth.outlier_kv(8, L, 1, d, ch)
    R = rot.to_f32(rot.hadamard(d) @ rot.bitrev_matrix(d))
    lv = codebook.lloyd_max(codebook.calibration_values(K[:, 0], R, 0.9, 128))
    assert np.all(np.diff(lv) > 0) and not np.array_equal(lv, codebook.UNIFORM)
    err = {}
    for name, cb in (("uniform", None), ("lloyd", lv[None])):
        P = opool.Pool(1, 4, 1, d, 128, 10, 10, R[None], R[None], [0.9], [0.9], codebook_k=cb, codebook_v=cb)
        P.page_table[0] = np.arange(10, dtype=np.int32)
        P.prefill(0, K, K)
        _, _, hk, _, _, _ = P.segments(0, 0)
        exact = quant.rotate_exact_many(K[64:L - 256, 0], R).astype(np.float64)
        err[name] = np.mean((hk - exact) ** 2)
    assert err["lloyd"] < err["uniform"]


def test_calibration_values_hand_computed_rows():
    """calibration_values on rows whose t are known by hand (R = I, so x_hat = x):
    row A: min -3, max 6, clip 1: scale 3, zero -3, t = (x + 3) / 3;
    row B: min -4, max 8, clip 0.5: the clip scales the extremes only (lo -2, hi 4, scale 2, zero -2), so
           x = -4 gives t = -1 and x = 8 gives t = 5 (no clamp of x);
    row C: min 0, max 1, clip 1: scale = bf16(fp32(1/3)) = 0.333984375 (0x3EAB), so x = 1 gives
           t = fp32(1 / 0.333984375) = 2.9941520..., not 3 (the stored bf16 scale is the divisor);
    row D: constant: scale 0, the group is left out."""
    d = 128
    I = np.eye(d, dtype=np.float32)
    base = np.zeros(d, np.float32)
    A = base.copy(); A[[0, 1, 2, 3]] = [-3.0, 6.0, 0.0, 1.5]
    B = base.copy(); B[[0, 1, 2]] = [-4.0, 8.0, 0.0]
    C = base.copy(); C[[5, 9]] = [1.0, 0.5]
    Dc = np.full(d, 2.0, np.float32)
    rows = lambda *r: synth.to_bf16_bits(np.stack(r))
    tA = codebook.calibration_values(rows(A), I, 1.0, 128)
    assert tA.shape == (128,)
    np.testing.assert_array_equal(tA[:4], np.array([0.0, 3.0, 1.0, 1.5], np.float32))
    assert np.all(tA[4:] == np.float32(1.0))                       # x = 0 -> (0 + 3) / 3
    tB = codebook.calibration_values(rows(B), I, 0.5, 128)
    np.testing.assert_array_equal(tB[:3], np.array([-1.0, 5.0, 1.0], np.float32))
    tC = codebook.calibration_values(rows(C), I, 1.0, 128)
    assert tC[5] == np.float32(1.0) / np.float32(0.333984375) and tC[5] != np.float32(3.0)
    assert tC[0] == 0.0 and tC[9] == np.float32(0.5) / np.float32(0.333984375)
    assert codebook.calibration_values(rows(Dc), I, 1.0, 128).size == 0
    # group 32: the constant group of a row is left out, the others kept in order
    E = base.copy(); E[:32] = 7.0; E[32:64] = np.linspace(-1, 2, 32).round(2); E[64] = -6.0; E[127] = 3.0
    tE = codebook.calibration_values(rows(E), I, 1.0, 32)
    assert tE.size == 96                                           # groups 1, 2, 3 of 4
    g3 = tE[64:]                                                   # group 3: min 0, max 3 -> scale 1, zero 0
    assert g3[-1] == np.float32(3.0) and np.all(g3[:-1] == 0.0)
    g2 = tE[32:64]                                                 # group 2: min -6, max 0 -> scale 2, zero -6
    assert g2[0] == 0.0 and np.all(g2[1:] == np.float32(3.0))

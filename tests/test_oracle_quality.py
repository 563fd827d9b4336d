"""Pins for oracle.quality: the score KL and output error of an INT2 pool against exact attention
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的动机", Fig. 1)."""
import numpy as np
import pytest
from scipy.special import rel_entr

from oracle import pool as opool
from oracle import quality
from oracle import rotation as rot
import synth


def test_kl_matches_scipy_and_is_zero_on_equal_inputs():
    g = np.random.default_rng(0)
    p, q = g.dirichlet(np.ones(50)), g.dirichlet(np.ones(50))
    assert quality.kl_divergence(p, q) == pytest.approx(float(np.sum(rel_entr(p, q))), rel=1e-12)
    assert quality.kl_divergence(p, p) == 0.0
    assert quality.kl_divergence(p, q) > 0


def _pool(R, clip, L, Hq=4, Hkv=1, d=128, g=128):
    pages = -(-(L - 320) // 64) + 1
    Rs = np.stack([R] * Hkv).astype(np.float32)
    P = opool.Pool(1, Hq, Hkv, d, g, pages, pages, Rs, Rs, [clip] * Hkv, [clip] * Hkv)
    P.page_table[0] = np.arange(pages, dtype=np.int32)
    return P


def test_lossless_history_gives_zero_error():
    """History vectors whose every channel is one of 4 evenly spaced levels (spacing a power of two,
    R = I, no clipping) are stored exactly: KL and output error vanish."""
    L, d = 320 + 200, 128
    g = np.random.default_rng(1)
    lv = np.array([-1.5, -0.5, 0.5, 1.5], np.float32)
    K = np.empty((L, 1, d), np.float32)
    V = np.empty((L, 1, d), np.float32)
    for X in (K, V):
        X[:] = lv[g.integers(0, 4, size=X.shape)]
        X[:, :, 0] = -1.5   # every vector spans all four levels, so min/max are the end levels
        X[:, :, 1] = 1.5
    Kb, Vb = synth.to_bf16_bits(K), synth.to_bf16_bits(V)
    P = _pool(np.eye(d), 1.0, L)
    P.prefill(0, Kb, Vb)
    q = synth.to_bf16_bits(g.standard_normal((4, d)))
    kl, err = quality.metrics(P, 0, Kb, Vb, q)
    assert abs(kl) < 1e-12 and err < 1e-24


def test_rotations_reduce_the_distortion_on_outlier_activations():
    """Anisotropic activations (calibration-style draws) with four outlier channels in K and V: the
    Hadamard / bit-reversal rotation cuts the distortion of naive INT2 (R = I), and the covariance-
    aligned rotation with clipping cuts it further (the ordering of the pages' Fig. 1 on this recipe)."""
    d, G, T, L = 128, 4, 2048, 320 + 640
    ch = synth.outlier_channels(3, 1, d, 4)
    Qs = synth.calib_samples(10, T + 1, G, d, ch, heads_per_channel_set=G, factor=4.0)
    KV = synth.calib_samples(11, T + L, 2, d, ch, heads_per_channel_set=2, factor=10.0)
    f = lambda b: synth.bf16_bits_to_f32(b).astype(np.float64)
    K, V, q = KV[T:, 0][:, None], KV[T:, 1][:, None], Qs[T]
    HP = rot.to_f32(rot.hadamard(d) @ rot.bitrev_matrix(d))
    Rk = rot.to_f32(rot.rotation_from_covariance(rot.covariance_k(f(Qs[:T]))))
    Rv = rot.to_f32(rot.rotation_from_covariance(rot.covariance_v(f(Qs[:T]), f(KV[:T, 0]), f(KV[:T, 1]))))
    res = {}
    for name, rk, rv, c in (("naive", np.eye(d), np.eye(d), 1.0), ("hadamard", HP, HP, 1.0), ("oscar", Rk, Rv, 0.9)):
        pages = -(-(L - 320) // 64) + 1
        P = opool.Pool(1, G, 1, d, 128, pages, pages, rk[None].astype(np.float32), rv[None].astype(np.float32),
                       [c], [c])
        P.page_table[0] = np.arange(pages, dtype=np.int32)
        P.prefill(0, K, V)
        res[name] = quality.metrics(P, 0, K, V, q)
    assert res["naive"][0] > 0 and res["naive"][1] > 0
    assert res["oscar"][1] < res["hadamard"][1] < res["naive"][1]
    assert res["hadamard"][0] < res["naive"][0] and res["oscar"][0] < res["naive"][0]

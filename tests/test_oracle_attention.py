"""Pins for oracle.attention: library softmax attention, segment merge, rotation invariance.

BF16 sink/recent and INT2 history handled separately and combined by an online-softmax merge
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计").
"""
import numpy as np
import pytest
import torch

from oracle import attention as att
from oracle import rotation as rot
import synth


def _sdpa(q, K, V, scale):
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        t(q[None]), t(K), t(V), scale=scale)[0, 0, 0].numpy()


def test_softmax_attend_matches_library():
    g = np.random.default_rng(0)
    q, K, V = g.standard_normal(64) * 4, g.standard_normal((300, 64)) * 3, g.standard_normal((300, 64))
    assert np.max(np.abs(att.softmax_attend(q, K, V, 0.125) - _sdpa(q, K, V, 0.125))) < 1e-13


@pytest.mark.parametrize("cuts", [(0, 10, 10, 300), (0, 0, 150, 300), (0, 1, 299, 300), (0, 64, 128, 300)])
def test_segment_merge_equals_brute_force(cuts):
    g = np.random.default_rng(1)
    q, K, V = g.standard_normal(32) * 30, g.standard_normal((300, 32)), g.standard_normal((300, 32))
    parts = [att.segment_partial(q, K[a:b], V[a:b], 0.1) for a, b in zip(cuts[:-1], cuts[1:])]
    m, l, o = att.lse_merge(parts)
    assert np.max(np.abs(o / l - att.softmax_attend(q, K, V, 0.1))) < 1e-12
    m2, l2, o2 = att.online_segment(q, K, V, 0.1, tile=17)
    assert np.max(np.abs(o2 / l2 - att.softmax_attend(q, K, V, 0.1))) < 1e-12


def _rotation(d, seed):
    return rot.rotation_from_gaussian(synth.gaussian_matrix(seed, d))


def test_rotated_history_is_invariant():
    """History stored as exact K·R_k and V·R_v: the decode equals plain attention over all tokens."""
    g = np.random.default_rng(2)
    d = 128
    Rk, Rv = _rotation(d, 1), _rotation(d, 2)
    q = g.standard_normal(d) * 3
    sk, sv = g.standard_normal((5, d)), g.standard_normal((5, d))
    hk, hv = g.standard_normal((70, d)), g.standard_normal((70, d))
    rk, rv = g.standard_normal((9, d)), g.standard_normal((9, d))
    s = 1 / np.sqrt(d)
    ref = att.softmax_attend(q, np.concatenate([sk, hk, rk]), np.concatenate([sv, hv, rv]), s)
    got = att.decode_one_head(q, sk, sv, hk @ Rk, hv @ Rv, rk, rv, Rk, Rv, s)
    assert np.max(np.abs(got - ref)) < 1e-12
    got2 = att.decode_one_head_merged(q, sk, sv, hk @ Rk, hv @ Rv, rk, rv, Rk, Rv, s, tile=16)
    assert np.max(np.abs(got2 - ref)) < 1e-12


def test_empty_history_is_plain_bf16_attention():
    g = np.random.default_rng(3)
    d = 128
    q = g.standard_normal(d)
    sk, sv, rk, rv = (g.standard_normal((n, d)) for n in (64, 64, 256, 256))
    R = _rotation(d, 3)
    got = att.decode_one_head(q, sk, sv, np.zeros((0, d)), np.zeros((0, d)), rk, rv, R, R, 1 / np.sqrt(d))
    ref = _sdpa(q, np.concatenate([sk, rk]), np.concatenate([sv, rv]), 1 / np.sqrt(d))
    assert np.max(np.abs(got - ref)) < 1e-13


def test_single_history_token_closed_form():
    g = np.random.default_rng(4)
    d = 128
    R = _rotation(d, 4)
    hv = g.standard_normal((1, d))
    got = att.decode_one_head(g.standard_normal(d), np.zeros((0, d)), np.zeros((0, d)),
                              g.standard_normal((1, d)), hv, np.zeros((0, d)), np.zeros((0, d)), R, R, 0.3)
    assert np.max(np.abs(got - hv[0] @ R.T)) < 1e-13


def test_wrong_unrotation_would_fail():
    """Guards the orientation: using R_v instead of R_v^T changes the result."""
    g = np.random.default_rng(5)
    d = 128
    R = _rotation(d, 5)
    hv = g.standard_normal((1, d))
    got = att.decode_one_head(g.standard_normal(d), np.zeros((0, d)), np.zeros((0, d)),
                              g.standard_normal((1, d)), hv @ R, np.zeros((0, d)), np.zeros((0, d)), R, R, 0.3)
    assert np.max(np.abs(got - hv[0])) < 1e-12
    assert np.max(np.abs((hv[0] @ R) @ R - hv[0])) > 1e-3

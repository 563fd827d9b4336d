"""Pins for oracle.pool: segment placement, demotion order, ring wrap-around, lossless round trip.

Three-segment pool "BF16 sink (64 tokens) | INT2 history | BF16 recent (256 tokens)"; new tokens
enter the recent window and the oldest recent token is demoted
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计").
"""
import numpy as np
import pytest
import torch

from oracle import pool as opool
from oracle import quant
from oracle import rotation as rot
import synth


def _make(B, Hq, Hkv, d, g, pages, R=None, clip=1.0, seed=0):
    if R is None:
        R = rot.to_f32(rot.rotation_from_gaussian(synth.gaussian_matrix(seed, d)))
    Rk = np.stack([R] * Hkv)
    P = opool.Pool(B, Hq, Hkv, d, g, pages, pages, Rk, Rk, [clip] * Hkv, [clip] * Hkv)
    P.page_table[:] = synth.page_tables(seed, [pages // B] * B, pages, pages)[0]
    return P


@pytest.mark.parametrize("L", [1, 63, 64, 65, 320, 321, 385, 700])
def test_prefill_segment_lengths(L):
    P = _make(1, 2, 1, 32, 32, 8)
    x = synth.outlier_kv(1, L, 1, 32, np.array([[3]]))
    P.prefill(0, x, x)
    assert P.sink_len[0] == min(L, 64)
    assert P.recent_len[0] == min(max(L - 64, 0), 256)
    assert P.hist_len[0] == max(L - 320, 0)
    assert np.array_equal(P.sink_k[0, 0, :P.sink_len[0]], x[:P.sink_len[0], 0])
    if L > 320:
        assert np.array_equal(P.recent_k[0, 0, :256], x[L - 256:, 0])


def test_append_equals_prefill_of_longer_sequence():
    """prefill(L) followed by n appends leaves the same pool as prefill(L + n) (history order, ring wrap)."""
    d, L, n = 32, 330, 300
    x = synth.outlier_kv(2, L + n, 2, d, np.array([[1, 5], [2, 9]]))
    y = synth.outlier_kv(3, L + n, 2, d, np.array([[1, 5], [2, 9]]))
    A = _make(1, 4, 2, d, 16, 8)
    A.prefill(0, x[:L], y[:L])
    for t in range(L, L + n):
        A.append(x[t][None], y[t][None])
    Bp = _make(1, 4, 2, d, 16, 8)
    Bp.prefill(0, x, y)
    assert A.hist_len[0] == Bp.hist_len[0] == L + n - 320
    for name in ("codes_k", "codes_v", "scale_k", "zero_k", "scale_v", "zero_v", "sink_k", "sink_v"):
        assert np.array_equal(getattr(A, name), getattr(Bp, name)), name
    segA, segB = A.segments(0, 1), Bp.segments(0, 1)
    for a, b in zip(segA, segB):
        assert np.array_equal(a, b)


def test_append_from_empty_fills_sink_then_recent():
    d = 32
    x = synth.outlier_kv(4, 70, 1, d, np.array([[0]]))
    P = _make(1, 1, 1, d, 32, 4)
    for t in range(70):
        P.append(x[t][None], x[t][None])
    assert (P.sink_len[0], P.hist_len[0], P.recent_len[0]) == (64, 0, 6)
    assert np.array_equal(P.recent_k[0, 0, :6], x[64:70, 0])


def test_lossless_tokens_round_trip_through_decode():
    """Tokens whose rotated groups already sit on a 4-level grid survive quantization exactly,
    so decode over the pool equals library attention over the original tokens."""
    d, Hkv, g = 32, 1, 32
    R = np.eye(d, dtype=np.float32)[::-1].copy()        # exact signed permutation (reversal)
    rng = np.random.default_rng(5)
    L = 400
    codes = rng.integers(0, 4, (L, Hkv, d))
    codes[:, :, 0], codes[:, :, 1] = 0, 3                # every group spans its range
    x = (codes * 0.5 - 0.75).astype(np.float32)          # values -0.75, -0.25, 0.25, 0.75 (exact bf16)
    xb = synth.to_bf16_bits(x)
    P = _make(1, 2, Hkv, d, g, 4, R=R, clip=1.0)
    P.prefill(0, xb, xb)
    sk, sv, hk, hv, rk, rv = P.segments(0, 0)
    assert np.array_equal(hk, x[64:144, 0] @ R.astype(np.float64))
    q = synth.to_bf16_bits(rng.standard_normal((1, 2, d)))
    out = P.decode(q)
    X = quant.bf16_bits_to_f64(xb)[:, 0]
    for h in range(2):
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(quant.bf16_bits_to_f64(q[0, h]))[None, None, None],
            torch.from_numpy(X)[None, None], torch.from_numpy(X)[None, None], scale=1 / np.sqrt(d))[0, 0, 0].numpy()
        assert np.max(np.abs(out[0, h] - ref)) < 1e-12


def test_demote_mask_moves_exactly_flagged_sequences():
    d = 32
    x = synth.outlier_kv(6, 400, 1, d, np.array([[7]]))
    P = _make(2, 1, 1, d, 32, 8)
    P.prefill(0, x, x)
    P.prefill(1, x[:300], x[:300])
    P.demote(np.array([0, 1]))
    assert (P.hist_len[0], P.recent_len[0]) == (80, 256)
    assert (P.hist_len[1], P.recent_len[1], P.recent_start[1]) == (1, 235, 1)


def test_shared_prefix_pages_equal_private_copies():
    """Two sequences with the same first 64 * P history tokens: the second one's page table points at
    the first one's prefix pages (written once).  Its decode equals, exactly, that of a pool where it has
    private pages holding the same tokens; sharing pages whose tokens differ would change it."""
    d, P, L = 32, 3, 320 + 64 * 5 + 10          # 5 full history pages + 10 tokens
    shared = synth.outlier_kv(11, L, 1, d, np.array([[2]]))
    tail = synth.outlier_kv(12, L, 1, d, np.array([[2]]))
    K1 = np.concatenate([shared[:64 + 64 * P], tail[64 + 64 * P:]])
    V0 = synth.outlier_kv(13, L, 1, d, np.array([[2]]))
    V1 = np.concatenate([V0[:64 + 64 * P], tail[64 + 64 * P:][:, :, ::-1]])
    q = synth.outlier_q(14, 2, 2, 1, d, np.array([[2]]))

    def make(share):
        Pl = _make(2, 2, 1, d, 16, 12)
        pt = np.full((2, 12), -1, np.int32)
        pt[:, :6] = np.arange(12, dtype=np.int32).reshape(2, 6)
        if share:
            pt[1, :P] = pt[0, :P]
        Pl.page_table[:] = pt
        Pl.prefill(0, shared, V0)
        Pl.prefill(1, K1, V1, shared_pages=P if share else 0)
        return Pl

    A, B = make(True), make(False)
    np.testing.assert_array_equal(A.decode(q), B.decode(q))
    # the pages seq 1 would have written for its prefix are byte-identical to the shared ones
    for name in ("codes_k", "codes_v", "scale_k", "zero_k", "scale_v", "zero_v"):
        arr = getattr(B, name)
        np.testing.assert_array_equal(arr[:P], arr[6:6 + P])
    bad = make(True)
    bad.prefill(0, tail, V0)                     # the prefix pages now hold other tokens
    assert np.abs(bad.decode(q)[1] - A.decode(q)[1]).max() > 1e-3

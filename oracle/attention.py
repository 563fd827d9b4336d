"""Oracle: float64 decode attention over the three-segment pool (test infrastructure only).

[Article, "OSCAR 的设计"]: at decode the BF16 segments (sink and recent) and
the INT2 history are handled separately — the INT2 side unpacks, dequantizes
with scale/zero point and accumulates in floating point, the BF16 side handles
sink/recent — and an online-softmax merge combines the two results.

Readings:
* Score of a BF16 token: (q . k) * softmax_scale in the original space.
* Score of a history token: (q · R_k) . k_tilde_rot * softmax_scale, where
  k_tilde_rot = code * scale + zero is the stored (rotated) key; its value
  enters the output as v_tilde_rot · R_v^T.  R_k and R_v are the float32
  device copies, widened to float64.  softmax_scale defaults to 1/sqrt(d).
* Query head h reads KV head h // (Hq/Hkv).
* The result is exact softmax attention in float64 over every token of the
  pool: the segment split and the merge change nothing mathematically.
"""
from __future__ import annotations

import numpy as np


def softmax_attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Brute force: softmax(K q * scale) @ V, all float64."""
    s = (np.asarray(K, np.float64) @ np.asarray(q, np.float64)) * scale
    p = np.exp(s - s.max())
    return (p / p.sum()) @ np.asarray(V, np.float64)


def segment_partial(q, K, V, scale):
    """(m, l, o_unnormalised) of one segment; m = -inf, l = 0, o = 0 for an empty segment."""
    K = np.asarray(K, np.float64)
    d = np.asarray(V).shape[-1] if np.asarray(V).ndim == 2 else len(q)
    if K.shape[0] == 0:
        return -np.inf, 0.0, np.zeros(d)
    s = (K @ np.asarray(q, np.float64)) * scale
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ np.asarray(V, np.float64)


def online_segment(q, K, V, scale, tile: int):
    """Streaming online softmax over tiles of one segment (running max, rescaled sum and output)."""
    m, l, o = -np.inf, 0.0, np.zeros(np.asarray(V).shape[1])
    for t0 in range(0, K.shape[0], tile):
        mt, lt, ot = segment_partial(q, K[t0:t0 + tile], V[t0:t0 + tile], scale)
        m, l, o = lse_merge([(m, l, o), (mt, lt, ot)])
    return m, l, o


def lse_merge(parts):
    """Combine (m_i, l_i, o_i) partials: m = max m_i, l = sum e^{m_i-m} l_i, o = sum e^{m_i-m} o_i."""
    m = max(p[0] for p in parts)
    if m == -np.inf:
        return -np.inf, 0.0, np.zeros_like(parts[0][2])
    l = sum(np.exp(p[0] - m) * p[1] for p in parts if p[0] != -np.inf)
    o = sum(np.exp(p[0] - m) * p[2] for p in parts if p[0] != -np.inf)
    return m, l, o


def decode_one_head(q, sink_k, sink_v, hist_k_rot, hist_v_rot, recent_k, recent_v, R_k, R_v, scale):
    """Exact attention of one query head over sink + history + recent, float64, one softmax."""
    q = np.asarray(q, np.float64)
    R_k = np.asarray(R_k, np.float64)
    R_v = np.asarray(R_v, np.float64)
    q_rot = q @ R_k
    s = np.concatenate([
        (np.asarray(sink_k, np.float64) @ q) * scale,
        (np.asarray(hist_k_rot, np.float64) @ q_rot) * scale,
        (np.asarray(recent_k, np.float64) @ q) * scale,
    ])
    p = np.exp(s - s.max())
    p /= p.sum()
    n0, n1 = len(sink_k), len(sink_k) + len(hist_k_rot)
    out = p[:n0] @ np.asarray(sink_v, np.float64) + p[n1:] @ np.asarray(recent_v, np.float64)
    if n1 > n0:
        out = out + (p[n0:n1] @ np.asarray(hist_v_rot, np.float64)) @ R_v.T
    return out


def decode_one_head_merged(q, sink_k, sink_v, hist_k_rot, hist_v_rot, recent_k, recent_v, R_k, R_v,
                           scale, tile: int = 64):
    """The same attention computed the split way: history in rotated space with a streaming online
    softmax, one BF16 partial over sink + recent, the history output un-rotated by R_v^T, then an
    LSE merge."""
    q = np.asarray(q, np.float64)
    R_k = np.asarray(R_k, np.float64)
    R_v = np.asarray(R_v, np.float64)
    mh, lh, oh = online_segment(q @ R_k, np.asarray(hist_k_rot, np.float64),
                                np.asarray(hist_v_rot, np.float64), scale, tile)
    oh = oh @ R_v.T
    kb = np.concatenate([np.asarray(sink_k, np.float64), np.asarray(recent_k, np.float64)])
    vb = np.concatenate([np.asarray(sink_v, np.float64), np.asarray(recent_v, np.float64)])
    mb, lb, ob = segment_partial(q, kb, vb, scale)
    m, l, o = lse_merge([(mh, lh, oh), (mb, lb, ob)])
    return o / l

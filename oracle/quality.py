"""Oracle: attention quality of an INT2 pool against exact attention (test infrastructure only).

[Article, "OSCAR 的动机" (Fig. 1)]: INT2 quantization of the KV cache distorts the attention that the
model computes, and rotations and clipping reduce that distortion (naive INT2 and Hadamard-only
rotation degrade; OSCAR's attention-aware rotation keeps the attention close to BF16).  The pages
measure this on real models; here the two attention-level quantities it rests on are computed in
float64 for one decode query per head:

* score KL: KL(p || p_hat) with p = softmax of the exact scores (q . k * scale over the BF16 tokens)
  and p_hat = softmax of the scores the pool attends with (history keys dequantized in the rotated
  space against q . R_k; sink and recent keys exact), summed over tokens, averaged over query heads;
* output error: sum over heads of ||o_hat - o||^2 divided by sum of ||o||^2, with o the exact
  attention output and o_hat the pool's (history values dequantized and un-rotated by R_v^T).

Readings: natural log; the mean over query heads of the per-head KL; one relative squared error over
all heads (not a mean of ratios).
"""
from __future__ import annotations

import numpy as np

from . import attention, quant


def _softmax(s):
    e = np.exp(s - s.max())
    return e / e.sum()


def kl_divergence(p, p_hat) -> float:
    """sum_t p_t log(p_t / p_hat_t), terms with p_t = 0 contributing 0."""
    p, p_hat = np.asarray(p, np.float64), np.asarray(p_hat, np.float64)
    m = p > 0
    return float(np.sum(p[m] * (np.log(p[m]) - np.log(p_hat[m]))))


def pool_scores(pool, b, kvh, q):
    """Scores (times softmax scale) the pool attends with for query q (float64 [d]) of KV head kvh of
    sequence b, in token order sink | history | recent."""
    sk, sv, hk, hv, rk, rv = pool.segments(b, kvh)
    q_rot = q @ pool.R_k[kvh].astype(np.float64)
    return np.concatenate([sk @ q, hk @ q_rot, rk @ q])


def metrics(pool, b, K_bits, V_bits, q_bits, softmax_scale=None):
    """(mean score KL, relative output error) of sequence b of `pool`, whose tokens in order are the bf16
    rows K_bits, V_bits [L][Hkv][d], for the bf16 queries q_bits [Hq][d]."""
    scale = 1.0 / np.sqrt(pool.d) if softmax_scale is None else softmax_scale
    G = pool.Hq // pool.Hkv
    f = quant.bf16_bits_to_f64
    q_all = np.zeros((pool.B,) + q_bits.shape, np.uint16)
    q_all[b] = q_bits
    o_hat = pool.decode(q_all, scale, batch=[b])[b]
    kls, num, den = [], 0.0, 0.0
    for h in range(pool.Hq):
        kvh = h // G
        q = f(q_bits[h])
        K, V = f(K_bits[:, kvh]), f(V_bits[:, kvh])
        p = _softmax((K @ q) * scale)
        p_hat = _softmax(pool_scores(pool, b, kvh, q) * scale)
        kls.append(kl_divergence(p, p_hat))
        o = attention.softmax_attend(q, K, V, scale)
        num += float(np.sum((o_hat[h] - o) ** 2))
        den += float(np.sum(o ** 2))
    return float(np.mean(kls)), num / den

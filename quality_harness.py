"""Attention-quality harness (a measurement beside the benchmark, not part of the library's decode path):
attention quality of INT2 history variants, measured with the library's own kernels.

"超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的动机" (Fig. 1): naive INT2
and Hadamard-only rotation distort the attention at two bits, OSCAR's covariance-aligned rotation
with clipping keeps it close to BF16.  This module measures the two attention-level quantities behind
that figure for one decode query per head, on any K, V, q held on the GPU:

* score KL: KL(p || p_hat), p = softmax of the exact scores q . k * scale over the BF16 tokens, p_hat =
  softmax of the scores the INT2 pool attends with, averaged over query heads;
* output error: sum over heads of ||o_hat - o||^2 / sum of ||o||^2, o exact attention, o_hat the
  pool's decode-attention output.

The pool is filled by oscar_prefill_pool and attended by oscar_decode_attention (the library's CUDA
kernels); the exact attention, the dequantization of the stored history for p_hat and the reductions
are plain float64 tensor arithmetic on the same device (measurement, not part of the decode path).

Variants (rotation R, clip ratio c): naive INT2 (I, 1), Hadamard-only (H . P, 1), clip-only (I, c),
OSCAR (U . H . P with U from the calibration covariances, c); OSCAR's rotation may further carry
Lloyd-Max codebooks calibrated on the same keys and values (the closing comparison with TurboQuant).
"""
from __future__ import annotations

import math

import torch

from bit_rotated_kv_02_gb300 import (HEAD_DIM, PAGE, RECENT, SINK, ROT_COVARIANCE, ROT_HAAR, Pool,
                                     oscar_calib_covariance_k, oscar_calib_covariance_v, oscar_decode_attention,
                                     oscar_lloyd_max_codebook, oscar_make_rotation, oscar_prefill_pool)


def identity_rotation(num_kv_heads: int, device="cuda") -> torch.Tensor:
    return torch.eye(HEAD_DIM, dtype=torch.float32, device=device).expand(num_kv_heads, -1, -1).contiguous()


def hadamard_rotation(num_kv_heads: int, device="cuda") -> torch.Tensor:
    """H . P: the library's rotation with U the Q factor of the identity (U = I)."""
    eye = torch.eye(HEAD_DIM, dtype=torch.float64, device=device)
    R = oscar_make_rotation(eye, ROT_HAAR)[1]
    return R.expand(num_kv_heads, -1, -1).contiguous()


def covariance_rotations(Qc: torch.Tensor, Kc: torch.Tensor, Vc: torch.Tensor, softmax_scale=None):
    """Per KV head R_k, R_v = U . H . P from the calibration covariances: Qc bf16 [T][Hq][d] (query heads
    h*G .. h*G+G-1 belong to KV head h), Kc, Vc bf16 [T][Hkv][d]."""
    Hq, Hkv = Qc.shape[1], Kc.shape[1]
    G = Hq // Hkv
    Rk, Rv = [], []
    for h in range(Hkv):
        Qh = Qc[:, h * G:(h + 1) * G].contiguous()
        Kh, Vh = Kc[:, h].contiguous(), Vc[:, h].contiguous()
        Rk.append(oscar_make_rotation(oscar_calib_covariance_k(Qh), ROT_COVARIANCE)[1])
        Rv.append(oscar_make_rotation(oscar_calib_covariance_v(Qh, Kh, Vh, softmax_scale), ROT_COVARIANCE)[1])
    return torch.stack(Rk), torch.stack(Rv)


def _dequant_history(P: Pool, kvh: int, which: str) -> torch.Tensor:
    """float64 [hist_len][d] rotated history vectors of sequence 0, KV head kvh, in token order."""
    hl = int(P.hist_len[0])
    t = torch.arange(hl, device=P.page_table.device)
    pages, rows = P.page_table[0, t // PAGE].long(), t % PAGE
    codes = getattr(P, "codes_" + which)[pages, kvh, rows]                      # u8 [hl][d/4]
    shifts = torch.arange(4, device=codes.device, dtype=torch.uint8) * 2
    c = ((codes[..., None] >> shifts) & 3).reshape(hl, HEAD_DIM)               # channel 4b+i: byte b, bits 2i
    cb = getattr(P, "codebook_" + which)
    c = c.double() if cb is None else cb[kvh].double()[c.long()]               # level of each code
    scale = getattr(P, "scale_" + which)[pages, kvh, rows].double()            # [hl][d/g]
    zero = getattr(P, "zero_" + which)[pages, kvh, rows].double()
    g = HEAD_DIM // scale.shape[1]
    return c * scale.repeat_interleave(g, 1) + zero.repeat_interleave(g, 1)


def measure(K: torch.Tensor, V: torch.Tensor, q: torch.Tensor, R_k: torch.Tensor, R_v: torch.Tensor, clip_k,
            clip_v, group_size: int = HEAD_DIM, softmax_scale=None, codebook_k=None, codebook_v=None):
    """(mean score KL, relative output error) of one sequence of tokens K, V (bf16 [L][Hkv][d], CUDA)
    stored in an INT2 pool with rotations R_k, R_v (fp32 [Hkv][d][d]), clip ratios clip_k, clip_v
    ([Hkv]) and optional codebooks (fp32 [Hkv][4]), for the queries q (bf16 [Hq][d])."""
    L, Hkv, d = K.shape
    Hq = q.shape[0]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(d) if softmax_scale is None else float(softmax_scale)
    pages = max(1, -(-max(L - SINK - RECENT, 0) // PAGE))
    clip_k = torch.as_tensor(clip_k, dtype=torch.float32).reshape(Hkv)
    clip_v = torch.as_tensor(clip_v, dtype=torch.float32).reshape(Hkv)
    P = Pool(1, Hq, Hkv, group_size, pages, pages, R_k, R_v, clip_k, clip_v, device=K.device, codebook_k=codebook_k,
             codebook_v=codebook_v)
    P.set_page_table(torch.arange(pages, dtype=torch.int32)[None])
    oscar_prefill_pool(P, 0, K.contiguous(), V.contiguous())
    o_hat = oscar_decode_attention(P, q[None].contiguous(), softmax_scale=scale)[0].double()
    if P.err():
        raise RuntimeError(f"pool device error {P.err():#x}")
    ns, hl = int(P.sink_len[0]), int(P.hist_len[0])
    kls, num, den = [], 0.0, 0.0
    for kvh in range(Hkv):
        Kf, Vf = K[:, kvh].double(), V[:, kvh].double()
        hk = _dequant_history(P, kvh, "k")
        Rk64 = P.R_k[kvh].double()
        for h in range(kvh * G, (kvh + 1) * G):
            qh = q[h].double()
            s = Kf @ qh * scale
            p = torch.softmax(s, 0)
            s_hat = torch.cat([Kf[:ns] @ qh, hk @ (qh @ Rk64), Kf[ns + hl:] @ qh]) * scale
            log_p_hat = torch.log_softmax(s_hat, 0)
            m = p > 0
            kls.append(float(torch.sum(p[m] * (torch.log(p[m]) - log_p_hat[m]))))
            o = p @ Vf
            num += float(torch.sum((o_hat[h] - o) ** 2))
            den += float(torch.sum(o ** 2))
    return sum(kls) / len(kls), num / den


def lloyd_max_codebooks(Kc: torch.Tensor, Vc: torch.Tensor, R_k: torch.Tensor, R_v: torch.Tensor, clip: float = 0.9,
                        group_size: int = HEAD_DIM):
    """Per-head Lloyd-Max levels (fp32 [Hkv][4]) of the calibration keys and values under R_k, R_v."""
    c = torch.full((Kc.shape[1],), float(clip), dtype=torch.float32, device=Kc.device)
    return (oscar_lloyd_max_codebook(Kc.contiguous(), R_k, c, group_size),
            oscar_lloyd_max_codebook(Vc.contiguous(), R_v, c, group_size))


def variants(Qc, Kc, Vc, clip: float = 0.9):
    """{name: (R_k, R_v, clip)} of the four variants of Fig. 1 for calibration data Qc, Kc, Vc."""
    Hkv = Kc.shape[1]
    dev = Kc.device
    I, HP = identity_rotation(Hkv, dev), hadamard_rotation(Hkv, dev)
    Rk, Rv = covariance_rotations(Qc, Kc, Vc)
    return {"naive_int2": (I, I, 1.0), "hadamard_only": (HP, HP, 1.0), "clip_only": (I, I, clip),
            "oscar": (Rk, Rv, clip)}

"""Oracle: the BF16 paged KV cache that INT2 decoding is compared against (test infrastructure only).

[Article, "评估结果" (Fig. 5)] and [Abstract]: OSCAR's decode speed-up (up to about 3x at
100k context and batch size 1) is measured against the same serving engine keeping its whole
history in BF16; the gain comes from reading fewer bytes of KV per decoded token.  This module is
that BF16 cache, kept the way a paged serving engine keeps it.

Readings (the pages give no layout for the BF16 cache):
* Every token of a sequence is stored in BF16, in pages of 64 tokens: token t of sequence b sits at
  page page_table[b][t // 64], row t % 64; k_pages and v_pages are [num_pages][Hkv][64][d].
* seq_len[b] tokens are held; appending writes position seq_len[b] and increments it.
* Decode attention is exact softmax attention in float64 over all held tokens, score
  (q . k) * softmax_scale, query head h reading KV head h // (Hq/Hkv); no rotation.
"""
from __future__ import annotations

import numpy as np

from . import attention, quant

PAGE = 64


class BF16Cache:
    def __init__(self, batch, num_q_heads, num_kv_heads, d, num_pages, max_pages):
        self.B, self.Hq, self.Hkv, self.d = batch, num_q_heads, num_kv_heads, d
        self.num_pages, self.max_pages = num_pages, max_pages
        self.k_pages = np.zeros((num_pages, num_kv_heads, PAGE, d), np.uint16)
        self.v_pages = np.zeros_like(self.k_pages)
        self.page_table = np.full((batch, max_pages), -1, np.int32)
        self.seq_len = np.zeros(batch, np.int32)

    def _place(self, b, t):
        """(physical page, row) of token position(s) t of sequence b."""
        t = np.asarray(t)
        return self.page_table[b, t // PAGE], t % PAGE

    def prefill(self, b, K_bits, V_bits):
        """K_bits, V_bits: bf16 [L][Hkv][d] of one sequence; replaces its contents."""
        L = K_bits.shape[0]
        pages, rows = self._place(b, np.arange(L))
        self.k_pages[pages, :, rows] = K_bits
        self.v_pages[pages, :, rows] = V_bits
        self.seq_len[b] = L

    def append(self, k_new, v_new):
        """k_new, v_new: bf16 [B][Hkv][d]: one new token per sequence, at position seq_len[b]."""
        for b in range(self.B):
            page, row = self._place(b, int(self.seq_len[b]))
            self.k_pages[page, :, row] = k_new[b]
            self.v_pages[page, :, row] = v_new[b]
            self.seq_len[b] += 1

    def tokens(self, b, kvh):
        """bf16 bits (K [L][d], V [L][d]) of one (sequence, KV head), in token order."""
        pages, rows = self._place(b, np.arange(int(self.seq_len[b])))
        return self.k_pages[pages, kvh, rows], self.v_pages[pages, kvh, rows]

    def decode(self, q_bits, softmax_scale=None, heads=None, batch=None):
        """float64 out [B][Hq][d] for bf16 queries q_bits [B][Hq][d] (optionally a subset of b / heads)."""
        scale = 1.0 / np.sqrt(self.d) if softmax_scale is None else softmax_scale
        G = self.Hq // self.Hkv
        f = quant.bf16_bits_to_f64
        out = np.full((self.B, self.Hq, self.d), np.nan)
        for b in (range(self.B) if batch is None else batch):
            if self.seq_len[b] == 0:
                out[b] = 0.0
                continue
            cache = {}
            for h in (range(self.Hq) if heads is None else heads):
                kvh = h // G
                if kvh not in cache:
                    K, V = self.tokens(b, kvh)
                    cache[kvh] = (f(K), f(V))
                out[b, h] = attention.softmax_attend(f(q_bits[b, h]), *cache[kvh], scale)
        return out

"""Oracle: the three-segment KV pool and its bookkeeping (test infrastructure only).

[Article, "OSCAR 的设计"]: the runtime keeps a three-segment token pool
"BF16 sink (64 tokens) | INT2 history | BF16 recent (256 tokens)"; a new token
is first written into the recent window; as decoding advances the oldest
recent token is rotated, clipped, quantized, packed and demoted into the INT2
history; the history is paged (compatible with paged KV).

Readings (the pages give no layout):
* Token positions 0..63 of a sequence go to the sink, in order.
* Later tokens go to the recent ring: slot (recent_start + recent_len) % 256.
* Demotion moves the token in slot recent_start to history position hist_len
  (page page_table[b][hist_len // 64], row hist_len % 64), so the history keeps
  token order; then hist_len += 1, recent_start += 1 (mod 256), recent_len -= 1.
* Appending to a full recent window first demotes its oldest token.
* Bulk prefill of L tokens: [0, 64) -> sink, [64, L-256) -> history,
  [L-256, L) -> recent (recent_start = 0); L <= 320 leaves the history empty.
* Layouts (mirroring the device arrays): sink/recent [B][Hkv][64|256][d] bf16,
  history codes [num_pages][Hkv][64][d/4] u8, scale/zero
  [num_pages][Hkv][64][d/g] bf16, page_table [B][max_pages] int32.
"""
from __future__ import annotations

import numpy as np

from . import attention, codebook, quant

PAGE, SINK, RECENT = 64, 64, 256


class Pool:
    def __init__(self, batch, num_q_heads, num_kv_heads, d, group, num_pages, max_pages,
                 R_k32, R_v32, clip_k, clip_v, codebook_k=None, codebook_v=None):
        """codebook_k, codebook_v: float32 [Hkv][4] levels (oracle.codebook), or None for the uniform
        levels (0, 1, 2, 3)."""
        self.B, self.Hq, self.Hkv, self.d, self.g = batch, num_q_heads, num_kv_heads, d, group
        self.ng = d // group
        self.num_pages, self.max_pages = num_pages, max_pages
        self.R_k = np.asarray(R_k32, np.float32).reshape(num_kv_heads, d, d)
        self.R_v = np.asarray(R_v32, np.float32).reshape(num_kv_heads, d, d)
        self.clip_k = np.asarray(clip_k, np.float32).reshape(num_kv_heads)
        self.clip_v = np.asarray(clip_v, np.float32).reshape(num_kv_heads)
        self.cb_k = None if codebook_k is None else np.asarray(codebook_k, np.float32).reshape(num_kv_heads, 4)
        self.cb_v = None if codebook_v is None else np.asarray(codebook_v, np.float32).reshape(num_kv_heads, 4)
        self.sink_k = np.zeros((batch, num_kv_heads, SINK, d), np.uint16)
        self.sink_v = np.zeros_like(self.sink_k)
        self.recent_k = np.zeros((batch, num_kv_heads, RECENT, d), np.uint16)
        self.recent_v = np.zeros_like(self.recent_k)
        self.codes_k = np.zeros((num_pages, num_kv_heads, PAGE, d // 4), np.uint8)
        self.codes_v = np.zeros_like(self.codes_k)
        self.scale_k = np.zeros((num_pages, num_kv_heads, PAGE, self.ng), np.uint16)
        self.zero_k = np.zeros_like(self.scale_k)
        self.scale_v = np.zeros_like(self.scale_k)
        self.zero_v = np.zeros_like(self.scale_k)
        self.page_table = np.full((batch, max_pages), -1, np.int32)
        self.sink_len = np.zeros(batch, np.int32)
        self.hist_len = np.zeros(batch, np.int32)
        self.recent_start = np.zeros(batch, np.int32)
        self.recent_len = np.zeros(batch, np.int32)

    # -- writes ----------------------------------------------------------
    def _store_history(self, b, pos, kvh, k_bits, v_bits):
        page = int(self.page_table[b, pos // PAGE])
        row = pos % PAGE
        pk, sk, zk = self._quantize(k_bits[None, :], self.R_k[kvh], self.clip_k[kvh], self.cb_k, kvh)
        pv, sv, zv = self._quantize(v_bits[None, :], self.R_v[kvh], self.clip_v[kvh], self.cb_v, kvh)
        self.codes_k[page, kvh, row], self.scale_k[page, kvh, row], self.zero_k[page, kvh, row] = pk[0], sk[0], zk[0]
        self.codes_v[page, kvh, row], self.scale_v[page, kvh, row], self.zero_v[page, kvh, row] = pv[0], sv[0], zv[0]

    def _quantize(self, X, R, clip, cb, kvh):
        if cb is None:
            return quant.quantize_vectors_many(X, R, clip, self.g)
        return codebook.quantize_vectors_cb(X, R, clip, self.g, cb[kvh])

    def _dequantize(self, packed, scale, zero, cb, kvh):
        if cb is None:
            return quant.dequantize(packed, scale, zero, self.g)
        return codebook.dequantize_cb(packed, scale, zero, self.g, cb[kvh])

    def prefill(self, b, K_bits, V_bits, heads=None, shared_pages=0):
        """K_bits, V_bits: bf16 [L][Hkv][d] of one sequence; fills its three segments (history of the
        KV heads in `heads` only, when given: each head's history is independent of the others).
        shared_pages: the first history pages are already in place (the page table points at pages
        another sequence with the same prefix filled) and are not written."""
        L = K_bits.shape[0]
        ns = min(L, SINK)
        nr = min(max(L - SINK, 0), RECENT)
        nh = L - ns - nr
        self.sink_k[b, :, :ns] = K_bits[:ns].transpose(1, 0, 2)
        self.sink_v[b, :, :ns] = V_bits[:ns].transpose(1, 0, 2)
        t = np.arange(shared_pages * PAGE, nh)
        pages, rows = self.page_table[b, t // PAGE], t % PAGE
        for kvh in (range(self.Hkv) if heads is None else heads):
            for X, R, clip, cb, codes, scale, zero in (
                    (K_bits, self.R_k, self.clip_k, self.cb_k, self.codes_k, self.scale_k, self.zero_k),
                    (V_bits, self.R_v, self.clip_v, self.cb_v, self.codes_v, self.scale_v, self.zero_v)):
                pc, sc, zc = self._quantize(X[ns + t, kvh], R[kvh], clip[kvh], cb, kvh)
                codes[pages, kvh, rows], scale[pages, kvh, rows], zero[pages, kvh, rows] = pc, sc, zc
        self.recent_k[b, :, :nr] = K_bits[ns + nh:].transpose(1, 0, 2)
        self.recent_v[b, :, :nr] = V_bits[ns + nh:].transpose(1, 0, 2)
        self.sink_len[b], self.hist_len[b], self.recent_start[b], self.recent_len[b] = ns, nh, 0, nr

    def demote(self, mask=None):
        """Demote the oldest recent token of every sequence whose recent window is full, or, when a
        mask is given, of every sequence with mask[b] != 0 and a non-empty recent window."""
        for b in range(self.B):
            want = (self.recent_len[b] == RECENT) if mask is None else (mask[b] != 0 and self.recent_len[b] > 0)
            if not want:
                continue
            slot = int(self.recent_start[b])
            for kvh in range(self.Hkv):
                self._store_history(b, int(self.hist_len[b]), kvh,
                                    self.recent_k[b, kvh, slot], self.recent_v[b, kvh, slot])
            self.hist_len[b] += 1
            self.recent_start[b] = (slot + 1) % RECENT
            self.recent_len[b] -= 1

    def append(self, k_new, v_new):
        """k_new, v_new: bf16 [B][Hkv][d]: one new token per sequence (demoting first where full)."""
        self.demote(None)
        for b in range(self.B):
            if self.sink_len[b] < SINK and self.hist_len[b] == 0 and self.recent_len[b] == 0:
                r = int(self.sink_len[b])
                self.sink_k[b, :, r], self.sink_v[b, :, r] = k_new[b], v_new[b]
                self.sink_len[b] += 1
            else:
                slot = int((self.recent_start[b] + self.recent_len[b]) % RECENT)
                self.recent_k[b, :, slot], self.recent_v[b, :, slot] = k_new[b], v_new[b]
                self.recent_len[b] += 1

    # -- reads -----------------------------------------------------------
    def segments(self, b, kvh):
        """Float64 (sink_k, sink_v, hist_k_rot, hist_v_rot, recent_k, recent_v) of one (sequence, KV head)."""
        f = quant.bf16_bits_to_f64
        ns, nh, rs, nr = int(self.sink_len[b]), int(self.hist_len[b]), int(self.recent_start[b]), int(self.recent_len[b])
        slots = [(rs + i) % RECENT for i in range(nr)]
        t = np.arange(nh)
        pages, rows = self.page_table[b, t // PAGE], t % PAGE
        hk = self._dequantize(self.codes_k[pages, kvh, rows], self.scale_k[pages, kvh, rows],
                              self.zero_k[pages, kvh, rows], self.cb_k, kvh)
        hv = self._dequantize(self.codes_v[pages, kvh, rows], self.scale_v[pages, kvh, rows],
                              self.zero_v[pages, kvh, rows], self.cb_v, kvh)
        return (f(self.sink_k[b, kvh, :ns]), f(self.sink_v[b, kvh, :ns]), hk, hv,
                f(self.recent_k[b, kvh, slots]), f(self.recent_v[b, kvh, slots]))

    def decode(self, q_bits, softmax_scale=None, heads=None, batch=None):
        """float64 out [B][Hq][d] for bf16 queries q_bits [B][Hq][d] (optionally a subset of b / heads)."""
        scale = 1.0 / np.sqrt(self.d) if softmax_scale is None else softmax_scale
        G = self.Hq // self.Hkv
        out = np.full((self.B, self.Hq, self.d), np.nan)
        for b in (range(self.B) if batch is None else batch):
            cache = {}
            for h in (range(self.Hq) if heads is None else heads):
                kvh = h // G
                if kvh not in cache:
                    cache[kvh] = self.segments(b, kvh)
                sk, sv, hk, hv, rk, rv = cache[kvh]
                out[b, h] = attention.decode_one_head(quant.bf16_bits_to_f64(q_bits[b, h]), sk, sv, hk, hv,
                                                      rk, rv, self.R_k[kvh], self.R_v[kvh], scale)
        return out

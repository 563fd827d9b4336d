"""GPU parity: the BF16 paged KV cache (the baseline INT2 decoding is compared against,
"超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "评估结果", Fig. 5) against its
float64 oracle.

Placement (prefill, append) is compared byte for byte; attention within max-abs 2e-3 and relative L2
1e-3 of exact float64 attention.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import bit_rotated_kv_02_gb300 as ok
import synth
from oracle import bf16_cache as obc
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _setup(lens, Hq, Hkv, seed, extra_pages=1, fill=None):
    """(oracle cache, device cache, q, outlier channels) with the same shuffled page tables and tokens.
    fill: a bf16 bit pattern written over every page before the prefill (what a reused page holds)."""
    B = len(lens)
    max_pages = max((L + 63) // 64 for L in lens) + extra_pages
    pt, num_pages = synth.page_tables(seed, [max_pages] * B, max_pages)
    O = obc.BF16Cache(B, Hq, Hkv, 128, num_pages, max_pages)
    O.page_table[:] = pt
    P = ok.BF16Cache(B, Hq, Hkv, num_pages, max_pages)
    P.set_page_table(pt)
    if fill is not None:
        P.k_pages.view(torch.int16).fill_(fill)
        P.v_pages.view(torch.int16).fill_(fill)
        O.k_pages[:] = np.uint16(fill & 0xffff)
        O.v_pages[:] = np.uint16(fill & 0xffff)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for b, L in enumerate(lens):
        K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
        V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
        O.prefill(b, K, V)
        ok.oscar_bf16_prefill(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    q = synth.outlier_q(seed + 7, B, Hq, Hkv, 128, ch)
    torch.cuda.synchronize()
    return O, P, q, ch


def _assert_cache_equal(O, P):
    assert np.array_equal(O.k_pages, helpers.bits_of(P.k_pages))
    assert np.array_equal(O.v_pages, helpers.bits_of(P.v_pages))
    assert np.array_equal(O.seq_len, P.seq_len.cpu().numpy())


@pytest.mark.parametrize("lens,Hq,Hkv", [
    ([1000], 8, 2),                    # GQA 4, a partial last page
    ([1, 64, 777], 8, 1),              # GQA 8, one-token and exact-page sequences
    ([65, 4000], 2, 2),                # GQA 1
    ([0, 130, 2000, 63], 4, 2),        # GQA 2, an empty sequence
])
def test_decode_matches_oracle(lens, Hq, Hkv):
    O, P, q, _ = _setup(lens, Hq, Hkv, 700 + sum(lens) % 97)
    _assert_cache_equal(O, P)
    out = ok.oscar_bf16_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    assert P.err() == 0


def test_rows_past_the_sequence_end_are_ignored():
    """Pages filled with NaN before the prefill: the rows past seq_len in each last page must not reach
    the result (their scores are masked and their value rows zeroed before the P.V products)."""
    O, P, q, _ = _setup([100, 1, 191], 8, 2, 720, fill=0x7fc0)
    out = ok.oscar_bf16_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))


def test_decode_step_equals_append_then_decode():
    seed, Hq, Hkv = 730, 8, 2
    O, P, q, ch = _setup([60, 1000], Hq, Hkv, seed, extra_pages=2)
    P2 = ok.BF16Cache(2, Hq, Hkv, P.num_pages, P.max_pages)
    P2.set_page_table(O.page_table)
    for name in ("k_pages", "v_pages", "seq_len"):
        getattr(P2, name).copy_(getattr(P, name))
    for t in range(70):   # the first sequence crosses two page boundaries
        kn = synth.outlier_kv(seed + 900 + t, 2, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 1900 + t, 2, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 2900 + t, 2, Hq, Hkv, 128, ch)
        O.append(kn, vn)
        a = ok.oscar_bf16_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        ok.oscar_bf16_append_kv(P2, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn))
        b = ok.oscar_bf16_decode_attention(P2, helpers.to_dev_bf16(qt))
        assert torch.equal(a, b)
        if t % 23 == 0 or t == 69:
            helpers.assert_attention_close(a.cpu().numpy(), O.decode(qt))
    torch.cuda.synchronize()
    _assert_cache_equal(O, P)
    _assert_cache_equal(O, P2)
    assert P.err() == 0 and P2.err() == 0


def test_full_size_100k_context():
    """The 100k-context, 32 query / 8 KV head layer the INT2 headline is quoted on, every head checked."""
    L, Hq, Hkv = 100_000, 32, 8
    O, P, q, _ = _setup([L], Hq, Hkv, 740)
    out = ok.oscar_bf16_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    assert P.err() == 0


def test_device_errors_are_flagged_not_faulted():
    O, P, q, ch = _setup([64], 4, 1, 750, extra_pages=0)
    kn = helpers.to_dev_bf16(synth.outlier_kv(751, 1, 1, 128, ch))
    ok.oscar_bf16_append_kv(P, kn, kn)   # the one page is full: no room for token 64
    torch.cuda.synchronize()
    assert P.err() & ok.DEVERR_HISTORY_FULL and int(P.seq_len[0]) == 64
    P.err_word.zero_()
    P.page_table[0, 0] = P.num_pages + 5
    out = ok.oscar_bf16_decode_attention(P, helpers.to_dev_bf16(q))
    torch.cuda.synchronize()
    assert P.err() & ok.DEVERR_PAGE_INDEX
    assert torch.isfinite(out).all()

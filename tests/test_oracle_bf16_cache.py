"""Pins for oracle.bf16_cache: the BF16 paged cache that INT2 decoding is compared against
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "评估结果", Fig. 5; the OSCAR
arXiv listing, Abstract: batch-1 decoding up to 3x faster than BF16).

The cache's placement is pinned by round trips and by equality with a contiguous sequence; its
attention by torch's own scaled-dot-product attention and by the three-segment pool oracle, which
computes the same thing through different code when no token is quantized.
"""
import numpy as np
import pytest
import torch

from oracle import bf16_cache as obc
from oracle import pool as opool
from oracle import quant
from oracle import rotation as rot
import synth


def _cache(B, Hq, Hkv, lens, seed, extra=1):
    max_pages = max((L + 63) // 64 for L in lens) + extra
    pt, num_pages = synth.page_tables(seed, [max_pages] * B, max_pages)
    C = obc.BF16Cache(B, Hq, Hkv, 128, num_pages, max_pages)
    C.page_table[:] = pt
    return C


def _seq(seed, L, Hkv):
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    return synth.outlier_kv(seed + 1, L, Hkv, 128, ch), synth.outlier_kv(seed + 2, L, Hkv, 128, ch), ch


@pytest.mark.parametrize("L", [1, 63, 64, 65, 200])
def test_prefill_round_trip_on_shuffled_pages(L):
    C = _cache(2, 4, 2, [L, L], seed=3)
    K, V, _ = _seq(5, L, 2)
    C.prefill(1, K, V)
    assert C.seq_len[1] == L and C.seq_len[0] == 0
    for kvh in range(2):
        k, v = C.tokens(1, kvh)
        assert np.array_equal(k, K[:, kvh]) and np.array_equal(v, V[:, kvh])
    # every written row is where the page table says, and nothing else was written
    touched = np.zeros(C.num_pages, bool)
    touched[C.page_table[1, :(L + 63) // 64]] = True
    assert not C.k_pages[~touched].any()


def test_append_equals_prefill_of_longer_sequence():
    L, n = 60, 70   # crosses two page boundaries
    K, V, _ = _seq(7, L + n, 2)
    A = _cache(1, 4, 2, [L + n], seed=8)
    A.prefill(0, K[:L], V[:L])
    for t in range(L, L + n):
        A.append(K[t][None], V[t][None])
    B = _cache(1, 4, 2, [L + n], seed=8)
    B.prefill(0, K, V)
    assert A.seq_len[0] == B.seq_len[0] == L + n
    assert np.array_equal(A.k_pages, B.k_pages) and np.array_equal(A.v_pages, B.v_pages)


def test_decode_matches_torch_sdpa():
    """Against torch's scaled_dot_product_attention in float64 on the contiguous sequences (GQA 4)."""
    lens = [130, 64, 1]
    B, Hq, Hkv = 3, 8, 2
    C = _cache(B, Hq, Hkv, lens, seed=11)
    seqs = []
    for b, L in enumerate(lens):
        K, V, ch = _seq(20 + b, L, Hkv)
        C.prefill(b, K, V)
        seqs.append((K, V, ch))
    q = np.concatenate([synth.outlier_q(30 + b, 1, Hq, Hkv, 128, seqs[b][2]) for b in range(B)])
    scale = 0.0625
    out = C.decode(q, scale)
    f = quant.bf16_bits_to_f64
    for b, (K, V, _) in enumerate(seqs):
        qt = torch.from_numpy(f(q[b])).view(1, Hq, 1, 128)
        kt = torch.from_numpy(f(K)).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)[None]
        vt = torch.from_numpy(f(V)).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("L", [1, 64, 200, 320])
def test_decode_equals_three_segment_pool_without_history(L):
    """Up to 320 tokens the OSCAR pool quantizes nothing (sink + recent only): both oracles agree."""
    Hq, Hkv = 8, 2
    K, V, ch = _seq(40, L, Hkv)
    q = synth.outlier_q(41, 1, Hq, Hkv, 128, ch)
    C = _cache(1, Hq, Hkv, [L], seed=42)
    C.prefill(0, K, V)
    R = np.stack([rot.to_f32(rot.rotation_from_gaussian(synth.gaussian_matrix(43 + h, 128))) for h in range(Hkv)])
    P = opool.Pool(1, Hq, Hkv, 128, 128, 4, 4, R, R, [0.9] * Hkv, [0.9] * Hkv)
    P.prefill(0, K, V)
    assert P.hist_len[0] == 0
    np.testing.assert_allclose(C.decode(q), P.decode(q), rtol=0, atol=1e-12)


def test_page_placement_does_not_change_the_result():
    L = 333
    K, V, ch = _seq(50, L, 2)
    q = synth.outlier_q(51, 1, 8, 2, 128, ch)
    A = _cache(1, 8, 2, [L], seed=52)
    B = _cache(1, 8, 2, [L], seed=53)
    assert not np.array_equal(A.page_table, B.page_table)
    A.prefill(0, K, V)
    B.prefill(0, K, V)
    assert np.array_equal(A.decode(q), B.decode(q))


def test_mismatched_value_pages_would_fail():
    """A planted mistake (values read through a shifted page table) moves the result far outside the
    attention tolerance, so the comparison with a contiguous sequence can see page-placement bugs."""
    L = 256
    K, V, ch = _seq(60, L, 1)
    q = synth.outlier_q(61, 1, 4, 1, 128, ch)
    C = _cache(1, 4, 1, [L], seed=62)
    C.prefill(0, K, V)
    good = C.decode(q)
    pages, rows = C._place(0, np.arange(L))
    bad_v = C.v_pages[np.roll(pages, 64), 0, rows]   # value rows of another page
    f = quant.bf16_bits_to_f64
    from oracle import attention
    bad = attention.softmax_attend(f(q[0, 0]), f(C.tokens(0, 0)[0]), f(bad_v), 1 / np.sqrt(128))
    assert np.abs(bad - good[0, 0]).max() > 1e-2

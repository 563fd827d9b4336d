"""GPU parity: prefill, demotion and append bookkeeping of the three-segment pool, byte for byte.

New tokens enter the BF16 recent window; the oldest recent token is rotated, clipped, quantized,
packed and demoted into the paged INT2 history ("超越TurboQuant！OSCAR：面向真实服务的2-bit KV
Cache量化", section "OSCAR 的设计").
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import bit_rotated_kv_02_gb300 as ok
import synth
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _kv(seed, L, Hkv):
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    return synth.outlier_kv(seed + 1, L, Hkv, 128, ch), synth.outlier_kv(seed + 2, L, Hkv, 128, ch)


@pytest.mark.parametrize("g", [32, 128])
def test_prefill_lengths(g):
    lens = [1, 63, 64, 200, 320, 321, 385, 1100]
    B, Hkv = len(lens), 2
    pages = [max(0, -(-(L - 320) // 64)) for L in lens]
    O, P = helpers.make_pools(B, 8, Hkv, g, pages, 31 + g)
    for b, L in enumerate(lens):
        K, V = _kv(40 + b, L, Hkv)
        O.prefill(b, K, V)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0


def test_append_demote_sequence_crosses_pages_and_wraps():
    B, Hkv, steps = 2, 2, 150
    lens = [330, 700]
    O, P = helpers.make_pools(B, 8, Hkv, 64, [12, 12], 77)
    seqs = []
    for b, L in enumerate(lens):
        K, V = _kv(80 + b, L + steps, Hkv)
        seqs.append((K, V))
        O.prefill(b, K[:L], V[:L])
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K[:L]), helpers.to_dev_bf16(V[:L]))
    for t in range(steps):
        kn = np.stack([seqs[b][0][lens[b] + t] for b in range(B)])
        vn = np.stack([seqs[b][1][lens[b] + t] for b in range(B)])
        O.append(kn, vn)
        ok.oscar_append_kv(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn))
        if t in (0, 63, 149):
            torch.cuda.synchronize()
            helpers.assert_pools_equal(O, P)
    assert P.err() == 0


def test_append_from_empty_fills_sink_then_recent_then_history():
    B, Hkv, n = 1, 2, 64 + 256 + 70
    O, P = helpers.make_pools(B, 4, Hkv, 128, [2], 91)
    K, V = _kv(92, n, Hkv)
    for t in range(n):
        O.append(K[t][None], V[t][None])
        ok.oscar_append_kv(P, helpers.to_dev_bf16(K[t][None]), helpers.to_dev_bf16(V[t][None]))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    c = P.counters()
    assert (c["sink_len"][0], c["hist_len"][0], c["recent_len"][0]) == (64, 70, 256)


def test_masked_demote():
    B, Hkv = 3, 1
    O, P = helpers.make_pools(B, 2, Hkv, 128, [3, 3, 3], 95)
    for b, L in enumerate([400, 300, 64]):
        K, V = _kv(96 + b, L, Hkv)
        O.prefill(b, K, V)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    mask = np.array([1, 1, 1], np.int32)
    for _ in range(3):
        O.demote(mask)
        ok.oscar_demote(P, torch.from_numpy(mask).cuda())
    O.demote(None)
    ok.oscar_demote(P)
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)


def test_bad_page_entry_is_flagged_and_sequence_left_unchanged():
    """A page-table entry outside the pool: the kernel's bounds check skips the write and sets a flag."""
    B, Hkv = 2, 2
    O, P = helpers.make_pools(B, 4, Hkv, 128, [2, 2], 99, extra_pages=1)
    for b in range(B):
        K, V = _kv(100 + b, 320 + 128, Hkv)      # history exactly fills 2 pages
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    pt = P.page_table.cpu().numpy()
    pt[0, 2] = P.num_pages + 5                   # the page the next demotion of sequence 0 needs
    P.set_page_table(pt)
    before = P.counters()
    kn = helpers.to_dev_bf16(_kv(103, 1, Hkv)[0].repeat(B, 0))
    ok.oscar_append_kv(P, kn, kn)
    torch.cuda.synchronize()
    after = P.counters()
    assert P.err() & ok.DEVERR_PAGE_INDEX
    for k in after:
        assert after[k][0] == before[k][0]       # sequence 0 untouched
    assert after["hist_len"][1] == before["hist_len"][1] + 1


def test_history_full_is_flagged():
    O, P = helpers.make_pools(1, 2, 1, 128, [1], 105)
    K, V = _kv(106, 320 + 64, 1)
    ok.oscar_prefill_pool(P, 0, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    kn = helpers.to_dev_bf16(_kv(107, 1, 1)[0])
    ok.oscar_append_kv(P, kn, kn)
    torch.cuda.synchronize()
    assert P.err() & ok.DEVERR_HISTORY_FULL
    assert P.counters()["hist_len"][0] == 64

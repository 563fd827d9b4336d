"""GPU: shared-prefix history pages (the paged, prefix-cache-compatible history of "OSCAR: Offline
Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract, and
"超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", sections "OSCAR 的设计" and "评估结果" Fig. 6).

Sequences whose prompts start with the same tokens point their page tables at the same physical
history pages, written once.  The pool bytes must equal the oracle's, the attention must match the
oracle, and it must equal bit for bit the attention of a pool where every sequence holds private
copies of the same pages; decode steps must never write a shared page.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import bit_rotated_kv_02_gb300 as ok
import synth
from oracle import pool as opool
from tests import helpers

pytestmark = pytest.mark.gpu

HQ, HKV = 8, 2


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def _tokens(seed, lens, shared_tokens):
    """K, V per sequence: the first shared_tokens[b] tokens equal sequence 0's."""
    ch = synth.outlier_channels(seed, HKV, 128, 4)
    K0 = synth.outlier_kv(seed + 1, lens[0], HKV, 128, ch)
    V0 = synth.outlier_kv(seed + 2, lens[0], HKV, 128, ch)
    out = []
    for b, L in enumerate(lens):
        if b == 0:
            out.append((K0, V0))
            continue
        K = synth.outlier_kv(seed + 10 + b, L, HKV, 128, ch)
        V = synth.outlier_kv(seed + 20 + b, L, HKV, 128, ch)
        n = shared_tokens[b]
        K[:n], V[:n] = K0[:n], V0[:n]
        out.append((K, V))
    return out, ch


def _pools(seed, lens, share, extra_pages=2):
    """share[b] = number of history pages sequence b shares with sequence 0 (share[0] = 0).
    Returns (oracle, device pool with shared pages, device pool with private copies, q, ch, page tables)."""
    B = len(lens)
    hist = [max(0, L - 320) for L in lens]
    own = [-(-h // 64) + extra_pages for h in hist]
    max_pages = max(own)
    perm = synth.shuffled_pages(seed, sum(own))
    pt_priv = np.full((B, max_pages), -1, np.int32)
    o = 0
    for b in range(B):
        pt_priv[b, :own[b]] = perm[o:o + own[b]]
        o += own[b]
    pt_shared = pt_priv.copy()
    for b in range(1, B):
        pt_shared[b, :share[b]] = pt_priv[0, :share[b]]
    toks, ch = _tokens(seed, lens, [64 + 64 * s for s in share])
    Rk, Rv = helpers.oracle_rotations(seed, HKV), helpers.oracle_rotations(seed + 1000, HKV)
    clip = np.full(HKV, 0.9, np.float32)
    O = opool.Pool(B, HQ, HKV, 128, 128, sum(own), max_pages, Rk, Rv, clip, clip)
    O.page_table[:] = pt_shared
    dev = []
    for pt in (pt_shared, pt_priv):
        P = ok.Pool(B, HQ, HKV, 128, sum(own), max_pages, torch.from_numpy(Rk), torch.from_numpy(Rv),
                    torch.from_numpy(clip), torch.from_numpy(clip))
        P.set_page_table(pt)
        dev.append(P)
    for b, (K, V) in enumerate(toks):
        O.prefill(b, K, V, shared_pages=share[b])
        kd, vd = helpers.to_dev_bf16(K), helpers.to_dev_bf16(V)
        ok.oscar_prefill_pool_shared(dev[0], b, kd, vd, share[b])
        ok.oscar_prefill_pool(dev[1], b, kd, vd)
    q = synth.outlier_q(seed + 7, B, HQ, HKV, 128, ch)
    torch.cuda.synchronize()
    return O, dev[0], dev[1], q, ch, pt_shared


def _shared_page_bytes(P, pages):
    return {n: helpers.device_array(P, n)[pages].copy() for n in ("codes_k", "codes_v", "scale_k", "zero_k",
                                                                  "scale_v", "zero_v")}


@pytest.mark.parametrize("lens,share", [
    ([2000, 2000, 1500], [0, 26, 10]),      # whole prefixes and a partial one
    ([1000, 4000], [0, 10]),                # the sharer is longer than the owner's history
])
def test_shared_pages_match_oracle_and_private_copies(lens, share):
    O, P, Ppriv, q, _, _ = _pools(800 + sum(share), lens, share)
    helpers.assert_pools_equal(O, P)
    qd = helpers.to_dev_bf16(q)
    out = ok.oscar_decode_attention(P, qd)
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    out_priv = ok.oscar_decode_attention(Ppriv, qd)
    assert torch.equal(out, out_priv)
    assert P.err() == 0 and Ppriv.err() == 0


def test_decode_steps_never_write_shared_pages():
    lens, share = [1700, 1700], [0, 20]
    O, P, _, q, ch, pt = _pools(830, lens, share)
    shared = pt[0, :share[1]]
    before = _shared_page_bytes(P, shared)
    for t in range(90):   # both histories grow by 90 tokens (each crosses a page boundary)
        kn = synth.outlier_kv(831 + t, 2, HKV, 128, ch)
        vn = synth.outlier_kv(931 + t, 2, HKV, 128, ch)
        qt = synth.outlier_q(1031 + t, 2, HQ, HKV, 128, ch)
        O.append(kn, vn)
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        if t % 30 == 29:
            helpers.assert_attention_close(out.cpu().numpy(), O.decode(qt))
    torch.cuda.synchronize()
    after = _shared_page_bytes(P, shared)
    for n in before:
        assert np.array_equal(before[n], after[n]), n
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0

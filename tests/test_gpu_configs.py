"""GPU parity at the workload sizes of the batch sweep and the long-context mixed batch, batches above
32 sequences, and a long run of consecutive decode steps.

Paged INT2 history, demotion of the oldest window token ahead of every step's attention, split-K decode
attention with an LSE merge ("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的
设计"; "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract).
Bar: pool bytes identical to the oracle's; attention within max-abs 2e-3 and relative L2 1e-3 of float64
attention over the oracle's pool.  At full sizes the oracle holds a few sampled sequences (and, for the
mixed batch, sampled KV heads); the other sequences load the kernels and exercise the indexing.
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


def _pages(L, extra_tokens=0):
    return max(0, -(-(max(L - 320, 0) + extra_tokens) // 64))


def _check_sampled_attention(O, out, q, sampled, heads=None):
    got = out.cpu().numpy()[sampled]
    ref = O.decode(q[sampled], heads=heads)
    if heads is not None:
        got, ref = got[:, heads], ref[:, heads]
    return helpers.assert_attention_close(got, ref)


@pytest.mark.parametrize("B", [33, 64])
def test_batches_above_32_uneven_contexts(B):
    """Qwen3-8B head shapes with more than 32 sequences (the attention kernel's range location and the
    merge's partial location scan the sequences in chunks of 32): uneven contexts, some without history,
    some ending on a page boundary; attention, then decode steps that cross page boundaries."""
    seed, Hq, Hkv = 900 + B, 32, 8
    g = synth.rng(seed)
    lens = [int(x) for x in g.integers(1, 2600, size=B)]
    lens[0], lens[1], lens[2], lens[B - 1] = 5, 320, 320 + 64 * 7, 321
    steps = 70
    O, P = helpers.make_pools(B, Hq, Hkv, 128, [_pages(L, steps) for L in lens], seed)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for b, L in enumerate(lens):
        K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
        V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
        O.prefill(b, K, V)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    q = synth.outlier_q(seed + 7, B, Hq, Hkv, 128, ch)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    for t in range(steps):
        kn = synth.outlier_kv(seed + 2000 + t, B, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, B, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, B, Hq, Hkv, 128, ch)
        O.append(kn, vn)
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        if t in (0, 33, steps - 1):
            helpers.assert_attention_close(out.cpu().numpy(), O.decode(qt))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0 and int(P.sync.abs().sum()) == 0


def test_one_long_sequence_among_many_short():
    """40 sequences, one with a 60k-token context and 39 short ones: the merge grid then merges four query
    heads per CTA, and the long sequence's segments hold more partials (about 52) than one staging round
    of the wide merge (48), so the merge stages them head by head in two rounds; attention, then decode
    steps."""
    seed, B, Hq, Hkv = 960, 40, 32, 8
    g = synth.rng(seed)
    lens = [int(x) for x in g.integers(300, 400, size=B)]
    lens[5] = 60_000
    steps = 3
    O, P = helpers.make_pools(B, Hq, Hkv, 128, [_pages(L, steps) for L in lens], seed)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for b, L in enumerate(lens):
        K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
        V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
        O.prefill(b, K, V)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    torch.cuda.synchronize()
    q = synth.outlier_q(seed + 7, B, Hq, Hkv, 128, ch)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    for t in range(steps):
        kn = synth.outlier_kv(seed + 2000 + t, B, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, B, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, B, Hq, Hkv, 128, ch)
        O.append(kn, vn)
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        helpers.assert_attention_close(out.cpu().numpy(), O.decode(qt))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0 and int(P.sync.abs().sum()) == 0


def _fill_sampled(O, P, lens, sampled, seed, ch, Hkv, heads=None):
    """Prefill: sampled sequences from seeded host draws (both pools), the rest from GPU draws."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    j = {b: i for i, b in enumerate(sampled)}
    for b, L in enumerate(lens):
        if b in j:
            K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
            V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
            O.prefill(j[b], K, V, heads=heads)
            ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
            del K, V
        else:
            ok.oscar_prefill_pool(P, b, helpers.gpu_outlier_kv(gen, L, Hkv, ch),
                                  helpers.gpu_outlier_kv(gen, L, Hkv, ch))
    torch.cuda.synchronize()


@pytest.mark.parametrize("B", [64, 256])
def test_batch_sweep_shape_32k_sampled(B):
    """The batch sweep's shapes: B sequences x 32,768 tokens (64 sink + 32,448 INT2 history on random page
    tables + 256 recent), Qwen3-8B layer (32 query / 8 KV heads), group 128, clip 0.9; three decode steps
    (append + demotion + attention).  Three sampled sequences are compared in full (all KV heads, pool
    bytes and attention of all 32 query heads)."""
    seed, Hq, Hkv, L, steps = 1100 + B, 32, 8, 32_768, 3
    lens = [L] * B
    sampled = [0, B // 2 - 1, B - 1]
    O, P, pt = helpers.make_sampled_pools(B, Hq, Hkv, 128, [_pages(L, steps) for L in lens], sampled, seed)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    _fill_sampled(O, P, lens, sampled, seed, ch, Hkv)
    helpers.assert_sampled_pools_equal(O, P, pt, sampled)
    for t in range(steps):
        kn = synth.outlier_kv(seed + 2000 + t, B, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, B, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, B, Hq, Hkv, 128, ch)
        O.append(kn[sampled], vn[sampled])
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        _check_sampled_attention(O, out, qt, sampled)
    torch.cuda.synchronize()
    helpers.assert_sampled_pools_equal(O, P, pt, sampled)
    assert P.err() == 0 and int(P.sync.abs().sum()) == 0


def test_mixed_long_context_batch_shape_sampled():
    """The long-context mixed batch: 8 sequences with lengths drawn in [8k, 128k], Qwen3-32B heads (64
    query / 8 KV heads), group 32 along head_dim, per-(head, K/V) clip ratios in [0.8, 1.0]; attention, then
    two decode steps.  The shortest, the longest and one middle sequence are compared on KV heads 0 and 5
    (pool bytes and their 16 query heads)."""
    wl = synth.mixed_long()
    Hq, Hkv, B, g = wl.num_q_heads, wl.num_kv_heads, wl.batch, wl.group_size
    lens = list(wl.context)
    order = np.argsort(lens)
    sampled = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2])})
    heads = [0, 5]
    qheads = [h for kv in heads for h in range(kv * wl.group, (kv + 1) * wl.group)]
    clip_k = synth.clip_ratios(wl.seed, Hkv, *wl.clip)
    clip_v = synth.clip_ratios(wl.seed + 1, Hkv, *wl.clip)
    steps = 2
    O, P, pt = helpers.make_sampled_pools(B, Hq, Hkv, g, [_pages(L, steps) for L in lens], sampled, wl.seed,
                                          clip_k, clip_v)
    ch = synth.outlier_channels(wl.seed, Hkv, 128, wl.n_outliers)
    _fill_sampled(O, P, lens, sampled, wl.seed, ch, Hkv, heads=heads)
    helpers.assert_sampled_pools_equal(O, P, pt, sampled, heads=heads)
    q = synth.outlier_q(wl.seed + 7, B, Hq, Hkv, 128, ch)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    _check_sampled_attention(O, out, q, sampled, heads=qheads)
    for t in range(steps):
        kn = synth.outlier_kv(wl.seed + 2000 + t, B, Hkv, 128, ch)
        vn = synth.outlier_kv(wl.seed + 3000 + t, B, Hkv, 128, ch)
        qt = synth.outlier_q(wl.seed + 4000 + t, B, Hq, Hkv, 128, ch)
        O.append(kn[sampled], vn[sampled])
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        _check_sampled_attention(O, out, qt, sampled, heads=qheads)
    torch.cuda.synchronize()
    helpers.assert_sampled_pools_equal(O, P, pt, sampled, heads=heads)
    assert P.err() == 0


def test_one_thousand_consecutive_decode_steps():
    """1,000 decode steps (append + demotion + attention) on the batch sweep's shapes at batch 16 x 32k:
    every 100 steps two sampled sequences are compared with the oracle, which has appended every token
    of theirs in turn (pool bytes of all KV heads, attention of all 32 query heads)."""
    seed, B, Hq, Hkv, L, steps = 1300, 16, 32, 8, 32_768, 1000
    lens = [L] * B
    sampled = [0, 9]
    O, P, pt = helpers.make_sampled_pools(B, Hq, Hkv, 128, [_pages(L, steps) for L in lens], sampled, seed)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    _fill_sampled(O, P, lens, sampled, seed, ch, Hkv)
    ws = torch.empty(ok.oscar_decode_workspace_size(P), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    checks = 0
    for t in range(steps):
        kn = synth.outlier_kv(seed + 20000 + t, B, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 30000 + t, B, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 40000 + t, B, Hq, Hkv, 128, ch)
        O.append(kn[sampled], vn[sampled])
        ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt),
                             out=out, ws=ws)
        if t % 100 == 99:
            torch.cuda.synchronize()
            _check_sampled_attention(O, out, qt, sampled)
            helpers.assert_sampled_pools_equal(O, P, pt, sampled)
            checks += 1
    assert checks == 10
    assert P.err() == 0 and int(P.sync.abs().sum()) == 0

"""GPU parity: decode attention over the three-segment pool against the float64 oracle.

INT2 history unpacked and dequantized with scale/zero point, BF16 sink/recent, online softmax merge
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计"; "OSCAR: Offline
Spectral Covariance-Aware Rotation for 2-bit KV Cache Quantization", Abstract).
Bar: max-abs error <= 2e-3 and relative L2 error <= 1e-3 against exact float64 attention over the
oracle's own pool (whose bytes must first equal the GPU pool's).
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


def _setup(lens, Hq, Hkv, g, seed, clip=None, heads=None, check_pool=True, extra_pages=0, rotation="haar"):
    B = len(lens)
    pages = [max(0, -(-(L - 320) // 64)) for L in lens]
    clip_k, clip_v = (None, None) if clip is None else clip
    O, P = helpers.make_pools(B, Hq, Hkv, g, pages, seed, clip_k, clip_v, extra_pages=extra_pages, rotation=rotation)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for b, L in enumerate(lens):
        K = synth.outlier_kv(seed + 10 + b, L, Hkv, 128, ch)
        V = synth.outlier_kv(seed + 500 + b, L, Hkv, 128, ch)
        O.prefill(b, K, V, heads=heads)
        ok.oscar_prefill_pool(P, b, helpers.to_dev_bf16(K), helpers.to_dev_bf16(V))
    q = synth.outlier_q(seed + 7, B, Hq, Hkv, 128, ch)
    torch.cuda.synchronize()
    if check_pool:
        helpers.assert_pools_equal(O, P, heads=heads)
    return O, P, q


def test_tiny_workload():
    """Batch 1, 8 query / 2 KV heads, context 1024 = 64 sink + 704 history + 256 recent, group 128, clip 0.9."""
    wl = synth.TINY
    O, P, q = _setup(list(wl.context), wl.num_q_heads, wl.num_kv_heads, wl.group_size, wl.seed)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    assert P.err() == 0


def test_edge_lengths():
    lens = [1, 40, 64, 65, 300, 320, 321, 384, 385, 449, 2000]
    O, P, q = _setup(lens, 8, 2, 128, 300)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))


@pytest.mark.parametrize("G,g", [(4, 32), (8, 64), (1, 32)])
def test_edge_lengths_group_sizes(G, g):
    """Groups of 32 and 64 (the tensor-memory kernel): empty histories, one history token, tiles whose
    second page is empty or partial, ragged last pages, sequences that end a CTA's range mid-page."""
    lens = [1, 64, 321, 384, 385, 449, 513, 577, 1000, 2000, 3333]
    O, P, q = _setup(lens, 2 * G, 2, g, 700 + 10 * G + g)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    assert P.err() == 0


@pytest.mark.parametrize("G,g", [(1, 32), (2, 64), (8, 32), (4, 64)])
def test_gqa_ratios_and_group_sizes(G, g):
    Hkv = 2
    clip = (np.array([0.8, 0.95], np.float32), np.array([0.9, 0.85], np.float32))
    O, P, q = _setup([900, 1500], G * Hkv, Hkv, g, 400 + G * 10 + g, clip=clip)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))


@pytest.mark.parametrize("splits", [1, 2, 5, 64, 0])
def test_split_counts(splits):
    O, P, q = _setup([3000, 700], 8, 2, 128, 500)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q), num_splits=splits)
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))


def test_decode_after_appends():
    seed, Hkv, Hq = 600, 2, 8
    O, P, q = _setup([340, 1000], Hq, Hkv, 128, seed, extra_pages=2)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for t in range(70):
        kn = synth.outlier_kv(seed + 2000 + t, 2, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, 2, Hkv, 128, ch)
        O.append(kn, vn)
        ok.oscar_append_kv(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn))
        if t % 23 == 0:
            out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
            helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)


@pytest.mark.parametrize("G,g", [(4, 128), (8, 128), (2, 32), (8, 32), (1, 64)])
def test_decode_step_matches_oracle_and_separate_calls(G, g):
    """oscar_decode_step gives the oracle's result at every step and, up to float32 rounding, what
    oscar_append_kv followed by oscar_decode_attention gives (for group 128 the step's attention runs
    alongside its demotion and takes the demoted token as a partial of its own); both leave the pool
    byte for byte as the oracle does."""
    seed, Hkv = 640 + G + g, 2
    Hq = G * Hkv
    O, P, q = _setup([330, 1100], Hq, Hkv, g, seed, extra_pages=2)
    _, P2, _ = _setup([330, 1100], Hq, Hkv, g, seed, extra_pages=2)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for t in range(20):
        kn = synth.outlier_kv(seed + 2000 + t, 2, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, 2, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, 2, Hq, Hkv, 128, ch)
        O.append(kn, vn)
        kd, vd, qd = helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt)
        out = ok.oscar_decode_step(P, kd, vd, qd)
        ok.oscar_append_kv(P2, kd, vd)
        out2 = ok.oscar_decode_attention(P2, qd)
        torch.testing.assert_close(out, out2, rtol=1e-5, atol=1e-4)
        if t % 7 == 0 or t == 19:
            helpers.assert_attention_close(out.cpu().numpy(), O.decode(qt))
            helpers.assert_pools_equal(O, P)
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    helpers.assert_pools_equal(O, P2)
    assert P.err() == 0 and P2.err() == 0


@pytest.mark.parametrize("g", [128, 32])
def test_decode_step_with_pinned_host_inputs_and_output(g):
    """q, k_new, v_new and out in page-locked host memory: the step's kernels read and write them in place over
    the host link (no separate copy) and give what the call with device buffers gives, pool bytes included; a
    pageable host buffer is refused on the host before any launch."""
    import ctypes as C
    seed, Hkv, Hq = 660 + g, 2, 8
    O, P, q = _setup([330, 1100], Hq, Hkv, g, seed, extra_pages=2)
    _, P2, _ = _setup([330, 1100], Hq, Hkv, g, seed, extra_pages=2)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for t in range(6):
        kn = synth.outlier_kv(seed + 2000 + t, 2, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, 2, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, 2, Hq, Hkv, 128, ch)
        O.append(kn, vn)
        kd, vd, qd = helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt)
        out_dev = ok.oscar_decode_step(P, kd, vd, qd)
        kh, vh, qh = kd.cpu().pin_memory(), vd.cpu().pin_memory(), qd.cpu().pin_memory()
        outh = torch.full(tuple(out_dev.shape), float("nan"), dtype=torch.float32).pin_memory()
        ok.oscar_decode_step(P2, kh, vh, qh, out=outh)
        torch.cuda.synchronize()
        torch.testing.assert_close(outh, out_dev.cpu(), rtol=1e-6, atol=1e-6)
        helpers.assert_attention_close(outh.numpy(), O.decode(qt))
    helpers.assert_pools_equal(O, P2)
    assert P2.err() == 0
    lib = ok.lib()
    ws = torch.empty(ok.oscar_decode_workspace_size(P2, 0), dtype=torch.uint8, device="cuda")
    pageable = qd.cpu()
    assert not pageable.is_pinned()
    st = lib.oscar_decode_step(P2.ref, C.c_void_p(kd.data_ptr()), C.c_void_p(vd.data_ptr()),
                               C.c_void_p(pageable.data_ptr()), C.c_void_p(out_dev.data_ptr()), 0.088,
                               C.c_void_p(ws.data_ptr()), ws.numel(), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 1 and b"page-locked" in lib.oscar_last_error_string()


def test_100k_context_sampled_heads():
    """Qwen3-8B layer shapes at 100k context: 99,680 history tokens on a shuffled page table (partial
    last page); the oracle rebuilds KV heads 0 and 5 and checks their 8 query heads."""
    wl = synth.DECODE_100K
    heads = [0, 5]
    O, P, q = _setup(list(wl.context), wl.num_q_heads, wl.num_kv_heads, wl.group_size, wl.seed, heads=heads)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q)).cpu().numpy()
    qh = [h for kv in heads for h in range(kv * wl.group, (kv + 1) * wl.group)]
    ref = O.decode(q, heads=qh)
    helpers.assert_attention_close(out[:, qh], ref[:, qh])


def test_100k_context_covariance_rotations_sampled_head():
    """The same shapes with the rotations of the covariance mode (eigenvectors of the calibration covariances
    Q^T Q and (S V)^T (S V), as the 100k workload specifies), KV head 3 rebuilt by the oracle."""
    wl = synth.DECODE_100K
    heads = [3]
    O, P, q = _setup(list(wl.context), wl.num_q_heads, wl.num_kv_heads, wl.group_size, wl.seed + 1, heads=heads,
                     rotation="covariance")
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q)).cpu().numpy()
    qh = [h for kv in heads for h in range(kv * wl.group, (kv + 1) * wl.group)]
    ref = O.decode(q, heads=qh)
    helpers.assert_attention_close(out[:, qh], ref[:, qh])


def test_decode_step_with_a_merge_grid_of_several_waves():
    """Qwen3-8B head shapes (32 query / 8 KV heads) with 8 sequences: the merge grid (4 x 8 x 8 CTAs of
    512 threads) takes more than one wave, and the histories cross page boundaries at different steps,
    so a late merge CTA must locate its partials from the counters before the step."""
    seed, Hkv, Hq = 700, 8, 32
    lens = [330 + 9 * b for b in range(8)]
    O, P, _ = _setup(lens, Hq, Hkv, 128, seed, extra_pages=2)
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for t in range(70):
        kn = synth.outlier_kv(seed + 2000 + t, len(lens), Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, len(lens), Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, len(lens), Hq, Hkv, 128, ch)
        O.append(kn, vn)
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        if t % 10 == 9:
            helpers.assert_attention_close(out.cpu().numpy(), O.decode(qt))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0 and int(P.sync.abs().sum()) == 0


def test_many_partials_per_segment_merge_in_several_rounds():
    """One KV head with a 20k-token history: every history CTA of the launch works on the same segment,
    so the merge stages its partial slots in several rounds (running maximum across rounds)."""
    seed, Hkv, Hq = 720, 1, 4
    O, P, q = _setup([20000], Hq, Hkv, 128, seed, extra_pages=1)
    out = ok.oscar_decode_attention(P, helpers.to_dev_bf16(q))
    helpers.assert_attention_close(out.cpu().numpy(), O.decode(q))
    ch = synth.outlier_channels(seed, Hkv, 128, 4)
    for t in range(3):
        kn = synth.outlier_kv(seed + 2000 + t, 1, Hkv, 128, ch)
        vn = synth.outlier_kv(seed + 3000 + t, 1, Hkv, 128, ch)
        qt = synth.outlier_q(seed + 4000 + t, 1, Hq, Hkv, 128, ch)
        O.append(kn, vn)
        out = ok.oscar_decode_step(P, helpers.to_dev_bf16(kn), helpers.to_dev_bf16(vn), helpers.to_dev_bf16(qt))
        helpers.assert_attention_close(out.cpu().numpy(), O.decode(qt))
    torch.cuda.synchronize()
    helpers.assert_pools_equal(O, P)
    assert P.err() == 0

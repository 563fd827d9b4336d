"""Shared test plumbing: numpy <-> torch bf16 bit conversion, pool construction for both sides,
and the parity checks the tests apply (bit-exact bytes; attention within the stated tolerance)."""
from __future__ import annotations

import numpy as np
import torch

from oracle import pool as opool
from oracle import quant as oquant
from oracle import rotation as orot
import synth

# Attention tolerance: max-abs 2e-3 and relative-L2 1e-3 against the float64 oracle.
ATOL, RTOL_L2 = 2e-3, 1e-3


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_rotations(seed: int, Hkv: int, d: int = 128):
    """Per-head float32 rotations R32 = fp32(U·H·P) with Haar U, from the oracle (kernel test inputs)."""
    return np.stack([orot.to_f32(orot.rotation_from_gaussian(synth.gaussian_matrix(seed + h, d))) for h in range(Hkv)])


def oracle_covariance_rotations(seed: int, Hq: int, Hkv: int, n_tokens: int = 512, d: int = 128):
    """Per-head float32 (R_k, R_v) from the oracle's covariance mode: U = the eigenvectors of C_k = sum Q^T Q
    over the group's query heads and of C_v = sum (S V)^T (S V), on seeded calibration-style activations."""
    G = Hq // Hkv
    ch = synth.outlier_channels(seed, Hkv, d, 4)
    Q = synth.bf16_bits_to_f32(synth.calib_samples(seed + 1, n_tokens, Hq, d, ch, heads_per_channel_set=G))
    K = synth.bf16_bits_to_f32(synth.calib_samples(seed + 2, n_tokens, Hkv, d, ch))
    V = synth.bf16_bits_to_f32(synth.calib_samples(seed + 3, n_tokens, Hkv, d, ch))
    Rk = np.stack([orot.to_f32(orot.rotation_from_covariance(orot.covariance_k(Q[:, h * G:(h + 1) * G])))
                   for h in range(Hkv)])
    Rv = np.stack([orot.to_f32(orot.rotation_from_covariance(orot.covariance_v(Q[:, h * G:(h + 1) * G], K[:, h], V[:, h])))
                   for h in range(Hkv)])
    return Rk, Rv


def make_pools(B, Hq, Hkv, g, pages_per_seq, seed, clip_k=None, clip_v=None, extra_pages=0, codebook_k=None,
               codebook_v=None, rotation="haar"):
    """(oracle Pool, device Pool) with identical rotations (Haar U, or the covariance mode's eigenvectors),
    clips, codebooks and shuffled page tables."""
    import bit_rotated_kv_02_gb300 as ok
    if rotation == "covariance":
        Rk, Rv = oracle_covariance_rotations(seed, Hq, Hkv)
    else:
        Rk = oracle_rotations(seed, Hkv)
        Rv = oracle_rotations(seed + 1000, Hkv)
    clip_k = np.full(Hkv, 0.9, np.float32) if clip_k is None else np.asarray(clip_k, np.float32)
    clip_v = np.full(Hkv, 0.9, np.float32) if clip_v is None else np.asarray(clip_v, np.float32)
    max_pages = max(max(pages_per_seq) + extra_pages, 1)
    pt, num_pages = synth.page_tables(seed, [p + extra_pages for p in pages_per_seq], max_pages)
    O = opool.Pool(B, Hq, Hkv, 128, g, num_pages, max_pages, Rk, Rv, clip_k, clip_v, codebook_k=codebook_k,
                   codebook_v=codebook_v)
    O.page_table[:] = pt
    P = ok.Pool(B, Hq, Hkv, g, num_pages, max_pages, torch.from_numpy(Rk), torch.from_numpy(Rv),
                torch.from_numpy(clip_k), torch.from_numpy(clip_v), codebook_k=codebook_k, codebook_v=codebook_v)
    P.set_page_table(pt)
    return O, P


POOL_ARRAYS = ("sink_k", "sink_v", "recent_k", "recent_v", "codes_k", "codes_v", "scale_k", "zero_k", "scale_v",
               "zero_v")


def device_array(P, name):
    t = getattr(P, name)
    return bits_of(t) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def assert_pools_equal(O, P, heads=None):
    for name in POOL_ARRAYS:
        a, b = getattr(O, name), device_array(P, name)
        if heads is not None and name.startswith(("codes", "scale", "zero")):
            a, b = a[:, heads], b[:, heads]
        assert np.array_equal(a, b), f"pool array {name} differs ({np.count_nonzero(a != b)} entries)"
    for name in ("sink_len", "hist_len", "recent_start", "recent_len"):
        assert np.array_equal(getattr(O, name), getattr(P, name).cpu().numpy()), name


def assert_attention_close(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert np.isfinite(got).all(), "non-finite attention output"
    assert err.max() <= ATOL, f"max-abs error {err.max():.3e} > {ATOL}"
    assert rel <= RTOL_L2, f"relative L2 error {rel:.3e} > {RTOL_L2}"
    return err.max(), rel


# ---- sampled-sequence parity at full workload sizes ---------------------------------------------------
# At the batch sweep's and the mixed batch's sizes the oracle cannot hold or quantize every sequence, so
# it builds a pool of a few sampled sequences (the other sequences are in the device pool only, with
# GPU-drawn contents that nothing compares).  Each sampled sequence has the same page-table row length
# in both pools; the oracle's pages are numbered compactly, and the device pages are gathered through
# the device page table before a byte comparison.

def make_sampled_pools(B, Hq, Hkv, g, pages_per_seq, sampled, seed, clip_k=None, clip_v=None, extra_pages=0):
    """(oracle Pool of the sampled sequences, device Pool of all B, device page table as numpy)."""
    import bit_rotated_kv_02_gb300 as ok
    Rk = oracle_rotations(seed, Hkv)
    Rv = oracle_rotations(seed + 1000, Hkv)
    clip_k = np.full(Hkv, 0.9, np.float32) if clip_k is None else np.asarray(clip_k, np.float32)
    clip_v = np.full(Hkv, 0.9, np.float32) if clip_v is None else np.asarray(clip_v, np.float32)
    own = [p + extra_pages for p in pages_per_seq]
    max_pages = max(max(own), 1)
    pt, num_pages = synth.page_tables(seed, own, max_pages)
    sub_own = [own[b] for b in sampled]
    O = opool.Pool(len(sampled), Hq, Hkv, 128, g, max(sum(sub_own), 1), max_pages, Rk, Rv, clip_k, clip_v)
    o = 0
    for j, n in enumerate(sub_own):
        O.page_table[j, :n] = np.arange(o, o + n, dtype=np.int32)
        o += n
    P = ok.Pool(B, Hq, Hkv, g, num_pages, max_pages, torch.from_numpy(Rk), torch.from_numpy(Rv),
                torch.from_numpy(clip_k), torch.from_numpy(clip_v))
    P.set_page_table(pt)
    return O, P, pt


def assert_sampled_pools_equal(O, P, pt, sampled, heads=None):
    """Byte equality of the sampled sequences' sink, window, history pages (gathered through the device
    page table) and counters; `heads` restricts the history comparison to those KV heads."""
    hs = slice(None) if heads is None else list(heads)
    dev = {name: device_array(P, name) for name in POOL_ARRAYS}
    cnt = {name: getattr(P, name).cpu().numpy() for name in ("sink_len", "hist_len", "recent_start", "recent_len")}
    for j, b in enumerate(sampled):
        for name in ("sink_len", "hist_len", "recent_start", "recent_len"):
            assert getattr(O, name)[j] == cnt[name][b], f"{name} of sequence {b}"
        for name in ("sink_k", "sink_v", "recent_k", "recent_v"):
            assert np.array_equal(getattr(O, name)[j], dev[name][b]), f"{name} of sequence {b}"
        np_ = -(-int(O.hist_len[j]) // 64)
        dp, op = pt[b, :np_], O.page_table[j, :np_]
        for name in ("codes_k", "codes_v", "scale_k", "zero_k", "scale_v", "zero_v"):
            a, d = getattr(O, name)[op][:, hs], dev[name][dp][:, hs]
            assert np.array_equal(a, d), f"{name} of sequence {b}: {np.count_nonzero(a != d)} entries differ"


def gpu_outlier_kv(gen, n, Hkv, channels, factor=20.0):
    """bf16 [n][Hkv][128] on the GPU: N(0,1) draws of a seeded torch generator with the given outlier
    channels scaled; the contents of unsampled sequences (never compared, never seen by the oracle)."""
    x = torch.randn((n, Hkv, 128), generator=gen, device="cuda")
    idx = torch.as_tensor(np.asarray(channels, np.int64), device="cuda")[None].expand(n, -1, -1)
    x.scatter_(2, idx, x.gather(2, idx) * factor)
    return x.to(torch.bfloat16)

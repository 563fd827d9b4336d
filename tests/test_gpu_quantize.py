"""GPU parity: bulk rotate/clip/quantize/pack (oscar_quantize_kv) against the oracle, bit for bit.

Rotate, clip, quantize and pack 4 two-bit values per byte with a scale and zero point
("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化", section "OSCAR 的设计").
Bar: packed bytes, scales and zeros identical; a differing code is tolerated only when the oracle's
pre-round value lies within one float32 ulp of a rounding boundary, for at most 1e-5 of the codes.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import bit_rotated_kv_02_gb300 as ok
from oracle import quant as oq
from oracle import rotation as orot
import synth
from tests import helpers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


def run_gpu(xb, R32, clip, g):
    N, Hkv, d = xb.shape
    stats = torch.zeros(4, dtype=torch.int32, device="cuda")
    codes, scale, zero = ok.oscar_quantize_kv(helpers.to_dev_bf16(xb), torch.from_numpy(R32).cuda(),
                                              torch.from_numpy(np.asarray(clip, np.float32)).cuda(), g, stats=stats)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), helpers.bits_of(scale), helpers.bits_of(zero), stats.cpu().numpy()


def check_rows(xb, R32, clip, g, gc, gs, gz, rows=None):
    """Compare GPU output rows with the oracle's (all rows, or the sampled `rows`)."""
    N, Hkv, d = xb.shape
    rows = np.arange(N) if rows is None else rows
    n_codes = n_bad = 0
    for h in range(Hkv):
        xh = oq.rotate_exact_many(xb[rows, h], R32[h])
        codes, s, z = oq.quantize_rotated_many(xh, clip[h], g)
        assert np.array_equal(gs[rows, h], s), f"scale differs in head {h}: {np.count_nonzero(gs[rows, h] != s)}"
        assert np.array_equal(gz[rows, h], z), f"zero differs in head {h}: {np.count_nonzero(gz[rows, h] != z)}"
        gcodes = oq.unpack_codes(gc[rows, h])
        diff = gcodes != codes
        n_codes += codes.size
        if diff.any():
            t = oq.pre_round_value(xh, s, z, g)[diff]
            dist = np.abs(t - (np.floor(t) + 0.5))
            ulp = np.spacing(np.abs(t).astype(np.float32)).astype(np.float64)
            assert np.all(dist <= ulp), "a differing code is not within one ulp of a rounding boundary"
            n_bad += int(diff.sum())
    assert n_bad <= 1e-5 * n_codes, f"{n_bad} differing codes of {n_codes}"
    return n_bad


def test_dyadic_tier_bit_exact():
    """Grid inputs k/64 and an orthogonal R with entries 0, +-1/2 make every float32 step exact."""
    d, Hkv, N = 128, 2, 777
    H4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]]) / 2.0
    base = np.kron(np.eye(32), H4) @ orot.bitrev_matrix(d)
    R32 = np.stack([base, base[:, ::-1]]).astype(np.float32)
    g_ = np.random.default_rng(0)
    xb = synth.to_bf16_bits(g_.integers(-256, 257, (N, Hkv, d)) / 64.0)
    for g in (32, 64, 128):
        for clip in ((1.0, 1.0), (0.9, 0.75)):
            gc, gs, gz, st = run_gpu(xb, R32, clip, g)
            assert check_rows(xb, R32, clip, g, gc, gs, gz) == 0
            assert st[2] == 0, "a result could not be proven correctly rounded"


@pytest.mark.parametrize("g", [32, 64, 128])
def test_production_rotation_ragged(g):
    d, Hkv, N = 128, 2, 2048 + 37
    R32 = helpers.oracle_rotations(50 + g, Hkv)
    ch = synth.outlier_channels(g, Hkv, d, 4)
    xb = synth.outlier_kv(60 + g, N, Hkv, d, ch)
    clip = (0.9, 0.8)
    gc, gs, gz, st = run_gpu(xb, R32, clip, g)
    check_rows(xb, R32, clip, g, gc, gs, gz)
    assert st[2] == 0, "a result could not be proven correctly rounded"


def test_single_row_and_empty():
    R32 = helpers.oracle_rotations(3, 1)
    xb = synth.outlier_kv(4, 1, 1, 128, synth.outlier_channels(4, 1, 128, 4))
    gc, gs, gz, st = run_gpu(xb, R32, (0.9,), 128)
    check_rows(xb, R32, (0.9,), 128, gc, gs, gz)
    assert st[2] == 0
    empty = torch.zeros((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    ok.oscar_quantize_kv(empty, torch.from_numpy(R32).cuda(), torch.ones(1, device="cuda"), 128)


def test_bulk_full_size_sampled():
    """Qwen3-32B bulk shapes: 131,072 tokens x 8 KV heads, 2 outlier channels (1%); sampled rows checked."""
    wl = synth.BULK_128K
    N, Hkv, d = wl.context[0], wl.num_kv_heads, 128
    ch = synth.outlier_channels(wl.seed, Hkv, d, wl.n_outliers)
    R32 = helpers.oracle_rotations(wl.seed, Hkv)
    xb = synth.outlier_kv(wl.seed + 1, N, Hkv, d, ch)
    gc, gs, gz, st = run_gpu(xb, R32, (0.9,) * Hkv, 128)
    rows = np.sort(np.random.default_rng(5).choice(N, 384, replace=False))
    rows = np.concatenate([[0, 1, N - 2, N - 1], rows])
    check_rows(xb, R32, (0.9,) * Hkv, 128, gc, gs, gz, rows)
    assert st[2] == 0


@pytest.mark.parametrize("g,Hkv", [(32, 3), (128, 2)])
def test_many_tiles_per_block_every_row(g, Hkv):
    """Enough rows that each block runs several tiles through its pipeline and crosses into the next
    head's rotation (head switches, ring wrap-around, both epilogue groups); every row checked."""
    d, N = 128, 50_000 + 17
    R32 = helpers.oracle_rotations(90 + g, Hkv)
    ch = synth.outlier_channels(91 + g, Hkv, d, 4)
    xb = synth.outlier_kv(92 + g, N, Hkv, d, ch)
    clip = (0.9, 0.8, 0.95)[:Hkv]
    gc, gs, gz, st = run_gpu(xb, R32, clip, g)
    check_rows(xb, R32, clip, g, gc, gs, gz)
    assert st[2] == 0 and st[3] == 0

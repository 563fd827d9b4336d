"""Seeded synthetic inputs shared by the CUDA path's tests/benchmarks and the CPU oracle.

This module holds none of the method's arithmetic: only random draws, the
rounding of those draws to bf16 (a storage-format conversion done with torch's
own cast), and plain shape presets.  Both sides receive the same arrays from
here; neither side's computation lives here.

Value recipe (the overview article "超越TurboQuant！OSCAR：面向真实服务的2-bit KV
Cache量化", section "OSCAR 的设计", says KV activations carry a few channels of
very large magnitude; the workload presets name "N(0,1) with 4 fixed outlier
channels scaled x20" and "N(0,1) + 1% channels x20"):

* q, K, V entries are N(0, 1) draws; a fixed, seeded set of channel indices per
  KV head is multiplied by the outlier factor (the same indices scale K, V and
  every query head of that KV head's group); values are then rounded to bf16.
* Page tables are seeded permutations of a physical page pool.
* Calibration samples for the covariance-aligned rotation are N(0,1) draws
  shaped by an anisotropic spectrum lambda_i proportional to 1/(i+1), mixed by
  a seeded orthogonal basis, with the same outlier channels, rounded to bf16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

PAGE = 64          # tokens per history page
SINK = 64          # BF16 sink tokens
RECENT = 256       # BF16 recent-window tokens


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(seed))


def to_bf16_bits(x) -> np.ndarray:
    """Round float values to bf16 (torch's round-to-nearest-even cast) and return the raw uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def outlier_channels(seed: int, num_kv_heads: int, d: int, n_outliers: int) -> np.ndarray:
    """[Hkv][n_outliers] distinct channel indices per KV head."""
    g = rng(seed)
    return np.stack([np.sort(g.choice(d, size=n_outliers, replace=False)) for _ in range(num_kv_heads)])


def outlier_kv(seed: int, n_tokens: int, num_kv_heads: int, d: int, channels: np.ndarray,
               factor: float = 20.0) -> np.ndarray:
    """bf16 bits [n_tokens][Hkv][d]: N(0,1) with the given channels of each head scaled by `factor`."""
    g = rng(seed)
    x = g.standard_normal((n_tokens, num_kv_heads, d), dtype=np.float32)
    for h in range(num_kv_heads):
        x[:, h, channels[h]] *= factor
    return to_bf16_bits(x)


def outlier_q(seed: int, batch: int, num_q_heads: int, num_kv_heads: int, d: int,
              channels: np.ndarray, factor: float = 20.0) -> np.ndarray:
    """bf16 bits [B][Hq][d]; query head h uses the outlier channels of KV head h // (Hq/Hkv)."""
    g = rng(seed)
    x = g.standard_normal((batch, num_q_heads, d), dtype=np.float32)
    grp = num_q_heads // num_kv_heads
    for h in range(num_q_heads):
        x[:, h, channels[h // grp]] *= factor
    return to_bf16_bits(x)


def gaussian_matrix(seed: int, d: int) -> np.ndarray:
    """float64 [d][d] of N(0,1) draws: the random input of a Haar-distributed orthogonal U."""
    return rng(seed).standard_normal((d, d))


def calib_samples(seed: int, n_tokens: int, num_heads: int, d: int, channels: np.ndarray,
                  heads_per_channel_set: int = 1, factor: float = 20.0) -> np.ndarray:
    """bf16 bits [n_tokens][num_heads][d]: anisotropic calibration activations.

    Each head draws Z ~ N(0,1), scales column i by sqrt(1/(i+1)), mixes the
    columns by a seeded orthogonal basis (the Q factor of a Gaussian matrix,
    taken from numpy's QR; it is a draw, not a step of the method), then scales
    the outlier channels of its channel set (head // heads_per_channel_set).
    """
    g = rng(seed)
    spec = np.sqrt(1.0 / (np.arange(d) + 1.0))
    out = np.empty((n_tokens, num_heads, d), np.float32)
    for h in range(num_heads):
        basis, _ = np.linalg.qr(g.standard_normal((d, d)))
        z = g.standard_normal((n_tokens, d)) * spec
        x = (z @ basis.T) * math.sqrt(d / spec.dot(spec))
        x[:, channels[h // heads_per_channel_set]] *= factor
        out[:, h, :] = x
    return to_bf16_bits(out)


def shuffled_pages(seed: int, num_pages: int) -> np.ndarray:
    return rng(seed).permutation(num_pages).astype(np.int32)


def page_tables(seed: int, pages_per_seq: list[int], max_pages: int, num_pages: int | None = None) -> tuple[np.ndarray, int]:
    """Random page tables drawn from one shuffled physical pool. Returns ([B][max_pages] int32, num_pages).

    Unused table slots hold -1."""
    total = int(sum(pages_per_seq))
    num_pages = max(total, 1) if num_pages is None else num_pages
    perm = shuffled_pages(seed, num_pages)
    pt = np.full((len(pages_per_seq), max_pages), -1, np.int32)
    o = 0
    for b, n in enumerate(pages_per_seq):
        pt[b, :n] = perm[o:o + n]
        o += n
    return pt, num_pages


def context_lengths(seed: int, batch: int, lo: int, hi: int) -> np.ndarray:
    return rng(seed).integers(lo, hi + 1, size=batch).astype(np.int64)


def clip_ratios(seed: int, num_kv_heads: int, lo: float, hi: float) -> np.ndarray:
    return rng(seed).uniform(lo, hi, size=num_kv_heads).astype(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape preset of one named synthetic workload (sizes only)."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    group_size: int
    context: tuple          # per-sequence total context lengths
    n_outliers: int
    clip: tuple             # (lo, hi) per-(head, K/V) clip ratio range; lo == hi for a fixed ratio
    rotation: str           # "haar" or "covariance"
    seed: int

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def hist_len(context: int) -> int:
    return max(context - SINK - RECENT, 0)


# Tiny single-layer decode: 1024 = 64 sink + 704 history + 256 recent, GQA 4.
TINY = Workload("tiny-gqa4-L1024", 1, 8, 2, 128, 128, (1024,), 4, (0.9, 0.9), "haar", 1001)
# Qwen3-8B-shaped layer at 100k context (99,680 history tokens), batch 1.
DECODE_100K = Workload("qwen3-8b-layer-L100000-b1", 1, 32, 8, 128, 128, (100_000,), 4, (0.9, 0.9),
                       "covariance", 1002)
# Batch sweep, Qwen3-8B shapes, 32k context per sequence.
def batch_sweep(batch: int) -> Workload:
    return Workload(f"qwen3-8b-layer-L32768-b{batch}", batch, 32, 8, 128, 128, (32_768,) * batch, 4,
                    (0.9, 0.9), "haar", 1003 + batch)
# Bulk prefill quantize, Qwen3-32B KV shapes: 131,072 tokens x 8 KV heads, 1% outlier channels.
BULK_128K = Workload("qwen3-32b-bulk-N131072", 1, 64, 8, 128, 128, (131_072,), 2, (0.9, 0.9), "haar", 1004)
# Long-context mixed batch, Qwen3-32B shapes, lengths U[8k,128k], group 32, clip U[0.8,1.0].
def mixed_long(seed: int = 1005) -> Workload:
    lens = tuple(int(v) for v in context_lengths(seed, 8, 8_192, 131_072))
    return Workload("qwen3-32b-mixed-b8-L8k-128k-g32", 8, 64, 8, 128, 32, lens, 4, (0.8, 1.0), "haar", seed)

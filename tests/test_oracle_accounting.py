"""Pins for oracle.accounting against the bits-per-element figures the pages print.

2.28 effective bits per KV element ("超越TurboQuant！OSCAR：面向真实服务的2-bit KV Cache量化",
evaluation summary; "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
Quantization", Abstract) and 2.38 on the 32K AIME25 run (Fig. 4 caption).
"""
import os

from oracle import accounting

HERE = os.path.dirname(__file__)


def test_printed_bits_per_element():
    rows = [l.split() for l in open(os.path.join(HERE, "golden", "bits_per_element.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for ctx, group, printed, _ in rows:
        assert round(accounting.bits_per_element(int(ctx), int(group)), 2) == float(printed)


def test_history_bytes_and_memory_ratio():
    assert accounting.history_bytes_per_token_head(128, 128) == 36
    assert accounting.history_bytes_per_token_head(128, 32) == 48
    # "约8倍": 16-bit vs 2-bit codes, metadata ignored
    assert 16 / 2 == 8 and abs(16 / (accounting.history_bytes_per_token_head() * 8 / 128) - 7.11) < 0.01

"""Oracle: effective bits per KV element of the three-segment pool (test infrastructure only).

[Article, "OSCAR 的动机"/"OSCAR 的设计"] and [Abstract]: OSCAR runs at about
2.28 effective bits per KV element; the AIME25 run at 32K reports 2.38.
Reading: each history element costs 2 bits plus one bf16 scale and one bf16
zero per group of g elements; sink (64) and recent (256) tokens cost 16 bits
per element.
"""
from __future__ import annotations


def bits_per_element(context: int, group: int = 128, sink: int = 64, recent: int = 256) -> float:
    bf16_tokens = min(context, sink + recent)
    hist = context - bf16_tokens
    return (hist * (2.0 + 32.0 / group) + bf16_tokens * 16.0) / context


def history_bytes_per_token_head(d: int = 128, group: int = 128) -> int:
    """Packed codes plus scale and zero of one (token, head) vector, K or V."""
    return d // 4 + 4 * (d // group)

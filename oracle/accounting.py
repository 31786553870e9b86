"""Closed-form storage accounting per token and tier.

Pages (Minima-KV abstract, mlsanity.com paper page): deployment accounting
reports 18.3 KiB of attention KV per live token, 3.50x less than BF16 and
1.75x less than FP8, for Qwen3.6-27B profiles with 16 full-attention layers;
the direct-decode canary (two 59,008-token requests) reports 3.625x
active-KV compression.

Under this library's formats a row (one token, one kv head, K or V) costs
  BF16: 2*d bytes;  FP8: d + 2 bytes;  TQ3: 3*d/8 + 2 bytes,
so with d = 256, 4 kv heads and K+V: 4096 / 2064 / 784 bytes per token per
layer.  The pages' own ratios are checked for internal consistency only;
reproducing 3.50x / 3.625x from this spec is NOT possible (the spec's mix is
more compact), so those two numbers are "parity unpinned" and reported side
by side.
"""
from __future__ import annotations


def row_bytes(fmt: str, d: int) -> int:
    if fmt == "bf16":
        return 2 * d
    if fmt == "fp8":
        return d + 2
    if fmt == "tq3":
        return 3 * d // 8 + 2
    raise ValueError(fmt)


def bytes_per_token_layer(fmt: str, d: int = 256, n_kv_heads: int = 4) -> int:
    return 2 * n_kv_heads * row_bytes(fmt, d)


def bytes_per_token(fmt: str, d: int = 256, n_kv_heads: int = 4, n_layers: int = 16) -> int:
    return n_layers * bytes_per_token_layer(fmt, d, n_kv_heads)


def mixed_bytes_per_token(fp8_tokens: int, tq3_tokens: int, d: int = 256,
                          n_kv_heads: int = 4, n_layers: int = 16) -> float:
    tot = fp8_tokens * bytes_per_token("fp8", d, n_kv_heads, n_layers) + \
        tq3_tokens * bytes_per_token("tq3", d, n_kv_heads, n_layers)
    return tot / (fp8_tokens + tq3_tokens)


def fp8_fraction_for_ratio_vs_bf16(ratio: float, d: int = 256) -> float:
    """Fraction f of FP8 tokens that gives BF16/mixed = ratio under this spec:
    f*fp8 + (1-f)*tq3 = bf16/ratio."""
    bf, f8, t3 = row_bytes("bf16", d), row_bytes("fp8", d), row_bytes("tq3", d)
    return (bf / ratio - t3) / (f8 - t3)

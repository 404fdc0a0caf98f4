"""Algorithmic byte and FLOP counts for one MLA decode step (roofline inputs).

Cache sizes follow the MLA operator write-up (nxmr.cn/news/151634) §1: one
token of one layer stores d_c + d_R = 576 elements (1.125 KB in bf16), against
2 x 128 heads x 128 dims for multi-head attention.  Page sizes follow §3.

Only work the method needs is credited: cache rows of visible tokens, the
absorbed query, the latent output and its log-sum-exp.  Split-KV partials,
padding rows of a page and the zero blocks of the grouped-latent query are
implementation overhead and are not counted.

kv="fp8": the cache row is the FP8 one of mla_decode_paged_fp8, 512 E4M3
codes + 64 bf16 RoPE key + 4 fp32 scales = 656 bytes a token.
"""
from __future__ import annotations

BF16 = 2
FP32 = 4
FP8_ROW_BYTES = 512 + 64 * BF16 + 4 * FP32


def row_bytes(kv: str = "bf16", d_c: int = 512, d_R: int = 64) -> int:
    """Cache bytes of one token in one layer for a cache format."""
    if kv == "fp8":
        return d_c + d_R * BF16 + (d_c // 128) * FP32
    return (d_c + d_R) * BF16


def bytes_per_token(d_c: int = 512, d_R: int = 64, elem_bytes: int = BF16) -> int:
    """Latent cache bytes of one token in one layer."""
    return (d_c + d_R) * elem_bytes


def mha_bytes_per_token(heads: int = 128, head_dim: int = 128, elem_bytes: int = BF16) -> int:
    """K and V of full multi-head attention for one token in one layer."""
    return 2 * heads * head_dim * elem_bytes


def gqa_bytes_per_token(groups: int, head_dim: int = 128, elem_bytes: int = BF16) -> int:
    return 2 * groups * head_dim * elem_bytes


def page_bytes(page_size: int, d_c: int = 512, d_R: int = 64, elem_bytes: int = BF16) -> int:
    return page_size * bytes_per_token(d_c, d_R, elem_bytes)


def compression_ratio(d_c: int = 512, d_R: int = 64, heads: int = 128, head_dim: int = 128) -> float:
    """Fraction of the MHA cache that the latent cache saves."""
    return 1.0 - bytes_per_token(d_c, d_R) / mha_bytes_per_token(heads, head_dim)


def latent_kv_bytes(seq_lens, d_c: int = 512, d_R: int = 64, kv: str = "bf16") -> int:
    """Latent KV cache bytes one decode step of one layer reads: every cached
    row of every sequence once (the new tokens' rows included)."""
    return sum(int(n) for n in seq_lens) * row_bytes(kv, d_c, d_R)


def decode_bytes(seq_lens, Lq: int, H: int, G: int = 1, d_c: int = 512, d_R: int = 64, kv: str = "bf16") -> int:
    """Algorithmic HBM bytes of mla_decode_paged + mla_combine_splits: every
    visible cache row once, q_cat in, o_lat (bf16) and lse (fp32) out."""
    d_g = d_c // G
    B = len(seq_lens)
    cache = sum(int(n) for n in seq_lens) * row_bytes(kv, d_c, d_R)
    q = B * Lq * H * (d_g + d_R) * BF16
    o = B * Lq * H * d_g * BF16 + B * Lq * H * FP32
    return cache + q + o


def decode_flops(seq_lens, Lq: int, H: int, G: int = 1, d_c: int = 512, d_R: int = 64,
                 causal: bool = True) -> int:
    """2*(d_g + d_R) (scores) + 2*d_g (weighted latent sum) per (query row,
    visible key)."""
    d_g = d_c // G
    keys = 0
    for n in seq_lens:
        n = int(n)
        for l in range(Lq):
            keys += (n - Lq + l + 1) if causal else n
    return keys * H * (2 * (d_g + d_R) + 2 * d_g)


def absorb_bytes(B: int, Lq: int, H: int, d_hc: int = 128, d_g: int = 512, d_R: int = 64) -> int:
    """W_UK + q_nope + q_rope in, q_cat out."""
    return (H * d_hc * d_g + B * Lq * H * (d_hc + d_R) + B * Lq * H * (d_g + d_R)) * BF16


def project_bytes(B: int, Lq: int, H: int, d_hc: int = 128, d_g: int = 512) -> int:
    """W_UV + o_lat in, out written."""
    return (H * d_hc * d_g + B * Lq * H * d_g + B * Lq * H * d_hc) * BF16


def step_bytes(seq_lens, Lq: int, H: int, G: int = 1, kv: str = "bf16") -> int:
    """One whole decode step of one layer: absorb, decode+combine, project."""
    B = len(seq_lens)
    d_g = 512 // G
    return (absorb_bytes(B, Lq, H, d_g=d_g) + decode_bytes(seq_lens, Lq, H, G, kv=kv)
            + project_bytes(B, Lq, H, d_g=d_g))


def step_flops(seq_lens, Lq: int, H: int, G: int = 1) -> int:
    B = len(seq_lens)
    d_g = 512 // G
    gemm = 2 * (2 * B * Lq * H * 128 * d_g)
    return decode_flops(seq_lens, Lq, H, G) + gemm

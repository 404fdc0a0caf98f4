"""Seeded synthetic inputs for MLA decode over a paged latent KV cache.

This module only draws random inputs: it holds none of the method's
arithmetic, and it is the one piece shared by the CUDA path's tests and the
oracle's.  Every tensor is drawn on the host from one ``torch.Generator``
seeded per workload, in a fixed order (seq_lens, q_nope, q_rope, cache,
W_UK, W_UV, block_table), and rounded to bf16 once.

Shapes and distributions follow the MLA operator write-up
(nxmr.cn/news/151634): §1 and §3 fix the cache row (512-d latent + 64-d RoPE
key, 576 bf16) and the 64-token page; the DeepSeek-V2/V3 dims of §3
(128 heads, 128-d content head) set H and d_hc.  Queries and cache entries are
N(0, 1); the projection matrices are N(0, 1/d_g) so logits have unit scale.

An FP8 cache (kv="fp8") is drawn as its bytes: per latent code a random
sign, an exponent field from a rounded normal (mean 13, sd 1.5, clipped to
0..15) and a uniform mantissa (never the NaN pattern), so the code values
spread over the E4M3 range as those of a Gaussian block scaled to fill it
do; per token and 128-column block a scale 2^k, k uniform in -8..-6 (the
latent then has about the size of the bf16 cache's); the RoPE key N(0, 1)
in bf16.  Row layout: 512 codes | 64 bf16 | 4 fp32 scales (656 bytes).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D_HC, D_C, D_R, PAGE = 128, 512, 64, 64
SEED_BASE = 20261200
FP8_ROW = D_C + 2 * D_R + 4 * (D_C // 128)  # bytes of an FP8 cache row

# name -> (index, spec).  Index i gives seed SEED_BASE + i.
WORKLOADS = {
    # tiny MLA decode: H=16, lengths 37 and 200 (1 + 4 pages), permuted pages
    "tiny": dict(index=1, B=2, Lq=1, H=16, G=1, seq_lens=[37, 200], table="perm"),
    # DeepSeek-V3 dims, one layer: B=16, all lengths 4096, contiguous tables
    "dsv3": dict(index=2, B=16, Lq=1, H=128, G=1, seq_lens=[4096] * 16, table="contig"),
    # long context: B=16, lengths uniform in [32768, 65536], shuffled pages
    "long": dict(index=3, B=16, Lq=1, H=128, G=1, seq_range=(32768, 65536), table="perm"),
    # speculative decode: B=64, Lq=2 causal, lengths uniform in [1024, 16384]
    "spec": dict(index=4, B=64, Lq=2, H=128, G=1, seq_range=(1024, 16384), table="perm"),
    # grouped latent (GLA): G=2 groups of 64 heads, 256-d latent each + shared k_R
    "gla": dict(index=5, B=32, Lq=1, H=128, G=2, seq_lens=[8192] * 32, table="contig"),
    # a long query chunk (the decompress branch): 1024 new tokens after 3072 cached ones, H=128
    "prefill": dict(index=6, B=1, Lq=1024, H=128, G=1, seq_lens=[4096], table="contig"),
}


@dataclass
class Case:
    name: str
    dims: dict
    q_nope: torch.Tensor       # bf16 [B,Lq,H,d_hc]
    q_rope: torch.Tensor       # bf16 [B,Lq,H,d_R]
    cache: torch.Tensor        # bf16 [num_pages,P,d_c+d_R], or uint8 [num_pages,P,656] (FP8)
    W_UK: torch.Tensor         # bf16 [H,d_hc,d_g]
    W_UV: torch.Tensor         # bf16 [H,d_hc,d_g]
    block_table: torch.Tensor  # int32 [B,max_pages] (-1 = unused)
    seq_lens: torch.Tensor     # int32 [B]
    meta: dict = field(default_factory=dict)

    def tensors(self):
        return dict(q_nope=self.q_nope, q_rope=self.q_rope, cache=self.cache,
                    W_UK=self.W_UK, W_UV=self.W_UV, block_table=self.block_table,
                    seq_lens=self.seq_lens)


def make_case(name: str = "custom", *, B: int, Lq: int = 1, H: int = 128, G: int = 1,
              seq_lens=None, seq_range=None, table: str = "contig", seed: int,
              max_pages: int | None = None, extra_pages: int = 0,
              q_zero: bool = False, causal: int = 1, kv: str = "bf16") -> Case:
    """Draw one synthetic decode problem.

    seq_lens: explicit list of lengths, or seq_range=(lo, hi) inclusive uniform.
    table: "contig" (sequence b owns pages b*max_pages + i), or "perm" (the
    pool of all needed pages handed out in a seeded random order).
    extra_pages: unused pages appended to the pool (never referenced).
    q_zero: all-zero queries (uniform attention), a test special case.
    kv: "bf16" (rows of 576 bf16) or "fp8" (rows of 656 bytes, see above).
    """
    gen = torch.Generator(device="cpu").manual_seed(int(seed))
    if seq_lens is None:
        lo, hi = seq_range
        seq = torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64)
    else:
        assert len(seq_lens) == B
        seq = torch.tensor(list(seq_lens), dtype=torch.int64)
    npages = [(int(n) + PAGE - 1) // PAGE for n in seq]
    if max_pages is None:
        cap = seq_range[1] if seq_range is not None else int(seq.max())
        max_pages = (cap + PAGE - 1) // PAGE
    assert max(npages) <= max_pages
    d_g = D_C // G
    if table == "contig":
        num_pages = B * max_pages + extra_pages
    else:
        num_pages = sum(npages) + extra_pages

    def normal(shape, std):
        t = torch.randn(shape, generator=gen, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(torch.bfloat16)

    q_nope = normal((B, Lq, H, D_HC), 1.0)
    q_rope = normal((B, Lq, H, D_R), 1.0)
    if q_zero:
        q_nope.zero_()
        q_rope.zero_()
    if kv == "bf16":
        cache = normal((num_pages, PAGE, D_C + D_R), 1.0)
    elif kv == "fp8":
        cache = fp8_cache(gen, num_pages)
    else:
        raise ValueError(kv)
    w_std = 1.0 / math.sqrt(d_g)
    W_UK = normal((H, D_HC, d_g), w_std)
    W_UV = normal((H, D_HC, d_g), w_std)

    bt = torch.full((B, max_pages), -1, dtype=torch.int32)
    if table == "contig":
        for b in range(B):
            bt[b, : npages[b]] = torch.arange(b * max_pages, b * max_pages + npages[b], dtype=torch.int32)
    elif table == "perm":
        pool = torch.randperm(sum(npages), generator=gen).to(torch.int32)
        off = 0
        for b in range(B):
            bt[b, : npages[b]] = pool[off: off + npages[b]]
            off += npages[b]
    else:
        raise ValueError(table)

    dims = dict(B=B, Lq=Lq, H=H, d_hc=D_HC, d_c=D_C, d_R=D_R, G=G, page_size=PAGE,
                max_pages=max_pages, num_pages=num_pages,
                scale=1.0 / math.sqrt(D_HC + D_R), causal=int(causal))
    return Case(name=name, dims=dims, q_nope=q_nope, q_rope=q_rope, cache=cache,
                W_UK=W_UK, W_UV=W_UV, block_table=bt, seq_lens=seq.to(torch.int32),
                meta=dict(seed=int(seed), table=table, kv=kv))


def fp8_rows(codes: torch.Tensor, rope: torch.Tensor, scales: torch.Tensor) -> torch.Tensor:
    """Pack FP8 cache rows: codes uint8 [..., 512], rope bf16 [..., 64],
    scales fp32 [..., 4] -> uint8 [..., 656]."""
    lead = codes.shape[:-1]
    return torch.cat([codes, rope.contiguous().view(torch.uint8).reshape(*lead, 2 * D_R),
                      scales.contiguous().view(torch.uint8).reshape(*lead, 16)], dim=-1).contiguous()


def fp8_cache(gen: torch.Generator, num_pages: int) -> torch.Tensor:
    """Random FP8 cache pages (uint8 [num_pages, P, 656]); see the module text."""
    shape = (num_pages, PAGE, D_C)
    sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.int32)
    expo = torch.randn(shape, generator=gen).mul_(1.5).add_(13.0).round_().clamp_(0, 15).to(torch.int32)
    mant = torch.randint(0, 8, shape, generator=gen, dtype=torch.int32)
    mant = torch.where((expo == 15) & (mant == 7), torch.full_like(mant, 6), mant)  # 0x7f / 0xff are NaN
    codes = (sign * 128 + expo * 8 + mant).to(torch.uint8)
    k = torch.randint(-8, -5, (num_pages, PAGE, D_C // 128), generator=gen, dtype=torch.int32)
    scales = torch.pow(2.0, k.to(torch.float32))
    rope = torch.randn((num_pages, PAGE, D_R), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return fp8_rows(codes, rope, scales)


def workload(name: str, **override) -> Case:
    """One of the named workloads (see WORKLOADS), seeded SEED_BASE + index."""
    spec = dict(WORKLOADS[name])
    idx = spec.pop("index")
    spec.update(override)
    return make_case(name, seed=SEED_BASE + idx, **spec)

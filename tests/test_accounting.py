"""The byte/FLOP accounting used for roofline numbers, pinned to the figures
the pages print (tests/golden/page_figures.json, each entry cited)."""
import json
import os

import pytest

from mla_latent_kv_10_gb300 import accounting as acc

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))
KB, GB, TB = 1024, 1024 ** 3, 1024 ** 4


def close(value, key, scale=1.0):
    g = GOLDEN[key]
    return value / scale == pytest.approx(g["value"], rel=max(g["rounding"], 1e-12))


def test_per_token_sizes():
    assert acc.bytes_per_token() == 1152
    assert close(acc.bytes_per_token(), "bytes_per_token_kb", KB)
    assert close(acc.mha_bytes_per_token(), "mha_bytes_per_token_kb", KB)
    assert round(100 * acc.compression_ratio(), 2) == GOLDEN["compression_percent"]["value"]


def test_page_sizes():
    assert acc.page_bytes(64) == 73728
    assert close(acc.page_bytes(64), "page64_kb", KB)
    assert close(acc.page_bytes(16), "page16_kb", KB)


def test_hopper_smem_budget_figure():
    tile, stages = 64, 3
    smem = (tile * 512 + tile * 64) * 2 * stages
    assert close(smem, "smem_tile64_stage3_kb", KB)


def test_cache_footprint_at_64k_batch16():
    tokens = 16 * 65536 * GOLDEN["cache_b16_64k_mla_gb"]["layers"]
    assert close(tokens * acc.mha_bytes_per_token(), "cache_b16_64k_mha_tb", TB)
    assert close(tokens * acc.gqa_bytes_per_token(8), "cache_b16_64k_gqa8_gb", GB)
    assert close(tokens * acc.bytes_per_token(), "cache_b16_64k_mla_gb", GB)


def test_ridge_and_mqa_ratio():
    assert close(989e12 / 3.35e12, "h100_ridge_flop_per_byte")
    # one MQA head stores K and V of 128 dims: 256 elements
    assert 576 / (2 * 128) == GOLDEN["latent_vs_mqa"]["value"]


def test_decode_counts():
    # DeepSeek-V3 dims, B=16, n=4096: 16*4096 rows of 1152 B + q_cat + o_lat + lse
    b = acc.decode_bytes([4096] * 16, 1, 128)
    assert b == 16 * 4096 * 1152 + 16 * 128 * 576 * 2 + 16 * 128 * 512 * 2 + 16 * 128 * 4
    f = acc.decode_flops([4096] * 16, 1, 128)
    assert f == 16 * 4096 * 128 * (2 * 576 + 2 * 512)
    # causal Lq=2: query 0 sees n-1 keys, query 1 sees n
    assert acc.decode_flops([10], 2, 1) == (9 + 10) * 2176
    # grouped latent: d_g = 256 -> 2*(256+64) + 2*256 = 1152 per (row, key)
    assert acc.decode_flops([8], 1, 2, G=2) == 8 * 2 * 1152

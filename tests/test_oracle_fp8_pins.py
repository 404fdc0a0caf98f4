"""Pins of the oracle's FP8 cache reading (CPU only).

The MLA operator write-up names a low-precision latent cache (introduction,
§5 tail) without fixing its format; the oracle reads the FP8 cache as OCP
8-bit floating point E4M3 codes (sign, 4 exponent bits with bias 7, 3
mantissa bits; exponent 0 subnormal; S.1111.111 NaN; no infinities), each
times the power-of-two scale of its 128-column block.  Pinned here to the
values the format definition fixes, to PyTorch's own float8_e4m3fn
conversion for all 256 codes, and to the bf16 decode it must reduce to.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_10_gb300.inputs import FP8_ROW, fp8_rows, make_case


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),      # subnormals: m/8 * 2^-6
    (0x08, 2.0 ** -6), (0x0F, 1.875 * 2.0 ** -6),              # smallest normal binade
    (0x30, 0.5), (0x38, 1.0), (0x3C, 1.5), (0x40, 2.0),
    (0x77, 240.0), (0x78, 256.0), (0x7E, 448.0),                # largest finite: S.1111.110
    (0xB8, -1.0), (0xFE, -448.0), (0x81, -(2.0 ** -9)),
])
def test_e4m3_values_of_the_format_definition(code, value):
    assert oracle.e4m3(code) == value


def test_e4m3_nan_codes_and_signed_zero():
    assert np.isnan(oracle.e4m3(0x7F)) and np.isnan(oracle.e4m3(0xFF))
    assert oracle.e4m3(0x80) == 0.0 and np.signbit(oracle.e4m3(0x80))
    finite = [c for c in range(256) if np.isfinite(oracle.e4m3(c))]
    assert len(finite) == 254


def test_e4m3_matches_torch_float8_for_every_code():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3(c) for c in range(256)])
    assert np.array_equal(ours, ref, equal_nan=True)


def test_e4m3_order_and_sign_symmetry():
    pos = np.array([oracle.e4m3(c) for c in range(0x7F)])
    assert np.all(np.diff(pos) > 0)
    for c in range(0x7F):
        assert oracle.e4m3(c | 0x80) == -oracle.e4m3(c)


def test_dequant_applies_each_blocks_scale():
    """Every 128-column block its own scale; codes checked against torch's
    float8 conversion times that scale; the RoPE key passes through."""
    gen = torch.Generator().manual_seed(5)
    codes = torch.randint(0, 256, (3, 7, 512), generator=gen, dtype=torch.int32).to(torch.uint8)
    codes[(codes == 0x7F) | (codes == 0xFF)] = 0x3C
    scales = torch.pow(2.0, torch.randint(-15, 8, (3, 7, 4), generator=gen).float())
    rope = torch.randn(3, 7, 64, generator=gen).to(torch.bfloat16)
    rows = fp8_rows(codes, rope, scales)
    assert rows.shape == (3, 7, FP8_ROW) and FP8_ROW == 656
    lat, rope_bits = oracle.dequant_fp8(rows)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64) * scales.double().repeat_interleave(128, dim=-1)
    assert np.array_equal(lat, want.numpy())
    assert np.array_equal(rope_bits, rope.view(torch.int16).numpy().view(np.uint16))


def test_fp8_decode_is_the_bf16_decode_of_the_dequantised_cache():
    """decode_fp8 equals decode over a bf16 cache built independently (torch's
    float8 conversion, scale, bf16) from the same FP8 rows: bit for bit."""
    c = make_case(B=3, Lq=2, H=16, G=2, seq_lens=[2, 90, 200], table="perm", seed=61, kv="fp8")
    codes, rope_b, sc_b = c.cache[..., :512], c.cache[..., 512:640], c.cache[..., 640:656]
    lat = codes.contiguous().view(torch.float8_e4m3fn).to(torch.float64) * \
        sc_b.contiguous().view(torch.float32).double().repeat_interleave(128, dim=-1)
    bf = torch.cat([lat.to(torch.bfloat16), rope_b.contiguous().view(torch.bfloat16)], dim=-1)
    assert torch.equal(bf[..., :512].double(), lat)  # exact in bf16
    t = c.tensors()
    got = oracle.decode_fp8(c.dims, **t)
    t["cache"] = bf
    ref = oracle.decode(c.dims, **t)
    for g, r in zip(got, ref):
        assert np.array_equal(g, r, equal_nan=True)


def test_fp8_reading_refuses_a_value_bf16_cannot_hold():
    codes = torch.full((1, 1, 512), 0x3F, dtype=torch.uint8)  # 1.875
    rope = torch.zeros(1, 1, 64, dtype=torch.bfloat16)
    ok = fp8_rows(codes, rope, torch.full((1, 1, 4), 3.0))  # 5.625: 6 significant bits, a bf16 value
    oracle.fp8_as_bf16_cache(ok)
    bad = fp8_rows(codes, rope, torch.full((1, 1, 4), 1.0 + 2.0 ** -10))
    with pytest.raises(ValueError):
        oracle.fp8_as_bf16_cache(bad)


def test_fp8_inputs_hold_no_nan_code_and_power_of_two_scales():
    c = make_case(B=2, Lq=1, H=16, seq_lens=[100, 300], table="perm", seed=62, kv="fp8")
    codes = c.cache[..., :512]
    assert not torch.any((codes == 0x7F) | (codes == 0xFF))
    sc = c.cache[..., 640:656].contiguous().view(torch.float32)
    m, e = torch.frexp(sc)
    assert torch.all(m == 0.5) and torch.all((e - 1 >= -15) & (e - 1 <= 7))

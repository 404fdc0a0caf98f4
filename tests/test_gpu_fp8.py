"""The FP8 latent cache (mla_decode_paged_fp8) against the fp64 oracle.

The oracle reads an FP8 cache by its definition: the latent is
e4m3(code) * scale of the code's 128-column block (OCP 8-bit floating point,
E4M3), the RoPE key is bf16; attention is then the same as for a bf16 cache.
The low-precision cache is the MLA operator write-up's (introduction and the
tail of §5: an NVFP4 cache read with 16-byte vector loads); FP8 E4M3 with
power-of-two scales is the reading implemented.

Tolerance: that of the bf16 path (max|err| <= 2e-2 max|ref|, cosine >=
0.9999).  The dequantisation itself is checked bit for bit: a sequence of
one token attends to that token alone, so its latent output is the token's
dequantised latent, which bf16 holds exactly.
"""
import numpy as np
import pytest
import torch

import mla_latent_kv_10_gb300 as mla
import oracle
from mla_latent_kv_10_gb300.inputs import fp8_rows, make_case, workload
from parity_util import assert_close, check_case, run_decode_only, run_gpu, sample_pairs

pytestmark = pytest.mark.gpu

MLA_ERR_RANGE = -9


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_latent_kv_10_gb300 import _build
    _build.build()
    mla.load_library()


def fp8_case(**kw):
    return make_case(kv="fp8", **kw)


SMALL = {
    "tiny": lambda: workload("tiny", kv="fp8"),
    "mla_ragged": lambda: fp8_case(B=4, Lq=1, H=128, seq_lens=[1, 65, 300, 700], table="perm", seed=131),
    "mla_lq2": lambda: fp8_case(B=3, Lq=2, H=128, seq_lens=[2, 64, 129], table="perm", seed=132),
    "gla_small": lambda: fp8_case(B=2, Lq=1, H=128, G=2, seq_lens=[100, 513], table="perm", seed=133),
    "h16_lq2": lambda: fp8_case(B=3, Lq=2, H=16, seq_lens=[3, 190, 64], table="perm", seed=134),
    "gla4": lambda: fp8_case(B=2, Lq=1, H=128, G=4, seq_lens=[100, 513], table="perm", seed=137),
    "gla8_h64_lq2": lambda: fp8_case(B=3, Lq=2, H=64, G=8, seq_lens=[2, 190, 700], table="perm", seed=138),
    "mla_lq4_h32": lambda: fp8_case(B=2, Lq=4, H=32, seq_lens=[4, 333], table="perm", seed=140),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_fp8_decode_step_matches_oracle(name):
    c = SMALL[name]()
    got = run_gpu(c)
    assert got["status"] == 0
    heads = None if c.dims["H"] <= 32 else 10
    check_case(c, got, sample_pairs(c, heads))


@pytest.mark.parametrize("B,Lq,G,launches", [(448, 2, 1, 1), (449, 1, 1, 2), (353, 1, 2, 2)])
def test_fp8_large_batch(B, Lq, G, launches):
    """The in-kernel split at its largest batch and the plan kernel above it."""
    rng = np.random.default_rng(B + 1000)
    lens = [int(x) for x in rng.integers(Lq, 200, size=B)]
    lens[0], lens[-1] = Lq, 64
    c = fp8_case(B=B, Lq=Lq, H=16, G=G, seq_lens=lens, table="perm", seed=147 + B)
    assert mla.mla_decode_kernel_launches(c.dims) == launches
    got = run_gpu(c)
    assert got["status"] == 0
    check_case(c, got, [(b, h) for b in range(B) for h in (0, 7, 15)])


def test_fp8_dsv3_full_size_sampled():
    """DeepSeek-V3 dims (B=16, 4096 tokens each, 128 heads), the launch the
    benchmark times, on sampled (sequence, head) pairs."""
    c = workload("dsv3", kv="fp8")
    got = run_gpu(c)
    assert got["status"] == 0
    check_case(c, got, sample_pairs(c, 2, seqs=[0, 7, 15]))


FINITE = [k for k in range(256) if k not in (0x7F, 0xFF)]
SCALES = [2.0 ** -15, 2.0 ** -9, 2.0 ** -3, 1.0, 2.0 ** 7]


def one_token_case(G, H, seed):
    """Sequences of one token whose cache row runs through every finite E4M3
    code (subnormals and signed zero included) with the extreme scales of the
    exact range, [2^-15, 2^7]."""
    B = 10
    c = fp8_case(B=B, Lq=1, H=H, G=G, seq_lens=[1] * B, table="perm", seed=seed)
    for b in range(B):
        codes = torch.tensor([FINITE[(37 * b + i) % len(FINITE)] for i in range(512)], dtype=torch.uint8)
        scales = torch.tensor([SCALES[(b + j) % len(SCALES)] for j in range(4)], dtype=torch.float32)
        page = int(c.block_table[b, 0])
        rope = c.cache[page, 0, 512:640].clone().view(torch.bfloat16)
        c.cache[page, 0] = fp8_rows(codes, rope, scales)
    return c


@pytest.mark.parametrize("G,H", [(1, 16), (1, 128), (2, 128), (8, 64)])
def test_fp8_dequantisation_is_exact(G, H):
    c = one_token_case(G, H, seed=150 + G)
    got = run_gpu(c)
    assert got["status"] == 0
    lat, _ = oracle.dequant_fp8(c.cache)
    d_g = 512 // G
    for b in range(c.dims["B"]):
        page = int(c.block_table[b, 0])
        for h in range(H):
            g = h * G // H
            want = lat[page, 0, g * d_g:(g + 1) * d_g]
            have = got["o_lat"][b, 0, h].to(torch.float64).numpy()
            assert np.array_equal(have, want), "b=%d h=%d: %d of %d differ" % (b, h, np.sum(have != want), d_g)
    pairs = [(b, h) for b in range(c.dims["B"]) for h in (0, H - 1)]
    _, _, ref_lse = oracle.decode_fp8(c.dims, **c.tensors(), sel=pairs)
    bi, hi = np.array([p[0] for p in pairs]), np.array([p[1] for p in pairs])
    assert_close(got["lse"].to(torch.float64).numpy()[bi, :, hi], ref_lse[bi, :, hi], "lse")


@pytest.mark.parametrize("G", [1, 2])
def test_fp8_scale_range(G):
    """Scales of 0 (a zero-filled row) past a sequence's end: fine, outputs
    as the oracle's.  A scale above 2^7 overflows the f16 operands, on a
    token of a sequence or on a row past its end (that row enters the
    products with weight 0, and 0 * inf is NaN): MLA_ERR_RANGE."""
    c = fp8_case(B=2, Lq=1, H=128, G=G, seq_lens=[70, 100], table="perm", seed=160 + G)
    page = int(c.block_table[1, 1])  # tokens 64..127 of sequence 1: rows 0..35 in the sequence

    def set_scale(row, j, value):
        rows = c.cache[page].clone()
        sc = rows[:, 640:656].clone().view(torch.float32)
        sc[row, j] = value
        rows[:, 640:656] = sc.view(torch.uint8)
        c.cache[page] = rows

    for row in range(36, 64):
        for j in range(4):
            set_scale(row, j, 0.0)
    got = run_gpu(c)
    assert got["status"] == 0
    check_case(c, got, [(b, h) for b in range(2) for h in (0, 63, 64, 127)])
    set_scale(50, 2, 2.0 ** 9)  # token 114: past the end
    assert run_gpu(c)["status"] == MLA_ERR_RANGE
    set_scale(50, 2, 0.0)
    set_scale(20, 1, 2.0 ** 8)  # token 84: in the sequence
    assert run_gpu(c)["status"] == MLA_ERR_RANGE


def test_fp8_query_beyond_f16_range_sets_status():
    c = fp8_case(B=2, Lq=1, H=128, seq_lens=[70, 100], table="perm", seed=170)
    q_cat = torch.randn(2, 1, 128, 576, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    assert run_decode_only(c, q_cat)["status"] == 0
    q_cat[1, 0, 5, 300] = 7.0e4
    assert run_decode_only(c, q_cat)["status"] == MLA_ERR_RANGE


def test_fp8_decode_from_given_query_matches_latent_oracle():
    """mla_decode_paged_fp8 + mla_combine_splits on a given q_cat against the
    oracle's latent-space decode over the same FP8 cache."""
    c = fp8_case(B=3, Lq=2, H=128, seq_lens=[2, 500, 1300], table="perm", seed=171)
    q_cat = (torch.randn(3, 2, 128, 576, generator=torch.Generator().manual_seed(4)) * 0.5).to(torch.bfloat16)
    got = run_decode_only(c, q_cat)
    assert got["status"] == 0
    pairs = sample_pairs(c, 12)
    ref_lat, ref_lse = oracle.decode_latent_fp8(c.dims, q_cat, c.cache, c.block_table, c.seq_lens, sel=pairs)
    bi, hi = np.array([p[0] for p in pairs]), np.array([p[1] for p in pairs])
    assert_close(got["o_lat"].to(torch.float64).numpy()[bi, :, hi], ref_lat[bi, :, hi], "o_lat")
    assert_close(got["lse"].to(torch.float64).numpy()[bi, :, hi], ref_lse[bi, :, hi], "lse")


def test_fp8_bad_table_entry_sets_status_without_fault():
    c = fp8_case(B=2, Lq=1, H=16, seq_lens=[70, 150], table="perm", seed=172)
    c.block_table[1, 2] = c.dims["num_pages"] + 3
    assert run_gpu(c)["status"] == -6  # MLA_ERR_BAD_TABLE

"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, per step and end to end, plus invariants of the split-KV
machinery and the device status word."""
import math

import numpy as np
import pytest
import torch

import mla_latent_kv_10_gb300 as mla
import oracle
from mla_latent_kv_10_gb300.inputs import make_case, workload
from parity_util import assert_close, check_case, run_gpu, sample_pairs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_latent_kv_10_gb300 import _build
    _build.build()
    mla.load_library()


# ---------------------------------------------------------------- step: absorb

@pytest.mark.parametrize("B,Lq,H,G", [(2, 1, 16, 1), (16, 1, 128, 1), (64, 2, 128, 1), (3, 2, 128, 2),
                                      (130, 1, 16, 1)])
def test_absorb_q_matches_oracle(B, Lq, H, G):
    c = make_case(B=B, Lq=Lq, H=H, G=G, seq_lens=[1] * B, seed=100 + B)
    d_g = 512 // G
    q_cat = torch.empty(B, Lq, H, d_g + 64, dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_q(c.dims, c.q_nope.cuda(), c.q_rope.cuda(), c.W_UK.cuda(), q_cat)
    torch.cuda.synchronize()
    ref = oracle.absorb(c.q_nope, c.W_UK)
    got = q_cat.cpu()
    assert_close(got[..., :d_g], ref, "q_abs")
    # per-element: one bf16 rounding of an fp32 sum
    err = np.abs(got[..., :d_g].double().numpy() - ref)
    assert np.all(err <= 2.0 ** -7 * np.abs(ref) + 1e-3)
    assert torch.equal(got[..., d_g:], c.q_rope)


# ---------------------------------------------------------------- step: project

@pytest.mark.parametrize("B,Lq,H,G", [(2, 1, 16, 1), (16, 1, 128, 1), (64, 2, 128, 1), (5, 1, 128, 2)])
def test_project_uv_matches_oracle(B, Lq, H, G):
    c = make_case(B=B, Lq=Lq, H=H, G=G, seq_lens=[1] * B, seed=200 + B)
    d_g = 512 // G
    gen = torch.Generator().manual_seed(7)
    o_lat = torch.randn(B, Lq, H, d_g, generator=gen).to(torch.bfloat16)
    out = torch.empty(B, Lq, H, 128, dtype=torch.bfloat16, device="cuda")
    mla.mla_project_uv(c.dims, o_lat.cuda(), c.W_UV.cuda(), out)
    torch.cuda.synchronize()
    ref = oracle.project_uv(o_lat, c.W_UV)
    assert_close(out.cpu(), ref, "out")


# ---------------------------------------------------------------- end to end, small

SMALL = {
    "tiny": lambda: workload("tiny"),
    "mla_ragged": lambda: make_case(B=4, Lq=1, H=128, seq_lens=[1, 65, 300, 700], table="perm", seed=31),
    "mla_lq2": lambda: make_case(B=3, Lq=2, H=128, seq_lens=[2, 64, 129], table="perm", seed=32),
    "gla_small": lambda: make_case(B=2, Lq=1, H=128, G=2, seq_lens=[100, 513], table="perm", seed=33),
    "h16_lq2": lambda: make_case(B=3, Lq=2, H=16, seq_lens=[3, 190, 64], table="perm", seed=34),
    "h64": lambda: make_case(B=2, Lq=1, H=64, seq_lens=[77, 128], table="contig", seed=35),
    "gla_h32_lq2": lambda: make_case(B=2, Lq=2, H=32, G=2, seq_lens=[45, 260], table="perm", seed=36),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_step_small(name):
    c = SMALL[name]()
    got = run_gpu(c)
    assert got["status"] == 0
    heads = None if c.dims["H"] <= 32 else 10
    check_case(c, got, sample_pairs(c, heads))


@pytest.mark.parametrize("B,Lq,launches", [(448, 2, 1), (449, 2, 2), (600, 1, 2)])
def test_decode_large_batch(B, Lq, launches):
    """Batches at the largest size the decode kernel splits by itself (448),
    just above it and well above it (split by the separate plan kernel):
    ragged lengths, shuffled pages, every sequence checked on a few heads."""
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(Lq, 200, size=B)]
    lens[0], lens[-1] = Lq, 64
    c = make_case(B=B, Lq=Lq, H=16, seq_lens=lens, table="perm", seed=47 + B)
    assert mla.mla_decode_kernel_launches(c.dims) == launches
    got = run_gpu(c)
    assert got["status"] == 0
    pairs = [(b, h) for b in range(B) for h in (0, 7, 15)]
    check_case(c, got, pairs)


@pytest.mark.parametrize("splits", [1, 3, 7])
def test_split_count_invariance(splits):
    """Any number of work units gives the same result (fp32 merge order
    aside) as the automatic split."""
    c = make_case(B=3, Lq=2, H=128, seq_lens=[300, 2, 1000], table="perm", seed=41)
    auto = run_gpu(c)
    got = run_gpu(c, num_splits=splits)
    assert got["status"] == 0
    assert_close(got["o_lat"], auto["o_lat"], "o_lat", rel=1e-2, cos=0.99999)
    np.testing.assert_allclose(got["lse"].numpy(), auto["lse"].numpy(), rtol=0, atol=1e-3)


def test_single_key_closed_form_on_gpu():
    """n = 1: the latent output is exactly the one cache row (rounded to
    bf16), lse is its score."""
    c = make_case(B=5, Lq=1, H=128, seq_lens=[1] * 5, table="perm", seed=42)
    got = run_gpu(c)
    for b in range(5):
        row = c.cache[int(c.block_table[b, 0]), 0, :512]
        assert torch.equal(got["o_lat"][b, 0], row.expand(128, 512))


def test_zero_query_uniform_mean_on_gpu():
    """q = 0: uniform weights over exactly n keys, lse = log n (masking of the
    ragged last page and the causal window)."""
    c = make_case(B=3, Lq=2, H=16, seq_lens=[65, 3, 200], table="perm", seed=43, q_zero=True)
    got = run_gpu(c)
    for b, n in enumerate([65, 3, 200]):
        for l in range(2):
            assert np.allclose(got["lse"][b, l].numpy(), math.log(n - 1 + l), atol=1e-4)
    check_case(c, got, sample_pairs(c))


def test_page_permutation_invariance_on_gpu():
    c = make_case(B=2, Lq=1, H=128, seq_lens=[333, 64], table="contig", seed=44)
    a = run_gpu(c)
    perm = torch.randperm(c.dims["num_pages"], generator=torch.Generator().manual_seed(1))
    cache2 = torch.empty_like(c.cache)
    cache2[perm] = c.cache
    bt2 = c.block_table.clone()
    m = bt2 >= 0
    bt2[m] = perm.to(torch.int32)[bt2[m].long()]
    c.cache, c.block_table = cache2, bt2
    b = run_gpu(c)
    assert torch.equal(a["o_lat"], b["o_lat"]) and torch.equal(a["lse"], b["lse"])


# ---------------------------------------------------------------- device status

def test_bad_table_entry_sets_status_without_fault():
    c = make_case(B=2, Lq=1, H=16, seq_lens=[70, 10], table="perm", seed=45)
    c.block_table[0, 1] = c.dims["num_pages"] + 5      # out of range: clamped, reported
    got = run_gpu(c)
    assert got["status"] == -6


def test_bad_seq_len_sets_status_without_fault():
    c = make_case(B=2, Lq=2, H=16, seq_lens=[70, 10], table="perm", seed=46)
    c.seq_lens[1] = 1                                  # fewer keys than new tokens
    got = run_gpu(c)
    assert got["status"] == -8
    c = make_case(B=2, Lq=1, H=16, seq_lens=[70, 10], table="perm", seed=46)
    c.seq_lens[0] = 10 ** 6                            # more than the table can hold
    got = run_gpu(c)
    assert got["status"] == -8

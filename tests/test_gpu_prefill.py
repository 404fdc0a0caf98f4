"""The decompress branch (long query chunks) against the fp64 oracle.

mla_decompress_kv expands the latent cache into per-head keys and values;
mla_prefill_attend runs causal attention of the Lq new tokens over them.
Their result is the oracle's non-absorbed decode ("path A" of the MLA
operator write-up §4) for the same inputs, for any Lq: out and lse are
compared on sampled (sequence, head) pairs at the tolerance of the decode
path (max|err| <= 2e-2 max|ref|, cosine >= 0.9999)."""
import numpy as np
import pytest
import torch

import mla_latent_kv_10_gb300 as mla
import oracle
from mla_latent_kv_10_gb300.inputs import make_case
from parity_util import assert_close, sample_pairs

pytestmark = pytest.mark.gpu


def run_prefill(c, device="cuda"):
    t = {k: v.to(device) for k, v in c.tensors().items()}
    bufs = mla.PrefillBuffers(c.dims, device)
    mla.prefill_step(c.dims, bufs, t["q_nope"], t["q_rope"], t["W_UK"], t["W_UV"], t["cache"], t["block_table"],
                     t["seq_lens"])
    status = mla.mla_get_device_status(bufs.workspace)
    return dict(status=status, out=bufs.out.cpu(), lse=bufs.lse.cpu(), k_nope=bufs.k_nope.cpu(), v=bufs.v.cpu())


def gathered_latents(c, b, g):
    """Cache rows of sequence b's tokens, latent of group g: [n, d_g] bf16."""
    d = c.dims
    d_g = d["d_c"] // d["G"]
    n = int(c.seq_lens[b])
    pages = c.block_table[b, : (n + 63) // 64].tolist()
    rows = torch.cat([c.cache[p] for p in pages], 0)[:n]
    return rows[:, g * d_g:(g + 1) * d_g].contiguous()


@pytest.mark.parametrize("G,H", [(1, 16), (2, 32), (8, 16)])
def test_decompress_matches_the_up_projections(G, H):
    """k_nope[b,h,s] = W_UK[h] . c_g(h)[s] and v[b,h,s] = W_UV[h] . c_g(h)[s]
    (the oracle's projection routine on the gathered rows), zeros on the
    rest of each sequence's last page."""
    c = make_case(B=2, Lq=1, H=H, G=G, seq_lens=[70, 200], table="perm", seed=71 + G)
    got = run_prefill(c)
    assert got["status"] == 0
    d = c.dims
    for b in range(2):
        n = int(c.seq_lens[b])
        for h in (0, H // 2 - 1, H // 2, H - 1):
            g = h * G // H
            lat = gathered_latents(c, b, g)                      # [n, d_g]
            o = lat[:, None, :].expand(n, 1, lat.shape[1]).contiguous()
            for name, W in (("k_nope", c.W_UK), ("v", c.W_UV)):
                ref = oracle.project_uv(o, W[h:h + 1])[:, 0, :]  # [n, 128]
                assert_close(got[name][b, h, :n], ref, "%s b=%d h=%d" % (name, b, h))
            tail = ((n + 63) // 64) * 64
            assert torch.all(got["k_nope"][b, :, n:tail] == 0) and torch.all(got["v"][b, :, n:tail] == 0)


CASES = {
    # Lq new tokens at the end of each sequence; query blocks of 128 rows with a ragged tail
    "lq130_full": dict(B=2, Lq=130, H=16, G=1, seq_lens=[130, 700], table="perm", seed=81),
    "lq256_gla": dict(B=1, Lq=256, H=32, G=2, seq_lens=[600], table="perm", seed=82),
    "lq300_h128": dict(B=1, Lq=300, H=128, G=1, seq_lens=[1000], table="perm", seed=83),
    "lq5_short": dict(B=3, Lq=5, H=16, G=1, seq_lens=[5, 64, 333], table="perm", seed=84),
    "lq200_gla4": dict(B=2, Lq=200, H=64, G=4, seq_lens=[260, 520], table="perm", seed=85),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_matches_oracle(name):
    c = make_case(**CASES[name])
    got = run_prefill(c)
    assert got["status"] == 0
    heads = None if c.dims["H"] <= 16 else 6
    pairs = sample_pairs(c, heads)
    ref_out, _, ref_lse = oracle.decode(c.dims, **c.tensors(), sel=pairs)
    bi = np.array([p[0] for p in pairs])
    hi = np.array([p[1] for p in pairs])
    assert_close(got["out"].to(torch.float64).numpy()[bi, :, hi], ref_out[bi, :, hi], name + " out")
    assert_close(got["lse"].to(torch.float64).numpy()[bi, :, hi], ref_lse[bi, :, hi], name + " lse")


def test_prefill_one_key_closed_form():
    """The first new token of a sequence of exactly Lq tokens sees one key:
    its output is v of key 0 (up to one bf16 rounding of the weight sum's
    reciprocal), its lse the scaled score of that key."""
    c = make_case(B=1, Lq=140, H=16, seq_lens=[140], table="perm", seed=86)
    got = run_prefill(c)
    assert got["status"] == 0
    v0 = got["v"][0, :, 0].to(torch.float64)                    # [H, 128]
    assert_close(got["out"][0, 0].to(torch.float64).numpy(), v0.numpy(), "out of one key", rel=2 ** -8)
    ref_out, _, ref_lse = oracle.decode(c.dims, **c.tensors(), sel=[(0, h) for h in range(16)])
    assert_close(got["lse"][0, 0].to(torch.float64).numpy(), ref_lse[0, 0], "lse of one key")


def test_prefill_bad_table_entry_sets_status_without_fault():
    c = make_case(B=2, Lq=70, H=16, seq_lens=[70, 150], table="perm", seed=87)
    c.block_table[1, 1] = c.dims["num_pages"] + 5
    got = run_prefill(c)
    assert got["status"] == -6  # MLA_ERR_BAD_TABLE

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
from parity_util import assert_close, check_case, run_decode_only, run_gpu, sample_pairs, scaled_queries

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_latent_kv_10_gb300 import _build
    _build.build()
    mla.load_library()


# ---------------------------------------------------------------- step: absorb

@pytest.mark.parametrize("B,Lq,H,G", [(2, 1, 16, 1), (16, 1, 128, 1), (64, 2, 128, 1), (3, 2, 128, 2),
                                      (130, 1, 16, 1), (5, 4, 128, 4), (3, 3, 64, 8)])
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

@pytest.mark.parametrize("B,Lq,H,G", [(2, 1, 16, 1), (16, 1, 128, 1), (64, 2, 128, 1), (5, 1, 128, 2),
                                      (4, 4, 128, 4), (3, 2, 64, 8), (130, 1, 16, 1), (67, 2, 16, 2)])
def test_project_uv_matches_oracle(B, Lq, H, G):
    """Query rows: a few (one 16-row MMA), 128 (the W_UV ring refilled
    through fewer slots than chunks) and more than 128 (a second, ragged
    row block)."""
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
    "gla4": lambda: make_case(B=2, Lq=1, H=128, G=4, seq_lens=[100, 513], table="perm", seed=37),
    "gla8_h64_lq2": lambda: make_case(B=3, Lq=2, H=64, G=8, seq_lens=[2, 190, 700], table="perm", seed=38),
    "mla_lq3": lambda: make_case(B=3, Lq=3, H=128, seq_lens=[3, 64, 200], table="perm", seed=39),
    "mla_lq4_h32": lambda: make_case(B=2, Lq=4, H=32, seq_lens=[4, 333], table="perm", seed=40),
    "gla4_lq4": lambda: make_case(B=2, Lq=4, H=128, G=4, seq_lens=[260, 1100], table="perm", seed=41),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_step_small(name):
    c = SMALL[name]()
    got = run_gpu(c)
    assert got["status"] == 0
    heads = None if c.dims["H"] <= 32 else 10
    check_case(c, got, sample_pairs(c, heads))


@pytest.mark.parametrize("B,Lq,G,launches", [(448, 2, 1, 1), (449, 2, 1, 2), (600, 1, 1, 2),
                                             (352, 1, 2, 1), (353, 2, 2, 2)])
def test_decode_large_batch(B, Lq, G, launches):
    """Batches at the largest size the decode kernel splits by itself (448
    for one latent group, 352 for grouped latents, whose kernel has fewer
    threads), just above it and well above it (split by the separate plan
    kernel): ragged lengths, shuffled pages, every sequence checked on a few
    heads of both latent halves."""
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(Lq, 200, size=B)]
    lens[0], lens[-1] = Lq, 64
    c = make_case(B=B, Lq=Lq, H=16, G=G, seq_lens=lens, table="perm", seed=47 + B)
    assert mla.mla_decode_kernel_launches(c.dims) == launches
    got = run_gpu(c)
    assert got["status"] == 0
    pairs = [(b, h) for b in range(B) for h in (0, 7, 15)]
    check_case(c, got, pairs)


def _expected_split(lens, Lq, units):
    """The work split restated from its rule: pages per sequence; the
    balanced cut (equal contiguous ranges of the flattened page list, cost =
    pages per unit + 4 per extra sequence a unit touches) against the
    sequence-aligned one (units shared out in proportion to pages, cost =
    most pages a unit gets); the cheaper one, ties to sequence-aligned."""
    nps = [(max(n, Lq, 1) + 63) // 64 for n in lens]
    off = np.concatenate([[0], np.cumsum(nps)]).astype(np.int64)
    B, total = len(lens), int(off[-1])
    chunk = -(-total // units)
    segs = 1
    for k in range(units):
        st, en = min(k * chunk, total), min(k * chunk + chunk, total)
        if st < en:
            segs = max(segs, int(np.sum((off[:-1] < en) & (off[1:] > st))))
    cost_bal = chunk + 4 * (segs - 1)
    u = [min(n, max(1, units * n // total)) for n in nps]
    worst = max(-(-n // x) for n, x in zip(nps, u))
    cost_al = worst if (B <= units and sum(u) <= units) else math.inf
    mode = 1 if cost_al <= cost_bal else 0
    if mode == 1:
        slot0, nslot = list(np.concatenate([[0], np.cumsum(u)[:-1]])), u
    else:
        kf = [int(off[b]) // chunk for b in range(B)]
        kl = [(int(off[b]) + nps[b] - 1) // chunk for b in range(B)]
        slot0, nslot = [b + kf[b] for b in range(B)], [kl[b] - kf[b] + 1 for b in range(B)]
    return dict(total=total, chunk=chunk, mode=mode, off=list(off), slot0=slot0, nslot=nslot)


@pytest.mark.parametrize("B", [32, 33])
@pytest.mark.parametrize("mix", ["skew", "one_long"])
def test_split_matches_rule(B, mix):
    """The split the decode kernel writes to the workspace (one planning warp
    up to 32 sequences, the whole block above) against the rule restated in
    Python; the outputs against the oracle on a few heads."""
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(1, 3000, size=B)] if mix == "skew" else [64] * (B - 1) + [20000]
    c = make_case(B=B, Lq=1, H=16, seq_lens=lens, table="perm", seed=60 + B)
    t = {k: v.cuda() for k, v in c.tensors().items()}
    bufs = mla.DecodeBuffers(c.dims)
    mla.decode_step(c.dims, bufs, t["q_nope"], t["q_rope"], t["W_UK"], t["W_UV"], t["cache"],
                    t["block_table"], t["seq_lens"])
    assert mla.mla_get_device_status(bufs.workspace) == 0
    ws = bufs.workspace.cpu().view(torch.int32).numpy()
    status, total, chunk, units, wB, mode = ws[:6]
    assert wB == B
    want = _expected_split(lens, 1, int(units))
    assert (total, chunk, mode) == (want["total"], want["chunk"], want["mode"])
    body = ws[8:]
    assert list(body[:B + 1]) == want["off"]
    assert list(body[B + 1:2 * B + 1]) == lens
    assert list(body[2 * B + 1:3 * B + 1]) == want["slot0"]
    assert list(body[3 * B + 1:4 * B + 1]) == want["nslot"]
    got = dict(o_lat=bufs.o_lat.cpu(), lse=bufs.lse.cpu(), out=bufs.out.cpu())
    check_case(c, got, [(b, h) for b in (0, B // 2, B - 1) for h in (0, 15)])


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


# ---------------------------------------------------------------- large logits

@pytest.mark.parametrize("mag", [4.0, 8.0])
@pytest.mark.parametrize("name", ["tiny", "mla_three_seqs"])
def test_large_logits_end_to_end(name, mag):
    """Queries scaled x4 and x8 before the bf16 rounding (scores in the tens
    to hundreds): the whole step still matches the fp64 non-absorbed oracle.
    (At x32 the bf16 absorbed query alone leaves the tolerance; the oracle's
    own pins show that, and the decode is checked there from a given q_cat.)"""
    c = workload("tiny") if name == "tiny" else make_case(
        B=3, Lq=1, H=128, seq_lens=[4096, 1500, 333], table="perm", seed=91)
    got = run_gpu(scaled_queries(c, mag))
    assert got["status"] == 0
    heads = None if c.dims["H"] <= 32 else 8
    errs = check_case(c, got, sample_pairs(c, heads))
    print(name, mag, {k: "%.2e" % v for k, v in errs.items()})


@pytest.mark.parametrize("mag", [1.0, 16.0, 64.0])
@pytest.mark.parametrize("shape", ["mla_lq2", "gla", "gla8_lq4"])
def test_decode_from_large_query_matches_latent_oracle(shape, mag):
    """The decode step alone on a q_cat drawn directly with element scale
    `mag` (x64: scores hundreds of nats apart): o_lat and lse against the
    oracle's latent-space decode from the same q_cat.  The two CTAs of a pair
    exchange partial scores as 16-bit fixed point scaled per row, so the
    error stays at the level of the bf16 weights P whatever the logit
    scale."""
    if shape == "mla_lq2":
        c = make_case(B=3, Lq=2, H=128, seq_lens=[4096, 700, 66], table="perm", seed=92)
    elif shape == "gla8_lq4":
        c = make_case(B=2, Lq=4, H=128, G=8, seq_lens=[1500, 4], table="perm", seed=97)
    else:
        c = make_case(B=2, Lq=1, H=128, G=2, seq_lens=[4096, 513], table="perm", seed=93)
    d = c.dims
    d_g = 512 // d["G"]
    gen = torch.Generator().manual_seed(int(mag) + 5)
    q_cat = (torch.randn(d["B"], d["Lq"], d["H"], d_g + 64, generator=gen) * mag).to(torch.bfloat16)
    got = run_decode_only(c, q_cat)
    assert got["status"] == 0
    pairs = sample_pairs(c, 10)
    ref_lat, ref_lse = oracle.decode_latent(d, q_cat, c.cache, c.block_table, c.seq_lens, sel=pairs)
    bi = np.array([p[0] for p in pairs])
    hi = np.array([p[1] for p in pairs])
    e = assert_close(got["o_lat"].to(torch.float64).numpy()[bi, :, hi], ref_lat[bi, :, hi], "o_lat")
    gl, rl = got["lse"].to(torch.float64).numpy()[bi, :, hi], ref_lse[bi, :, hi]
    # lse per element: the peer's partial crosses the pair in 16-bit fixed
    # point (step 2^-14 of the row's largest partial, which can exceed the
    # total score when the halves cancel), so each score, and the
    # log-sum-exp, may move by a few 1e-5 of the scores' scale
    assert_close(gl, rl, "lse")
    assert np.all(np.abs(gl - rl) <= 1e-4 * np.abs(rl).max() + 2e-3), np.abs(gl - rl).max()
    print(shape, mag, "o_lat %.2e" % e, "lse %.2e" % np.abs(gl - rl).max())


# ---------------------------------------------------------------- many partials per sequence

@pytest.mark.parametrize("B,Lq,H,lens", [(1, 1, 16, [20000]), (2, 1, 128, [30000, 100])])
def test_combine_with_more_than_64_partials(B, Lq, H, lens):
    """A sequence split over more than 64 work units: the combine takes its
    path without the per-CTA weight table (log-sum-exps read again from
    memory); checked against the oracle."""
    c = make_case(B=B, Lq=Lq, H=H, seq_lens=lens, table="perm", seed=94 + B)
    t = {k: v.cuda() for k, v in c.tensors().items()}
    bufs = mla.DecodeBuffers(c.dims)
    mla.decode_step(c.dims, bufs, t["q_nope"], t["q_rope"], t["W_UK"], t["W_UV"], t["cache"],
                    t["block_table"], t["seq_lens"])
    assert mla.mla_get_device_status(bufs.workspace) == 0
    ws = bufs.workspace.cpu().view(torch.int32).numpy()
    nslot = ws[8 + 3 * B + 1: 8 + 4 * B + 1]
    if int(ws[3]) <= 64:
        pytest.skip("this GPU has %d work units; the case needs more than 64" % int(ws[3]))
    assert nslot[0] > 64, nslot
    got = dict(o_lat=bufs.o_lat.cpu(), lse=bufs.lse.cpu(), out=bufs.out.cpu())
    check_case(c, got, sample_pairs(c, 6))



# ---------------------------------------------------------------- fused combine + project

@pytest.mark.parametrize("name", list(SMALL))
def test_fused_combine_project_matches_two_calls_and_oracle(name):
    """mla_combine_project gives exactly what mla_combine_splits followed by
    mla_project_uv gives (same merge order, same bf16 rounding of o_lat, same
    MMA), and so matches the oracle."""
    c = SMALL[name]()
    two = run_gpu(c)
    one = run_gpu(c, fused=True)
    assert one["status"] == 0
    assert torch.equal(one["o_lat"], two["o_lat"])
    assert torch.equal(one["lse"], two["lse"])
    assert torch.equal(one["out"], two["out"])
    heads = None if c.dims["H"] <= 32 else 10
    check_case(c, one, sample_pairs(c, heads))


def test_fused_combine_project_without_optional_outputs():
    """o_lat and lse are optional outputs of the fused call."""
    c = make_case(B=3, Lq=2, H=128, seq_lens=[300, 2, 1000], table="perm", seed=48)
    ref = run_gpu(c, fused=True)
    t = {k: v.cuda() for k, v in c.tensors().items()}
    bufs = mla.DecodeBuffers(c.dims)
    mla.mla_absorb_q(c.dims, t["q_nope"], t["q_rope"], t["W_UK"], bufs.q_cat)
    mla.mla_decode_paged(c.dims, bufs.q_cat, t["cache"], t["block_table"], t["seq_lens"], 0,
                         bufs.o_part, bufs.lse_part, bufs.workspace)
    mla.mla_combine_project(c.dims, bufs.o_part, bufs.lse_part, bufs.workspace, t["W_UV"], bufs.out)
    assert mla.mla_get_device_status(bufs.workspace) == 0
    assert torch.equal(bufs.out.cpu(), ref["out"])


# ---------------------------------------------------------------- cache rows past a sequence's end

def _fill_tails(c, value=None, seed=0):
    """Fill every cache row past a sequence's end on its last page: with
    `value`, or (value None) with stale rows of another part of the cache,
    as a page pool that is reused would hold."""
    gen = torch.Generator().manual_seed(seed)
    for b in range(c.dims["B"]):
        n = int(c.seq_lens[b])
        if n % 64:
            page = int(c.block_table[b, (n - 1) // 64])
            if value is None:
                src = torch.randint(0, c.dims["num_pages"], (64 - n % 64,), generator=gen)
                c.cache[page, n % 64:, :] = c.cache[src, torch.arange(64 - n % 64) % 64, :]
            else:
                c.cache[page, n % 64:, :] = value


def _tail_case(shape):
    if shape == "mla":
        return make_case(B=3, Lq=1, H=128, seq_lens=[70, 1, 333], table="perm", seed=61)
    if shape == "mla_lq2":
        return make_case(B=2, Lq=2, H=64, seq_lens=[130, 7], table="perm", seed=62)
    return make_case(B=2, Lq=1, H=128, G=2, seq_lens=[100, 513], table="perm", seed=63)


@pytest.mark.parametrize("shape", ["mla", "mla_lq2", "gla"])
def test_decode_with_stale_rows_past_sequence_end(shape):
    """The decode reads whole pages: rows past a sequence's end take part in
    the MMAs (masked, weight 0).  With stale rows there (a reused page pool)
    the results match the oracle, which reads only the sequence's own rows.
    (Such rows must hold finite values of the cache's usual size: a NaN
    there would reach O through 0 * NaN, and a huge value would set the
    16-bit exchange's row scale.)"""
    c = _tail_case(shape)
    _fill_tails(c, None, seed=5)
    got = run_gpu(c)
    assert got["status"] == 0
    check_case(c, got, sample_pairs(c, 8))


@pytest.mark.parametrize("value", [float("nan"), 3e38, -3e38])
@pytest.mark.parametrize("shape", ["mla", "mla_lq2", "gla"])
def test_decompress_branch_ignores_anything_past_sequence_end(shape, value):
    """The decompress branch writes zeros for K and V past a sequence's end
    and masks those scores, so even NaN or huge values in the cache rows
    there leave out and lse equal to the oracle's."""
    c = _tail_case(shape)
    _fill_tails(c, value)
    t = {k: v.cuda() for k, v in c.tensors().items()}
    bufs = mla.PrefillBuffers(c.dims)
    mla.prefill_step(c.dims, bufs, t["q_nope"], t["q_rope"], t["W_UK"], t["W_UV"], t["cache"], t["block_table"],
                     t["seq_lens"])
    assert mla.mla_get_device_status(bufs.workspace) == 0
    pairs = sample_pairs(c, 8)
    ref_out, _, ref_lse = oracle.decode(c.dims, **c.tensors(), sel=pairs)
    bi = np.array([p[0] for p in pairs])
    hi = np.array([p[1] for p in pairs])
    assert_close(bufs.out.cpu().to(torch.float64).numpy()[bi, :, hi], ref_out[bi, :, hi], "prefill out")
    assert_close(bufs.lse.cpu().to(torch.float64).numpy()[bi, :, hi], ref_lse[bi, :, hi], "prefill lse")


@pytest.mark.parametrize("kv,fused", [("bf16", False), ("bf16", True), ("fp8", False)])
def test_one_call_step_equals_the_separate_calls(kv, fused):
    """mla_decode_step launches the same kernels as the four calls (three
    with the fused merge), so its outputs are bit-equal; the second round
    runs on other buffers of the same dims, so the tensor maps the library
    remembers must follow the buffers."""
    c = make_case(B=3, Lq=2, H=128, seq_lens=[2, 300, 900], table="perm", seed=191, kv=kv)
    fp8 = kv == "fp8"
    for _ in range(2):
        t = {k: v.cuda() for k, v in c.tensors().items()}
        one = mla.DecodeBuffers(c.dims, "cuda")
        sep = mla.DecodeBuffers(c.dims, "cuda")
        mla.mla_decode_step(c.dims, t["q_nope"], t["q_rope"], t["W_UK"], t["W_UV"], t["cache"], fp8, t["block_table"],
                            t["seq_lens"], one.q_cat, one.o_part, one.lse_part, one.workspace, one.o_lat, one.lse,
                            one.out, fused)
        mla.mla_absorb_q(c.dims, t["q_nope"], t["q_rope"], t["W_UK"], sep.q_cat)
        decode = mla.mla_decode_paged_fp8 if fp8 else mla.mla_decode_paged
        decode(c.dims, sep.q_cat, t["cache"], t["block_table"], t["seq_lens"], 0, sep.o_part, sep.lse_part,
               sep.workspace)
        if fused:
            mla.mla_combine_project(c.dims, sep.o_part, sep.lse_part, sep.workspace, t["W_UV"], sep.out, sep.o_lat,
                                    sep.lse)
        else:
            mla.mla_combine_splits(c.dims, sep.o_part, sep.lse_part, sep.workspace, sep.o_lat, sep.lse)
            mla.mla_project_uv(c.dims, sep.o_lat, t["W_UV"], sep.out)
        assert mla.mla_get_device_status(one.workspace) == 0 and mla.mla_get_device_status(sep.workspace) == 0
        for name in ("q_cat", "o_lat", "lse", "out"):
            assert torch.equal(getattr(one, name), getattr(sep, name)), name
    got = dict(o_lat=one.o_lat.cpu(), lse=one.lse.cpu(), out=one.out.cpu())
    check_case(c, got, sample_pairs(c, 8))

"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI, compare with the oracle under the stated tolerance.

Tolerance (bf16 inputs, fp32 accumulation): max|err| <= 2e-2 * max|ref| and
cosine similarity >= 0.9999, per compared tensor.
"""
import numpy as np
import torch

import mla_latent_kv_10_gb300 as mla
import oracle

REL_MAX = 2e-2
COS_MIN = 0.9999


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def assert_close(got, ref, what, rel=REL_MAX, cos=COS_MIN):
    g, r = to64(got).ravel(), to64(ref).ravel()
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), "%s: non-finite values" % what
    scale = np.max(np.abs(r))
    err = np.max(np.abs(g - r))
    assert err <= rel * scale, "%s: max|err| %.3e > %.1e * max|ref| %.3e" % (what, err, rel, scale)
    denom = np.linalg.norm(g) * np.linalg.norm(r)
    if denom > 0:
        c = float(np.dot(g, r) / denom)
        assert c >= cos, "%s: cosine %.7f < %.5f" % (what, c, cos)
    return err / max(scale, 1e-300)


def is_fp8(case):
    return case.meta.get("kv") == "fp8"


def run_gpu(case, num_splits=0, device="cuda", fused=False):
    """Upload a case, run the four entry points (or three, with the fused
    combine + project; the FP8 decode for an FP8 cache), return host copies."""
    t = {k: v.to(device) for k, v in case.tensors().items()}
    bufs = mla.DecodeBuffers(case.dims, device)
    mla.decode_step(case.dims, bufs, t["q_nope"], t["q_rope"], t["W_UK"], t["W_UV"], t["cache"],
                    t["block_table"], t["seq_lens"], num_splits=num_splits, fused=fused, fp8=is_fp8(case))
    status = mla.mla_get_device_status(bufs.workspace)
    torch.cuda.synchronize()
    return dict(q_cat=bufs.q_cat.cpu(), o_lat=bufs.o_lat.cpu(), lse=bufs.lse.cpu(), out=bufs.out.cpu(),
                status=status, slots=bufs.slots)


def sample_pairs(case, heads_per_seq=None, seqs=None):
    B, H = case.dims["B"], case.dims["H"]
    bs = range(B) if seqs is None else seqs
    if heads_per_seq is None:
        return [(b, h) for b in bs for h in range(H)]
    rng = np.random.default_rng(case.meta.get("seed", 0))
    pairs = []
    for b in bs:
        hs = sorted(set([0, H - 1, H // 2 - 1, H // 2] + list(rng.choice(H, heads_per_seq, replace=False))))
        pairs += [(b, int(h)) for h in hs]
    return pairs


def check_case(case, got, pairs, nthreads=0):
    """Compare o_lat, lse, out of the selected (b, h) pairs with the oracle."""
    ref_decode = oracle.decode_fp8 if is_fp8(case) else oracle.decode
    ref_out, ref_lat, ref_lse = ref_decode(case.dims, **case.tensors(), sel=pairs, nthreads=nthreads)
    bi = np.array([p[0] for p in pairs])
    hi = np.array([p[1] for p in pairs])
    errs = {}
    errs["o_lat"] = assert_close(got["o_lat"].to(torch.float64).numpy()[bi, :, hi], ref_lat[bi, :, hi], "o_lat")
    errs["lse"] = assert_close(got["lse"].to(torch.float64).numpy()[bi, :, hi], ref_lse[bi, :, hi], "lse")
    errs["out"] = assert_close(got["out"].to(torch.float64).numpy()[bi, :, hi], ref_out[bi, :, hi], "out")
    return errs


def run_decode_only(case, q_cat, num_splits=0, device="cuda"):
    """mla_decode_paged + mla_combine_splits on a given q_cat (bf16
    [B,Lq,H,d_g+64]); returns host copies of o_lat, lse and the status."""
    t = {k: v.to(device) for k, v in case.tensors().items()}
    bufs = mla.DecodeBuffers(case.dims, device)
    bufs.q_cat.copy_(q_cat.to(device))
    decode = mla.mla_decode_paged_fp8 if is_fp8(case) else mla.mla_decode_paged
    decode(case.dims, bufs.q_cat, t["cache"], t["block_table"], t["seq_lens"], num_splits, bufs.o_part,
           bufs.lse_part, bufs.workspace)
    mla.mla_combine_splits(case.dims, bufs.o_part, bufs.lse_part, bufs.workspace, bufs.o_lat, bufs.lse)
    status = mla.mla_get_device_status(bufs.workspace)
    torch.cuda.synchronize()
    return dict(o_lat=bufs.o_lat.cpu(), lse=bufs.lse.cpu(), status=status,
                ws=bufs.workspace.cpu().view(torch.int32).numpy())


def scaled_queries(case, mag):
    """Scale q_nope and q_rope by `mag` (in fp64) and round to bf16 once:
    logits grow by mag (scores in the tens to hundreds)."""
    case.q_nope = (case.q_nope.double() * mag).to(torch.bfloat16)
    case.q_rope = (case.q_rope.double() * mag).to(torch.bfloat16)
    return case

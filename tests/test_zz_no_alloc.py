"""The allocation-free decode entry point (mla_decode_attend_noalloc).

It serves callers that cannot give the library scratch memory; it must give
the same result as the regular mla_decode_paged + mla_combine_splits pair, on
repeated calls (the fixed scratch array keeps the previous call's contents),
and refuse work that does not fit its fixed scratch.  Named to run last."""
import ctypes

import pytest
import torch

import mla_latent_kv_10_gb300 as mla
from mla_latent_kv_10_gb300.inputs import make_case, workload
from parity_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from mla_latent_kv_10_gb300 import _build
    _build.build()
    return mla.load_library()


def noalloc(lib, dims, q_cat, cache, bt, sl, o_lat, lse, status):
    f = lib.mla_decode_attend_noalloc
    f.argtypes = [ctypes.POINTER(mla.Dims)] + [ctypes.c_void_p] * 8
    f.restype = ctypes.c_int
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(ctypes.byref(mla.make_dims(dims)), p(q_cat), p(cache), p(bt), p(sl), p(o_lat), p(lse),
             p(status), stream)


CASES = {
    "dsv3": lambda: workload("dsv3"),
    "gla": lambda: workload("gla"),
    "lq2_ragged": lambda: make_case(B=3, Lq=2, H=128, seq_lens=[2, 700, 129], table="perm", seed=51),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_regular_entry_points(lib, name):
    c = CASES[name]()
    t = {k: v.cuda() for k, v in c.tensors().items()}
    bufs = mla.DecodeBuffers(c.dims)
    mla.mla_absorb_q(c.dims, t["q_nope"], t["q_rope"], t["W_UK"], bufs.q_cat)
    mla.mla_decode_paged(c.dims, bufs.q_cat, t["cache"], t["block_table"], t["seq_lens"], 0,
                         bufs.o_part, bufs.lse_part, bufs.workspace)
    mla.mla_combine_splits(c.dims, bufs.o_part, bufs.lse_part, bufs.workspace, bufs.o_lat, bufs.lse)
    assert mla.mla_get_device_status(bufs.workspace) == 0
    ref_lat, ref_lse = bufs.o_lat.clone(), bufs.lse.clone()
    for call in range(2):
        o_lat = torch.full_like(ref_lat, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
        rc = noalloc(lib, c.dims, bufs.q_cat, t["cache"], t["block_table"], t["seq_lens"], o_lat, lse, status)
        assert rc == 0, mla.mla_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(o_lat, ref_lat, "o_lat call %d" % call)
        assert_close(lse, ref_lse, "lse call %d" % call)


def test_noalloc_refuses_work_beyond_its_scratch(lib):
    c = make_case(B=1024, Lq=1, H=128, seq_lens=[64] * 1024, seed=52)
    dev = torch.empty(16, dtype=torch.uint8, device="cuda")   # never touched: refused before launch
    rc = noalloc(lib, c.dims, dev, dev, dev, dev, dev, None, None)
    assert rc == -4   # MLA_ERR_WORKSPACE


def test_noalloc_reports_device_errors_and_starts_clean(lib):
    """The fixed scratch keeps the last call's contents, so every call clears
    its status word: a call with an out-of-range block-table entry reports
    MLA_ERR_BAD_TABLE (the entry is clamped, never dereferenced), and the
    next clean call on the same scratch reports MLA_OK and matches the
    regular entry points.  A batch above the decode kernel's own planning
    limit (the plan kernel runs first) goes through the same scratch."""
    for c, bad in ((make_case(B=3, Lq=1, H=128, seq_lens=[70, 300, 5], table="perm", seed=53), True),
                   (make_case(B=449, Lq=1, H=16, seq_lens=[1 + (7 * i) % 190 for i in range(449)],
                              table="perm", seed=54), False)):
        t = {k: v.cuda() for k, v in c.tensors().items()}
        bufs = mla.DecodeBuffers(c.dims)
        mla.mla_absorb_q(c.dims, t["q_nope"], t["q_rope"], t["W_UK"], bufs.q_cat)
        status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
        o_lat = torch.empty_like(bufs.o_lat)
        lse = torch.empty_like(bufs.lse)
        if bad:
            bt = t["block_table"].clone()
            bt[1, 2] = c.dims["num_pages"] + 3
            assert noalloc(lib, c.dims, bufs.q_cat, t["cache"], bt, t["seq_lens"], o_lat, lse, status) == 0
            torch.cuda.synchronize()
            assert int(status.item()) == -6   # MLA_ERR_BAD_TABLE
        mla.mla_decode_paged(c.dims, bufs.q_cat, t["cache"], t["block_table"], t["seq_lens"], 0,
                             bufs.o_part, bufs.lse_part, bufs.workspace)
        mla.mla_combine_splits(c.dims, bufs.o_part, bufs.lse_part, bufs.workspace, bufs.o_lat, bufs.lse)
        assert mla.mla_get_device_status(bufs.workspace) == 0
        rc = noalloc(lib, c.dims, bufs.q_cat, t["cache"], t["block_table"], t["seq_lens"], o_lat, lse, status)
        assert rc == 0, mla.mla_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(o_lat, bufs.o_lat, "o_lat")
        assert_close(lse, bufs.lse, "lse")

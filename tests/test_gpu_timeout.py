"""The decode kernel's timeout path on the GPU, made to happen without a
fault: a testing hook shortens the limit of the waits between the kernel's
warps and makes the MMA-issuing thread of every CTA wait, before a chosen
page, on a barrier that nothing completes.  That wait gives up; the kernel
must record MLA_ERR_TIMEOUT, wait for the copies, MMAs and exchange stores
already in flight, free its tensor memory and return, leaving the context
usable: the next call on a fresh workspace matches the oracle."""
import pytest

import mla_latent_kv_10_gb300 as mla
from mla_latent_kv_10_gb300.inputs import make_case
from parity_util import check_case, run_gpu, sample_pairs

pytestmark = pytest.mark.gpu

MLA_ERR_TIMEOUT = -7


@pytest.fixture(scope="module", autouse=True)
def built():
    from mla_latent_kv_10_gb300 import _build
    _build.build()
    mla.load_library()
    yield
    mla.mla_set_timeout_test(0, -1)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("stall_page", [0, 2])
@pytest.mark.parametrize("Lq,G", [(1, 1), (2, 1), (4, 4)])
def test_wait_that_gives_up_sets_timeout_and_context_stays_usable(Lq, G, stall_page, kv):
    """Clusters of 2, 4 and 8 CTAs (one, two and four 128-row blocks), over
    the bf16 cache and over the FP8 cache (whose teardown also waits for the
    raw-slot copies)."""
    c = make_case(B=2, Lq=Lq, H=128, G=G, seq_lens=[700, 300], table="perm", seed=95 + Lq, kv=kv)
    mla.mla_set_timeout_test(50_000, stall_page)   # 50 us
    try:
        got = run_gpu(c, num_splits=2)
    finally:
        mla.mla_set_timeout_test(0, -1)
    assert got["status"] == MLA_ERR_TIMEOUT
    again = run_gpu(c, num_splits=2)
    assert again["status"] == 0
    check_case(c, again, sample_pairs(c, 6))


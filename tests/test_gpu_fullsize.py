"""Parity at the full workload sizes, in the launch configuration the
benchmark times (automatic split count), on sampled (sequence, head) pairs
that the oracle computes one by one."""
import pytest

from mla_latent_kv_10_gb300.inputs import workload
from parity_util import check_case, run_gpu, sample_pairs

pytestmark = pytest.mark.gpu

FULL = {
    # name: sequences sampled, extra random heads per sampled sequence
    "dsv3": ([0, 7, 15], 4),
    "long": ([0, 15], 2),
    "spec": ([0, 31, 63], 3),
    "gla": ([0, 31], 4),
}


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", list(FULL))
def test_full_size_workload(name, fused):
    case = workload(name)
    got = run_gpu(case, fused=fused)
    assert got["status"] == 0
    seqs, heads = FULL[name]
    errs = check_case(case, got, sample_pairs(case, heads, seqs))
    print(name, "fused" if fused else "", {k: "%.2e" % v for k, v in errs.items()})

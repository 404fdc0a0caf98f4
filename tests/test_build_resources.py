"""Compile-time resource checks of the hot-path CUDA kernels (no GPU): the
compiler's resource report (-Xptxas -v).  Register spills go to local memory,
which these kernels cannot afford (shared memory leaves almost no L1, so a
spill becomes an L2 round trip), and the decode kernel (480 threads for one
latent group, 352 for grouped latents) and the 512-thread combine kernel
must fit their one-CTA-per-SM budgets: four warps of an SM sub-partition
share its 64K registers.  The plan
kernel (one CTA, only for batches above the decode kernel's own planning
limit) is not on the hot path and is not checked."""
import os
import re
import shutil
import subprocess

import pytest

from mla_latent_kv_10_gb300 import _build

NVCC = _build.nvcc()
pytestmark = pytest.mark.skipif(shutil.which(NVCC) is None and not os.path.exists(NVCC), reason="nvcc not found")

ENTRY = re.compile(r"Compiling entry function '([^']+)'")
SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")
REGS = re.compile(r"Used (\d+) registers")
HOT = ("decode_kernel", "combine_kernel", "combine_project_kernel", "absorb_kernel", "project_kernel")


def resource_report(source, tmp_path):
    out = tmp_path / (os.path.basename(source) + ".cubin")
    flags = [f for f in _build.NVCC_FLAGS if f not in ("-Xcompiler", "-fPIC")]
    r = subprocess.run([NVCC, *flags, "-Xptxas", "-v", "-cubin", source, "-o", str(out)],
                       capture_output=True, text=True, check=True)
    kernels, name = {}, None
    for line in (r.stdout + r.stderr).splitlines():
        m = ENTRY.search(line)
        if m:
            name = m.group(1)
            kernels[name] = {}
            continue
        if name is None:
            continue
        m = SPILL.search(line)
        if m:
            kernels[name]["spill"] = int(m.group(1)) + int(m.group(2))
        m = REGS.search(line)
        if m:
            kernels[name]["regs"] = int(m.group(1))
    return kernels


@pytest.mark.parametrize("source,limits", [
    ("mla_decode.cu", {"decode_kernelILb0E": 128, "decode_kernelILb1E": 168,
                       "decode_kernelILb0ELb1E": 128, "decode_kernelILb1ELb1E": 168}),
    ("mla_combine.cu", {"combine_kernel": 128}),
    ("mla_gemm.cu", {}),
])
def test_hot_kernels_do_not_spill(source, limits, tmp_path):
    kernels = resource_report(os.path.join(_build.CSRC, source), tmp_path)
    kernels = {n: r for n, r in kernels.items() if any(k in n for k in HOT)}
    assert kernels, "no hot-path kernel entries in the compiler's report"
    for name, res in kernels.items():
        assert res.get("spill", 0) == 0, (name, res)
        for key, cap in limits.items():
            if key in name:
                assert res["regs"] <= cap, (name, res)
    for key in limits:
        assert any(key in n for n in kernels), key

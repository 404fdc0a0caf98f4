"""Host-only checks of the C ABI: the library builds, loads without a GPU,
exports every function include/mla.h declares, and rejects bad arguments
with the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest

import mla_latent_kv_10_gb300 as mla
from mla_latent_kv_10_gb300 import _build
from mla_latent_kv_10_gb300.inputs import workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mla.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_absorb_q", "mla_decode_paged", "mla_combine_splits", "mla_project_uv",
              "mla_decode_workspace_size", "mla_get_device_status", "mla_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert mla.mla_status_string(0) == "MLA_OK"
    assert mla.mla_status_string(-7) == "MLA_ERR_TIMEOUT"
    assert mla.mla_status_string(-6) == "MLA_ERR_BAD_TABLE"
    assert mla.mla_status_string(123) == "MLA_ERR_UNKNOWN"


def dims(**kw):
    d = dict(workload("tiny").dims)
    d.update(kw)
    return mla.make_dims(d)


P = ctypes.c_void_p
A16 = P(0x10000)      # aligned fake device addresses (never dereferenced)
A8 = P(0x10008)


def decode(lib, d, q=A16, cache=A16, bt=A16, sl=A16, splits=0, op=A16, lp=A16, ws=A16, wsb=1 << 20):
    return lib.mla_decode_paged(ctypes.byref(d), q, cache, bt, sl, splits, op, lp, ws, wsb, None)


def test_decode_rejects_bad_arguments(lib):
    d = dims()
    assert lib.mla_decode_paged(None, A16, A16, A16, A16, 0, A16, A16, A16, 4096, None) == -1
    assert decode(lib, d, q=None) == -1
    assert decode(lib, d, bt=None) == -1
    assert decode(lib, d, splits=-1) == -1
    assert decode(lib, d, ws=None) == -4
    assert decode(lib, d, wsb=8) == -4
    assert decode(lib, d, cache=A8) == -3
    assert decode(lib, d, q=A8) == -3
    assert decode(lib, d, op=A8) == -3
    # int32 and fp32 arrays need 4-byte alignment only
    assert decode(lib, d, bt=P(0x10002)) == -3
    assert decode(lib, d, sl=P(0x10001)) == -3
    assert decode(lib, d, lp=P(0x10002)) == -3


def test_fp8_decode_rejects_bad_arguments(lib):
    """mla_decode_paged_fp8 validates exactly as mla_decode_paged does."""
    def decode8(d, q=A16, cache=A16, bt=A16, sl=A16, splits=0, op=A16, lp=A16, ws=A16, wsb=1 << 20):
        return lib.mla_decode_paged_fp8(ctypes.byref(d), q, cache, bt, sl, splits, op, lp, ws, wsb, None)
    d = dims()
    assert lib.mla_decode_paged_fp8(None, A16, A16, A16, A16, 0, A16, A16, A16, 4096, None) == -1
    assert decode8(d, cache=None) == -1
    assert decode8(d, splits=-1) == -1
    assert decode8(d, wsb=8) == -4
    assert decode8(d, cache=A8) == -3
    assert decode8(d, q=A8) == -3
    assert decode8(d, lp=P(0x10002)) == -3
    for field, value in (("G", 3), ("Lq", 5), ("d_c", 256)):
        d = dims()
        setattr(d, field, value)
        assert decode8(d) == -2
    assert mla.mla_status_string(-9) == "MLA_ERR_RANGE"


def test_decode_step_checks_arguments_before_any_launch(lib):
    """mla_decode_step validates like the calls it chains: the first failing
    call's code comes back and nothing is launched (no GPU needed here)."""
    def step(d, q=A16, out=A16, o_lat=A16, fused=0, wsb=1 << 20, kv_fp8=0):
        return lib.mla_decode_step(ctypes.byref(d), q, A16, A16, A16, A16, kv_fp8, A16, A16, A16, A16, A16, A16,
                                   wsb, o_lat, None, out, fused, None)
    d = dims()
    assert step(d, out=None) == -1
    assert step(d, o_lat=None) == -1     # the two-call merge needs o_lat
    assert step(d, q=None) == -1         # absorb
    assert step(d, q=A8) == -3
    bad = dims()
    bad.G = 3
    assert step(bad) == -2
    assert step(bad, kv_fp8=1, fused=1, o_lat=None) == -2


def test_decode_rejects_index_overflow(lib):
    """Token and table indices are 32-bit on the device: dims whose cache rows
    or table entries would not fit are refused before any launch."""
    d = dims()
    d.num_pages = (1 << 31) // 64
    assert decode(lib, d) == -2
    d = dims()
    d.max_pages_per_seq = (1 << 31) // 64
    assert decode(lib, d) == -2


@pytest.mark.parametrize("field,value,code", [
    ("d_hc", 64, -2), ("d_c", 256, -2), ("d_R", 32, -2), ("page_size", 16, -2),
    ("G", 3, -2), ("G", 16, -2), ("Lq", 5, -2), ("H", 24, -2), ("H", 256, -2),
    ("B", 0, -1), ("num_pages", 0, -1), ("scale", 0.0, -1), ("scale", float("nan"), -1),
    ("max_pages_per_seq", 0, -1)])
def test_unsupported_or_invalid_dims(lib, field, value, code):
    d = dims()
    setattr(d, field, value)
    assert decode(lib, d) == code
    assert lib.mla_absorb_q(ctypes.byref(d), A16, A16, A16, A16, None) == code
    assert lib.mla_project_uv(ctypes.byref(d), A16, A16, A16, None) == code
    n = ctypes.c_size_t()
    assert lib.mla_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == code


def test_gemm_entry_points_check_pointers(lib):
    d = dims()
    assert lib.mla_absorb_q(ctypes.byref(d), None, A16, A16, A16, None) == -1
    assert lib.mla_absorb_q(ctypes.byref(d), A16, A16, A8, A16, None) == -3
    assert lib.mla_project_uv(ctypes.byref(d), A16, None, A16, None) == -1
    assert lib.mla_project_uv(ctypes.byref(d), A16, A16, A8, None) == -3
    assert lib.mla_combine_splits(ctypes.byref(d), A16, A16, None, 4096, A16, None, None) == -4
    assert lib.mla_combine_splits(ctypes.byref(d), None, A16, A16, 4096, A16, None, None) == -1
    assert lib.mla_get_device_status(None, None) == -1


def test_workspace_size_grows_with_batch(lib):
    a = mla.mla_decode_workspace_size(dims(B=2))
    b = mla.mla_decode_workspace_size(dims(B=5000))
    assert a >= 32 + 4 * 5 and a % 256 == 0
    assert b >= 32 + 4 * 10001 and b > a


def test_python_binding_raises_mla_error(lib):
    with pytest.raises(mla.MLAError) as e:
        mla.mla_decode_workspace_size(dims(G=3))
    assert e.value.code == -2


def test_timeout_test_hook_arguments(lib):
    """The testing hook of the decode kernel's timeout path validates its
    arguments on the host (no GPU needed) and restores the defaults."""
    assert lib.mla_set_timeout_test(-1, -1) == -1
    assert lib.mla_set_timeout_test(0, -2) == -1
    assert lib.mla_set_timeout_test(1000, 3) == 0
    assert lib.mla_set_timeout_test(0, -1) == 0


def prefill(lib, d, qn=A16, qr=A16, cache=A16, bt=A16, sl=A16, k=A16, v=A16, out=A16, lse=A16, ws=A16, wsb=32):
    return lib.mla_prefill_attend(ctypes.byref(d), qn, qr, cache, bt, sl, k, v, out, lse, ws, wsb, None)


def decompress(lib, d, cache=A16, bt=A16, sl=A16, wk=A16, wv=A16, k=A16, v=A16, ws=A16, wsb=32):
    return lib.mla_decompress_kv(ctypes.byref(d), cache, bt, sl, wk, wv, k, v, ws, wsb, None)


@pytest.mark.parametrize("field,value,code", [
    ("d_hc", 64, -2), ("G", 3, -2), ("H", 24, -2), ("B", 0, -1), ("Lq", 0, -1), ("scale", 0.0, -1),
    ("Lq", 1 << 20, -1)])  # more new tokens than the table can hold
def test_decompress_branch_checks_dims(lib, field, value, code):
    d = dims()
    setattr(d, field, value)
    n = ctypes.c_size_t()
    assert lib.mla_decompressed_kv_size(ctypes.byref(d), ctypes.byref(n)) == code
    assert decompress(lib, d) == code
    assert prefill(lib, d) == code


def test_decompress_branch_accepts_long_chunks_and_sizes_its_buffers(lib):
    """Lq beyond the decode's 4 is fine for the decompress branch, up to the
    cached length; each of k_nope and v holds B*H*max_pages*64*d_hc bf16."""
    d = dims(Lq=300, max_pages=8)
    n = ctypes.c_size_t()
    assert lib.mla_decompressed_kv_size(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value == d.B * d.H * 8 * 64 * 128 * 2
    assert mla.PREFILL_THRESHOLD == 256


def test_decompress_branch_checks_pointers_alignment_and_workspace(lib):
    d = dims(Lq=130, max_pages=4)
    assert decompress(lib, d, cache=None) == -1
    assert decompress(lib, d, k=A8) == -3
    assert decompress(lib, d, ws=None) == -4
    assert decompress(lib, d, wsb=16) == -4
    assert prefill(lib, d, lse=None) == -1
    assert prefill(lib, d, qn=A8) == -3
    assert prefill(lib, d, bt=P(0x10002)) == -3
    assert prefill(lib, d, wsb=8) == -4

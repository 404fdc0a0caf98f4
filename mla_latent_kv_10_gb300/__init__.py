"""MLA decode with matrix absorption over a paged latent KV cache, on GB300.

The compute lives in ``libmla.so`` (hand-written CUDA for sm_103a behind the
C ABI of ``include/mla.h``).  This package is its thin Python binding: the
functions below carry the C names, marshal torch tensors into pointers and
sizes, and raise ``MLAError`` on a non-zero status.  There is no fallback:
if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MLAError", "Dims", "load_library", "library_path",
    "mla_absorb_q", "mla_decode_paged", "mla_decode_paged_fp8", "mla_decode_step", "mla_combine_splits",
    "mla_project_uv", "mla_combine_project",
    "mla_decode_workspace_size", "mla_decode_num_slots", "mla_decode_kernel_launches",
    "launches_per_step", "mla_get_device_status", "mla_set_timeout_test",
    "mla_status_string", "make_dims", "DecodeBuffers", "decode_step",
    "mla_decompressed_kv_size", "mla_decompress_kv", "mla_prefill_attend", "PrefillBuffers", "prefill_step",
    "PREFILL_THRESHOLD",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libmla.so")


class MLAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (where, mla_status_string(code), code))


class Dims(ctypes.Structure):
    """Mirror of ``mla_dims``."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "Lq", "H", "d_hc", "d_c", "d_R", "G", "page_size", "max_pages_per_seq", "num_pages")] + [
        ("scale", ctypes.c_float), ("causal", ctypes.c_int)]


_lib = None
_STATUS = {0: "MLA_OK", -1: "MLA_ERR_INVALID_ARG", -2: "MLA_ERR_UNSUPPORTED", -3: "MLA_ERR_MISALIGNED",
           -4: "MLA_ERR_WORKSPACE", -5: "MLA_ERR_CUDA", -6: "MLA_ERR_BAD_TABLE",
           -7: "MLA_ERR_TIMEOUT", -8: "MLA_ERR_BAD_SEQLEN"}


def load_library():
    """Load libmla.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError("libmla.so is not built (run __graft_entry__.build()); "
                           "there is no fallback implementation")
    lib = ctypes.CDLL(library_path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    DP = ctypes.POINTER(Dims)
    sig = {
        "mla_absorb_q": [DP, P, P, P, P, P],
        "mla_decode_num_slots": [DP, ctypes.POINTER(I)],
        "mla_decode_kernel_launches": [DP, ctypes.POINTER(I)],
        "mla_decode_workspace_size": [DP, ctypes.POINTER(S)],
        "mla_decode_paged": [DP, P, P, P, P, I, P, P, P, S, P],
        "mla_decode_paged_fp8": [DP, P, P, P, P, I, P, P, P, S, P],
        "mla_decode_step": [DP, P, P, P, P, P, I, P, P, P, P, P, P, S, P, P, P, I, P],
        "mla_combine_splits": [DP, P, P, P, S, P, P, P],
        "mla_project_uv": [DP, P, P, P, P],
        "mla_combine_project": [DP, P, P, P, S, P, P, P, P, P],
        "mla_get_device_status": [P, P],
        "mla_set_timeout_test": [ctypes.c_longlong, I],
        "mla_decompressed_kv_size": [DP, ctypes.POINTER(S)],
        "mla_decompress_kv": [DP, P, P, P, P, P, P, P, P, S, P],
        "mla_prefill_attend": [DP, P, P, P, P, P, P, P, P, P, P, S, P],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = I
    lib.mla_status_string.argtypes = [I]
    lib.mla_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def mla_status_string(code: int) -> str:
    if _lib is not None:
        return _lib.mla_status_string(int(code)).decode()
    return _STATUS.get(int(code), "MLA_ERR_UNKNOWN")


def make_dims(d: dict) -> Dims:
    """dims dict (as produced by ``inputs.make_case``) -> ``mla_dims``."""
    return Dims(B=d["B"], Lq=d["Lq"], H=d["H"], d_hc=d["d_hc"], d_c=d["d_c"], d_R=d["d_R"],
                G=d["G"], page_size=d["page_size"], max_pages_per_seq=d["max_pages"],
                num_pages=d["num_pages"], scale=float(d["scale"]), causal=int(d.get("causal", 1)))


def _dims(d):
    return ctypes.byref(d if isinstance(d, Dims) else make_dims(d))


def _ptr(t):
    return None if t is None else t.data_ptr()  # an int: ctypes makes it a void*


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _check(rc, where):
    if rc != 0:
        raise MLAError(rc, where)


def mla_absorb_q(dims, q_nope, q_rope, W_UK, q_cat, stream=None):
    _check(load_library().mla_absorb_q(_dims(dims), _ptr(q_nope), _ptr(q_rope), _ptr(W_UK),
                                       _ptr(q_cat), _stream(stream)), "mla_absorb_q")


def mla_decode_workspace_size(dims) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().mla_decode_workspace_size(_dims(dims), ctypes.byref(n)), "mla_decode_workspace_size")
    return n.value


def mla_decode_num_slots(dims) -> int:
    n = ctypes.c_int(0)
    _check(load_library().mla_decode_num_slots(_dims(dims), ctypes.byref(n)), "mla_decode_num_slots")
    return n.value


def mla_decode_kernel_launches(dims) -> int:
    n = ctypes.c_int(0)
    _check(load_library().mla_decode_kernel_launches(_dims(dims), ctypes.byref(n)),
           "mla_decode_kernel_launches")
    return n.value


def launches_per_step(dims, fused=False) -> int:
    """Kernel launches of one decode_step: absorb, decode (+ plan), then
    combine and project (two) or the fused combine + project (one)."""
    return (2 if fused else 3) + mla_decode_kernel_launches(dims)


def mla_decode_paged(dims, q_cat, kv_cache, block_table, seq_lens, num_splits, o_part, lse_part,
                     workspace, stream=None):
    _check(load_library().mla_decode_paged(
        _dims(dims), _ptr(q_cat), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), int(num_splits),
        _ptr(o_part), _ptr(lse_part), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "mla_decode_paged")


def mla_decode_paged_fp8(dims, q_cat, kv_cache_fp8, block_table, seq_lens, num_splits, o_part, lse_part,
                         workspace, stream=None):
    """kv_cache_fp8: uint8 [num_pages, 64, 656] rows of 512 e4m3 codes, the
    bf16 RoPE key and four fp32 scales (see include/mla.h)."""
    _check(load_library().mla_decode_paged_fp8(
        _dims(dims), _ptr(q_cat), _ptr(kv_cache_fp8), _ptr(block_table), _ptr(seq_lens), int(num_splits),
        _ptr(o_part), _ptr(lse_part), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "mla_decode_paged_fp8")


def mla_decode_step(dims, q_nope, q_rope, W_UK, W_UV, kv_cache, kv_fp8, block_table, seq_lens, q_cat, o_part,
                    lse_part, workspace, o_lat, lse, out, fused=False, stream=None):
    """The whole decode step in one C call (absorb, decode over the bf16 or
    FP8 cache, merge and projection)."""
    _check(load_library().mla_decode_step(
        _dims(dims), _ptr(q_nope), _ptr(q_rope), _ptr(W_UK), _ptr(W_UV), _ptr(kv_cache), int(bool(kv_fp8)),
        _ptr(block_table), _ptr(seq_lens), _ptr(q_cat), _ptr(o_part), _ptr(lse_part), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o_lat), _ptr(lse), _ptr(out), int(bool(fused)),
        _stream(stream)), "mla_decode_step")


def mla_combine_splits(dims, o_part, lse_part, workspace, o_lat, lse=None, stream=None):
    _check(load_library().mla_combine_splits(
        _dims(dims), _ptr(o_part), _ptr(lse_part), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(o_lat), _ptr(lse), _stream(stream)),
        "mla_combine_splits")


def mla_project_uv(dims, o_lat, W_UV, out, stream=None):
    _check(load_library().mla_project_uv(_dims(dims), _ptr(o_lat), _ptr(W_UV), _ptr(out), _stream(stream)),
           "mla_project_uv")


def mla_set_timeout_test(wait_limit_ns: int, stall_page: int):
    """Testing hook of the decode kernel's timeout path (process-wide; 0, -1
    restores the defaults)."""
    _check(load_library().mla_set_timeout_test(int(wait_limit_ns), int(stall_page)), "mla_set_timeout_test")


def mla_combine_project(dims, o_part, lse_part, workspace, W_UV, out, o_lat=None, lse=None, stream=None):
    _check(load_library().mla_combine_project(
        _dims(dims), _ptr(o_part), _ptr(lse_part), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(W_UV), _ptr(out), _ptr(o_lat), _ptr(lse),
        _stream(stream)), "mla_combine_project")


def mla_get_device_status(workspace, stream=None) -> int:
    return load_library().mla_get_device_status(_ptr(workspace), _stream(stream))


class DecodeBuffers:
    """Device buffers of one decode step for fixed dims (torch allocations;
    the library itself never allocates)."""

    def __init__(self, dims: dict, device="cuda"):
        import torch
        self.dims = dict(dims)
        B, Lq, H, G = dims["B"], dims["Lq"], dims["H"], dims["G"]
        d_g = dims["d_c"] // G
        self.slots = mla_decode_num_slots(dims)
        rows = Lq * H
        self.q_cat = torch.empty(B, Lq, H, d_g + dims["d_R"], dtype=torch.bfloat16, device=device)
        self.o_part = torch.empty(self.slots, rows, dims["d_c"], dtype=torch.float32, device=device)
        self.lse_part = torch.empty(self.slots, rows, dtype=torch.float32, device=device)
        self.workspace = torch.zeros(mla_decode_workspace_size(dims), dtype=torch.uint8, device=device)
        self.o_lat = torch.empty(B, Lq, H, d_g, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(B, Lq, H, dtype=torch.float32, device=device)
        self.out = torch.empty(B, Lq, H, dims["d_hc"], dtype=torch.bfloat16, device=device)
        self.dims_c = make_dims(self.dims)  # the C struct of these dims, built once


def decode_step(dims, bufs: DecodeBuffers, q_nope, q_rope, W_UK, W_UV, cache, block_table, seq_lens,
                num_splits=0, stream=None, fused=False, fp8=False):
    """The whole hot path of one layer's decode step: absorb, paged decode,
    then combine and project (or, with ``fused``, the fused combine +
    project, which also writes o_lat and lse).  With ``fp8`` the cache is
    the FP8 layout of mla_decode_paged_fp8.  All tensors on the device;
    results land in ``bufs``."""
    if num_splits == 0:  # one C call for the whole step
        dc = bufs.dims_c if (dims is bufs.dims or dims == bufs.dims) else dims
        mla_decode_step(dc, q_nope, q_rope, W_UK, W_UV, cache, fp8, block_table, seq_lens, bufs.q_cat, bufs.o_part,
                        bufs.lse_part, bufs.workspace, bufs.o_lat, bufs.lse, bufs.out, fused, stream)
        return bufs.out
    mla_absorb_q(dims, q_nope, q_rope, W_UK, bufs.q_cat, stream)
    decode = mla_decode_paged_fp8 if fp8 else mla_decode_paged
    decode(dims, bufs.q_cat, cache, block_table, seq_lens, num_splits, bufs.o_part, bufs.lse_part,
           bufs.workspace, stream)
    if fused:
        mla_combine_project(dims, bufs.o_part, bufs.lse_part, bufs.workspace, W_UV, bufs.out, bufs.o_lat,
                            bufs.lse, stream)
    else:
        mla_combine_splits(dims, bufs.o_part, bufs.lse_part, bufs.workspace, bufs.o_lat, bufs.lse, stream)
        mla_project_uv(dims, bufs.o_lat, W_UV, bufs.out, stream)
    return bufs.out


PREFILL_THRESHOLD = 256  # mirror of MLA_PREFILL_THRESHOLD: from this many new tokens on, the decompress branch


def mla_decompressed_kv_size(dims) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().mla_decompressed_kv_size(_dims(dims), ctypes.byref(n)), "mla_decompressed_kv_size")
    return n.value


def mla_decompress_kv(dims, kv_cache, block_table, seq_lens, W_UK, W_UV, k_nope, v, workspace, stream=None):
    _check(load_library().mla_decompress_kv(
        _dims(dims), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), _ptr(W_UK), _ptr(W_UV), _ptr(k_nope),
        _ptr(v), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "mla_decompress_kv")


def mla_prefill_attend(dims, q_nope, q_rope, kv_cache, block_table, seq_lens, k_nope, v, out, lse, workspace,
                       stream=None):
    _check(load_library().mla_prefill_attend(
        _dims(dims), _ptr(q_nope), _ptr(q_rope), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), _ptr(k_nope),
        _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)), "mla_prefill_attend")


class PrefillBuffers:
    """Device buffers of the decompress branch for fixed dims (torch
    allocations; the library itself never allocates)."""

    def __init__(self, dims: dict, device="cuda"):
        import torch
        self.dims = dict(dims)
        B, Lq, H = dims["B"], dims["Lq"], dims["H"]
        S = dims["max_pages"] * dims["page_size"]
        assert mla_decompressed_kv_size(dims) == B * H * S * dims["d_hc"] * 2
        self.k_nope = torch.empty(B, H, S, dims["d_hc"], dtype=torch.bfloat16, device=device)
        self.v = torch.empty(B, H, S, dims["d_hc"], dtype=torch.bfloat16, device=device)
        self.out = torch.empty(B, Lq, H, dims["d_hc"], dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(B, Lq, H, dtype=torch.float32, device=device)
        self.workspace = torch.zeros(32, dtype=torch.uint8, device=device)  # the status word


def prefill_step(dims, bufs: PrefillBuffers, q_nope, q_rope, W_UK, W_UV, cache, block_table, seq_lens,
                 stream=None):
    """The decompress branch of one layer: per-head keys and values from the
    latent cache, then causal attention of the Lq new tokens over them."""
    mla_decompress_kv(dims, cache, block_table, seq_lens, W_UK, W_UV, bufs.k_nope, bufs.v, bufs.workspace, stream)
    mla_prefill_attend(dims, q_nope, q_rope, cache, block_table, seq_lens, bufs.k_nope, bufs.v, bufs.out, bufs.lse,
                       bufs.workspace, stream)

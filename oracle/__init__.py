"""ctypes wrapper of the fp64 CPU oracle (``oracle/mla_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline / reference legs, never by the library.
It shares no code with the CUDA path; both receive the same seeded inputs.

Inputs are bf16 torch tensors (any device; they are copied to host and their
raw 16-bit storage is handed to C) or uint16 numpy arrays holding bf16 bits.
Outputs are float64 numpy arrays.
"""
import ctypes
import math

import numpy as np

from .build import build_oracle

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        I, D = ctypes.c_int, ctypes.c_double
        lib.mla_oracle_decode.argtypes = [I] * 10 + [D, I] + [_u16p] * 5 + [_i32p] * 3 + [I] + [_f64p] * 3 + [I]
        lib.mla_oracle_decode.restype = I
        lib.mla_oracle_decode_latent.argtypes = [I] * 9 + [D, I] + [_u16p] * 2 + [_i32p] * 3 + [I] + [_f64p] * 2 + [I]
        lib.mla_oracle_decode_latent.restype = I
        lib.mla_oracle_scores_both.argtypes = [I] * 9 + [D] + [_u16p] * 4 + [_i32p] * 2 + [I] * 3 + [_f64p] * 2
        lib.mla_oracle_scores_both.restype = I
        lib.mla_oracle_absorb.argtypes = [I] * 4 + [_u16p] * 2 + [_f64p]
        lib.mla_oracle_project_uv.argtypes = [I] * 4 + [_u16p] * 2 + [_f64p]
        lib.mla_oracle_lse_merge.argtypes = [I] * 3 + [_f64p] * 4
        lib.mla_oracle_num_threads.restype = I
        lib.mla_oracle_e4m3.argtypes = [I]
        lib.mla_oracle_e4m3.restype = D
        lib.mla_oracle_dequant_fp8.argtypes = [ctypes.c_long, I, I, I, ctypes.POINTER(ctypes.c_uint8), _f64p]
        lib.mla_oracle_dequant_fp8.restype = I
        _lib = lib
    return _lib


def num_threads() -> int:
    return load().mla_oracle_num_threads()


def _bits(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous uint16 numpy array of bf16 bits."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.int32)
    return np.ascontiguousarray(x.detach().to("cpu").numpy(), dtype=np.int32)


def _p(a, t):
    return a.ctypes.data_as(t)


def decode(dims, q_nope, q_rope, W_UK, W_UV, cache, block_table, seq_lens,
           sel=None, nthreads=0):
    """Naive-path decode.  ``dims`` is a dict with B, Lq, H, d_hc, d_c, d_R, G,
    page_size, max_pages, num_pages, scale, causal.  ``sel`` is an optional
    list of (b, h) pairs; only those entries of the outputs are computed
    (others stay NaN).  Returns (out [B,Lq,H,d_hc], o_lat [B,Lq,H,d_g],
    lse [B,Lq,H]) as float64 arrays."""
    lib = load()
    B, Lq, H = dims["B"], dims["Lq"], dims["H"]
    d_hc, d_c, d_R, G = dims["d_hc"], dims["d_c"], dims["d_R"], dims["G"]
    d_g = d_c // G
    out = np.full((B, Lq, H, d_hc), np.nan)
    o_lat = np.full((B, Lq, H, d_g), np.nan)
    lse = np.full((B, Lq, H), np.nan)
    qn, qr, wk, wv, kc = map(_bits, (q_nope, q_rope, W_UK, W_UV, cache))
    bt, sl = _i32(block_table), _i32(seq_lens)
    if sel is None:
        selp, nsel = None, 0
    else:
        s = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
        selp, nsel = _p(s, _i32p), s.shape[0]
    rc = lib.mla_oracle_decode(
        B, Lq, H, d_hc, d_c, d_R, G, dims["page_size"], dims["max_pages"],
        dims["num_pages"], float(dims["scale"]), int(dims.get("causal", 1)),
        _p(qn, _u16p), _p(qr, _u16p), _p(wk, _u16p), _p(wv, _u16p), _p(kc, _u16p),
        _p(bt, _i32p), _p(sl, _i32p), selp, nsel,
        _p(out, _f64p), _p(o_lat, _f64p), _p(lse, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the inputs (seq_lens / block_table)")
    return out, o_lat, lse


def decode_latent(dims, q_cat, cache, block_table, seq_lens, sel=None, nthreads=0):
    """Latent-space decode from a given absorbed query q_cat [B,Lq,H,d_g+d_R]
    (bf16): the absorbed scores q_cat . [c_g | k_R] * scale through the
    softmax.  Returns (o_lat [B,Lq,H,d_g], lse [B,Lq,H]) as float64; with
    ``sel`` only those (b, h) pairs are computed (others stay NaN)."""
    lib = load()
    B, Lq, H = dims["B"], dims["Lq"], dims["H"]
    d_c, d_R, G = dims["d_c"], dims["d_R"], dims["G"]
    d_g = d_c // G
    o_lat = np.full((B, Lq, H, d_g), np.nan)
    lse = np.full((B, Lq, H), np.nan)
    qc, kc = _bits(q_cat), _bits(cache)
    assert qc.shape == (B, Lq, H, d_g + d_R), qc.shape
    bt, sl = _i32(block_table), _i32(seq_lens)
    if sel is None:
        selp, nsel = None, 0
    else:
        s = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
        selp, nsel = _p(s, _i32p), s.shape[0]
    rc = lib.mla_oracle_decode_latent(
        B, Lq, H, d_c, d_R, G, dims["page_size"], dims["max_pages"], dims["num_pages"],
        float(dims["scale"]), int(dims.get("causal", 1)), _p(qc, _u16p), _p(kc, _u16p),
        _p(bt, _i32p), _p(sl, _i32p), selp, nsel, _p(o_lat, _f64p), _p(lse, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the inputs (seq_lens / block_table)")
    return o_lat, lse


def scores_both(dims, q_nope, q_rope, W_UK, cache, block_table, seq_lens, b, l, h):
    """(naive, absorbed) scores of query row (b, l, h) over all seq_lens[b] keys."""
    lib = load()
    n = int(_i32(seq_lens)[b])
    sa, sb = np.empty(n), np.empty(n)
    qn, qr, wk, kc = map(_bits, (q_nope, q_rope, W_UK, cache))
    bt, sl = _i32(block_table), _i32(seq_lens)
    rc = lib.mla_oracle_scores_both(
        dims["B"], dims["Lq"], dims["H"], dims["d_hc"], dims["d_c"], dims["d_R"],
        dims["G"], dims["page_size"], dims["max_pages"], float(dims["scale"]),
        _p(qn, _u16p), _p(qr, _u16p), _p(wk, _u16p), _p(kc, _u16p),
        _p(bt, _i32p), _p(sl, _i32p), b, l, h, _p(sa, _f64p), _p(sb, _f64p))
    if rc != 0:
        raise ValueError("bad row index")
    return sa, sb


def absorb(q_nope, W_UK):
    """q_abs[..., h, :] = q_nope[..., h, :] . W_UK[h]; q_nope [..., H, d_hc]."""
    qn, wk = _bits(q_nope), _bits(W_UK)
    H, d_hc, d_g = wk.shape
    lead = qn.shape[:-2]
    R = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (H, d_g))
    load().mla_oracle_absorb(R, H, d_hc, d_g, _p(qn, _u16p), _p(wk, _u16p), _p(out, _f64p))
    return out


def project_uv(o_lat, W_UV):
    """out[..., h, :] = W_UV[h] . o_lat[..., h, :]; o_lat [..., H, d_g]."""
    ol, wv = _bits(o_lat), _bits(W_UV)
    H, d_hc, d_g = wv.shape
    lead = ol.shape[:-2]
    R = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (H, d_hc))
    load().mla_oracle_project_uv(R, H, d_hc, d_g, _p(ol, _u16p), _p(wv, _u16p), _p(out, _f64p))
    return out


def lse_merge(o_part, lse):
    """Merge partials o_part [S,R,D], lse [S,R] -> (o [R,D], L [R])."""
    o_part = np.ascontiguousarray(o_part, dtype=np.float64)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    S, R, D = o_part.shape
    o, L = np.empty((R, D)), np.empty(R)
    load().mla_oracle_lse_merge(S, R, D, _p(o_part, _f64p), _p(lse, _f64p), _p(o, _f64p), _p(L, _f64p))
    return o, L


def e4m3(code: int) -> float:
    """Value of one FP8 E4M3 code (OCP 8-bit floating point; NaN for 0x7f, 0xff)."""
    return load().mla_oracle_e4m3(int(code))


FP8_ROW_BYTES = 512 + 2 * 64 + 4 * 4  # 512 codes | 64 bf16 RoPE key | 4 fp32 scales


def dequant_fp8(cache8, d_c: int = 512, d_R: int = 64, blk: int = 128):
    """FP8 cache rows (uint8 tensor / array [..., 656]) -> (latent float64
    [..., d_c] = e4m3(code) * scale of the code's blk-column block, RoPE key
    as bf16 bits uint16 [..., d_R])."""
    a = cache8 if isinstance(cache8, np.ndarray) else cache8.detach().to("cpu").contiguous().numpy()
    a = np.ascontiguousarray(a, dtype=np.uint8)
    lead = a.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    assert a.shape[-1] == d_c + 2 * d_R + 4 * (d_c // blk), a.shape
    lat = np.empty(lead + (d_c,))
    rc = load().mla_oracle_dequant_fp8(n, d_c, d_R, blk, _p(a, ctypes.POINTER(ctypes.c_uint8)), _p(lat, _f64p))
    if rc != 0:
        raise ValueError("bad FP8 layout")
    rope = np.ascontiguousarray(a[..., d_c:d_c + 2 * d_R]).view(np.uint16)
    return lat, rope


def fp8_as_bf16_cache(cache8, d_c: int = 512, d_R: int = 64, blk: int = 128) -> np.ndarray:
    """The bf16 cache (bits, uint16 [..., d_c + d_R]) holding exactly the
    dequantised latent of an FP8 cache and its RoPE key.  Every E4M3 value
    times a power-of-two scale has at most 4 significant bits, so it is a
    bf16 value unless it leaves the bf16 range; this is checked, never
    rounded."""
    lat, rope = dequant_fp8(cache8, d_c, d_R, blk)
    f32 = lat.astype(np.float32)
    if not np.array_equal(f32.astype(np.float64), lat, equal_nan=True):
        raise ValueError("dequantised latent not exact in fp32")
    u = f32.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("dequantised latent not exact in bf16 (a scale outside the power-of-two range)")
    return np.ascontiguousarray(np.concatenate([(u >> 16).astype(np.uint16), rope], axis=-1))


def decode_fp8(dims, q_nope, q_rope, W_UK, W_UV, cache, block_table, seq_lens, sel=None, nthreads=0):
    """decode() over an FP8 cache (uint8 [num_pages, P, 656]): the attention
    of the dequantised latent, c = e4m3(code) * scale, and the bf16 RoPE key."""
    return decode(dims, q_nope, q_rope, W_UK, W_UV, fp8_as_bf16_cache(cache), block_table, seq_lens,
                  sel=sel, nthreads=nthreads)


def decode_latent_fp8(dims, q_cat, cache, block_table, seq_lens, sel=None, nthreads=0):
    """decode_latent() over an FP8 cache (uint8 [num_pages, P, 656])."""
    return decode_latent(dims, q_cat, fp8_as_bf16_cache(cache), block_table, seq_lens, sel=sel,
                         nthreads=nthreads)


def default_scale(d_hc: int = 128, d_R: int = 64) -> float:
    """(d_hc + d_R)^-1/2, the softmax scale of the §4 equivalence script."""
    return 1.0 / math.sqrt(d_hc + d_R)

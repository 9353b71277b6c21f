"""Oracle for the FP8-KV attention library -- TEST INFRASTRUCTURE ONLY.

A plain, slow, single-threaded CPU statement (C, fp64 attention) of what the
GPU path computes.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library itself never
does, and it shares no code with the CUDA path.

Functions take numpy arrays.  bf16 data is passed as its raw uint16 bit
patterns so that nothing is rounded on the way in.

Sources (page title, section):
  * "FP8 KV cache (fp8_kv, opt-in)", bullets "Storage" and "Math": e4m3 codes,
    one fp32 scale amax/448 per (token, KV head), attention over the
    dequantised cache with grouped-query heads and per-sequence lengths, and
    the error report ``fp8_kv_error``.
  * "03 · 8n — FA-style tiled prefill attention", sections 2.1 and 3.1: causal
    prefill masking by position and GQA slicing.
  * "FP8 KV attention: hardware paths and tile preparation", section "Measure
    block-scaled QK": MXFP8 keys, one E8M0 scale per 32-element block.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        c_dbl_p = ctypes.POINTER(ctypes.c_double)
        c_u8_p = ctypes.POINTER(ctypes.c_uint8)
        c_u16_p = ctypes.POINTER(ctypes.c_uint16)
        c_f32_p = ctypes.POINTER(ctypes.c_float)
        c_i32_p = ctypes.POINTER(ctypes.c_int32)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        lib.fp8kv_oracle_e4m3_decode.restype = ctypes.c_double
        lib.fp8kv_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fp8kv_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.fp8kv_oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fp8kv_oracle_e4m3_decode_n.argtypes = [c_u8_p, i64, c_dbl_p]
        lib.fp8kv_oracle_e4m3_encode_n.argtypes = [c_f32_p, i64, c_u8_p]
        lib.fp8kv_oracle_bf16_to_double.argtypes = [c_u16_p, i64, c_dbl_p]
        lib.fp8kv_oracle_quantize.argtypes = [c_u16_p, i64, i32, c_u8_p, c_f32_p]
        lib.fp8kv_oracle_dequantize.argtypes = [c_u8_p, c_f32_p, i64, i32, c_dbl_p]
        lib.fp8kv_oracle_mx_quantize.argtypes = [c_u16_p, i64, i32, c_u8_p, c_u8_p]
        lib.fp8kv_oracle_quantize_residual.argtypes = [c_u16_p, c_f32_p, i64, i32, i64, i32, c_u8_p, c_f32_p]
        c_i32_p = ctypes.POINTER(ctypes.c_int32)
        lib.fp8kv_oracle_rope_bias.argtypes = [c_f32_p, c_f32_p, c_f32_p, c_i32_p, i32, i64, i32, c_f32_p]
        lib.fp8kv_oracle_quantize_residual_rope.argtypes = [c_u16_p, c_f32_p, c_f32_p, c_f32_p, c_i32_p, i32, i64,
                                                            i32, c_u8_p, c_f32_p]
        lib.fp8kv_oracle_mx_dequantize.argtypes = [c_u8_p, c_u8_p, i64, i32, c_dbl_p]
        lib.fp8kv_oracle_gather_paged.restype = ctypes.c_int
        lib.fp8kv_oracle_gather_paged.argtypes = [
            c_u8_p, i32, i32, i32, i32, c_i32_p, i32, i32, i32, c_u8_p]
        lib.fp8kv_oracle_decode.argtypes = [
            c_dbl_p, c_dbl_p, c_dbl_p, c_i32_p, i32, i32, i32, i32, i32,
            ctypes.c_double, c_dbl_p]
        lib.fp8kv_oracle_prefill.argtypes = [
            c_dbl_p, c_dbl_p, c_dbl_p, i32, i32, i32, i32, i32, i32,
            ctypes.c_double, c_dbl_p]
        _lib = lib
    return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ e4m3 --

def e4m3_decode(codes):
    """fp64 value of each E4M3 code (NaN for S.1111.111)."""
    lib = _load()
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib.fp8kv_oracle_e4m3_decode_n(_ptr(codes, ctypes.c_uint8), codes.size,
                                   _ptr(out, ctypes.c_double))
    return out


def e4m3_encode(values):
    """E4M3 code of each fp32 value: RNE, satfinite, sign-preserving zero."""
    lib = _load()
    vals = _c(values, np.float32)
    out = np.empty(vals.shape, dtype=np.uint8)
    lib.fp8kv_oracle_e4m3_encode_n(_ptr(vals, ctypes.c_float), vals.size,
                                   _ptr(out, ctypes.c_uint8))
    return out


# -------------------------------------------------------------- quantise --

def bf16_to_double(x_bits):
    lib = _load()
    x = _c(x_bits, np.uint16)
    out = np.empty(x.shape, dtype=np.float64)
    lib.fp8kv_oracle_bf16_to_double(_ptr(x, ctypes.c_uint16), x.size,
                                    _ptr(out, ctypes.c_double))
    return out


def quantize(x_bits):
    """Rows of bf16 (uint16 bits, shape [..., D]) -> (codes u8 [..., D], scales f32 [...])."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    d = x.shape[-1]
    rows = x.size // d if d else 0
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    lib.fp8kv_oracle_quantize(_ptr(x, ctypes.c_uint16), rows, d,
                              _ptr(codes, ctypes.c_uint8),
                              _ptr(scales, ctypes.c_float))
    return codes, scales


def dequantize(codes, scales):
    """codes [..., D] and scales [...] -> fp64 values [..., D]."""
    lib = _load()
    c = _c(codes, np.uint8)
    s = _c(scales, np.float32)
    d = c.shape[-1]
    rows = c.size // d if d else 0
    assert s.size == rows
    out = np.empty(c.shape, dtype=np.float64)
    lib.fp8kv_oracle_dequantize(_ptr(c, ctypes.c_uint8), _ptr(s, ctypes.c_float),
                                rows, d, _ptr(out, ctypes.c_double))
    return out


# ------------------------------------------------------ pre-bias residual --

def quantize_residual(x_bits, bias):
    """Key rows [Hkv, T, D] (bf16 bits) and a per-KV-head fp32 bias [Hkv, D] ->
    codes and fp32 scales of the residual fp32(k) - bias ("Fused KV-cache
    quantization", section "Bias-aware symmetric FP8")."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    b = _c(bias, np.float32)
    heads, T, d = x.shape
    assert b.shape == (heads, d)
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    lib.fp8kv_oracle_quantize_residual(_ptr(x, ctypes.c_uint16), _ptr(b, ctypes.c_float), heads * T, heads, T, d,
                                       _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_float))
    return codes, scales


def residual_keys(codes, scales, bias):
    """The keys a residual cache represents: dequant(r) + bias, fp64 [Hkv, T, D]."""
    return dequantize(codes, scales) + np.asarray(bias, dtype=np.float64)[:, None, :]


# ---------------------------------------- rotated pre-bias residual (rotary) --

def rope_bias(bias, cos, sin, positions):
    """The rotated bias R_t b of every (KV head, token): bias [Hkv, D] fp32,
    cos and sin [P, D/2] fp32 (rotary tables, "rotate half" pairs i and
    i + D/2), positions [T] -> fp32 [Hkv, T, D], evaluated as the appender
    does ("Fused KV-cache quantization", section "Bias-aware symmetric FP8":
    a bias added before the rotary embedding moves with the key's position)."""
    lib = _load()
    b = _c(bias, np.float32)
    c = _c(cos, np.float32)
    s = _c(sin, np.float32)
    p = _c(positions, np.int32)
    heads, d = b.shape
    assert c.shape == s.shape and c.shape[1] == d // 2 and p.ndim == 1
    assert p.size == 0 or (p.min() >= 0 and p.max() < c.shape[0])
    out = np.empty((heads, p.size, d), dtype=np.float32)
    lib.fp8kv_oracle_rope_bias(_ptr(b, ctypes.c_float), _ptr(c, ctypes.c_float), _ptr(s, ctypes.c_float),
                               _ptr(p, ctypes.c_int32), heads, p.size, d, _ptr(out, ctypes.c_float))
    return out


def quantize_residual_rope(x_bits, bias, cos, sin, positions):
    """Key rows [Hkv, T, D] (bf16 bits) at positions [T] -> codes and fp32
    scales of the residual fp32(k) - R_t b (the per-row rule)."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    b = _c(bias, np.float32)
    c = _c(cos, np.float32)
    s = _c(sin, np.float32)
    p = _c(positions, np.int32)
    heads, T, d = x.shape
    assert b.shape == (heads, d) and p.shape == (T,) and d <= 512
    assert T == 0 or (p.min() >= 0 and p.max() < c.shape[0])
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1], dtype=np.float32)
    lib.fp8kv_oracle_quantize_residual_rope(_ptr(x, ctypes.c_uint16), _ptr(b, ctypes.c_float),
                                            _ptr(c, ctypes.c_float), _ptr(s, ctypes.c_float),
                                            _ptr(p, ctypes.c_int32), heads, T, d,
                                            _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_float))
    return codes, scales


def residual_rope_keys(codes, scales, rb):
    """The keys a rotated-residual cache represents: dequant(r) + R_t b, fp64."""
    return dequantize(codes, scales) + np.asarray(rb, dtype=np.float64)


# ----------------------------------------------------------------- MXFP8 --

def mx_quantize(x_bits):
    """Rows of bf16 bits [..., D] (D a multiple of 32) -> (codes u8 [..., D],
    E8M0 bytes u8 [..., D/32]): one power-of-two scale per 32-element block,
    the smallest with amax <= 448 * scale ("FP8 KV attention: hardware paths
    and tile preparation", section "Measure block-scaled QK")."""
    lib = _load()
    x = _c(x_bits, np.uint16)
    d = x.shape[-1]
    assert d % 32 == 0
    rows = x.size // d if d else 0
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1] + (d // 32,), dtype=np.uint8)
    lib.fp8kv_oracle_mx_quantize(_ptr(x, ctypes.c_uint16), rows, d,
                                 _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    return codes, scales


def mx_dequantize(codes, scales):
    """codes [..., D] and E8M0 bytes [..., D/32] -> fp64 values [..., D]."""
    lib = _load()
    c = _c(codes, np.uint8)
    s = _c(scales, np.uint8)
    d = c.shape[-1]
    rows = c.size // d if d else 0
    assert s.size == rows * (d // 32)
    out = np.empty(c.shape, dtype=np.float64)
    lib.fp8kv_oracle_mx_dequantize(_ptr(c, ctypes.c_uint8), _ptr(s, ctypes.c_uint8),
                                   rows, d, _ptr(out, ctypes.c_double))
    return out


# ----------------------------------------------------------------- paged --

def gather_paged(pool, page_table, b, n_tokens):
    """Sequence b of a paged pool [num_pages, heads, page_size, ...] in token
    order -> [heads, n_tokens, ...] (any element type; rows copied as bytes)."""
    lib = _load()
    pool = np.ascontiguousarray(pool)
    num_pages, heads, page_size = pool.shape[:3]
    row_shape = pool.shape[3:]
    row_bytes = int(np.prod(row_shape, dtype=np.int64)) * pool.itemsize
    pt = _c(page_table, np.int32)
    out = np.empty((heads, n_tokens) + row_shape, dtype=pool.dtype)
    rc = lib.fp8kv_oracle_gather_paged(
        _ptr(pool.view(np.uint8), ctypes.c_uint8), num_pages, heads, page_size,
        row_bytes, _ptr(pt, ctypes.c_int32), pt.shape[1], b, n_tokens,
        _ptr(out.view(np.uint8), ctypes.c_uint8))
    if rc != 0:
        raise ValueError("page table entry out of range")
    return out


# ------------------------------------------------------------- attention --

def decode_attention(q, k, v, seq_lens, sm_scale):
    """q [B,Hq,D], k/v [B,Hkv,Tmax,D] (fp64 values), seq_lens [B] -> o [B,Hq,D] fp64."""
    lib = _load()
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    sl = _c(seq_lens, np.int32)
    B, Hq, D = q.shape
    _, Hkv, Tmax, _ = k.shape
    assert k.shape == v.shape == (B, Hkv, Tmax, D) and Hq % Hkv == 0
    assert sl.shape == (B,) and int(sl.max(initial=0)) <= Tmax
    out = np.empty_like(q)
    lib.fp8kv_oracle_decode(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                            _ptr(v, ctypes.c_double), _ptr(sl, ctypes.c_int32),
                            B, Hq, Hkv, Tmax, D, float(sm_scale),
                            _ptr(out, ctypes.c_double))
    return out


def prefill_attention(q, k, v, pos0, sm_scale):
    """Causal prefill of one sequence: q [n_q,Hq,D], k/v [Hkv,Tk,D] (fp64),
    query i at position pos0+i attends keys 0..pos0+i -> o [n_q,Hq,D] fp64."""
    lib = _load()
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    v = _c(v, np.float64)
    n_q, Hq, D = q.shape
    Hkv, Tk, _ = k.shape
    assert k.shape == v.shape and Hq % Hkv == 0 and pos0 + n_q <= Tk
    out = np.empty_like(q)
    lib.fp8kv_oracle_prefill(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                             _ptr(v, ctypes.c_double), n_q, int(pos0), Hq, Hkv,
                             Tk, D, float(sm_scale), _ptr(out, ctypes.c_double))
    return out


def fp8_kv_error(q_bits, k_bits, v_bits, seq_lens, sm_scale):
    """Relative L2 change of decode attention when the bf16 K/V of a
    contiguous cache [B,Hkv,T,D] are replaced by their e4m3 round trip
    ("FP8 KV cache (fp8_kv, opt-in)", bullet "Math": report fp8_kv_error)."""
    q = bf16_to_double(q_bits)
    k = bf16_to_double(k_bits)
    v = bf16_to_double(v_bits)
    kc, ks = quantize(k_bits)
    vc, vs = quantize(v_bits)
    o_ref = decode_attention(q, k, v, seq_lens, sm_scale)
    o_fp8 = decode_attention(q, dequantize(kc, ks), dequantize(vc, vs),
                             seq_lens, sm_scale)
    return float(np.linalg.norm(o_fp8 - o_ref) / max(np.linalg.norm(o_ref), 1e-300))


def attention_gate(out, ref, rel_l2=1e-2, max_abs=2e-2, axis=-1):
    """The parity gate: per head, relative L2 <= rel_l2 and max-abs <= max_abs.

    ``out``/``ref`` are [..., D]-shaped arrays; the gate is evaluated for every
    row along ``axis`` (decode: one D-vector per (b, q head)).  A row whose
    reference norm is below 1e-6 is held to max-abs only.  Returns
    (ok, worst_rel_l2, worst_max_abs)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = out - ref
    num = np.sqrt((diff ** 2).sum(axis=axis))
    den = np.sqrt((ref ** 2).sum(axis=axis))
    rel = np.where(den < 1e-6, 0.0, num / np.maximum(den, 1e-300))
    mab = np.abs(diff).max(axis=axis) if diff.size else np.zeros(())
    ok = bool(np.all(rel <= rel_l2) and np.all(mab <= max_abs)
              and np.all(np.isfinite(out)))
    worst_rel = float(rel.max()) if rel.size else 0.0
    worst_abs = float(mab.max()) if np.size(mab) else 0.0
    return ok, worst_rel, worst_abs

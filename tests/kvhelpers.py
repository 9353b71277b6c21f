"""Test helpers: fill GPU caches through the C ABI from seeded synthetic
inputs, and compute oracle references from the same bf16 bits.

Nothing here does method arithmetic of its own: the GPU side calls the
library, the reference side calls the oracle."""
import math

import numpy as np
import torch

import oracle
from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk


def fill_cache(inp: synth.DecodeInputs, dtype: str, device="cuda", capacity=None, k_bias=None, rope=None):
    """Append every token of a decode workload into a new cache (contiguous or
    paged per the workload) through fp8kv_append.  Returns the cache.
    k_bias: optional [Hkv, D] fp32 device tensor (pre-bias residual keys);
    rope: optional (cos, sin) [P, D/2] fp32 device tensors (the bias turns
    with the key's position)."""
    spec = inp.spec
    B = inp.seq_lens.numel()
    rc, rs = rope if rope is not None else (None, None)
    if spec.page_size is None:
        cap = capacity or max(16, ((inp.max_len + 63) // 64) * 64)
        cache = fk.Fp8KVCache.contiguous(B, spec.kv_heads, spec.head_dim, cap, dtype, device, k_bias=k_bias,
                                         rope_cos=rc, rope_sin=rs)
    else:
        cache = fk.Fp8KVCache.paged(inp.page_table, inp.num_pages, spec.kv_heads, spec.head_dim,
                                    spec.page_size, dtype, device, k_bias=k_bias, rope_cos=rc, rope_sin=rs)
    lens = inp.seq_lens.to(torch.int64)
    if int(lens.sum()) == 0:
        return cache
    seq_idx = torch.repeat_interleave(torch.arange(B), lens).to(torch.int32)
    pos = torch.cat([torch.arange(int(n)) for n in lens]).to(torch.int32) if B else torch.zeros(0, dtype=torch.int32)
    fk.fp8kv_append(cache, inp.k.to(device).contiguous(), inp.v.to(device).contiguous(),
                    seq_idx.to(device), pos.to(device))
    return cache


def k_fp8(dtype: str) -> bool:
    """Whether the cache dtype stores K as e4m3 codes with a per-row scale."""
    return dtype in ("k8v8", "k8v16")


def v_fp8(dtype: str) -> bool:
    """Whether the cache dtype stores V as e4m3 codes (else bf16)."""
    return dtype in ("k8v8", "k16v8", "mxk8v8")


def seq_bits(inp: synth.DecodeInputs, which: str, b: int):
    """bf16 bits of sequence b's K or V rows, as [Hkv, T_b, D]."""
    t = inp.k if which == "k" else inp.v
    s, e = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
    return synth.bf16_bits(t[s:e]).transpose(1, 0, 2)


def oracle_kv(inp: synth.DecodeInputs, dtype: str, b: int, k_bias=None, rope=None):
    """fp64 K and V of sequence b as the cache holds them: e4m3 round trip
    for an FP8 side, the bf16 value for a bf16 side, dequant(residual) + bias
    for pre-bias residual keys (+ R_t bias with rotary tables rope = (cos,
    sin), numpy).  [Hkv, T_b, D]."""
    out = []
    for which, fp8 in (("k", k_fp8(dtype)), ("v", v_fp8(dtype))):
        bits = seq_bits(inp, which, b)
        if which == "k" and k_bias is not None and rope is not None:
            pos = np.arange(bits.shape[1], dtype=np.int32)
            c, s = oracle.quantize_residual_rope(bits, k_bias, rope[0], rope[1], pos)
            out.append(oracle.residual_rope_keys(c, s, oracle.rope_bias(k_bias, rope[0], rope[1], pos)))
        elif which == "k" and k_bias is not None:
            c, s = oracle.quantize_residual(bits, k_bias)
            out.append(oracle.residual_keys(c, s, k_bias))
        elif which == "k" and dtype == "mxk8v8":
            out.append(oracle.mx_dequantize(*oracle.mx_quantize(bits)))
        elif fp8:
            c, s = oracle.quantize(bits)
            out.append(oracle.dequantize(c, s))
        else:
            out.append(oracle.bf16_to_double(bits))
    return out


def oracle_decode(inp: synth.DecodeInputs, dtype: str, batch_ids, sm_scale=None, k_bias=None, rope=None):
    """Oracle decode outputs [len(batch_ids), Hq, D] for the listed sequences."""
    spec = inp.spec
    D = spec.head_dim
    sm = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    q_all = oracle.bf16_to_double(synth.bf16_bits(inp.q))
    res = []
    for b in batch_ids:
        T = int(inp.seq_lens[b])
        k, v = oracle_kv(inp, dtype, b, k_bias, rope)
        Tc = max(T, 1)
        kk = np.zeros((1, spec.kv_heads, Tc, D))
        vv = np.zeros((1, spec.kv_heads, Tc, D))
        kk[0, :, :T] = k
        vv[0, :, :T] = v
        res.append(oracle.decode_attention(q_all[b:b + 1], kk, vv, np.array([T], np.int32), sm)[0])
    return np.stack(res) if res else np.zeros((0, spec.q_heads, D))


def gpu_decode(inp, cache, num_splits=0, out_dtype=torch.float32, kernel="auto"):
    q = inp.q.to("cuda").contiguous()
    lens = inp.seq_lens.to("cuda")
    return fk.fp8kv_decode_attention(q, cache, lens, num_splits=num_splits, out_dtype=out_dtype,
                                     kernel=kernel)


def assert_gate(out, ref, what, rel_l2=1e-2, max_abs=2e-2):
    ok, rel, mab = oracle.attention_gate(out, ref, rel_l2, max_abs)
    assert ok, f"{what}: worst rel-L2 {rel:.3e}, worst max-abs {mab:.3e}"
    return rel, mab


def split_last_token(inp: synth.DecodeInputs):
    """The workload minus each sequence's last token, and those tokens."""
    lens = inp.seq_lens.to(torch.int64)
    last = (inp.cu_seqlens[1:] - 1).clamp(min=0)
    keep = torch.ones(int(inp.cu_seqlens[-1]), dtype=torch.bool)
    has = lens > 0
    keep[last[has]] = False
    prev = synth.DecodeInputs(inp.spec, inp.q, inp.k[keep.to(inp.k.device)], inp.v[keep.to(inp.v.device)],
                              (inp.seq_lens - has.to(torch.int32)).to(torch.int32),
                              torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(lens - has.to(torch.int64), 0)]),
                              inp.page_table, inp.num_pages)
    B, Hkv, D = len(lens), inp.spec.kv_heads, inp.spec.head_dim
    knew = torch.zeros(B, Hkv, D, dtype=torch.bfloat16, device=inp.k.device)
    vnew = torch.zeros_like(knew)
    knew[has.to(knew.device)] = inp.k[last[has].to(inp.k.device)]
    vnew[has.to(vnew.device)] = inp.v[last[has].to(inp.v.device)]
    return prev, knew, vnew

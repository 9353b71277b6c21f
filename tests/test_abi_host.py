"""Host-side checks of the C ABI and of the workload generator.  No GPU: the
library is loaded and its argument checks are exercised, but no kernel runs."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from fp8_quantized_kv_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8kv.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_quantized_kv_gb300 import build as kbuild
    from fp8_quantized_kv_gb300._lib import get_lib
    kbuild.build()
    return get_lib()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"FP8KV_API\s+[\w\s\*]+?\b(fp8kv_\w+)\s*\(", text)


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    from fp8_quantized_kv_gb300._lib import EXPORTS
    assert set(EXPORTS) == set(names)


def test_status_strings(lib):
    for s in range(7):
        assert lib.fp8kv_status_string(s)
    assert lib.fp8kv_status_string(99) == b"unknown status"


def _cache(**kw):
    from fp8_quantized_kv_gb300._lib import CacheStruct
    base = dict(dtype=0, layout=0, batch=16, kv_heads=2, head_dim=128, max_tokens=8192,
                k=0x1000, v=0x2000, k_scale=0x3000, v_scale=0x4000)
    base.update(kw)
    return CacheStruct(**base)


def test_argument_checks_return_before_any_launch(lib):
    # every case below is rejected on the host, before any CUDA call
    c = _cache()
    r = ctypes.byref
    assert lib.fp8kv_quantize(None, -1, 128, None, None, None) == 1
    assert lib.fp8kv_quantize(None, 10, 96, None, None, None) == 2
    assert lib.fp8kv_quantize(None, 10, 128, None, None, None) == 1
    assert lib.fp8kv_decode_attention(None, None, None, 16, 0.1, 0, 0, None, 0, None, 0, None) == 1
    bad_dim = _cache(head_dim=96)
    out = 0x6000        # never dereferenced: each call is rejected first
    assert lib.fp8kv_decode_attention(None, r(bad_dim), None, 16, 0.1, 0, 0, None, 0, out, 0, None) == 2
    assert lib.fp8kv_decode_attention(None, r(c), None, 15, 0.1, 0, 0, None, 0, out, 0, None) == 1
    assert lib.fp8kv_decode_attention(None, r(c), None, 16, 0.1, 0, 0, None, 0, out, 7, None) == 1
    assert lib.fp8kv_decode_attention(0x7000, r(c), 0x8000, 16, 0.1, 0, 0, None, 0, out, 0, None) == 3
    no_scale = _cache(k_scale=None)
    assert lib.fp8kv_decode_attention(None, r(no_scale), None, 16, 0.1, 0, 0, None, 0, out, 0, None) == 1
    odd_cap = _cache(max_tokens=100)
    assert lib.fp8kv_append(r(odd_cap), None, None, None, None, 1, None) == 2
    paged_bad = _cache(layout=1, page_size=8, num_pages=4, max_pages_per_seq=2, page_table=0x5000)
    assert lib.fp8kv_append(r(paged_bad), None, None, None, None, 1, None) == 2
    paged_nopt = _cache(layout=1, page_size=16, num_pages=4, max_pages_per_seq=2)
    assert lib.fp8kv_decode_num_splits(r(paged_nopt), 16, 0, 0) == 0
    big_group = _cache(kv_heads=1)
    assert lib.fp8kv_decode_split(None, r(big_group), None, 16, 0.1, 0, 0, None, 0, None) == 2
    # the tensor-core kernel needs head_dim 128
    d64 = _cache(head_dim=64)
    assert lib.fp8kv_decode_split(None, r(d64), None, 16, 0.1, 0, 2, None, 0, None) == 2
    assert lib.fp8kv_decode_split(None, r(c), None, 16, 0.1, 0, 3, None, 0, None) == 1
    # decode step: unknown flag bits are rejected before anything else
    assert lib.fp8kv_decode_step(0x7000, 0x7000, 0x7000, r(c), 0x8000, 16, 0.1, 0, 2, 0x9000, 1 << 30,
                                 out, 0, 2, None) == 1
    # prefill: the tensor-core kernel is built for K8V8 at head_dim 128 only;
    # a bad kernel id is rejected
    k16 = _cache(dtype=1, k_scale=None)
    assert lib.fp8kv_prefill_attention(0x7000, r(k16), 0x8000, 64, 16, 0.1, 2, out, 0, None) == 2
    assert lib.fp8kv_prefill_attention(0x7000, r(d64), 0x8000, 64, 16, 0.1, 2, out, 0, None) == 2
    assert lib.fp8kv_prefill_attention(0x7000, r(c), 0x8000, 64, 16, 0.1, 5, out, 0, None) == 1
    assert lib.fp8kv_prefill_attention(0x7000, r(c), 0x8000, 0, 16, 0.1, 2, out, 0, None) == 0


def test_cache_dtype_and_scale_pointers(lib):
    # each dtype wants a scale row exactly for its e4m3 sides:
    # K8V8 both, K16V8 V only, K16V16 none, K8V16 K only, MXK8V8 both (the K
    # row's E8M0 bytes); ids past MXK8V8 are unknown
    r = ctypes.byref
    for dtype, k8, v8 in ((0, 1, 1), (1, 0, 1), (2, 0, 0), (3, 1, 0), (4, 1, 1)):
        for ks in (0, 1):
            for vs in (0, 1):
                c = _cache(dtype=dtype, k_scale=0x3000 if ks else None, v_scale=0x4000 if vs else None)
                want = 64 if (ks, vs) == (k8, v8) else 0
                assert lib.fp8kv_decode_num_splits(r(c), 16, 64, 2) == want, (dtype, ks, vs)
    assert lib.fp8kv_decode_num_splits(r(_cache(dtype=5)), 16, 64, 2) == 0
    assert lib.fp8kv_decode_num_splits(r(_cache(dtype=-1)), 16, 64, 2) == 0


def test_mxfp8_kernel_choice(lib):
    # MXFP8 keys: AUTO picks the tensor cores; the CUDA-core decode is built
    # too (planned like any CUDA-core decode); the transform paths and the
    # tensor-core prefill are not; head_dim 128 only
    r = ctypes.byref
    mx = _cache(dtype=4)
    assert lib.fp8kv_decode_num_splits(r(mx), 16, 0, 0) == lib.fp8kv_decode_num_splits(r(_cache()), 16, 0, 2)
    assert lib.fp8kv_decode_num_splits(r(mx), 16, 0, 2) > 0
    assert lib.fp8kv_decode_num_splits(r(mx), 16, 0, 1) == lib.fp8kv_decode_num_splits(r(_cache()), 16, 0, 1) > 0
    for kid in (3, 4):                           # transform paths
        assert lib.fp8kv_decode_num_splits(r(mx), 16, 0, kid) == 0
    assert lib.fp8kv_decode_split(None, r(mx), None, 16, 0.1, 0, 3, None, 0, None) == 2
    assert lib.fp8kv_decode_split(None, r(mx), None, 16, 0.1, 0, 1, None, 0, None) == 1   # null pointers
    assert lib.fp8kv_decode_num_splits(r(_cache(dtype=4, head_dim=64)), 16, 0, 0) == 0
    out = 0x6000
    assert lib.fp8kv_prefill_attention(0x7000, r(mx), 0x8000, 64, 16, 0.1, 2, out, 0, None) == 2
    # the standalone MX quantiser checks its arguments on the host
    assert lib.fp8kv_quantize_mx(None, -1, 128, None, None, None) == 1
    assert lib.fp8kv_quantize_mx(None, 10, 96, None, None, None) == 2
    assert lib.fp8kv_quantize_mx(None, 10, 128, None, None, None) == 1
    assert lib.fp8kv_quantize_mx(None, 0, 128, None, None, None) == 0


def test_key_bias_checks(lib):
    # pre-bias residual keys: K8V8 and K8V16 only, 16-byte aligned
    r = ctypes.byref
    assert lib.fp8kv_decode_num_splits(r(_cache(k_bias=0x5000)), 16, 0, 0) > 0
    assert lib.fp8kv_decode_num_splits(r(_cache(dtype=3, v_scale=None, k_bias=0x5000)), 16, 0, 0) > 0
    assert lib.fp8kv_decode_num_splits(r(_cache(dtype=1, k_scale=None, k_bias=0x5000)), 16, 0, 0) == 0
    assert lib.fp8kv_decode_num_splits(r(_cache(dtype=4, k_bias=0x5000)), 16, 0, 0) == 0
    assert lib.fp8kv_decode_num_splits(r(_cache(k_bias=0x5004)), 16, 0, 0) == 0


def test_rotated_bias_checks(lib):
    # rotary tables: both or neither, only with a bias, 16-byte aligned, and
    # at least as many rows as the cache has positions; such a cache runs on
    # the CUDA-core kernels (AUTO picks them), the tensor cores refuse it
    r = ctypes.byref
    ok = dict(k_bias=0x5000, rope_cos=0x6000, rope_sin=0x7000, rope_positions=8192)
    c = _cache(**ok)
    assert lib.fp8kv_decode_num_splits(r(c), 16, 0, 0) == lib.fp8kv_decode_num_splits(r(_cache()), 16, 0, 1) > 0
    assert lib.fp8kv_decode_num_splits(r(c), 16, 0, 1) > 0
    for kid in (2, 3, 4):
        assert lib.fp8kv_decode_num_splits(r(c), 16, 0, kid) == 0
    assert lib.fp8kv_decode_num_splits(r(_cache(**dict(ok, rope_sin=None))), 16, 0, 0) == 0
    assert lib.fp8kv_decode_num_splits(r(_cache(**dict(ok, k_bias=None))), 16, 0, 0) == 0
    assert lib.fp8kv_decode_num_splits(r(_cache(**dict(ok, rope_positions=8191))), 16, 0, 0) == 0
    assert lib.fp8kv_decode_num_splits(r(_cache(**dict(ok, rope_cos=0x6004))), 16, 0, 0) == 0
    paged = _cache(layout=1, page_size=16, num_pages=64, max_pages_per_seq=8, page_table=0x8000,
                   **dict(ok, rope_positions=128))
    assert lib.fp8kv_decode_num_splits(r(paged), 16, 0, 0) > 0
    assert lib.fp8kv_decode_num_splits(r(_cache(layout=1, page_size=16, num_pages=64, max_pages_per_seq=8,
                                                 page_table=0x8000, **dict(ok, rope_positions=127))), 16, 0, 0) == 0
    assert lib.fp8kv_prefill_attention(0x7000, r(c), 0x8000, 64, 16, 0.1, 2, 0x9000, 0, None) == 2


def test_transform_path_kernel_ids(lib):
    # kernels 3 and 4 (tensor cores, K converted to f16 on chip): K8V8 at
    # head_dim 128 only, planned like the tensor-core kernel; unknown ids rejected
    r = ctypes.byref
    c = _cache()
    for kid in (3, 4):
        assert lib.fp8kv_decode_num_splits(r(c), 16, 0, kid) == lib.fp8kv_decode_num_splits(r(c), 16, 0, 2)
        assert (lib.fp8kv_decode_workspace_bytes(r(c), 16, 0, kid)
                == lib.fp8kv_decode_workspace_bytes(r(c), 16, 0, 2))
        assert lib.fp8kv_decode_num_splits(r(_cache(dtype=1, k_scale=None)), 16, 0, kid) == 0
        assert lib.fp8kv_decode_num_splits(r(_cache(dtype=3, v_scale=None)), 16, 0, kid) == 0
        assert lib.fp8kv_decode_num_splits(r(_cache(head_dim=64)), 16, 0, kid) == 0
    assert lib.fp8kv_decode_num_splits(r(c), 16, 0, 5) == 0
    out = 0x6000
    assert lib.fp8kv_decode_split(None, r(c), None, 16, 0.1, 0, 5, None, 0, None) == 1
    assert lib.fp8kv_decode_split(None, r(_cache(dtype=2, k_scale=None, v_scale=None)), None, 16, 0.1, 0, 3,
                                  None, 0, None) == 2
    # the prefill has no transform-path kernel
    assert lib.fp8kv_prefill_attention(0x7000, r(c), 0x8000, 64, 16, 0.1, 3, out, 0, None) == 1


def test_split_plan_and_workspace(lib):
    c = _cache()
    r = ctypes.byref
    # explicit split counts: chunks are whole tiles anchored at 0; the CUDA-core
    # kernel walks 64-token tiles, the tensor-core kernel 128-token tiles
    for kern, tile in ((1, 64), (2, 128)):
        n_tiles = 8192 // tile
        assert lib.fp8kv_decode_num_splits(r(c), 16, 1, kern) == 1
        assert lib.fp8kv_decode_num_splits(r(c), 16, 7, kern) == 7
        assert lib.fp8kv_decode_num_splits(r(c), 16, 10 ** 6, kern) == n_tiles
        S = lib.fp8kv_decode_num_splits(r(c), 16, 0, kern)
        assert 1 <= S <= n_tiles
        ws = lib.fp8kv_decode_workspace_bytes(r(c), 16, 0, kern)
        assert ws == 16 * 16 * S * (128 + 2) * 4
    # automatic choice: group 8 at head_dim 128 runs on the tensor cores
    assert lib.fp8kv_decode_num_splits(r(c), 16, 10 ** 6, 0) == 64
    # more (sequence, KV-head) units than SMs (the paged batch-64 serving
    # decode: 64 sequences x 8 KV heads, group 4, so two KV heads per CTA and
    # 64-token tiles, 16-token pages up to 16,384 tokens): splits of about 56
    # tiles, 256 tiles -> 5 splits of 52
    paged = _cache(layout=1, batch=64, kv_heads=8, max_tokens=16384, page_size=16,
                   num_pages=64 * 1024, max_pages_per_seq=1024, page_table=0x7000)
    assert lib.fp8kv_decode_num_splits(r(paged), 32, 0, 2) == 5
    assert lib.fp8kv_decode_num_splits(r(paged), 32, 0, 0) == 5


def test_workloads_match_their_description():
    spec = synth.WORKLOADS["paged_b64_hostile"]
    # the lengths of the full paged workload, drawn as decode_inputs draws them
    cpu = torch.Generator().manual_seed(spec.seed)
    lens = torch.randint(1024, 16385, (64,), generator=cpu)
    assert lens.min() >= 1024 and lens.max() <= 16384
    small = synth.DecodeWorkload("s", 5, 8, 2, 64, seed=3, len_range=(1, 100), page_size=16,
                                 hostile_keys=True)
    inp = synth.decode_inputs(small)
    P = 16
    used = inp.page_table[inp.page_table >= 0]
    assert sorted(used.tolist()) == list(range(inp.num_pages))      # a permutation of the pool
    for b in range(5):
        n = (int(inp.seq_lens[b]) + P - 1) // P
        assert (inp.page_table[b, :n] >= 0).all() and (inp.page_table[b, n:] == -1).all()
    # hostile keys: the four biased channels sit near +20
    k = inp.k.float()
    for c in synth.HOSTILE_CHANNELS:
        if c < 64:
            assert abs(k[..., c].mean().item() - 20) < 1.0
    assert abs(inp.v.float().mean().item()) < 0.2
    # determinism
    again = synth.decode_inputs(small)
    assert torch.equal(again.k, inp.k) and torch.equal(again.page_table, inp.page_table)


def test_python_binding_rejects_host_tensors_before_any_call(lib):
    # the binding only marshals device tensors: host tensors and wrong dtypes
    # are refused before the library is called
    import fp8_quantized_kv_gb300 as fk
    x = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fk.fp8kv_quantize(x)
    with pytest.raises(ValueError):
        fk.fp8kv_quantize_mx(x)
    with pytest.raises(ValueError):
        fk.fp8kv_quantize_mx(torch.zeros(4, 128, dtype=torch.float32))
    assert fk.KERNELS["tensor_cores_k_f16"] == 3 and fk.KERNELS["tensor_cores_k_f16_producer"] == 4
    assert fk.DTYPES == {"k8v8": 0, "k16v8": 1, "k16v16": 2, "k8v16": 3, "mxk8v8": 4}


def test_mxfp8_and_bias_workspace_match_the_plain_cache(lib):
    # the MXFP8 dtype and a key bias change neither the split plan nor the
    # workspace: the scale slot is the same 4 bytes per row
    r = ctypes.byref
    for kern in (0, 2):
        base = lib.fp8kv_decode_workspace_bytes(r(_cache()), 16, 0, kern)
        assert lib.fp8kv_decode_workspace_bytes(r(_cache(dtype=4)), 16, 0, kern) == base
        assert lib.fp8kv_decode_workspace_bytes(r(_cache(k_bias=0x5000)), 16, 0, kern) == base
        assert (lib.fp8kv_decode_step_workspace_bytes(r(_cache(dtype=4)), 16, 0, kern)
                == lib.fp8kv_decode_step_workspace_bytes(r(_cache()), 16, 0, kern))

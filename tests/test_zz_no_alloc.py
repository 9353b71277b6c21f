"""The allocation-free decode entry point, fp8kv_decode_attention_static.

It serves callers that cannot call cudaMalloc (a runtime whose pool owns the
device memory, a plugin handed only its tensors): the partials live in a fixed
array inside the library instead of a caller-allocated workspace.  Checked
through the C ABI against fp8kv_decode_attention on the same inputs, on two
calls in a row (the array keeps the previous call's contents).  This file is
collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest
import torch

from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from fp8_quantized_kv_gb300._lib import get_lib
from kvhelpers import fill_cache

pytestmark = pytest.mark.gpu


def _static_call(lib, q, cache, lens, out):
    st = lib.fp8kv_decode_attention_static(
        ctypes.c_void_p(q.data_ptr()), cache.struct_ref, ctypes.c_void_p(lens.data_ptr()),
        q.shape[1], ctypes.c_float(1.0 / math.sqrt(q.shape[2])), 0,
        ctypes.c_void_p(out.data_ptr()), 1, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, fk.fp8kv_status_string(st)


def test_static_scratch_decode_matches_workspace_decode():
    lib = get_lib()
    assert lib.fp8kv_decode_static_scratch_bytes() == 16 << 20
    cases = [synth.WORKLOADS["decode_b16_ctx8192"], synth.WORKLOADS["tiny_decode"]]
    for spec in cases:                        # two different calls in a row
        inp = synth.decode_inputs(spec, device="cuda")
        cache = fill_cache(inp, "k8v8")
        q = inp.q.contiguous()
        lens = inp.seq_lens.cuda()
        ref = fk.fp8kv_decode_attention(q, cache, lens, out_dtype=torch.float32)
        for _ in range(2):
            out = torch.full_like(ref, float("nan"))
            _static_call(lib, q, cache, lens, out)
            torch.cuda.synchronize()
            o, r = out.double().cpu().numpy(), ref.double().cpu().numpy()
            rel = np.linalg.norm(o - r, axis=-1) / np.linalg.norm(r, axis=-1)
            assert np.all(np.isfinite(o))
            assert rel.max() <= 1e-5 and np.abs(o - r).max() <= 2e-2


def test_static_scratch_rejects_oversized_calls():
    lib = get_lib()
    # batch 32 x 16 query heads x 64 splits (128-token tiles over 8192 tokens)
    # of (128 + 2) fp32 partials is 17,039,360 bytes: just above the 16 MiB
    # array, so the call is refused before anything is launched
    cache = fk.Fp8KVCache.contiguous(32, 2, 128, 8192, "k8v8")
    q = torch.zeros(32, 16, 128, dtype=torch.bfloat16, device="cuda")
    lens = torch.full((32,), 8192, dtype=torch.int32, device="cuda")
    out = torch.empty(32, 16, 128, dtype=torch.float32, device="cuda")
    assert fk.fp8kv_decode_workspace_bytes(cache, 16, 64) == 17039360
    st = lib.fp8kv_decode_attention_static(
        ctypes.c_void_p(q.data_ptr()), cache.struct_ref, ctypes.c_void_p(lens.data_ptr()), 16,
        ctypes.c_float(0.1), 64, ctypes.c_void_p(out.data_ptr()), 1, None)
    assert st == 3
    # a few splits fewer fit
    assert fk.fp8kv_decode_workspace_bytes(cache, 16, 60) <= lib.fp8kv_decode_static_scratch_bytes()


def test_static_scratch_allocates_nothing_and_matches_the_oracle():
    """Once the library's kernels are loaded (the first call of the workspace
    entry point), two calls of the allocation-free entry point leave the
    device's free memory exactly as it was and the torch allocator untouched,
    and their output passes the attention bar against the oracle."""
    import oracle
    from kvhelpers import oracle_decode
    lib = get_lib()
    inp = synth.decode_inputs(synth.WORKLOADS["tiny_decode"], device="cuda")
    cache = fill_cache(inp, "k8v8")
    q = inp.q.contiguous()
    lens = inp.seq_lens.cuda()
    fk.fp8kv_decode_attention(q, cache, lens, out_dtype=torch.float32)      # loads the kernels
    out = torch.empty(2, 4, 64, dtype=torch.float32, device="cuda")
    _static_call(lib, q, cache, lens, out)                                 # first call on this device
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    n0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    for _ in range(2):
        _static_call(lib, q, cache, lens, out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == n0
    ok, rel, mab = oracle.attention_gate(out.cpu().numpy(), oracle_decode(inp, "k8v8", range(2)))
    assert ok, (rel, mab)


def test_static_scratch_lowers_the_automatic_split_count_to_fit():
    """256 sequences x 8 query heads over a paged cache of 131,072 tokens'
    capacity: the automatic plan (22 splits) needs 23.4 MB of partials, above
    the 16 MiB array, so the call takes the largest split count that fits and
    agrees with the workspace entry point (automatic splits) to 1e-5."""
    lib = get_lib()
    B, Hq, Hkv, D, P, max_pages = 256, 8, 1, 128, 16, 8192
    n_pages = 64
    g = torch.Generator().manual_seed(3)
    table = torch.randint(0, n_pages, (B, max_pages), generator=g, dtype=torch.int32)
    cache = fk.Fp8KVCache.paged(table, n_pages, Hkv, D, P, "k8v8")
    k = synth.bf16_normal((n_pages * P, Hkv, D), torch.Generator(device="cuda").manual_seed(4), "cuda")
    v = synth.bf16_normal((n_pages * P, Hkv, D), torch.Generator(device="cuda").manual_seed(5), "cuda")
    # fill the pool through sequence 0, whose table is set to pages 0..63 in order
    table[0, :n_pages] = torch.arange(n_pages, dtype=torch.int32)
    cache.page_table.copy_(table.cuda())
    fk.fp8kv_append(cache, k, v, torch.zeros(n_pages * P, dtype=torch.int32, device="cuda"),
                    torch.arange(n_pages * P, dtype=torch.int32, device="cuda"))
    lens = torch.randint(1, 300, (B,), generator=g, dtype=torch.int32).cuda()
    q = synth.bf16_normal((B, Hq, D), torch.Generator(device="cuda").manual_seed(6), "cuda")
    assert fk.fp8kv_decode_workspace_bytes(cache, Hq, 0) > lib.fp8kv_decode_static_scratch_bytes()
    ref = fk.fp8kv_decode_attention(q, cache, lens, out_dtype=torch.float32)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        _static_call(lib, q, cache, lens, out)
        torch.cuda.synchronize()
        rel = ((out.double() - ref.double()).norm(dim=-1) / ref.double().norm(dim=-1)).max().item()
        assert rel <= 1e-5, rel
    assert fk.fp8kv_get_device_error() == 0

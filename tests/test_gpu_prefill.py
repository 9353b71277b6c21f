"""GPU parity of causal prefill on the tensor cores (128-query tiles, K8V8,
head dim 128) against the oracle: batches with different prefix offsets,
contiguous capacities that end inside a 64-token KV tile, paged caches,
GQA group sizes, V scales spread over many binades, degenerate query counts
and the device-side length check.

Bars as in the other parity tests: relative L2 1e-2 and max-abs 2e-2 per
(query row block, head) of the fp64 oracle on the dequantised cache."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import assert_gate

pytestmark = pytest.mark.gpu
KERNELS = ["cuda_cores", "tensor_cores"]


@pytest.fixture(autouse=True)
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield


def _build(B, n_q, pos0s, Hq, Hkv, seed, page_size=None, cap_align=16, v_token_scale=None):
    """Seeded bf16 Q/K/V for B sequences (sequence b holds pos0s[b] + n_q
    tokens), appended into a contiguous or paged K8V8 cache."""
    D = 128
    qs, ks, vs = [], [], []
    for b in range(B):
        spec = synth.PrefillWorkload("pf", n_q, Hq, Hkv, D, seed=seed + b, pos0=pos0s[b])
        pin = synth.prefill_inputs(spec, device="cuda")
        v = pin.v
        if v_token_scale is not None:
            v = (v.float() * v_token_scale(b, v.shape[0]).to("cuda")[:, None, None]).to(torch.bfloat16)
        qs.append(pin.q)
        ks.append(pin.k)
        vs.append(v)
    totals = [p + n_q for p in pos0s]
    if page_size is None:
        cap = ((max(totals) + cap_align - 1) // cap_align) * cap_align
        cache = fk.Fp8KVCache.contiguous(B, Hkv, D, cap, "k8v8")
    else:
        gen = torch.Generator().manual_seed(seed)
        per = [(t + page_size - 1) // page_size for t in totals]
        num_pages = sum(per) + 3
        perm = torch.randperm(num_pages, generator=gen).to(torch.int32)
        table = torch.full((B, max(per)), -1, dtype=torch.int32)
        off = 0
        for b in range(B):
            table[b, :per[b]] = perm[off:off + per[b]]
            off += per[b]
        cache = fk.Fp8KVCache.paged(table, num_pages, Hkv, D, page_size, "k8v8")
    seq_idx = torch.cat([torch.full((t,), b, dtype=torch.int32) for b, t in enumerate(totals)])
    pos = torch.cat([torch.arange(t, dtype=torch.int32) for t in totals])
    fk.fp8kv_append(cache, torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), seq_idx.cuda(), pos.cuda())
    q = torch.stack(qs).contiguous()
    return cache, q, ks, vs


def _check(cache, q, ks, vs, pos0s, kernel, blocks=None):
    B, n_q, Hq, D = q.shape
    out = fk.fp8kv_prefill_attention(q, cache, torch.tensor(pos0s, dtype=torch.int32, device="cuda"),
                                     out_dtype=torch.float32, kernel=kernel).cpu().numpy()
    assert fk.fp8kv_get_device_error() == 0
    sm = 1 / math.sqrt(D)
    for b in range(B):
        kb = synth.bf16_bits(ks[b]).transpose(1, 0, 2)
        vb = synth.bf16_bits(vs[b]).transpose(1, 0, 2)
        k = oracle.dequantize(*oracle.quantize(kb))
        v = oracle.dequantize(*oracle.quantize(vb))
        qd = oracle.bf16_to_double(synth.bf16_bits(q[b]))
        p0 = pos0s[b]
        for a, e in (blocks or [(0, n_q)]):
            ref = oracle.prefill_attention(qd[a:e], k[:, :p0 + e], v[:, :p0 + e], p0 + a, sm)
            assert_gate(out[b, a:e].reshape(-1, D), ref.reshape(-1, D), f"seq {b} rows {a}:{e} {kernel}")
    return out


@pytest.mark.parametrize("kernel", KERNELS)
def test_batch_offsets_capacity_inside_tile(kernel):
    """Two sequences with prefixes 37 and 100 (query tiles not aligned to KV
    tiles), capacity a multiple of 16 but not of 64: the last KV tile runs
    past the sequence's rows."""
    pos0s = [37, 100]
    cache, q, ks, vs = _build(2, 300, pos0s, 8, 2, seed=41, cap_align=16)
    assert cache.max_tokens % 64 != 0
    _check(cache, q, ks, vs, pos0s, kernel)


@pytest.mark.parametrize("page_size", [16, 64])
@pytest.mark.parametrize("kernel", KERNELS)
def test_paged(kernel, page_size):
    pos0s = [0, 70]
    cache, q, ks, vs = _build(2, 150, pos0s, 4, 4, seed=43, page_size=page_size)
    _check(cache, q, ks, vs, pos0s, kernel)


@pytest.mark.parametrize("n_q", [1, 64, 128, 129])
def test_query_counts(n_q):
    """One query row, exactly one and two 64-row tiles, one 128-row tile, and
    one row past it."""
    pos0s = [5, 64]
    cache, q, ks, vs = _build(2, n_q, pos0s, 16, 2, seed=47 + n_q)
    _check(cache, q, ks, vs, pos0s, "tensor_cores")


def test_v_scales_across_binades():
    """Sequence 0: every V row scaled by 2^-18 (tiny V scales); sequence 1:
    per-token factors between 2^-12 and 2^3.  The P.V operand scaling must keep
    both inside the 16-bit operand's range."""
    def factor(b, n):
        if b == 0:
            return torch.full((n,), 2.0 ** -18)
        g = torch.Generator().manual_seed(5)
        return 2.0 ** torch.randint(-12, 4, (n,), generator=g).float()
    pos0s = [0, 33]
    cache, q, ks, vs = _build(2, 260, pos0s, 4, 1, seed=53, v_token_scale=factor)
    _check(cache, q, ks, vs, pos0s, "tensor_cores")


def test_large_scores_lazy_rescale():
    """Query rows scaled so scores span hundreds of log2 units: the running
    maximum moves often and the accumulator rescale path runs."""
    pos0s = [0]
    cache, q, ks, vs = _build(1, 512, pos0s, 2, 1, seed=59)
    g = torch.Generator(device="cuda").manual_seed(3)
    q = (q.float() * (1 + 30 * torch.rand(q.shape[:3] + (1,), generator=g, device="cuda"))).to(torch.bfloat16)
    _check(cache, q.contiguous(), ks, vs, pos0s, "tensor_cores")


def test_tensor_cores_match_cuda_cores():
    """Both prefill kernels on one cache agree within the attention bar."""
    pos0s = [11]
    cache, q, ks, vs = _build(1, 333, pos0s, 8, 2, seed=61)
    p0 = torch.tensor(pos0s, dtype=torch.int32, device="cuda")
    a = fk.fp8kv_prefill_attention(q, cache, p0, out_dtype=torch.float32, kernel="tensor_cores")
    b = fk.fp8kv_prefill_attention(q, cache, p0, out_dtype=torch.float32, kernel="cuda_cores")
    assert_gate(a.reshape(-1, 128).cpu().numpy(), b.reshape(-1, 128).double().cpu().numpy(), "tc vs cuda cores")


def test_repeatable():
    pos0s = [3]
    cache, q, ks, vs = _build(1, 700, pos0s, 4, 2, seed=67)
    p0 = torch.tensor(pos0s, dtype=torch.int32, device="cuda")
    first = fk.fp8kv_prefill_attention(q, cache, p0, out_dtype=torch.float32, kernel="tensor_cores")
    for _ in range(20):
        assert torch.equal(fk.fp8kv_prefill_attention(q, cache, p0, out_dtype=torch.float32,
                                                      kernel="tensor_cores"), first)


def test_prefix_beyond_capacity_flags_device_error():
    """q_pos0 + n_q past the cache capacity: the CTA skips the work and raises
    the length bit; nothing faults."""
    cache, q, ks, vs = _build(1, 64, [0], 2, 1, seed=71)
    p0 = torch.tensor([cache.max_tokens - 10], dtype=torch.int32, device="cuda")
    fk.fp8kv_prefill_attention(q, cache, p0, kernel="tensor_cores")
    assert fk.fp8kv_get_device_error() & fk.DEVERR_SEQ_TOO_LONG


def test_unsupported_dtype_rejected():
    cache = fk.Fp8KVCache.contiguous(1, 1, 128, 64, "k16v8")
    q = torch.zeros(1, 4, 1, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fk.Fp8KVError) as e:
        fk.fp8kv_prefill_attention(q, cache, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                   kernel="tensor_cores")
    assert e.value.status == 2


@pytest.mark.parametrize("page_size", [None, 32])
def test_several_items_per_cta(page_size):
    """More (query tile, sequence, query head) work items than SMs, of
    different lengths and sequences: three sequences with prefixes 0, 129 and
    700, 400 queries, 16 query heads."""
    pos0s = [0, 129, 700]
    cache, q, ks, vs = _build(3, 400, pos0s, 16, 2, seed=73, page_size=page_size)
    _check(cache, q, ks, vs, pos0s, "tensor_cores")


def test_many_items_sampled():
    """512 work items (1024 queries, 2 sequences, 32 query heads over 4 KV
    heads): sampled query blocks against the oracle."""
    pos0s = [0, 300]
    cache, q, ks, vs = _build(2, 1024, pos0s, 32, 4, seed=79)
    _check(cache, q, ks, vs, pos0s, "tensor_cores", blocks=[(0, 64), (448, 520), (960, 1024)])


def test_invalid_sequence_skipped_others_computed():
    """A sequence whose prefix runs past the capacity is skipped (length bit
    raised) while the other sequence's work items stay correct: 256 items, the
    skipped ones among valid ones."""
    pos0s = [0, 0]
    cache, q, ks, vs = _build(2, 256, pos0s, 64, 8, seed=83)
    bad = [0, cache.max_tokens - 10]
    out = fk.fp8kv_prefill_attention(q, cache, torch.tensor(bad, dtype=torch.int32, device="cuda"),
                                     out_dtype=torch.float32, kernel="tensor_cores").cpu().numpy()
    assert fk.fp8kv_get_device_error() & fk.DEVERR_SEQ_TOO_LONG
    D = q.shape[-1]
    kb = synth.bf16_bits(ks[0]).transpose(1, 0, 2)
    vb = synth.bf16_bits(vs[0]).transpose(1, 0, 2)
    k = oracle.dequantize(*oracle.quantize(kb))
    v = oracle.dequantize(*oracle.quantize(vb))
    qd = oracle.bf16_to_double(synth.bf16_bits(q[0]))
    ref = oracle.prefill_attention(qd, k[:, :256], v[:, :256], 0, 1 / math.sqrt(D))
    assert_gate(out[0].reshape(-1, D), ref.reshape(-1, D), "valid sequence beside a skipped one")

"""Paged tensor-core decode with several KV heads per CTA.

On a paged cache with fewer than 8 query heads per KV head, one tensor-core
CTA takes 8 / G neighbouring KV heads (as many as divide the head count and
fit 128 rows per page), so a 128-row tile holds several heads' tokens and
every score column is masked to its own head's rows.  Parity against the
oracle for every page size (16, 32, 64) and group size (1, 2, 4, 8), head
counts that force fewer heads per CTA, split invariance (cluster and global
merges), and the fused step, whose appender writes each of the CTA's heads."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import assert_gate, fill_cache, gpu_decode, oracle_decode, seq_bits, split_last_token

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield
    assert fk.fp8kv_get_device_error() == 0


def _spec(P, G, Hkv, seed, batch=4, len_range=(1, 600)):
    return synth.DecodeWorkload(f"paged_heads_P{P}_G{G}", batch, G * Hkv, Hkv, 128, seed=seed,
                                len_range=len_range, page_size=P, hostile_keys=True)


@pytest.mark.parametrize("dtype", ["k8v8", "k16v8", "k8v16", "k16v16", "mxk8v8"])
@pytest.mark.parametrize("G,Hkv", [(1, 8), (2, 4), (4, 2), (8, 2)])
@pytest.mark.parametrize("P", [16, 32, 64])
def test_paged_page_sizes_and_groups(P, G, Hkv, dtype):
    inp = synth.decode_inputs(_spec(P, G, Hkv, seed=100 + P + G), device="cuda")
    cache = fill_cache(inp, dtype)
    out = gpu_decode(inp, cache, kernel="tensor_cores").cpu().numpy()
    assert_gate(out, oracle_decode(inp, dtype, range(4)), f"paged P{P} G{G} {dtype}")


@pytest.mark.parametrize("P,G,Hkv", [(16, 2, 6), (16, 1, 3), (16, 1, 12), (32, 1, 6), (64, 4, 3)])
def test_paged_head_counts_that_limit_heads_per_cta(P, G, Hkv):
    """KV head counts that 8 / G does not divide: fewer heads per CTA."""
    inp = synth.decode_inputs(_spec(P, G, Hkv, seed=7 * P + Hkv, batch=3), device="cuda")
    cache = fill_cache(inp, "k8v8")
    out = gpu_decode(inp, cache, kernel="tensor_cores").cpu().numpy()
    assert_gate(out, oracle_decode(inp, "k8v8", range(3)), f"paged P{P} G{G} Hkv{Hkv}")


@pytest.mark.parametrize("P,G", [(16, 4), (32, 2), (64, 1)])
def test_paged_split_invariance(P, G):
    """Splits of the same tiles (cluster merge for 2-8 splits, global merge
    above): fp32 outputs within 1e-5 relative of the unsplit run."""
    Hkv = 8 // G
    inp = synth.decode_inputs(_spec(P, G, Hkv, seed=31, batch=2, len_range=(1500, 3000)), device="cuda")
    cache = fill_cache(inp, "k8v8")
    base = gpu_decode(inp, cache, num_splits=1, kernel="tensor_cores")
    for ns in (2, 3, 5, 8, 12):
        out = gpu_decode(inp, cache, num_splits=ns, kernel="tensor_cores")
        rel = float((out - base).norm() / base.norm())
        assert rel <= 1e-5, (P, G, ns, rel)
    # the fused step merges in the kernel: in a cluster for 2-8 splits,
    # through global partials above
    prev, knew, vnew = split_last_token(inp)
    for ns in (1, 2, 5, 8, 12):
        c2 = fill_cache(prev, "k8v8")
        out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, c2, inp.seq_lens.cuda(),
                                   num_splits=ns, out_dtype=torch.float32, kernel="tensor_cores")
        rel = float((out - base).norm() / base.norm())
        assert rel <= 1e-5, (P, G, "step", ns, rel)


@pytest.mark.parametrize("P,G,Hkv", [(16, 4, 2), (32, 2, 4), (64, 1, 8), (16, 1, 8)])
def test_paged_step_writes_every_head(P, G, Hkv):
    """The fused step on a paged cache: each sequence's new token lands in
    every KV head the CTA covers (codes and scales bit-exact against the
    oracle's quantiser), and the attention over it passes the gate."""
    inp = synth.decode_inputs(_spec(P, G, Hkv, seed=55 + P, batch=5, len_range=(1, 700)), device="cuda")
    prev, knew, vnew = split_last_token(inp)
    cache = fill_cache(prev, "k8v8")
    out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, cache, inp.seq_lens.cuda(),
                               out_dtype=torch.float32, kernel="tensor_cores")
    assert_gate(out.cpu().numpy(), oracle_decode(inp, "k8v8", range(5)), f"paged step P{P} G{G}")
    pt = inp.page_table.numpy()
    for b in range(5):
        T = int(inp.seq_lens[b])
        if T == 0:
            continue
        kc, ks = oracle.quantize(seq_bits(inp, "k", b))
        vc, vs = oracle.quantize(seq_bits(inp, "v", b))
        got_k = oracle.gather_paged(cache.k.cpu().numpy(), pt, b, T)
        got_v = oracle.gather_paged(cache.v.cpu().numpy(), pt, b, T)
        got_vs = oracle.gather_paged(cache.v_scale.cpu().numpy()[..., None], pt, b, T)[..., 0]
        assert np.array_equal(got_k[:, T - 1], kc[:, T - 1]), b
        assert np.array_equal(got_v[:, T - 1], vc[:, T - 1]), b
        assert np.array_equal(got_vs[:, T - 1].view(np.uint32), vs[:, T - 1].view(np.uint32)), b

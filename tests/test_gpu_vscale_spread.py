"""V scales that differ across tokens by many binades, on every decode path
that folds the V scale into P ("FP8 KV cache (fp8_kv, opt-in)", bullet
"Math": V scale folded into P, rounded to bf16 for P.V).

The tensor-core decode writes each bf16 P' = p * v_scale row as e4m3 terms
after one power-of-two scaling of a (tile, head) column, so the choice of that
power decides which tokens keep their precision.  The inputs here break any
choice that looks at the V scales alone:

* every V row of a sequence multiplied by 2^-18 (tiny scales throughout);
* per-token factors 2^-12 .. 2^3 drawn at random;
* dominance: in every 128-token tile one token has a score far above the rest
  for the first query head of each group (its key is a multiple of that
  head's query) and a V row 2^-14 or 2^-20 times smaller than its
  neighbours, whose V rows are 8x larger than N(0,1).  That head's output is
  then the small token's V row, and p * v_scale of the loud neighbours is
  tiny although their V scales are the tile's largest.

Checked element by element against the fp64 oracle on the dequantised cache
(relative L2 1e-2 and max-abs 2e-2 per sequence and query head), on the
split + merge calls (tensor cores and CUDA cores), and on the fused step with
the cluster merge (2-8 splits) and the global merge (12 splits)."""
import numpy as np
import pytest
import torch

from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import assert_gate, fill_cache, gpu_decode, oracle_decode, split_last_token

V8_DTYPES = ["k8v8", "k16v8", "mxk8v8"]
LENS = (1000, 300, 129, 2500)


@pytest.fixture
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield


def _with_v_factors(inp: synth.DecodeInputs, factor) -> synth.DecodeInputs:
    """The workload with V row n of sequence b multiplied by factor(b, T_b)[n]
    (powers of two: exact in bf16)."""
    v = inp.v.float().clone()
    for b in range(inp.seq_lens.numel()):
        s, e = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
        v[s:e] *= factor(b, e - s).to(v.device)[:, None, None]
    return synth.DecodeInputs(inp.spec, inp.q, inp.k, v.to(torch.bfloat16), inp.seq_lens, inp.cu_seqlens,
                              inp.page_table, inp.num_pages)


def _spread_inputs(page_size=None):
    spec = synth.DecodeWorkload("vspread", 4, 16, 2, 128, seed=81, seq_lens=LENS, page_size=page_size)

    def factor(b, n):
        if b == 0:
            return torch.full((n,), 2.0 ** -18)
        g = torch.Generator().manual_seed(100 + b)
        return 2.0 ** torch.randint(-12, 4, (n,), generator=g).float()
    return _with_v_factors(synth.decode_inputs(spec, device="cuda"), factor)


def _dominance_inputs(small_exp, page_size=None, device="cuda"):
    """One loud-score, small-V token per 128-token tile (see module doc)."""
    spec = synth.DecodeWorkload("vdominance", 4, 16, 2, 128, seed=83, seq_lens=LENS, page_size=page_size)
    inp = synth.decode_inputs(spec, device=device)
    G = spec.group
    k = inp.k.float().clone()
    v = inp.v.float().clone() * 8.0
    g = torch.Generator().manual_seed(7)
    for b in range(inp.seq_lens.numel()):
        s, T = int(inp.cu_seqlens[b]), int(inp.seq_lens[b])
        for t0 in range(0, T, 128):
            j = s + t0 + int(torch.randint(0, min(128, T - t0), (1,), generator=g))
            for hk in range(spec.kv_heads):
                k[j, hk] = 4.0 * inp.q[b, hk * G].float()
                v[j, hk] *= 2.0 ** small_exp / 8.0
    return synth.DecodeInputs(spec, inp.q, k.to(torch.bfloat16), v.to(torch.bfloat16), inp.seq_lens,
                              inp.cu_seqlens, inp.page_table, inp.num_pages)


def _cases():
    return [("spread", lambda **kw: _spread_inputs(**kw)),
            ("dominance_2^-14", lambda **kw: _dominance_inputs(-14, **kw)),
            ("dominance_2^-20", lambda **kw: _dominance_inputs(-20, **kw))]


@pytest.mark.gpu
@pytest.mark.usefixtures("_clear_device_error")
@pytest.mark.parametrize("dtype", V8_DTYPES)
def test_decode_tensor_cores(dtype):
    for name, make in _cases():
        inp = make()
        cache = fill_cache(inp, dtype, capacity=2560)
        ref = oracle_decode(inp, dtype, range(4))
        for ns in (0, 1, 3):
            out = gpu_decode(inp, cache, num_splits=ns, kernel="tensor_cores").cpu().numpy()
            assert_gate(out, ref, f"{name} {dtype} splits={ns}")
    assert fk.fp8kv_get_device_error() == 0


@pytest.mark.gpu
@pytest.mark.usefixtures("_clear_device_error")
@pytest.mark.parametrize("dtype", ["k8v8", "k16v8"])
def test_decode_cuda_cores(dtype):
    for name, make in _cases():
        inp = make()
        cache = fill_cache(inp, dtype, capacity=2560)
        out = gpu_decode(inp, cache, kernel="cuda_cores").cpu().numpy()
        assert_gate(out, oracle_decode(inp, dtype, range(4)), f"{name} {dtype} cuda cores")


@pytest.mark.gpu
@pytest.mark.usefixtures("_clear_device_error")
def test_decode_paged():
    for name, make in _cases():
        inp = make(page_size=16)
        cache = fill_cache(inp, "k8v8")
        out = gpu_decode(inp, cache, kernel="tensor_cores").cpu().numpy()
        assert_gate(out, oracle_decode(inp, "k8v8", range(4)), f"{name} paged")


@pytest.mark.gpu
@pytest.mark.usefixtures("_clear_device_error")
@pytest.mark.parametrize("dtype", V8_DTYPES)
def test_fused_step_cluster_and_global_merge(dtype):
    """The fused step: the new token of each sequence appended in the launch,
    its splits merged in a thread-block cluster (2, 5, 8) or through global
    partials (12), and the automatic plan."""
    for name, make in _cases():
        inp = make()
        prev, knew, vnew = split_last_token(inp)
        ref = oracle_decode(inp, dtype, range(4))
        for ns in (0, 2, 5, 8, 12):
            cache = fill_cache(prev, dtype, capacity=2560)
            out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, cache, inp.seq_lens.cuda(),
                                       num_splits=ns, out_dtype=torch.float32, kernel="tensor_cores")
            assert_gate(out.cpu().numpy(), ref, f"step {name} {dtype} splits={ns}")
    assert fk.fp8kv_get_device_error() == 0


def test_dominance_case_is_what_it_claims():
    """The dominance inputs do what the module doc says, checked on the
    oracle: head 0 of each group puts nearly all its weight on the small-V
    tokens (its output is small), while most other heads' outputs are
    dominated by the loud V rows."""
    inp = _dominance_inputs(-14, device="cpu")
    ref = oracle_decode(inp, "k16v16", range(4))
    norms = np.linalg.norm(ref, axis=-1)                 # [B, Hq]
    G = inp.spec.group
    first = norms[:, ::G]
    others = np.delete(norms, np.arange(0, 16, G), axis=1)
    assert first.max() < 2.0 ** -10 * np.median(others)


def _prefill_dominance(small_exp, n_q=300, pos0=20):
    """Causal prefill with, in every 64-key tile, one key that is a multiple
    of a query row's query (loud score for that row) and whose V row is
    2^small_exp times its N(0,1) neighbours'.  (Outputs stay O(1), the scale
    the absolute max-abs bar assumes.)"""
    Hq, Hkv, D = 4, 1, 128
    spec = synth.PrefillWorkload("pf_dominance", n_q, Hq, Hkv, D, seed=91, pos0=pos0)
    pin = synth.prefill_inputs(spec, device="cpu")
    k = pin.k.float().clone()
    v = pin.v.float().clone()
    g = torch.Generator().manual_seed(11)
    total = pos0 + n_q
    for t0 in range(0, total, 64):
        j = t0 + int(torch.randint(0, min(64, total - t0), (1,), generator=g))
        qi = max(j - pos0, 0)                  # a query row that sees key j
        k[j, 0] = 4.0 * pin.q[min(qi, n_q - 1), 0].float()
        v[j, 0] *= 2.0 ** small_exp
    return pin.q, k.to(torch.bfloat16), v.to(torch.bfloat16), pos0


@pytest.mark.gpu
@pytest.mark.usefixtures("_clear_device_error")
@pytest.mark.parametrize("small_exp", [-14, -20])
@pytest.mark.parametrize("kernel", ["tensor_cores", "cuda_cores"])
def test_prefill_dominance(small_exp, kernel):
    import math
    import oracle
    q, k, v, pos0 = _prefill_dominance(small_exp)
    n_q, Hq, D = q.shape
    total = pos0 + n_q
    cache = fk.Fp8KVCache.contiguous(1, 1, D, ((total + 63) // 64) * 64, "k8v8")
    fk.fp8kv_append(cache, k.cuda().contiguous(), v.cuda().contiguous(),
                    torch.zeros(total, dtype=torch.int32, device="cuda"),
                    torch.arange(total, dtype=torch.int32, device="cuda"))
    out = fk.fp8kv_prefill_attention(q[None].cuda().contiguous(), cache,
                                     torch.tensor([pos0], dtype=torch.int32, device="cuda"),
                                     out_dtype=torch.float32, kernel=kernel)[0].cpu().numpy()
    kk = oracle.dequantize(*oracle.quantize(synth.bf16_bits(k).transpose(1, 0, 2)))
    vv = oracle.dequantize(*oracle.quantize(synth.bf16_bits(v).transpose(1, 0, 2)))
    ref = oracle.prefill_attention(oracle.bf16_to_double(synth.bf16_bits(q)), kk, vv, pos0, 1 / math.sqrt(D))
    assert_gate(out.reshape(-1, D), ref.reshape(-1, D), f"prefill dominance 2^{small_exp} {kernel}")
    assert fk.fp8kv_get_device_error() == 0

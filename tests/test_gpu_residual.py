"""Pre-bias residual keys (fp8kv_cache.k_bias): appends quantise fp32(k) - b
per row, bit-exact against the oracle; decode, the fused step and prefill
attend over the residual codes and are held to the attention gate against the
oracle's attention over the keys the cache represents, dequant(r) + b (the
constant q.b cancels in the softmax).  On keys with a large fixed bias the
residual cache is also checked to be closer to the bf16 cache than the plain
per-row cache."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import assert_gate, fill_cache, gpu_decode, oracle_decode, seq_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield
    assert fk.fp8kv_get_device_error() == 0


def _bias(Hkv, D, seed):
    """The hostile keys' fixed offset on their channels, plus a random
    per-head bias of a few units elsewhere."""
    g = torch.Generator().manual_seed(seed)
    b = torch.randn(Hkv, D, generator=g) * 3
    for c in synth.HOSTILE_CHANNELS:
        b[:, c] = synth.HOSTILE_BIAS
    return b.float()


@pytest.mark.parametrize("dtype", ["k8v8", "k8v16"])
@pytest.mark.parametrize("paged", [False, True])
def test_append_bit_exact(dtype, paged):
    spec = synth.DecodeWorkload("append_res", 3, 4, 2, 128, seed=21, seq_lens=(77, 130, 16),
                                page_size=16 if paged else None, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    b = _bias(2, 128, 1)
    cache = fill_cache(inp, dtype, k_bias=b.cuda())
    for s in range(3):
        T = int(inp.seq_lens[s])
        if paged:
            pt = inp.page_table.numpy()
            kc = oracle.gather_paged(cache.k.cpu().numpy(), pt, s, T)
            ks = oracle.gather_paged(cache.k_scale.cpu().numpy()[..., None], pt, s, T)[..., 0]
        else:
            kc, ks = cache.k[s, :, :T].cpu().numpy(), cache.k_scale[s, :, :T].cpu().numpy()
        rc, rs = oracle.quantize_residual(seq_bits(inp, "k", s), b.numpy())
        assert np.array_equal(kc, rc), s
        assert np.array_equal(ks.view(np.uint32), rs.view(np.uint32)), s


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("dtype", ["k8v8", "k8v16"])
def test_decode_matches_reconstructed_keys(dtype, kernel):
    spec = synth.DecodeWorkload("res_dec", 6, 16, 2, 128, seed=9, len_range=(1, 1500), hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    b = _bias(2, 128, 2)
    cache = fill_cache(inp, dtype, k_bias=b.cuda())
    out = gpu_decode(inp, cache, kernel=kernel).cpu().numpy()
    assert_gate(out, oracle_decode(inp, dtype, range(6), k_bias=b.numpy()), f"residual {dtype} {kernel}")


def test_residual_is_closer_to_bf16_than_plain_fp8():
    """The numerical-safety claim on keys with a large fixed bias: measured
    on the GPU path against the oracle's bf16-cache attention."""
    spec = synth.DecodeWorkload("res_q", 16, 16, 2, 128, seed=1, seq_lens=(512,) * 16, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    b = torch.zeros(2, 128)                    # the keys' own fixed part: the hostile offset
    b[:, list(synth.HOSTILE_CHANNELS)] = synth.HOSTILE_BIAS
    ref = oracle_decode(inp, "k16v16", range(16))
    plain = gpu_decode(inp, fill_cache(inp, "k8v8")).cpu().numpy()
    resid = gpu_decode(inp, fill_cache(inp, "k8v8", k_bias=b.cuda())).cpu().numpy()
    e_plain = np.linalg.norm(plain - ref) / np.linalg.norm(ref)
    e_resid = np.linalg.norm(resid - ref) / np.linalg.norm(ref)
    assert e_resid < 0.6 * e_plain, (e_resid, e_plain)


def test_fused_step_appends_residual_row():
    from kvhelpers import split_last_token as _split_last_token
    spec = synth.DecodeWorkload("res_step", 8, 16, 2, 128, seed=2, seq_lens=(4096,) * 8, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    b = _bias(2, 128, 4)
    prev, knew, vnew = _split_last_token(inp)
    cache = fill_cache(prev, "k8v8", capacity=4096, k_bias=b.cuda())
    out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, cache, inp.seq_lens.cuda(),
                               out_dtype=torch.float32)
    assert_gate(out.cpu().numpy(), oracle_decode(inp, "k8v8", range(8), k_bias=b.numpy()), "residual step")
    rc, rs = oracle.quantize_residual(synth.bf16_bits(knew).transpose(1, 0, 2), b.numpy())
    assert np.array_equal(cache.k[:, :, 4095].cpu().numpy(), rc.transpose(1, 0, 2))
    assert np.array_equal(cache.k_scale[:, :, 4095].cpu().numpy().view(np.uint32), rs.T.view(np.uint32))


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
def test_prefill_matches_reconstructed_keys(kernel):
    n_q, Hq, Hkv, D = 300, 8, 2, 128
    spec = synth.PrefillWorkload("res_pf", n_q, Hq, Hkv, D, seed=33)
    pin = synth.prefill_inputs(spec, device="cuda")
    b = _bias(Hkv, D, 5)
    k = pin.k.float()
    k[:, :, list(synth.HOSTILE_CHANNELS)] += synth.HOSTILE_BIAS        # keys with the fixed offset
    k = k.to(torch.bfloat16)
    cache = fk.Fp8KVCache.contiguous(1, Hkv, D, 320, "k8v8", k_bias=b.cuda())
    fk.fp8kv_append(cache, k.contiguous(), pin.v.contiguous(), torch.zeros(n_q, dtype=torch.int32, device="cuda"),
                    torch.arange(n_q, dtype=torch.int32, device="cuda"))
    out = fk.fp8kv_prefill_attention(pin.q[None].contiguous(), cache, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                     out_dtype=torch.float32, kernel=kernel)[0].cpu().numpy()
    kb = synth.bf16_bits(k).transpose(1, 0, 2)
    kk = oracle.residual_keys(*oracle.quantize_residual(kb, b.numpy()), b.numpy())
    vv = oracle.dequantize(*oracle.quantize(synth.bf16_bits(pin.v).transpose(1, 0, 2)))
    ref = oracle.prefill_attention(oracle.bf16_to_double(synth.bf16_bits(pin.q)), kk, vv, 0, 1 / math.sqrt(D))
    assert_gate(out.reshape(-1, D), ref.reshape(-1, D), f"residual prefill {kernel}")


def test_bias_rejected_for_other_dtypes():
    b = torch.zeros(1, 128, device="cuda")
    for dtype in ("k16v8", "k16v16", "mxk8v8"):
        cache = fk.Fp8KVCache.contiguous(1, 1, 128, 64, dtype, k_bias=b)
        assert fk.fp8kv_decode_num_splits(cache, 8, 0) == 0

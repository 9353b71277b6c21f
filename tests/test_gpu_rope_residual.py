"""Rotated pre-bias residual keys (fp8kv_cache.k_bias with rope_cos and
rope_sin): the cache holds rotated keys, and the bias b, added before the
rotary embedding, turns with each key's position.  Appends quantise
fp32(k) - R_t b per row, bit-exact against the oracle; the CUDA-core decode
(AUTO picks it), the fused step and the CUDA-core prefill are held to the
attention gate against the oracle's attention over dequant(r) + R_t b; the
tensor-core kernels refuse such a cache.  On keys that carry a large rotated
bias the residual cache is closer to the bf16 cache than the plain per-row
cache and than a constant-bias residual."""
import math

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


def _tables(P, D, base=10000.0):
    """Rotary tables for positions 0..P-1: theta_{t,i} = t base^(-i/(D/2))."""
    h = D // 2
    th = np.arange(P)[:, None] * base ** (-np.arange(h)[None, :] / h)
    return np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)


def _bias(Hkv, D, seed):
    """A large bias on the hostile channels (and their rotary partners'
    pairs) plus a small random part."""
    g = np.random.default_rng(seed)
    b = (g.standard_normal((Hkv, D)) * 2).astype(np.float32)
    for c in synth.HOSTILE_CHANNELS:
        b[:, c % D] = synth.HOSTILE_BIAS
    return b


def _rotated(b, cos, sin, T):
    """R_t b for t < T in fp64 (the textbook rotate-half rotation)."""
    h = b.shape[1] // 2
    c, s = cos[:T].astype(np.float64), sin[:T].astype(np.float64)
    lo, hi = b[:, None, :h].astype(np.float64), b[:, None, h:].astype(np.float64)
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)      # [Hkv, T, D]


def _workload(name, B, Hq, Hkv, D, seed, page_size=None, seq_lens=None, len_range=None, P=4096):
    """A decode workload whose keys carry the rotated bias: k_t = noise + R_t b."""
    kw = dict(seed=seed, page_size=page_size)
    if seq_lens is not None:
        kw["seq_lens"] = seq_lens
    else:
        kw["len_range"] = len_range
    inp = synth.decode_inputs(synth.DecodeWorkload(name, B, Hq, Hkv, D, **kw), device="cuda")
    b = _bias(Hkv, D, seed)
    cos, sin = _tables(P, D)
    k = inp.k.float().cpu()
    for s in range(B):
        lo, hi = int(inp.cu_seqlens[s]), int(inp.cu_seqlens[s + 1])
        if hi > lo:
            k[lo:hi] += torch.from_numpy(_rotated(b, cos, sin, hi - lo).transpose(1, 0, 2)).float()
    inp.k.copy_(k.to(torch.bfloat16).to(inp.k.device))
    return inp, b, cos, sin


def _dev(b, cos, sin):
    return torch.from_numpy(b).cuda(), (torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda())


@pytest.mark.parametrize("dtype", ["k8v8", "k8v16"])
@pytest.mark.parametrize("paged", [False, True])
def test_append_bit_exact(dtype, paged):
    inp, b, cos, sin = _workload("rope_app", 3, 4, 2, 128, seed=11, page_size=16 if paged else None,
                                 seq_lens=(77, 300, 16), P=512)
    bd, rope = _dev(b, cos, sin)
    cache = fill_cache(inp, dtype, capacity=512, k_bias=bd, rope=rope)
    for s in range(3):
        T = int(inp.seq_lens[s])
        if paged:
            pt = inp.page_table.numpy()
            kc = oracle.gather_paged(cache.k.cpu().numpy(), pt, s, T)
            ks = oracle.gather_paged(cache.k_scale.cpu().numpy()[..., None], pt, s, T)[..., 0]
        else:
            kc, ks = cache.k[s, :, :T].cpu().numpy(), cache.k_scale[s, :, :T].cpu().numpy()
        rc, rs = oracle.quantize_residual_rope(seq_bits(inp, "k", s), b, cos, sin, np.arange(T, dtype=np.int32))
        assert np.array_equal(kc, rc), s
        assert np.array_equal(ks.view(np.uint32), rs.view(np.uint32)), s


@pytest.mark.parametrize("D,G", [(128, 8), (128, 1), (64, 4)])
@pytest.mark.parametrize("paged", [False, True])
def test_decode_matches_reconstructed_keys(D, G, paged):
    Hkv = 2
    inp, b, cos, sin = _workload("rope_dec", 5, G * Hkv, Hkv, D, seed=12 + G, len_range=(1, 1500),
                                 page_size=16 if paged else None, P=2048)
    bd, rope = _dev(b, cos, sin)
    cache = fill_cache(inp, "k8v8", capacity=1536, k_bias=bd, rope=rope)
    ref = oracle_decode(inp, "k8v8", range(5), k_bias=b, rope=(cos, sin))
    for kernel in ("auto", "cuda_cores"):
        for ns in (0, 1, 3):
            out = gpu_decode(inp, cache, num_splits=ns, kernel=kernel).cpu().numpy()
            assert_gate(out, ref, f"rope decode D{D} G{G} paged={paged} {kernel} splits={ns}")


def test_fused_step_appends_rotated_residual_row():
    inp, b, cos, sin = _workload("rope_step", 6, 16, 2, 128, seed=13, seq_lens=(1000, 1, 64, 65, 700, 999), P=1024)
    bd, rope = _dev(b, cos, sin)
    prev, knew, vnew = split_last_token(inp)
    cache = fill_cache(prev, "k8v8", capacity=1024, k_bias=bd, rope=rope)
    out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, cache, inp.seq_lens.cuda(),
                               out_dtype=torch.float32)
    assert_gate(out.cpu().numpy(), oracle_decode(inp, "k8v8", range(6), k_bias=b, rope=(cos, sin)), "rope step")
    kb = synth.bf16_bits(knew)
    for s in range(6):
        t = int(inp.seq_lens[s]) - 1
        rc, rs = oracle.quantize_residual_rope(kb[s][:, None, :], b, cos, sin, np.array([t], np.int32))
        assert np.array_equal(cache.k[s, :, t].cpu().numpy(), rc[:, 0]), s
        assert np.array_equal(cache.k_scale[s, :, t].cpu().numpy().view(np.uint32), rs[:, 0].view(np.uint32)), s


@pytest.mark.parametrize("page_size", [None, 16])
def test_prefill_matches_reconstructed_keys(page_size):
    n_q, Hq, Hkv, D = 300, 8, 2, 128
    pin = synth.prefill_inputs(synth.PrefillWorkload("rope_pf", n_q, Hq, Hkv, D, seed=34), device="cuda")
    b = _bias(Hkv, D, 34)
    cos, sin = _tables(320, D)
    k = (pin.k.float().cpu() + torch.from_numpy(_rotated(b, cos, sin, n_q).transpose(1, 0, 2)).float())
    k = k.to(torch.bfloat16)
    bd, rope = _dev(b, cos, sin)
    if page_size is None:
        cache = fk.Fp8KVCache.contiguous(1, Hkv, D, 320, "k8v8", k_bias=bd, rope_cos=rope[0], rope_sin=rope[1])
    else:
        perm = torch.randperm(20, generator=torch.Generator().manual_seed(3)).to(torch.int32)
        cache = fk.Fp8KVCache.paged(perm[None], 20, Hkv, D, page_size, "k8v8", k_bias=bd,
                                    rope_cos=rope[0], rope_sin=rope[1])
    fk.fp8kv_append(cache, k.cuda().contiguous(), pin.v.contiguous(), torch.zeros(n_q, dtype=torch.int32, device="cuda"),
                    torch.arange(n_q, dtype=torch.int32, device="cuda"))
    out = fk.fp8kv_prefill_attention(pin.q[None].contiguous(), cache, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                     out_dtype=torch.float32)[0].cpu().numpy()
    kb = synth.bf16_bits(k).transpose(1, 0, 2)
    pos = np.arange(n_q, dtype=np.int32)
    kk = oracle.residual_rope_keys(*oracle.quantize_residual_rope(kb, b, cos, sin, pos),
                                   oracle.rope_bias(b, cos, sin, pos))
    vv = oracle.dequantize(*oracle.quantize(synth.bf16_bits(pin.v).transpose(1, 0, 2)))
    ref = oracle.prefill_attention(oracle.bf16_to_double(synth.bf16_bits(pin.q)), kk, vv, 0, 1 / math.sqrt(D))
    assert_gate(out.reshape(-1, D), ref.reshape(-1, D), "rope prefill")


def test_tensor_cores_refuse_rotated_bias():
    b = torch.zeros(1, 128, device="cuda")
    c, s = torch.ones(64, 64, device="cuda"), torch.zeros(64, 64, device="cuda")
    cache = fk.Fp8KVCache.contiguous(1, 1, 128, 64, "k8v8", k_bias=b, rope_cos=c, rope_sin=s)
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(fk.Fp8KVError) as e:
        fk.fp8kv_decode_attention(q, cache, lens, kernel="tensor_cores")
    assert e.value.status == 2
    with pytest.raises(fk.Fp8KVError) as e:
        fk.fp8kv_prefill_attention(q[:, None].contiguous(), cache, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                   kernel="tensor_cores")
    assert e.value.status == 2


def test_rotated_residual_is_closer_to_bf16():
    """The numerical-safety claim for a bias that turns with position: the
    rotated residual beats both the plain per-row cache and a constant-bias
    residual (which cannot follow the rotation)."""
    inp, b, cos, sin = _workload("rope_q", 16, 16, 2, 128, seed=15, seq_lens=(512,) * 16, P=512)
    bd, rope = _dev(b, cos, sin)
    ref = oracle_decode(inp, "k16v16", range(16))
    plain = gpu_decode(inp, fill_cache(inp, "k8v8")).cpu().numpy()
    const = gpu_decode(inp, fill_cache(inp, "k8v8", k_bias=bd)).cpu().numpy()
    rot = gpu_decode(inp, fill_cache(inp, "k8v8", k_bias=bd, rope=rope)).cpu().numpy()
    err = lambda o: np.linalg.norm(o - ref) / np.linalg.norm(ref)
    assert err(rot) < 0.6 * err(plain), (err(rot), err(plain))
    assert err(rot) < 0.6 * err(const), (err(rot), err(const))

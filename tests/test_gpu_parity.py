"""GPU parity: the CUDA path through the C ABI against the oracle, element by
element on the same seeded bf16 inputs.

Bars (written here, from the method's statement): append/quantise codes and
scales bit-exact; attention within relative L2 1e-2 and max-abs 2e-2 per
(sequence, query head) of the fp64 oracle on the dequantised cache; split-KV
merge versus the unsplit run within 1e-5 relative (fp32 outputs)."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import (assert_gate, fill_cache, gpu_decode, k_fp8, oracle_decode, oracle_kv, seq_bits,
                       v_fp8)

pytestmark = pytest.mark.gpu
DTYPES = ["k8v8", "k16v8", "k16v16", "k8v16"]
KERNELS = ["cuda_cores", "tensor_cores"]


@pytest.fixture(autouse=True)
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield


# --------------------------------------------------------------- quantise --

@pytest.mark.parametrize("D", [64, 128])
def test_quantize_bit_exact(D):
    g = torch.Generator(device="cuda").manual_seed(11)
    rows = 4099                                  # several blocks and a ragged tail
    x = torch.randn(rows, D, generator=g, device="cuda")
    x = x * torch.exp(torch.randn(rows, 1, generator=g, device="cuda") * 4)
    x[5] = 0.0                                   # all-zero row
    x[6] = -0.0
    x[7, :] = 1e-30                              # subnormal-range quotients
    x[7, 3] = 2.0
    x[8, :] = -1e-7                              # values that round to -0
    x[8, 0] = 100.0
    xb = x.to(torch.bfloat16).contiguous()
    codes, scales = fk.fp8kv_quantize(xb)
    ref_c, ref_s = oracle.quantize(synth.bf16_bits(xb))
    got_c = codes.cpu().numpy()
    got_s = scales.cpu().numpy()
    bad = np.flatnonzero((got_c != ref_c).any(axis=1))
    assert bad.size == 0, f"code mismatch in rows {bad[:8]}: {got_c[bad[0]][:8]} vs {ref_c[bad[0]][:8]}"
    assert np.array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))


def test_quantize_every_code_and_tie():
    """Every E4M3 value and every midpoint between neighbours, as x/scale with
    scale = 1 (row amax 448): the hardware encode must match the oracle's."""
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    vals = np.concatenate([table, (table[:-1] + table[1:]) / 2])
    vals = np.concatenate([vals, -vals])
    n = (len(vals) + 126) // 127
    rows = np.zeros((n, 128), dtype=np.float32)
    rows[:, 0] = 448.0                           # amax 448 -> scale exactly 1
    flat = rows[:, 1:].reshape(-1)
    flat[:len(vals)] = vals
    rows[:, 1:] = flat.reshape(n, 127)
    xb = torch.tensor(rows).to(torch.bfloat16)
    assert torch.equal(xb.float(), torch.tensor(rows))   # all values exact in bf16
    codes, scales = fk.fp8kv_quantize(xb.cuda().contiguous())
    ref_c, ref_s = oracle.quantize(synth.bf16_bits(xb))
    assert np.all(ref_s == 1.0)
    assert np.array_equal(codes.cpu().numpy(), ref_c)


# ----------------------------------------------------------------- append --

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("paged", [False, True])
def test_append_bit_exact(dtype, paged):
    spec = synth.DecodeWorkload("append", 3, 4, 2, 128, seed=21, seq_lens=(77, 130, 16),
                                page_size=16 if paged else None)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, dtype)
    assert fk.fp8kv_get_device_error() == 0
    for b in range(3):
        T = int(inp.seq_lens[b])
        for which, fp8 in (("k", k_fp8(dtype)), ("v", v_fp8(dtype))):
            store = cache.k if which == "k" else cache.v
            if store.dtype == torch.bfloat16:
                store = store.view(torch.int16)
            sc = cache.k_scale if which == "k" else cache.v_scale
            if paged:
                got = oracle.gather_paged(store.cpu().numpy(), inp.page_table.numpy(), b, T)
                got_s = oracle.gather_paged(sc.cpu().numpy()[..., None], inp.page_table.numpy(), b, T)[..., 0] if fp8 else None
            else:
                got = store[b, :, :T].cpu().numpy()
                got_s = sc[b, :, :T].cpu().numpy() if fp8 else None
            bits = seq_bits(inp, which, b)
            if fp8:
                rc, rs = oracle.quantize(bits)
                assert np.array_equal(got, rc), (b, which)
                assert np.array_equal(got_s.view(np.uint32), rs.view(np.uint32)), (b, which)
            else:
                assert np.array_equal(got.view(np.uint16), bits), (b, which)


# ----------------------------------------------------------------- decode --

@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_tiny(dtype):
    """Batch 2, 4 q / 1 KV head, head_dim 64, lengths {77, 128}."""
    inp = synth.decode_inputs(synth.WORKLOADS["tiny_decode"], device="cuda")
    cache = fill_cache(inp, dtype)
    out = gpu_decode(inp, cache).cpu().numpy()
    ref = oracle_decode(inp, dtype, range(2))
    assert_gate(out, ref, f"tiny {dtype}")
    assert fk.fp8kv_get_device_error() == 0


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_ctx512(dtype, kernel):
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx512"], device="cuda")
    cache = fill_cache(inp, dtype)
    out = gpu_decode(inp, cache, kernel=kernel).cpu().numpy()
    ref = oracle_decode(inp, dtype, range(16))
    assert_gate(out, ref, f"ctx512 {dtype} {kernel}")


@pytest.mark.parametrize("kernel", ["auto"] + KERNELS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_ctx8192_full(dtype, kernel):
    """The benchmark workload at full size, in the benchmark's launch
    configuration (automatic splits, bf16 output)."""
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    cache = fill_cache(inp, dtype)
    out = gpu_decode(inp, cache, out_dtype=torch.bfloat16, kernel=kernel).float().cpu().numpy()
    ref = oracle_decode(inp, dtype, range(16))
    assert_gate(out, ref, f"ctx8192 {dtype} {kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_ragged_and_edge_lengths(dtype, kernel):
    lens = (0, 1, 2, 63, 64, 65, 127, 128, 129, 300, 1000, 17)
    spec = synth.DecodeWorkload("ragged", len(lens), 8, 1, 128, seed=5, seq_lens=lens)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, dtype, capacity=1024)
    for ns in (0, 1, 3):
        out = gpu_decode(inp, cache, num_splits=ns, kernel=kernel).cpu().numpy()
        ref = oracle_decode(inp, dtype, range(len(lens)))
        assert np.all(out[0] == 0), "zero-length sequence must give a zero row"
        assert_gate(out[1:], ref[1:], f"ragged {dtype} {kernel} splits={ns}")


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8])
def test_decode_group_sizes(G):
    spec = synth.DecodeWorkload("groups", 3, 2 * G, 2, 64, seed=6, seq_lens=(100, 257, 64))
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, "k8v8")
    out = gpu_decode(inp, cache).cpu().numpy()
    assert_gate(out, oracle_decode(inp, "k8v8", range(3)), f"G={G}")


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8])
def test_decode_group_sizes_tensor_cores(G):
    spec = synth.DecodeWorkload("groups128", 3, 2 * G, 2, 128, seed=16, seq_lens=(100, 257, 128))
    inp = synth.decode_inputs(spec, device="cuda")
    for dtype in DTYPES:
        cache = fill_cache(inp, dtype)
        out = gpu_decode(inp, cache, kernel="tensor_cores").cpu().numpy()
        assert_gate(out, oracle_decode(inp, dtype, range(3)), f"G={G} {dtype}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", DTYPES)
def test_decode_paged_small(dtype, kernel):
    spec = synth.DecodeWorkload("paged_small", 6, 16, 4, 128, seed=7, len_range=(1, 700),
                                page_size=16, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, dtype)
    out = gpu_decode(inp, cache, kernel=kernel).cpu().numpy()
    assert_gate(out, oracle_decode(inp, dtype, range(6)), f"paged small {dtype} {kernel}")


@pytest.mark.parametrize("kernel", ["auto"] + KERNELS)
@pytest.mark.parametrize("dtype", ["k8v8", "k16v8"])
def test_decode_paged_b64_full_sampled(dtype, kernel):
    """The paged serving workload at full size (64 sequences up to 16384
    tokens, hostile keys); the oracle checks a sample of sequences."""
    inp = synth.decode_inputs(synth.WORKLOADS["paged_b64_hostile"], device="cuda")
    cache = fill_cache(inp, dtype)
    out = gpu_decode(inp, cache, out_dtype=torch.bfloat16, kernel=kernel).float().cpu().numpy()
    lens = inp.seq_lens.numpy()
    sample = sorted({int(lens.argmin()), int(lens.argmax()), 7, 33})
    ref = oracle_decode(inp, dtype, sample)
    assert_gate(out[sample], ref, f"paged b64 {dtype} {kernel}")
    assert fk.fp8kv_get_device_error() == 0


@pytest.mark.parametrize("kernel", KERNELS)
def test_split_invariance_ctx8192(kernel):
    """Split-KV merge versus unsplit: fp32 outputs within 1e-5 relative."""
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    for dtype in DTYPES:
        cache = fill_cache(inp, dtype)
        one = gpu_decode(inp, cache, num_splits=1, kernel=kernel).double()
        for ns in (0, 7, 64):
            many = gpu_decode(inp, cache, num_splits=ns, kernel=kernel).double()
            rel = ((many - one).norm(dim=-1) / one.norm(dim=-1)).max().item()
            assert rel <= 1e-5, f"{dtype} {kernel} splits={ns}: rel {rel:.3e}"


def test_tensor_core_path_subnormal_codes_and_tiny_queries():
    """Rows whose amax is far above the rest put most codes in the E4M3
    subnormal range; queries with components spanning many binades exercise
    the two-term e4m3 split of Q and P.  Checked against the oracle."""
    g = torch.Generator(device="cuda").manual_seed(17)
    B, Hq, Hkv, D, T = 2, 8, 1, 128, 300
    # amax 2 per row: every other element (|x| < 2 * 2^-6 / 448) gets a
    # subnormal E4M3 code; outputs stay O(1), where the max-abs bar applies
    k = torch.randn(B * T, Hkv, D, generator=g, device="cuda") * 3e-5
    k[:, :, 5] = 2.0
    v = torch.randn(B * T, Hkv, D, generator=g, device="cuda") * 3e-5
    v[:, :, 9] = -2.0
    q = torch.randn(B, Hq, D, generator=g, device="cuda") * torch.exp(
        torch.randn(B, Hq, D, generator=g, device="cuda") * 3)
    q[:, :, 5] = 1e-3                                      # keep the huge channel from dominating
    spec = synth.DecodeWorkload("subnormal", B, Hq, Hkv, D, seed=0, seq_lens=(T, T))
    inp = synth.DecodeInputs(spec, q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
                             torch.tensor([T, T], dtype=torch.int32),
                             torch.tensor([0, T, 2 * T], dtype=torch.int64))
    for dtype in DTYPES:
        cache = fill_cache(inp, dtype)
        if dtype == "k8v8":
            codes = cache.k[:, :, :T].cpu().numpy()
            assert np.mean((codes & 0x78) == 0) > 0.5          # most K codes subnormal
        ref = oracle_decode(inp, dtype, range(B))
        for kernel in KERNELS:
            out = gpu_decode(inp, cache, kernel=kernel).cpu().numpy()
            assert_gate(out, ref, f"subnormal {dtype} {kernel}")


def test_gpu_output_fails_gate_against_broken_oracle_scales():
    """The gate has teeth ("FP8 KV cache (fp8_kv, opt-in)", bullet
    "Accuracy"): the GPU output passes against the oracle on the correct
    cache and fails against the oracle fed V scales x1.05, or one token's K
    scale for all tokens.  The mistakes are planted in the oracle's inputs."""
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx512"], device="cuda")
    cache = fill_cache(inp, "k8v8")
    out = gpu_decode(inp, cache).cpu().numpy()[:4]
    q = oracle.bf16_to_double(synth.bf16_bits(inp.q))[:4]
    D, T = 128, 512
    sm = 1 / math.sqrt(D)
    ks, vs, kc, vc = [], [], [], []
    for b in range(4):
        c, s = oracle.quantize(seq_bits(inp, "k", b)); kc.append(c); ks.append(s)
        c, s = oracle.quantize(seq_bits(inp, "v", b)); vc.append(c); vs.append(s)
    kc, ks, vc, vs = map(np.stack, (kc, ks, vc, vs))
    lens = np.full(4, T, np.int32)
    good = oracle.decode_attention(q, oracle.dequantize(kc, ks), oracle.dequantize(vc, vs), lens, sm)
    assert oracle.attention_gate(out, good)[0]
    bad_v = oracle.decode_attention(q, oracle.dequantize(kc, ks), oracle.dequantize(vc, vs * 1.05), lens, sm)
    assert not oracle.attention_gate(out, bad_v)[0]
    one = np.broadcast_to(ks[..., :1], ks.shape)
    bad_k = oracle.decode_attention(q, oracle.dequantize(kc, one), oracle.dequantize(vc, vs), lens, sm)
    assert not oracle.attention_gate(out, bad_k)[0]


@pytest.mark.parametrize("kernel", KERNELS)
def test_decode_repeat_is_bitwise_stable(kernel):
    """Standalone repeat harness ("03 · 8n", section 4): many launches on the
    same inputs give bitwise-identical outputs."""
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx512"], device="cuda")
    cache = fill_cache(inp, "k8v8")
    first = gpu_decode(inp, cache, kernel=kernel)
    for _ in range(200):
        assert torch.equal(gpu_decode(inp, cache, kernel=kernel), first)


# ---------------------------------------------------------------- prefill --

def _prefill_case(n_q, pos0, Hq, Hkv, D, dtype, seed, sample_blocks=None, kernel="auto"):
    spec = synth.PrefillWorkload("pf", n_q, Hq, Hkv, D, seed=seed, pos0=pos0)
    pin = synth.prefill_inputs(spec, device="cuda")
    total = pos0 + n_q
    cap = ((total + 63) // 64) * 64
    cache = fk.Fp8KVCache.contiguous(1, Hkv, D, cap, dtype)
    fk.fp8kv_append(cache, pin.k.contiguous(), pin.v.contiguous(),
                    torch.zeros(total, dtype=torch.int32, device="cuda"),
                    torch.arange(total, dtype=torch.int32, device="cuda"))
    out = fk.fp8kv_prefill_attention(pin.q[None].contiguous(), cache,
                                     torch.tensor([pos0], dtype=torch.int32, device="cuda"),
                                     out_dtype=torch.float32, kernel=kernel)[0].cpu().numpy()
    kb = synth.bf16_bits(pin.k).transpose(1, 0, 2)
    vb = synth.bf16_bits(pin.v).transpose(1, 0, 2)
    k = oracle.dequantize(*oracle.quantize(kb)) if k_fp8(dtype) else oracle.bf16_to_double(kb)
    v = oracle.dequantize(*oracle.quantize(vb)) if v_fp8(dtype) else oracle.bf16_to_double(vb)
    q = oracle.bf16_to_double(synth.bf16_bits(pin.q))
    sm = 1 / math.sqrt(D)
    blocks = sample_blocks or [(0, n_q)]
    for a, e in blocks:
        ref = oracle.prefill_attention(q[a:e], k[:, :pos0 + e], v[:, :pos0 + e], pos0 + a, sm)
        assert_gate(out[a:e].reshape(-1, D), ref.reshape(-1, D), f"prefill rows {a}:{e} {dtype}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_prefill_small_ragged(dtype):
    _prefill_case(200, 0, 4, 2, 128, dtype, seed=31, kernel="cuda_cores")


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_small_ragged_k8v8_both_kernels(kernel):
    _prefill_case(200, 0, 4, 2, 128, "k8v8", seed=31, kernel=kernel)


@pytest.mark.parametrize("dtype", DTYPES)
def test_prefill_with_prefix_offset(dtype):
    _prefill_case(77, 37, 6, 2, 64, dtype, seed=32)


@pytest.mark.parametrize("kernel", KERNELS)
def test_prefill_2048_full_sampled(kernel):
    """Causal prefill at full size (2048 tokens, 28 q / 4 KV heads), oracle on
    sampled query blocks that straddle tile boundaries."""
    _prefill_case(2048, 0, 28, 4, 128, "k8v8", seed=4, kernel=kernel,
                  sample_blocks=[(0, 70), (1000, 1090), (1980, 2048)])


# ------------------------------------------------------- device-side checks --

def test_device_error_on_length_beyond_capacity():
    spec = synth.DecodeWorkload("cap", 2, 4, 1, 64, seed=8, seq_lens=(50, 60))
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, "k8v8", capacity=64)
    lens = torch.tensor([50, 4096], dtype=torch.int32, device="cuda")
    out = fk.fp8kv_decode_attention(inp.q.cuda().contiguous(), cache, lens, out_dtype=torch.float32)
    bits = fk.fp8kv_get_device_error()
    assert bits & fk.DEVERR_SEQ_TOO_LONG
    assert torch.all(out[1] == 0)


def test_device_error_on_bad_page():
    spec = synth.DecodeWorkload("badpage", 2, 4, 1, 64, seed=9, seq_lens=(40, 40), page_size=16)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, "k8v8")
    assert fk.fp8kv_get_device_error() == 0
    cache.page_table[1, 1] = inp.num_pages + 1000          # out of range: skipped, flagged
    fk.fp8kv_decode_attention(inp.q.cuda().contiguous(), cache, inp.seq_lens.cuda())
    assert fk.fp8kv_get_device_error() & fk.DEVERR_BAD_PAGE


def test_abi_rejects_bad_arguments():
    inp = synth.decode_inputs(synth.WORKLOADS["tiny_decode"], device="cuda")
    cache = fill_cache(inp, "k8v8")
    q = inp.q.cuda().contiguous()
    lens = inp.seq_lens.cuda()
    with pytest.raises(fk.Fp8KVError) as e:
        fk.fp8kv_decode_attention(q, cache, lens, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3
    q9 = torch.zeros(2, 9, 64, dtype=torch.bfloat16, device="cuda")   # 9 heads over 1 KV head
    with pytest.raises(fk.Fp8KVError) as e:
        fk.fp8kv_decode_attention(q9, cache, lens)
    assert e.value.status == 2

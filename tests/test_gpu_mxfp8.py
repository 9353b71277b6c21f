"""MXFP8 keys (cache dtype "mxk8v8"): e4m3 codes with one E8M0 scale per
32-dim block of each K row, V as e4m3 with a per-row fp32 scale.  The
quantiser and the appends are bit-exact against the oracle; the decode on
both kernels (split, merge, fused step) and the CUDA-core prefill are held to
the attention gate against the oracle's fp64 attention over the
block-dequantised keys."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import assert_gate, fill_cache, gpu_decode, oracle_decode, seq_bits

pytestmark = pytest.mark.gpu
MX = "mxk8v8"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(autouse=True)
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield


def _wide_rows(seed, n, d):
    """bf16 rows whose 32-element blocks span 2^-140 .. 2^120, with zero
    blocks, negative zeros, spikes and subnormals."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g) * torch.exp2(torch.randint(-140, 120, (n, d // 32), generator=g)
                                                  .float().repeat_interleave(32, dim=1))
    x[::17, :32] = 0.0
    x[3::19, 32:64] = -0.0
    x[5::23, 40] = 1e30
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("D", [64, 128])
def test_quantize_mx_bit_exact(D):
    x = _wide_rows(31, 4099, D)
    codes, scales = fk.fp8kv_quantize_mx(x.cuda())
    rc, rs = oracle.mx_quantize(synth.bf16_bits(x))
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


def test_quantize_mx_worked_row_and_every_code():
    kv = {}
    with open(os.path.join(GOLDEN, "mx_quantize_worked_row.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                key, *vals = line.split()
                kv[key] = [int(h, 16) for h in vals]
    x = torch.from_numpy(np.array(kv["input"], dtype=np.uint16).view(np.int16)).view(torch.bfloat16)[None].cuda()
    codes, scales = fk.fp8kv_quantize_mx(x)
    assert codes[0].cpu().tolist() == kv["codes"] and scales[0].cpu().tolist() == kv["e8m0"]
    # every finite e4m3 value and every midpoint between neighbours, in
    # blocks whose largest magnitude pins the scale to 2^0 (amax 448)
    grid = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    pos = np.unique(grid[np.isfinite(grid) & (grid >= 0)])
    vals = np.concatenate([pos, (pos[1:] + pos[:-1]) / 2])
    vals = np.concatenate([vals, -vals])
    n = ((len(vals) + 30) // 31 + 3) // 4 * 4          # 32-element blocks, four per 128-wide row
    blocks = np.zeros((n, 32))
    blocks[:, 0] = 448.0
    blocks[:, 1:].flat[:len(vals)] = vals
    rows = blocks.reshape(n // 4, 128)
    bits = synth.bf16_bits(torch.from_numpy(rows).to(torch.bfloat16))
    codes, scales = fk.fp8kv_quantize_mx(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda())
    rc, rs = oracle.mx_quantize(bits)
    assert np.all(rs == 127)
    assert np.array_equal(codes.cpu().numpy(), rc)


@pytest.mark.parametrize("paged", [False, True])
def test_append_bit_exact(paged):
    spec = synth.DecodeWorkload("append_mx", 3, 4, 2, 128, seed=21, seq_lens=(77, 130, 16),
                                page_size=16 if paged else None, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, MX)
    assert fk.fp8kv_get_device_error() == 0
    for b in range(3):
        T = int(inp.seq_lens[b])
        if paged:
            pt = inp.page_table.numpy()
            kc = oracle.gather_paged(cache.k.cpu().numpy(), pt, b, T)
            ks = oracle.gather_paged(cache.k_scale.cpu().numpy(), pt, b, T)
            vc = oracle.gather_paged(cache.v.cpu().numpy(), pt, b, T)
            vs = oracle.gather_paged(cache.v_scale.cpu().numpy()[..., None], pt, b, T)[..., 0]
        else:
            kc, ks = cache.k[b, :, :T].cpu().numpy(), cache.k_scale[b, :, :T].cpu().numpy()
            vc, vs = cache.v[b, :, :T].cpu().numpy(), cache.v_scale[b, :, :T].cpu().numpy()
        rkc, rks = oracle.mx_quantize(seq_bits(inp, "k", b))
        rvc, rvs = oracle.quantize(seq_bits(inp, "v", b))
        assert np.array_equal(kc, rkc) and np.array_equal(ks, rks), b
        assert np.array_equal(vc, rvc) and np.array_equal(vs.view(np.uint32), rvs.view(np.uint32)), b


@pytest.mark.parametrize("wl", ["decode_b16_ctx512", "decode_b16_ctx8192"])
def test_decode_full(wl):
    inp = synth.decode_inputs(synth.WORKLOADS[wl], device="cuda")
    cache = fill_cache(inp, MX)
    out = gpu_decode(inp, cache, out_dtype=torch.bfloat16).float().cpu().numpy()
    assert_gate(out, oracle_decode(inp, MX, range(16)), f"{wl} mx")
    assert fk.fp8kv_get_device_error() == 0


def test_decode_ragged_edge_lengths_and_splits():
    lens = (0, 1, 2, 63, 64, 65, 127, 128, 129, 300, 1000, 17)
    spec = synth.DecodeWorkload("ragged_mx", len(lens), 8, 1, 128, seed=5, seq_lens=lens, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, MX, capacity=1024)
    ref = oracle_decode(inp, MX, range(len(lens)))
    for ns in (0, 1, 3):
        out = gpu_decode(inp, cache, num_splits=ns, kernel="tensor_cores").cpu().numpy()
        assert np.all(out[0] == 0)
        assert_gate(out[1:], ref[1:], f"ragged mx splits={ns}")


def test_decode_paged_hostile():
    spec = synth.DecodeWorkload("paged_mx", 6, 16, 4, 128, seed=7, len_range=(1, 700),
                                page_size=16, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, MX)
    out = gpu_decode(inp, cache).cpu().numpy()
    assert_gate(out, oracle_decode(inp, MX, range(6)), "paged mx")


def test_fused_step_appends_mx_row_and_matches_oracle():
    from test_gpu_decode_step import _run
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    cache, out, knew, _ = _run(inp, MX, "auto")
    assert fk.fp8kv_get_device_error() == 0
    assert_gate(out.cpu().numpy(), oracle_decode(inp, MX, range(16)), "step mx")
    codes, scales = oracle.mx_quantize(synth.bf16_bits(knew))
    assert np.array_equal(cache.k[:, :, 8191].cpu().numpy(), codes)
    assert np.array_equal(cache.k_scale[:, :, 8191].cpu().numpy(), scales)


def test_split_invariance():
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    cache = fill_cache(inp, MX)
    one = gpu_decode(inp, cache, num_splits=1).double()
    for ns in (0, 7, 64):
        many = gpu_decode(inp, cache, num_splits=ns).double()
        rel = ((many - one).norm(dim=-1) / one.norm(dim=-1)).max().item()
        assert rel <= 1e-5, f"splits={ns}: rel {rel:.3e}"


def test_unbuilt_kernels_rejected():
    """The transform paths (f16 K tiles) and the tensor-core prefill are not
    built for MXFP8 keys: FP8KV_ERR_UNSUPPORTED."""
    cache = fk.Fp8KVCache.contiguous(1, 1, 128, 64, MX)
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    for kernel in ("tensor_cores_k_f16", "tensor_cores_k_f16_producer"):
        with pytest.raises(fk.Fp8KVError) as e:
            fk.fp8kv_decode_attention(q, cache, lens, kernel=kernel)
        assert e.value.status == 2
    with pytest.raises(fk.Fp8KVError) as e:
        fk.fp8kv_prefill_attention(q[:, None].contiguous(), cache, torch.zeros(1, dtype=torch.int32, device="cuda"),
                                   kernel="tensor_cores")
    assert e.value.status == 2


# ---------------------------------------------------------------- CUDA cores

def test_cuda_cores_decode_full_and_hostile():
    """The CUDA-core split weights each 32-dim block's partial dot by its
    E8M0 scale (each thread's half row holds two blocks)."""
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx512"], device="cuda")
    cache = fill_cache(inp, MX)
    out = gpu_decode(inp, cache, kernel="cuda_cores").cpu().numpy()
    assert_gate(out, oracle_decode(inp, MX, range(16)), "ctx512 mx cuda cores")
    tc = gpu_decode(inp, cache, kernel="tensor_cores").cpu().numpy()
    assert_gate(out, tc, "mx cuda cores vs tensor cores")
    assert fk.fp8kv_get_device_error() == 0


@pytest.mark.parametrize("G", [1, 3, 8])
def test_cuda_cores_decode_ragged_paged(G):
    lens = (0, 1, 31, 64, 65, 200, 513)
    spec = synth.DecodeWorkload(f"mx_fma_G{G}", len(lens), 2 * G, 2, 128, seed=60 + G, seq_lens=lens,
                                page_size=16, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, MX)
    ref = oracle_decode(inp, MX, range(len(lens)))
    for ns in (0, 1, 5):
        out = gpu_decode(inp, cache, num_splits=ns, kernel="cuda_cores").cpu().numpy()
        assert np.all(out[0] == 0)
        assert_gate(out[1:], ref[1:], f"mx cuda cores G{G} splits={ns}")
    assert fk.fp8kv_get_device_error() == 0


def test_cuda_cores_fused_step():
    from test_gpu_decode_step import _run
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx512"], device="cuda")
    cache, out, knew, _ = _run(inp, MX, "cuda_cores")
    assert fk.fp8kv_get_device_error() == 0
    assert_gate(out.cpu().numpy(), oracle_decode(inp, MX, range(16)), "step mx cuda cores")
    T = int(inp.seq_lens[0])
    codes, scales = oracle.mx_quantize(synth.bf16_bits(knew))
    assert np.array_equal(cache.k[:, :, T - 1].cpu().numpy(), codes)
    assert np.array_equal(cache.k_scale[:, :, T - 1].cpu().numpy(), scales)


# ------------------------------------------------------------------ prefill

def _prefill_case(B, n_q, pos0s, Hq, Hkv, seed, page_size=None):
    D = 128
    qs, ks, vs = [], [], []
    for b in range(B):
        spec = synth.PrefillWorkload("pf_mx", n_q, Hq, Hkv, D, seed=seed + b, pos0=pos0s[b])
        pin = synth.prefill_inputs(spec, device="cuda")
        qs.append(pin.q)
        ks.append(pin.k)
        vs.append(pin.v)
    totals = [p + n_q for p in pos0s]
    if page_size is None:
        cache = fk.Fp8KVCache.contiguous(B, Hkv, D, (max(totals) + 15) // 16 * 16, MX)
    else:
        per = [(t + page_size - 1) // page_size for t in totals]
        num_pages = sum(per) + 2
        perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(seed)).to(torch.int32)
        table = torch.full((B, max(per)), -1, dtype=torch.int32)
        off = 0
        for b in range(B):
            table[b, :per[b]] = perm[off:off + per[b]]
            off += per[b]
        cache = fk.Fp8KVCache.paged(table, num_pages, Hkv, D, page_size, MX)
    seq_idx = torch.cat([torch.full((t,), b, dtype=torch.int32) for b, t in enumerate(totals)])
    pos = torch.cat([torch.arange(t, dtype=torch.int32) for t in totals])
    fk.fp8kv_append(cache, torch.cat(ks).contiguous(), torch.cat(vs).contiguous(), seq_idx.cuda(), pos.cuda())
    return cache, torch.stack(qs).contiguous(), ks, vs


@pytest.mark.parametrize("page_size", [None, 32])
@pytest.mark.parametrize("kernel", ["auto", "cuda_cores"])
def test_prefill_mx(kernel, page_size):
    """Causal prefill over MXFP8 keys (the CUDA-core kernel, which applies
    each block's scale where it converts the codes), two sequences with
    different prefixes, against the oracle over the block-dequantised keys."""
    pos0s = [0, 45]
    cache, q, ks, vs = _prefill_case(2, 150, pos0s, 8, 2, seed=71, page_size=page_size)
    out = fk.fp8kv_prefill_attention(q, cache, torch.tensor(pos0s, dtype=torch.int32, device="cuda"),
                                     out_dtype=torch.float32, kernel=kernel).cpu().numpy()
    assert fk.fp8kv_get_device_error() == 0
    D = 128
    for b in range(2):
        k = oracle.mx_dequantize(*oracle.mx_quantize(synth.bf16_bits(ks[b]).transpose(1, 0, 2)))
        v = oracle.dequantize(*oracle.quantize(synth.bf16_bits(vs[b]).transpose(1, 0, 2)))
        qd = oracle.bf16_to_double(synth.bf16_bits(q[b]))
        ref = oracle.prefill_attention(qd, k[:, :pos0s[b] + 150], v[:, :pos0s[b] + 150], pos0s[b], 1 / math.sqrt(D))
        assert_gate(out[b].reshape(-1, D), ref.reshape(-1, D), f"prefill mx seq {b} {kernel} P{page_size}")

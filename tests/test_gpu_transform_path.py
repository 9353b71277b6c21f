"""The tensor-core decode on the transform path: each landed e4m3 K tile is
converted to f16 in shared memory and QK runs as a 16-bit MMA on an f16 query,
the conversion done by the softmax warpgroup that owns the tile (kernel
"tensor_cores_k_f16") or by the producer warp ("tensor_cores_k_f16_producer").
The same parity gate as the native e4m3 path, on the same seeded inputs, at
the benchmark's size and at ragged, paged and fused-step shapes."""
import numpy as np
import pytest
import torch

from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import assert_gate, fill_cache, gpu_decode, oracle_decode

pytestmark = pytest.mark.gpu
XF = ["tensor_cores_k_f16", "tensor_cores_k_f16_producer"]


@pytest.fixture(autouse=True)
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield
    assert fk.fp8kv_get_device_error() == 0


@pytest.mark.parametrize("KF16", XF)
def test_ctx8192_full(KF16):
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    cache = fill_cache(inp, "k8v8")
    out = gpu_decode(inp, cache, out_dtype=torch.bfloat16, kernel=KF16).float().cpu().numpy()
    ref = oracle_decode(inp, "k8v8", range(16))
    assert_gate(out, ref, "ctx8192 k_f16")
    nat = gpu_decode(inp, cache, out_dtype=torch.bfloat16, kernel="tensor_cores").float().cpu().numpy()
    assert_gate(nat, ref, "ctx8192 native")
    again = gpu_decode(inp, cache, out_dtype=torch.bfloat16, kernel=KF16).float().cpu().numpy()
    assert np.array_equal(out, again), "transform path not repeatable"


@pytest.mark.parametrize("KF16", XF)
def test_ragged_and_edge_lengths(KF16):
    lens = (0, 1, 2, 63, 64, 65, 127, 128, 129, 300, 1000, 17)
    spec = synth.DecodeWorkload("ragged", len(lens), 8, 1, 128, seed=5, seq_lens=lens)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, "k8v8", capacity=1024)
    ref = oracle_decode(inp, "k8v8", range(len(lens)))
    for ns in (0, 1, 3):
        out = gpu_decode(inp, cache, num_splits=ns, kernel=KF16).cpu().numpy()
        assert np.all(out[0] == 0), "zero-length sequence must give a zero row"
        assert_gate(out[1:], ref[1:], f"ragged k_f16 splits={ns}")


@pytest.mark.parametrize("KF16", XF)
@pytest.mark.parametrize("G", [1, 4, 8])
def test_group_sizes_and_paged(G, KF16):
    spec = synth.DecodeWorkload("paged_kf16", 5, 2 * G, 2, 128, seed=17, len_range=(1, 900),
                                page_size=32, hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    cache = fill_cache(inp, "k8v8")
    out = gpu_decode(inp, cache, kernel=KF16).cpu().numpy()
    assert_gate(out, oracle_decode(inp, "k8v8", range(5)), f"paged k_f16 G={G}")


@pytest.mark.parametrize("KF16", XF)
def test_query_magnitudes(KF16):
    """Query rows from 1e-30 to 1e30: the f16 query's power-of-two row scale
    keeps every row in range."""
    spec = synth.DecodeWorkload("qmag", 2, 8, 1, 128, seed=23, seq_lens=(300, 129))
    inp = synth.decode_inputs(spec, device="cuda")
    scale = torch.tensor([1e-30, 1e-8, 1e-2, 1.0, 3.0, 1e4, 1e12, 1e30], device="cuda")
    q = (inp.q.float() * scale[None, :, None]).to(torch.bfloat16)
    inp = synth.DecodeInputs(spec, q, inp.k, inp.v, inp.seq_lens, inp.cu_seqlens)
    cache = fill_cache(inp, "k8v8")
    out = gpu_decode(inp, cache, kernel=KF16).cpu().numpy()
    assert np.all(np.isfinite(out))
    assert_gate(out, oracle_decode(inp, "k8v8", range(2)), "query magnitudes k_f16")


@pytest.mark.parametrize("KF16", XF)
def test_fused_step_matches_oracle_and_native_step(KF16):
    from test_gpu_decode_step import _run
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    cache, out, _, _ = _run(inp, "k8v8", KF16)
    assert_gate(out.cpu().numpy(), oracle_decode(inp, "k8v8", range(16)), "step k_f16")
    _, nat, _, _ = _run(inp, "k8v8", "tensor_cores")
    rel = ((out.double() - nat.double()).norm(dim=-1) / nat.double().norm(dim=-1)).max().item()
    assert rel < 1e-2, rel


@pytest.mark.parametrize("KF16", XF)
def test_other_dtypes_rejected(KF16):
    for dtype in ("k16v8", "k16v16", "k8v16"):
        cache = fk.Fp8KVCache.contiguous(1, 1, 128, 64, dtype)
        assert fk.fp8kv_decode_num_splits(cache, 8, 0, KF16) == 0
        q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(fk.Fp8KVError) as e:
            fk.fp8kv_decode_attention(q, cache, torch.ones(1, dtype=torch.int32, device="cuda"), kernel=KF16)
        assert e.value.status == 2

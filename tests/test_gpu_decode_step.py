"""fp8kv_decode_step: append the new token of every sequence and decode in
one call (one launch on the tensor-core kernel).  Checked against the oracle
over the full length, the appended rows bit-exact against the oracle's
quantiser, and against the separate append + decode calls."""
import numpy as np
import pytest
import torch

import oracle
from fp8_quantized_kv_gb300 import synth
import fp8_quantized_kv_gb300 as fk
from kvhelpers import assert_gate, fill_cache, oracle_decode, split_last_token as _split_last_token

pytestmark = pytest.mark.gpu
DTYPES = ["k8v8", "k16v8", "k16v16", "k8v16"]


@pytest.fixture(autouse=True)
def _clear_device_error():
    fk.fp8kv_get_device_error(clear=True)
    yield


def _run(inp, dtype, kernel, num_splits=0, capacity=None):
    prev, knew, vnew = _split_last_token(inp)
    cache = fill_cache(prev, dtype, capacity=capacity or max(16, ((inp.max_len + 127) // 128) * 128))
    lens = inp.seq_lens.cuda()
    out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, cache, lens, num_splits=num_splits,
                               out_dtype=torch.float32, kernel=kernel)
    return cache, out, knew, vnew


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_step_ctx8192_full(dtype, kernel):
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    cache, out, knew, vnew = _run(inp, dtype, kernel)
    assert fk.fp8kv_get_device_error() == 0
    assert_gate(out.cpu().numpy(), oracle_decode(inp, dtype, range(16)), f"step {dtype} {kernel}")
    # the appended row is exactly what the quantiser writes
    if dtype == "k8v8":
        codes, scales = oracle.quantize(synth.bf16_bits(knew))
        got = cache.k[:, :, 8191].cpu().numpy()
        assert np.array_equal(got, codes)
        assert np.array_equal(cache.k_scale[:, :, 8191].cpu().numpy().view(np.uint32), scales.view(np.uint32))


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
def test_step_matches_separate_calls_and_resets_counters(kernel):
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx512"], device="cuda")
    prev, knew, vnew = _split_last_token(inp)
    c1 = fill_cache(prev, "k8v8", capacity=512)
    c2 = fill_cache(prev, "k8v8", capacity=512)
    lens = inp.seq_lens.cuda()
    q = inp.q.cuda().contiguous()
    ws = torch.zeros(fk.fp8kv_decode_step_workspace_bytes(c1, 16, 0, kernel), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):                      # same workspace: the counters must come back to zero
        outs.append(fk.fp8kv_decode_step(q, knew, vnew, c1, lens, out_dtype=torch.float32, workspace=ws,
                                         kernel=kernel))
    torch.cuda.synchronize()
    assert torch.count_nonzero(ws[-(16 * 2 * 4):]) == 0 or kernel == "cuda_cores"
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    fk.fp8kv_append(c2, knew, vnew, torch.arange(16, dtype=torch.int32, device="cuda"),
                    (lens - 1).to(torch.int32))
    sep = fk.fp8kv_decode_attention(q, c2, lens, out_dtype=torch.float32, kernel=kernel)
    assert torch.equal(c1.k, c2.k) and torch.equal(c1.k_scale, c2.k_scale)
    rel = ((outs[0].double() - sep.double()).norm(dim=-1) / sep.double().norm(dim=-1)).max().item()
    assert rel <= 1e-5, rel


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_step_ragged_splits_and_empty(dtype, kernel):
    lens = (0, 1, 2, 127, 128, 129, 300, 1000, 17, 256)
    spec = synth.DecodeWorkload("ragged_step", len(lens), 8, 1, 128, seed=25, seq_lens=lens)
    inp = synth.decode_inputs(spec, device="cuda")
    # 2..8 splits: the tensor-core step merges inside a thread-block cluster;
    # more splits (12, and the automatic count here): through global partials
    for ns in (0, 1, 2, 3, 8, 12):
        cache, out, _, _ = _run(inp, dtype, kernel, num_splits=ns, capacity=1024)
        o = out.cpu().numpy()
        assert np.all(o[0] == 0)
        assert_gate(o[1:], oracle_decode(inp, dtype, range(1, len(lens))), f"step ragged {dtype} {kernel} {ns}")
    assert fk.fp8kv_get_device_error() == 0


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
def test_step_paged(kernel):
    spec = synth.DecodeWorkload("paged_step", 6, 16, 4, 128, seed=27, len_range=(1, 900), page_size=16,
                                hostile_keys=True)
    inp = synth.decode_inputs(spec, device="cuda")
    prev, knew, vnew = _split_last_token(inp)
    cache = fill_cache(prev, "k8v8")            # paged pool sized for the full lengths
    out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, cache, inp.seq_lens.cuda(),
                               out_dtype=torch.float32, kernel=kernel)
    assert_gate(out.cpu().numpy(), oracle_decode(inp, "k8v8", range(6)), f"step paged {kernel}")
    assert fk.fp8kv_get_device_error() == 0


def test_step_split_invariance_cluster_and_global_merge():
    """The fused tensor-core step at 1 split (no merge), 2-8 splits (merge in
    a thread-block cluster) and 12-16 splits (merge through global partials)
    agrees within the split-merge bar of 1e-5 relative."""
    spec = synth.DecodeWorkload("inv_step", 4, 16, 2, 128, seed=29, seq_lens=(4096, 3000, 2049, 1))
    inp = synth.decode_inputs(spec, device="cuda")
    prev, knew, vnew = _split_last_token(inp)
    q = inp.q.cuda().contiguous()
    lens = inp.seq_lens.cuda()
    outs = {}
    for ns in (1, 2, 4, 5, 8, 12, 16):
        cache = fill_cache(prev, "k8v8", capacity=4096)
        outs[ns] = fk.fp8kv_decode_step(q, knew, vnew, cache, lens, num_splits=ns, out_dtype=torch.float32,
                                        kernel="tensor_cores").double()
    assert fk.fp8kv_get_device_error() == 0
    ref = outs[1]
    for ns, o in outs.items():
        rel = ((o - ref).norm(dim=-1) / ref.norm(dim=-1)).max().item()
        assert rel <= 1e-5, (ns, rel)


@pytest.mark.parametrize("G", [4, 8])
def test_step_global_merge_many_partials(G):
    """The in-kernel global merge with more (query head, split) partials than
    the 128 merging threads, and with more splits than one staging chunk
    (44): one KV head, 8192 tokens, up to 64 one-tile splits."""
    spec = synth.DecodeWorkload("many_parts", 2, G, 1, 128, seed=61, seq_lens=(8192, 5000))
    inp = synth.decode_inputs(spec, device="cuda")
    ref = oracle_decode(inp, "k8v8", range(2))
    outs = {}
    for ns in (1, 17, 33, 45, 64):
        _, out, _, _ = _run(inp, "k8v8", "tensor_cores", num_splits=ns, capacity=8192)
        assert fk.fp8kv_get_device_error() == 0
        assert_gate(out.cpu().numpy(), ref, f"G{G} splits {ns}")
        outs[ns] = out.double()
    for ns, o in outs.items():
        rel = ((o - outs[1]).norm(dim=-1) / outs[1].norm(dim=-1)).max().item()
        assert rel <= 1e-5, (ns, rel)


def test_step_early_cache_read_matches_plain_launch():
    """Back-to-back steps over four layer caches with
    FP8KV_STEP_EARLY_CACHE_READ (each step streams its cache while the step
    before it finishes) give the same outputs and the same appended rows as
    plain launches."""
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx512"], device="cuda")
    prev, knew, vnew = _split_last_token(inp)
    q = inp.q.cuda().contiguous()
    lens = inp.seq_lens.cuda()
    results = {}
    for early in (False, True):
        caches = [fill_cache(prev, "k8v8", capacity=512) for _ in range(4)]
        outs = [torch.empty(16, 16, 128, dtype=torch.float32, device="cuda") for _ in range(4)]
        for rep in range(3):
            for i, c in enumerate(caches):
                fk.fp8kv_decode_step(q, knew, vnew, c, lens, out=outs[i], kernel="tensor_cores",
                                     early_cache_read=early)
        torch.cuda.synchronize()
        results[early] = (outs, caches)
    assert fk.fp8kv_get_device_error() == 0
    for i in range(4):
        assert torch.equal(results[False][0][i], results[True][0][i])
        assert torch.equal(results[False][1][i].k, results[True][1][i].k)
        assert torch.equal(results[False][1][i].v_scale, results[True][1][i].v_scale)
    assert_gate(results[True][0][0].cpu().numpy(), oracle_decode(inp, "k8v8", range(16)), "early cache read")


@pytest.mark.parametrize("kernel", ["cuda_cores", "tensor_cores"])
def test_step_with_pinned_host_buffers(kernel):
    """q, k_new, v_new, seq_lens and out in page-locked host memory, read and
    written by the kernels directly: the same output and cache as with device
    buffers."""
    spec = synth.DecodeWorkload("host_bufs", 3, 16, 2, 128, seed=37, seq_lens=(700, 129, 1))
    inp = synth.decode_inputs(spec, device="cuda")
    results = []
    for host in (False, True):
        prev, knew, vnew = _split_last_token(inp)
        cache = fill_cache(prev, "k8v8", capacity=768)
        q, lens = inp.q.cuda().contiguous(), inp.seq_lens.cuda()
        if host:
            q, knew, vnew, lens = (t.cpu().pin_memory() for t in (q, knew, vnew, lens))
            out = torch.empty((3, 16, 128), dtype=torch.float32).pin_memory()
        else:
            out = torch.empty((3, 16, 128), dtype=torch.float32, device="cuda")
        fk.fp8kv_decode_step(q, knew, vnew, cache, lens, out=out, kernel=kernel)
        torch.cuda.synchronize()
        assert fk.fp8kv_get_device_error() == 0
        results.append((out.cpu().clone(), cache.k.cpu().clone(), cache.v_scale.cpu().clone()))
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1]) and torch.equal(results[0][2], results[1][2])
    assert_gate(results[1][0].numpy(), oracle_decode(inp, "k8v8", range(3)), f"host buffers {kernel}")


def test_step_graph_replay_with_early_cache_read_full_size():
    """The headline's own launch configuration at full size: four layer
    caches of 16 sequences x 8192 tokens, the layers' fused steps captured
    in one CUDA graph, each launched as the previous one's programmatic
    dependent (early cache read), the graph replayed twice.  Every layer
    matches a plain eager step bit for bit, and a sample of sequences
    passes the gate against the oracle."""
    inp = synth.decode_inputs(synth.WORKLOADS["decode_b16_ctx8192"], device="cuda")
    prev, knew, vnew = _split_last_token(inp)
    q = inp.q.cuda().contiguous()
    lens = inp.seq_lens.cuda()
    n_layers = 4
    caches = [fill_cache(prev, "k8v8", capacity=8192) for _ in range(n_layers)]
    wss = [torch.zeros(fk.fp8kv_decode_step_workspace_bytes(c, 16, 0, "tensor_cores"), dtype=torch.uint8,
                       device="cuda") for c in caches]
    outs = [torch.empty(16, 16, 128, dtype=torch.float32, device="cuda") for _ in range(n_layers)]

    def steps(early):
        for j in range(n_layers):
            fk.fp8kv_decode_step(q, knew, vnew, caches[j], lens, out=outs[j], workspace=wss[j],
                                 kernel="tensor_cores", early_cache_read=early and j > 0)

    steps(False)                       # eager, plain launches: the reference outputs
    torch.cuda.synchronize()
    plain = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            steps(True)
    torch.cuda.current_stream().wait_stream(side)
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert fk.fp8kv_get_device_error() == 0
    for j in range(n_layers):
        assert torch.equal(outs[j], plain[j]), j
    sample = [0, 7, 15]
    assert_gate(outs[3].cpu().numpy()[sample], oracle_decode(inp, "k8v8", sample), "graph replay, early read")


@pytest.mark.parametrize("dtype", ["k8v8", "mxk8v8"])
def test_step_paged_b64_full_sampled(dtype):
    """The paged serving workload at full size (64 sequences of 1K-16K
    tokens, 16-token pages, hostile keys) through the fused step, as the
    bench runs it; the oracle checks a sample of sequences, and the appended
    rows of those sequences are the quantiser's."""
    inp = synth.decode_inputs(synth.WORKLOADS["paged_b64_hostile"], device="cuda")
    prev, knew, vnew = _split_last_token(inp)
    cache = fill_cache(prev, dtype)
    out = fk.fp8kv_decode_step(inp.q.cuda().contiguous(), knew, vnew, cache, inp.seq_lens.cuda(),
                               out_dtype=torch.float32)
    assert fk.fp8kv_get_device_error() == 0
    lens = inp.seq_lens.numpy()
    sample = sorted({int(lens.argmin()), int(lens.argmax()), 5, 40})
    assert_gate(out.cpu().numpy()[sample], oracle_decode(inp, dtype, sample), f"paged b64 step {dtype}")
    pt = inp.page_table.numpy()
    quant = oracle.mx_quantize if dtype == "mxk8v8" else oracle.quantize
    for b in sample:
        T = int(lens[b])
        codes, scales = quant(synth.bf16_bits(knew[b:b + 1]))
        got = oracle.gather_paged(cache.k.cpu().numpy(), pt, b, T)
        assert np.array_equal(got[:, T - 1], codes[0]), b

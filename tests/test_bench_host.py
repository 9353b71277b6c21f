"""The benchmark's host-side arithmetic on CPU: the algorithmic bytes of one
decode step (the numerator of the reported GB/s and of the roofline) for each
cache dtype at batch 16, 8,192 tokens, 16 query / 2 KV heads, head_dim 128,
worked out by hand below, and the argument parser's profiling mode."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from fp8_quantized_kv_gb300 import synth  # noqa: E402


def test_step_bytes_per_dtype():
    # per (token, KV head): K and V rows of 128 elements (1 byte each as e4m3,
    # 2 as bf16) plus a 4-byte scale per e4m3 side; 16 x 2 x 8192 rows.
    # Q in and O out: 2 x 16 x 16 x 128 x 2 bytes = 131,072.  The appended
    # token: 16 x 2 rows, 2 x 128 x 2 bf16 bytes in plus one cache row out.
    spec = synth.WORKLOADS["decode_b16_ctx8192"]
    rows, qo = 16 * 2 * 8192, 131072
    for dtype, row in (("k8v8", 264), ("mxk8v8", 264), ("k16v8", 388), ("k8v16", 388), ("k16v16", 512)):
        nb = bench.step_bytes(spec, dtype, 8192)
        assert nb["kv"] == rows * row, dtype
        assert nb["qo"] == qo
        assert nb["append"] == 32 * (512 + row)
        assert nb["step"] == rows * row + qo + 32 * (512 + row)
    assert bench.step_bytes(spec, "k8v8", 8192)["step"] == 69_361_920


def test_shape_mode_parses():
    a = bench.parse(["--shape", "paged_b64_hostile", "--dtype", "k16v16", "--steps", "10", "--warmup", "3"])
    assert a.shape == "paged_b64_hostile" and a.dtype == "k16v16" and a.steps == 10
    assert bench.parse([]).shape is None


def test_prefill_size_mode_and_flops():
    a = bench.parse(["--prefill-size", "8192,1,28,4", "--prefill-steps", "50"])
    assert a.prefill_size == "8192,1,28,4" and a.prefill_steps == 50
    assert bench.parse([]).prefill_size is None
    # 2048 tokens, 28 query heads, head_dim 128: 2,098,176 causal (query, key)
    # pairs per head, 4 x 128 FLOPs each, 28 heads
    assert bench.prefill_flops(2048, 1, 28, 128) == 2_098_176 * 512 * 28 == 30_079_451_136
    # a batch of 8 is 8 independent sequences
    assert bench.prefill_flops(2048, 8, 28, 128) == 8 * 30_079_451_136
    # one token attends only itself
    assert bench.prefill_flops(1, 1, 1, 128) == 512


def test_fp8_kv_error_report():
    """The bench's fp8_kv_error report on the tiny workload: the bf16 cache
    changes nothing; every 8-bit side adds error of the size an e4m3 round
    trip (3 mantissa bits) gives, a few percent; two 8-bit sides more than one
    of them."""
    err = bench.fp8_kv_errors(samples={"tiny_decode": (77, 128)}, dtypes=("k8v8", "k16v8", "k8v16", "k16v16"))
    e = err["tiny_decode"]
    assert e["k16v16"] == 0.0
    for dt in ("k8v8", "k16v8", "k8v16"):
        assert 1e-3 < e[dt] < 0.1, (dt, e[dt])
    assert e["k8v8"] > max(e["k16v8"], e["k8v16"])
    # head_dim 64 has two MXFP8 blocks of 32: the MXFP8 key cache is reported too
    mx = bench.fp8_kv_errors(samples={"tiny_decode": (77, 128)}, dtypes=("mxk8v8",))["tiny_decode"]["mxk8v8"]
    assert 1e-3 < mx < 0.1

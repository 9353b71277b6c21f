"""Seeded synthetic workloads for the FP8-KV attention path.

This module only draws random inputs and describes workload shapes; it holds
none of the method's arithmetic (no quantisation, no attention).  Both the CUDA
path and the oracle are fed from it, so it is the one module they share.

Workloads copy the shapes the pages measure on:
  * "FP8 KV cache (fp8_kv, opt-in)", bullet "Speed": batch 16, 16 query / 2 KV
    heads, head dim 128, contexts from 77 to 8192 tokens.
  * "03 · 8n — FA-style tiled prefill attention", section 3.1: a 7B-class
    model at 2K tokens, 28 query / 4 KV heads, head dim 128, causal prefill.
  * A paged serving decode (16-token pages, random permuted page table) with
    "hostile" keys: a fixed +20 bias on four channels of every KV head, the
    key-bias failure mechanism of "FP8 KV attention: hardware paths and tile
    preparation", section "Treat numerical safety and kernel speed as separate
    gates".

Recipe: fp32 N(0,1) from torch's seeded generator, rounded to bf16 (RNE) by
``Tensor.to(torch.bfloat16)``; hostile channels get +20 before that rounding.
Draw order per workload: (lengths, page permutation on a CPU generator), then
Q, then K, then V, each row-major in its logical layout.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch

HOSTILE_CHANNELS = (3, 17, 64, 111)
HOSTILE_BIAS = 20.0


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    seed: int
    seq_lens: Optional[Tuple[int, ...]] = None      # fixed lengths, or
    len_range: Optional[Tuple[int, int]] = None     # inclusive uniform range
    page_size: Optional[int] = None                 # None = contiguous cache
    hostile_keys: bool = False

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    n_tokens: int
    q_heads: int
    kv_heads: int
    head_dim: int
    seed: int
    pos0: int = 0


WORKLOADS = {
    "tiny_decode": DecodeWorkload("tiny_decode", 2, 4, 1, 64, seed=0, seq_lens=(77, 128)),
    "decode_b16_ctx512": DecodeWorkload("decode_b16_ctx512", 16, 16, 2, 128, seed=1,
                                        seq_lens=(512,) * 16),
    "decode_b16_ctx8192": DecodeWorkload("decode_b16_ctx8192", 16, 16, 2, 128, seed=2,
                                         seq_lens=(8192,) * 16),
    "paged_b64_hostile": DecodeWorkload("paged_b64_hostile", 64, 32, 8, 128, seed=3,
                                        len_range=(1024, 16384), page_size=16,
                                        hostile_keys=True),
}

PREFILL_WORKLOADS = {
    "prefill_2048": PrefillWorkload("prefill_2048", 2048, 28, 4, 128, seed=4),
}


def bf16_normal(shape, gen: torch.Generator, device, bias_channels=(), bias=0.0):
    """N(0,1) fp32 rounded to bf16; optional +bias on the last-dim channels."""
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    for c in bias_channels:
        if c < shape[-1]:
            x[..., c] += bias
    return x.to(torch.bfloat16)


@dataclass
class DecodeInputs:
    spec: DecodeWorkload
    q: torch.Tensor              # [B, Hq, D] bf16
    k: torch.Tensor              # [N, Hkv, D] bf16, sequences packed in order
    v: torch.Tensor              # [N, Hkv, D] bf16
    seq_lens: torch.Tensor       # [B] int32 (CPU)
    cu_seqlens: torch.Tensor     # [B+1] int64 (CPU)
    page_table: Optional[torch.Tensor] = None   # [B, max_pages] int32 (CPU)
    num_pages: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def max_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.numel() else 0


def decode_inputs(spec: DecodeWorkload, device="cpu", seq_lens=None) -> DecodeInputs:
    """Draw one decode workload.  ``seq_lens`` overrides the spec's lengths
    (used for shrunken copies of a workload in tests)."""
    cpu = torch.Generator(device="cpu").manual_seed(spec.seed)
    if seq_lens is not None:
        lens = torch.tensor(list(seq_lens), dtype=torch.int32)
    elif spec.seq_lens is not None:
        lens = torch.tensor(spec.seq_lens, dtype=torch.int32)
    else:
        lo, hi = spec.len_range
        lens = torch.randint(lo, hi + 1, (spec.batch,), generator=cpu, dtype=torch.int64)
        lens = lens.to(torch.int32)
    B = lens.numel()
    cu = torch.zeros(B + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens.to(torch.int64), 0)
    page_table, num_pages = None, 0
    if spec.page_size is not None:
        P = spec.page_size
        pages_per_seq = (lens.to(torch.int64) + P - 1) // P
        num_pages = int(pages_per_seq.sum())
        perm = torch.randperm(num_pages, generator=cpu).to(torch.int32)
        max_pages = int(pages_per_seq.max()) if B else 0
        page_table = torch.full((B, max(max_pages, 1)), -1, dtype=torch.int32)
        off = 0
        for b in range(B):
            n = int(pages_per_seq[b])
            page_table[b, :n] = perm[off:off + n]
            off += n
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(spec.seed)
    N = int(cu[-1])
    D, Hq, Hkv = spec.head_dim, spec.q_heads, spec.kv_heads
    q = bf16_normal((B, Hq, D), gen, dev)
    chans = HOSTILE_CHANNELS if spec.hostile_keys else ()
    k = bf16_normal((N, Hkv, D), gen, dev, chans, HOSTILE_BIAS)
    v = bf16_normal((N, Hkv, D), gen, dev)
    return DecodeInputs(spec, q, k, v, lens, cu, page_table, num_pages)


@dataclass
class PrefillInputs:
    spec: PrefillWorkload
    q: torch.Tensor    # [n_q, Hq, D] bf16 (the last n_q tokens)
    k: torch.Tensor    # [pos0 + n_q, Hkv, D] bf16 (all cached tokens)
    v: torch.Tensor


def prefill_inputs(spec: PrefillWorkload, device="cpu", n_tokens=None, pos0=None) -> PrefillInputs:
    n = spec.n_tokens if n_tokens is None else n_tokens
    p0 = spec.pos0 if pos0 is None else pos0
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(spec.seed)
    D = spec.head_dim
    q = bf16_normal((n, spec.q_heads, D), gen, dev)
    k = bf16_normal((p0 + n, spec.kv_heads, D), gen, dev)
    v = bf16_normal((p0 + n, spec.kv_heads, D), gen, dev)
    return PrefillInputs(spec, q, k, v)


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor as a numpy array (CPU)."""
    import numpy as np
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)

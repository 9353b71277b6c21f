"""GB300-native fused attention over an FP8 E4M3 KV cache.

Python binding of the C ABI in include/fp8kv.h.  The functions below carry
the C names and do argument marshalling only (torch tensors -> device
pointers, the current torch stream -> cudaStream_t); every step of the path
runs in the library's CUDA kernels.  torch provides device memory and streams.

    cache = Fp8KVCache.contiguous(batch, kv_heads, head_dim, max_tokens, "k8v8")
    fp8kv_append(cache, k_new, v_new, seq_idx, pos)
    out = fp8kv_decode_attention(q, cache, seq_lens)
    out = fp8kv_prefill_attention(q, cache, q_pos0)
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from ._lib import EXPORTS, CacheStruct, get_lib

K8V8, K16V8, K16V16, K8V16, MXK8V8 = 0, 1, 2, 3, 4
DTYPES = {"k8v8": K8V8, "k16v8": K16V8, "k16v16": K16V16, "k8v16": K8V16, "mxk8v8": MXK8V8}
LAYOUT_CONTIGUOUS, LAYOUT_PAGED = 0, 1
OUT_BF16, OUT_F32 = 0, 1

DEVERR_SEQ_TOO_LONG, DEVERR_BAD_PAGE, DEVERR_TIMEOUT = 0x1, 0x2, 0x4
STEP_EARLY_CACHE_READ = 0x1
KERNEL_AUTO, KERNEL_CUDA_CORES, KERNEL_TENSOR_CORES = 0, 1, 2
KERNEL_TENSOR_CORES_K_F16, KERNEL_TENSOR_CORES_K_F16_PRODUCER = 3, 4
KERNELS = {"auto": KERNEL_AUTO, "cuda_cores": KERNEL_CUDA_CORES, "tensor_cores": KERNEL_TENSOR_CORES,
           "tensor_cores_k_f16": KERNEL_TENSOR_CORES_K_F16,
           "tensor_cores_k_f16_producer": KERNEL_TENSOR_CORES_K_F16_PRODUCER}

STATUS_NAMES = {0: "FP8KV_OK", 1: "FP8KV_ERR_INVALID_ARG", 2: "FP8KV_ERR_UNSUPPORTED",
                3: "FP8KV_ERR_WORKSPACE", 4: "FP8KV_ERR_CUDA", 5: "FP8KV_ERR_TIMEOUT",
                6: "FP8KV_ERR_DEVICE_CHECK"}


class Fp8KVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = get_lib().fp8kv_status_string(status).decode()
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({msg})")


def _check(status: int, where: str):
    if status != 0:
        raise Fp8KVError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name, host_ok=False):
    """A contiguous CUDA tensor of `dtype` (or, where host_ok, a contiguous
    page-locked host tensor, which the kernels address directly)."""
    where_ok = t.is_cuda or (host_ok and t.is_pinned())
    if t.dtype != dtype or not where_ok or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor"
                         f"{' (or pinned host tensor)' if host_ok else ''}, got "
                         f"{t.dtype} on {t.device} (contiguous={t.is_contiguous()})")


class Fp8KVCache:
    """Device tensors of one KV cache (allocated with torch) and the C struct
    that describes them.  Layouts are those of include/fp8kv.h."""

    def __init__(self, *, dtype, layout, batch, kv_heads, head_dim, k, v, k_scale, v_scale,
                 max_tokens=0, page_size=0, num_pages=0, page_table=None, k_bias=None, rope_cos=None,
                 rope_sin=None):
        self.dtype = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
        self.layout = layout
        self.batch, self.kv_heads, self.head_dim = batch, kv_heads, head_dim
        self.max_tokens, self.page_size, self.num_pages = max_tokens, page_size, num_pages
        self.k, self.v, self.k_scale, self.v_scale = k, v, k_scale, v_scale
        self.page_table = page_table
        if k_bias is not None:
            _need(k_bias, torch.float32, "k_bias")
        self.k_bias = k_bias
        if (rope_cos is None) != (rope_sin is None):
            raise ValueError("rope_cos and rope_sin come together")
        if rope_cos is not None:
            for t, name in ((rope_cos, "rope_cos"), (rope_sin, "rope_sin")):
                _need(t, torch.float32, name)
                if t.dim() != 2 or t.shape[1] != head_dim // 2 or t.shape != rope_cos.shape:
                    raise ValueError(f"{name}: want [positions, head_dim / 2] fp32, got {tuple(t.shape)}")
        self.rope_cos, self.rope_sin = rope_cos, rope_sin
        self._struct = CacheStruct(
            dtype=self.dtype, layout=layout, batch=batch, kv_heads=kv_heads, head_dim=head_dim,
            max_tokens=max_tokens, page_size=page_size, num_pages=num_pages,
            max_pages_per_seq=0 if page_table is None else page_table.shape[1],
            rope_positions=0 if rope_cos is None else rope_cos.shape[0],
            k=k.data_ptr(), v=v.data_ptr(),
            k_scale=None if k_scale is None else k_scale.data_ptr(),
            v_scale=None if v_scale is None else v_scale.data_ptr(),
            page_table=None if page_table is None else page_table.data_ptr(),
            k_bias=None if k_bias is None else k_bias.data_ptr(),
            rope_cos=None if rope_cos is None else rope_cos.data_ptr(),
            rope_sin=None if rope_sin is None else rope_sin.data_ptr())

    @property
    def struct_ref(self):
        return ctypes.byref(self._struct)

    @property
    def capacity(self) -> int:
        if self.layout == LAYOUT_PAGED:
            return self.page_table.shape[1] * self.page_size
        return self.max_tokens

    @staticmethod
    def _alloc(dtype, lead, head_dim, device):
        dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
        k8, v8 = dt in (K8V8, K8V16, MXK8V8), dt in (K8V8, K16V8, MXK8V8)
        kel = torch.uint8 if k8 else torch.bfloat16
        vel = torch.uint8 if v8 else torch.bfloat16
        k = torch.zeros(lead + (head_dim,), dtype=kel, device=device)
        v = torch.zeros(lead + (head_dim,), dtype=vel, device=device)
        if dt == MXK8V8:    # the four E8M0 block bytes of each row in its 4-byte slot
            ks = torch.zeros(lead + (4,), dtype=torch.uint8, device=device)
        else:
            ks = torch.zeros(lead, dtype=torch.float32, device=device) if k8 else None
        vs = torch.zeros(lead, dtype=torch.float32, device=device) if v8 else None
        return k, v, ks, vs

    @classmethod
    def contiguous(cls, batch, kv_heads, head_dim, max_tokens, dtype="k8v8", device="cuda", k_bias=None,
                   rope_cos=None, rope_sin=None):
        """k_bias: optional [kv_heads, head_dim] fp32 key bias; the cache then
        holds pre-bias residual keys (include/fp8kv.h, fp8kv_cache.k_bias).
        rope_cos, rope_sin: optional [positions, head_dim / 2] fp32 rotary
        tables; the bias then turns with the key's position (rope_cos)."""
        k, v, ks, vs = cls._alloc(dtype, (batch, kv_heads, max_tokens), head_dim, device)
        return cls(dtype=dtype, layout=LAYOUT_CONTIGUOUS, batch=batch, kv_heads=kv_heads, k_bias=k_bias,
                   head_dim=head_dim, k=k, v=v, k_scale=ks, v_scale=vs, max_tokens=max_tokens,
                   rope_cos=rope_cos, rope_sin=rope_sin)

    @classmethod
    def paged(cls, page_table: torch.Tensor, num_pages, kv_heads, head_dim, page_size=16,
              dtype="k8v8", device="cuda", k_bias=None, rope_cos=None, rope_sin=None):
        pt = page_table.to(device=device, dtype=torch.int32).contiguous()
        k, v, ks, vs = cls._alloc(dtype, (num_pages, kv_heads, page_size), head_dim, device)
        return cls(dtype=dtype, layout=LAYOUT_PAGED, batch=pt.shape[0], kv_heads=kv_heads, k_bias=k_bias,
                   head_dim=head_dim, k=k, v=v, k_scale=ks, v_scale=vs, page_size=page_size,
                   num_pages=num_pages, page_table=pt, rope_cos=rope_cos, rope_sin=rope_sin)


# ------------------------------------------------------------ C-ABI calls --

def fp8kv_quantize(x: torch.Tensor, codes: Optional[torch.Tensor] = None,
                   scales: Optional[torch.Tensor] = None, stream=None):
    """bf16 rows [..., D] -> (uint8 codes [..., D], fp32 scales [...])."""
    _need(x, torch.bfloat16, "x")
    D = x.shape[-1]
    rows = x.numel() // D if D else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _check(get_lib().fp8kv_quantize(_ptr(x), rows, D, _ptr(codes), _ptr(scales), _stream(stream)),
           "fp8kv_quantize")
    return codes, scales


def fp8kv_quantize_mx(x: torch.Tensor, codes: Optional[torch.Tensor] = None,
                      scales: Optional[torch.Tensor] = None, stream=None):
    """bf16 rows [..., D] (D 64 or 128) -> (uint8 codes [..., D], uint8 E8M0
    block scales [..., D/32]): MXFP8, one power-of-two scale per 32 elements."""
    _need(x, torch.bfloat16, "x")
    D = x.shape[-1]
    rows = x.numel() // D if D else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (max(D // 32, 1),), dtype=torch.uint8, device=x.device)
    _check(get_lib().fp8kv_quantize_mx(_ptr(x), rows, D, _ptr(codes), _ptr(scales), _stream(stream)),
           "fp8kv_quantize_mx")
    return codes, scales


def fp8kv_append(cache: Fp8KVCache, k_new: torch.Tensor, v_new: torch.Tensor,
                 seq_idx: torch.Tensor, pos: torch.Tensor, stream=None):
    """Quantise and write K/V rows [n, kv_heads, D] (bf16) for tokens
    (seq_idx[i], pos[i])."""
    _need(k_new, torch.bfloat16, "k_new")
    _need(v_new, torch.bfloat16, "v_new")
    _need(seq_idx, torch.int32, "seq_idx")
    _need(pos, torch.int32, "pos")
    n = k_new.shape[0]
    _check(get_lib().fp8kv_append(cache.struct_ref, _ptr(k_new), _ptr(v_new), _ptr(seq_idx),
                                  _ptr(pos), n, _stream(stream)), "fp8kv_append")


def _kernel(kernel) -> int:
    return KERNELS[kernel] if isinstance(kernel, str) else int(kernel)


def fp8kv_decode_num_splits(cache: Fp8KVCache, q_heads: int, num_splits: int = 0, kernel=0) -> int:
    return int(get_lib().fp8kv_decode_num_splits(cache.struct_ref, q_heads, num_splits, _kernel(kernel)))


def fp8kv_decode_workspace_bytes(cache: Fp8KVCache, q_heads: int, num_splits: int = 0, kernel=0) -> int:
    return int(get_lib().fp8kv_decode_workspace_bytes(cache.struct_ref, q_heads, num_splits,
                                                      _kernel(kernel)))


def fp8kv_decode_attention(q: torch.Tensor, cache: Fp8KVCache, seq_lens: torch.Tensor,
                           sm_scale: Optional[float] = None, num_splits: int = 0,
                           out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                           workspace: Optional[torch.Tensor] = None, kernel=0, stream=None):
    """q [B, Hq, D] bf16, seq_lens [B] int32 -> out [B, Hq, D] (bf16 or fp32).
    kernel: "auto" / "cuda_cores" / "tensor_cores" / "tensor_cores_k_f16" /
    "tensor_cores_k_f16_producer" (or 0 .. 4)."""
    _need(q, torch.bfloat16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=q.device)
    odt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    k = _kernel(kernel)
    need = fp8kv_decode_workspace_bytes(cache, Hq, num_splits, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(get_lib().fp8kv_decode_attention(
        _ptr(q), cache.struct_ref, _ptr(seq_lens), Hq, float(sm_scale), num_splits, k,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), odt,
        _stream(stream)), "fp8kv_decode_attention")
    return out


def fp8kv_decode_split(q: torch.Tensor, cache: Fp8KVCache, seq_lens: torch.Tensor,
                       workspace: torch.Tensor, sm_scale: Optional[float] = None,
                       num_splits: int = 0, kernel=0, stream=None):
    """Kernel 1 of decode: fp32 partials of every split into `workspace`."""
    _need(q, torch.bfloat16, "q")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    _check(get_lib().fp8kv_decode_split(
        _ptr(q), cache.struct_ref, _ptr(seq_lens), Hq, float(sm_scale), num_splits, _kernel(kernel),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
        "fp8kv_decode_split")


def fp8kv_decode_merge(cache: Fp8KVCache, q_heads: int, workspace: torch.Tensor,
                       out: torch.Tensor, num_splits: int = 0, kernel=0, stream=None):
    """Kernel 2 of decode: merge the partials in `workspace` into `out`."""
    odt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(get_lib().fp8kv_decode_merge(
        cache.struct_ref, q_heads, num_splits, _kernel(kernel), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), odt, _stream(stream)),
        "fp8kv_decode_merge")
    return out


def fp8kv_decode_step_workspace_bytes(cache: Fp8KVCache, q_heads: int, num_splits: int = 0,
                                      kernel=0) -> int:
    return int(get_lib().fp8kv_decode_step_workspace_bytes(cache.struct_ref, q_heads, num_splits,
                                                           _kernel(kernel)))


def fp8kv_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, cache: Fp8KVCache,
                      seq_lens: torch.Tensor, sm_scale: Optional[float] = None, num_splits: int = 0,
                      out: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16,
                      workspace: Optional[torch.Tensor] = None, kernel=0, early_cache_read=False,
                      stream=None):
    """Append k_new/v_new [B, Hkv, D] at position seq_lens[b]-1 and decode
    q [B, Hq, D] over seq_lens[b] tokens.  `workspace` must start zero-filled
    (a fresh one is allocated that way when not given).  early_cache_read:
    FP8KV_STEP_EARLY_CACHE_READ (the kernel issued just before on the stream
    must not write this cache or seq_lens)."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, n, host_ok=True)
    _need(seq_lens, torch.int32, "seq_lens", host_ok=True)
    B, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    dev = cache.k.device                   # (q and the others may be pinned host tensors)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=out_dtype, device=dev)
    _need(out, out.dtype, "out", host_ok=True)
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"out: expected bf16 or fp32, got {out.dtype}")
    odt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    k = _kernel(kernel)
    if workspace is None:
        need = fp8kv_decode_step_workspace_bytes(cache, Hq, num_splits, k)
        workspace = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
    _need(workspace, torch.uint8, "workspace")
    _check(get_lib().fp8kv_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), cache.struct_ref, _ptr(seq_lens), Hq, float(sm_scale),
        num_splits, k, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(out), odt,
        STEP_EARLY_CACHE_READ if early_cache_read else 0, _stream(stream)), "fp8kv_decode_step")
    return out


def fp8kv_prefill_attention(q: torch.Tensor, cache: Fp8KVCache, q_pos0: torch.Tensor,
                            sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                            out_dtype=torch.bfloat16, kernel="auto", stream=None):
    """q [B, n_q, Hq, D] bf16, q_pos0 [B] int32 -> out [B, n_q, Hq, D].
    kernel: "auto", "tensor_cores" (K8V8, head_dim 128) or "cuda_cores"."""
    _need(q, torch.bfloat16, "q")
    _need(q_pos0, torch.int32, "q_pos0")
    B, n_q, Hq, D = q.shape
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, n_q, Hq, D), dtype=out_dtype, device=q.device)
    odt = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(get_lib().fp8kv_prefill_attention(
        _ptr(q), cache.struct_ref, _ptr(q_pos0), n_q, Hq, float(sm_scale), _kernel(kernel), _ptr(out),
        odt, _stream(stream)), "fp8kv_prefill_attention")
    return out


def fp8kv_get_device_error(clear: bool = True) -> int:
    """Synchronise the device and return (optionally clearing) the device
    error word (bits DEVERR_*)."""
    bits = ctypes.c_uint32(0)
    st = get_lib().fp8kv_get_device_error(ctypes.byref(bits), 1 if clear else 0)
    if st not in (0, 5, 6):
        raise Fp8KVError(st, "fp8kv_get_device_error")
    return int(bits.value)


def fp8kv_status_string(status: int) -> str:
    return get_lib().fp8kv_status_string(status).decode()


__all__ = ["Fp8KVCache", "Fp8KVError", "fp8kv_quantize", "fp8kv_quantize_mx", "fp8kv_append",
           "fp8kv_decode_num_splits", "fp8kv_decode_workspace_bytes", "fp8kv_decode_split",
           "fp8kv_decode_merge", "fp8kv_decode_attention", "fp8kv_decode_step",
           "fp8kv_decode_step_workspace_bytes",
           "fp8kv_prefill_attention", "fp8kv_get_device_error", "fp8kv_status_string",
           "EXPORTS", "K8V8", "K16V8", "K16V16", "K8V16", "MXK8V8"]

"""ctypes loader for libfp8kv.so (the C ABI declared in include/fp8kv.h).

Argument marshalling only: every computation runs in the CUDA kernels of the
library.  If the library is missing, the first call raises; there is no
fallback implementation.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfp8kv.so")

EXPORTS = (
    "fp8kv_quantize",
    "fp8kv_quantize_mx",
    "fp8kv_append",
    "fp8kv_decode_num_splits",
    "fp8kv_decode_workspace_bytes",
    "fp8kv_decode_split",
    "fp8kv_decode_merge",
    "fp8kv_decode_attention",
    "fp8kv_decode_step_workspace_bytes",
    "fp8kv_decode_step",
    "fp8kv_decode_attention_static",
    "fp8kv_decode_static_scratch_bytes",
    "fp8kv_prefill_attention",
    "fp8kv_get_device_error",
    "fp8kv_status_string",
)


class CacheStruct(ctypes.Structure):
    """Mirror of the C struct fp8kv_cache."""
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_tokens", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("rope_positions", ctypes.c_int32),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p),
        ("k_bias", ctypes.c_void_p),
        ("rope_cos", ctypes.c_void_p),
        ("rope_sin", ctypes.c_void_p),
    ]


_lib = None


def get_lib() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(the FP8-KV kernels have no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    u32 = ctypes.c_uint32
    cp = ctypes.POINTER(CacheStruct)
    sig = {
        "fp8kv_quantize": (i32, [vp, i64, i32, vp, vp, vp]),
        "fp8kv_quantize_mx": (i32, [vp, i64, i32, vp, vp, vp]),
        "fp8kv_append": (i32, [cp, vp, vp, vp, vp, i64, vp]),
        "fp8kv_decode_num_splits": (i32, [cp, i32, i32, i32]),
        "fp8kv_decode_workspace_bytes": (sz, [cp, i32, i32, i32]),
        "fp8kv_decode_split": (i32, [vp, cp, vp, i32, f32, i32, i32, vp, sz, vp]),
        "fp8kv_decode_merge": (i32, [cp, i32, i32, i32, vp, sz, vp, i32, vp]),
        "fp8kv_decode_attention": (i32, [vp, cp, vp, i32, f32, i32, i32, vp, sz, vp, i32, vp]),
        "fp8kv_decode_step_workspace_bytes": (sz, [cp, i32, i32, i32]),
        "fp8kv_decode_step": (i32, [vp, vp, vp, cp, vp, i32, f32, i32, i32, vp, sz, vp, i32, u32, vp]),
        "fp8kv_decode_attention_static": (i32, [vp, cp, vp, i32, f32, i32, vp, i32, vp]),
        "fp8kv_decode_static_scratch_bytes": (sz, []),
        "fp8kv_prefill_attention": (i32, [vp, cp, vp, i32, i32, f32, i32, vp, i32, vp]),
        "fp8kv_get_device_error": (i32, [ctypes.POINTER(ctypes.c_uint32), i32]),
        "fp8kv_status_string": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib

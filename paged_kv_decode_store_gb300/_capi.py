"""ctypes declarations of include/pkvd.h and tensor-to-argument helpers."""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkvd.so")

PATH_AUTO, PATH_FMA, PATH_MMA, PATH_TC = 0, 1, 2, 3
ERR_BLOCK_ID, ERR_SLOT, ERR_CONTEXT, ERR_TIMEOUT = 1, 2, 4, 8
NO_SPACE = 6
_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

c_void_p, c_int32, c_int64, c_size_t, c_float = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_size_t, ctypes.c_float)


class PkvdCache(ctypes.Structure):
    _fields_ = [("k_base", c_void_p), ("v_base", c_void_p), ("dtype", c_int32),
                ("block_size", c_int32), ("num_blocks", c_int64), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("block_stride", c_int64), ("token_stride", c_int64),
                ("head_stride", c_int64)]


class PkvdError(RuntimeError):
    def __init__(self, status: int, text: str):
        super().__init__(f"pkvd status {status}: {text}")
        self.status = status


# name -> (restype, argtypes)
SIGNATURES = {
    "pkvd_status_string": (ctypes.c_char_p, [c_int32]),
    "pkvd_version": (c_int32, []),
    "pkvd_slot_mapping": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_int32, c_int64,
                                    c_void_p, c_void_p]),
    "pkvd_kv_store": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, ctypes.POINTER(PkvdCache),
                                c_void_p, c_void_p]),
    "pkvd_kv_store_paged": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_int32, c_void_p,
                                      ctypes.POINTER(PkvdCache), c_void_p, c_void_p]),
    "pkvd_kv_store_prefill": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_int32,
                                        c_int32, c_void_p, ctypes.POINTER(PkvdCache), c_void_p, c_void_p]),
    "pkvd_prefill_attention": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(PkvdCache), c_void_p, c_int32,
                                         c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_float,
                                         c_int32, c_void_p, c_void_p]),
    "pkvd_prefill_attention_ex": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(PkvdCache), c_void_p, c_int32,
                                            c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_float,
                                            c_int32, c_void_p, c_void_p, c_int32]),
    "pkvd_bm_create": (c_int32, [c_int32, c_int32, ctypes.POINTER(c_void_p)]),
    "pkvd_bm_destroy": (None, [c_void_p]),
    "pkvd_bm_num_free": (c_int32, [c_void_p]),
    "pkvd_bm_ref_count": (c_int32, [c_void_p, c_int32]),
    "pkvd_bm_allocate": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_int32, ctypes.POINTER(c_int32),
                                   ctypes.POINTER(c_int32)]),
    "pkvd_bm_append": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, ctypes.POINTER(c_int32), c_int32,
                                 ctypes.POINTER(c_int32), ctypes.POINTER(c_int32), ctypes.POINTER(c_int32)]),
    "pkvd_bm_fork": (c_int32, [c_void_p, c_void_p, c_int32]),
    "pkvd_bm_shared_prefix": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_int32, ctypes.POINTER(c_int32)]),
    "pkvd_bm_release": (c_int32, [c_void_p, c_void_p, c_int32]),
    "pkvd_copy_blocks": (c_int32, [ctypes.POINTER(PkvdCache), c_void_p, c_void_p, c_void_p, c_int32, c_void_p,
                                   c_void_p]),
    "pkvd_decode_workspace_bytes": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32,
                                              ctypes.POINTER(c_size_t)]),
    "pkvd_paged_decode_attention": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(PkvdCache), c_void_p,
                                              c_int32, c_void_p, c_int32, c_int32, c_int32, c_float,
                                              c_void_p, c_size_t, c_void_p, c_void_p]),
    "pkvd_paged_decode_attention_ex": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(PkvdCache), c_void_p,
                                                 c_int32, c_void_p, c_int32, c_int32, c_int32, c_float,
                                                 c_void_p, c_size_t, c_void_p, c_void_p, c_int32]),
    "pkvd_paged_decode_attention_window": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(PkvdCache), c_void_p,
                                                     c_int32, c_void_p, c_int32, c_int32, c_int32, c_float,
                                                     c_int32, c_void_p, c_size_t, c_void_p, c_void_p, c_int32]),
    "pkvd_decode_prefix_workspace_bytes": (c_int32, [c_int32, c_int32, c_int32, c_int32, c_int32, c_int32, c_int32,
                                                     ctypes.POINTER(c_size_t)]),
    "pkvd_paged_decode_attention_prefix": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(PkvdCache), c_void_p, c_int32,
                                                     c_void_p, c_int32, c_int32, c_int32, c_float, c_int32, c_void_p,
                                                     c_size_t, c_void_p, c_void_p]),
    "pkvd_paged_decode_attention_noalloc": (c_int32, [c_void_p, c_void_p, ctypes.POINTER(PkvdCache), c_void_p,
                                                      c_int32, c_void_p, c_int32, c_int32, c_int32, c_float,
                                                      c_void_p, c_void_p]),
    "pkvd_sample_workspace_bytes": (c_int32, [c_int32, c_int32, ctypes.POINTER(c_size_t)]),
    "pkvd_sample": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int64, c_void_p, c_void_p,
                              c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "pkvd_sample_ex": (c_int32, [c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int64, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_size_t, c_void_p]),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def check(status: int) -> None:
    if status != 0:
        raise PkvdError(status, lib().pkvd_status_string(status).decode())


def dtype_code(dt: torch.dtype) -> int:
    if dt not in _DTYPES:
        raise TypeError(f"unsupported dtype {dt}")
    return _DTYPES[dt]


def ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on a CUDA device")
    return t.data_ptr()


def stream_handle(stream, like: torch.Tensor):
    if stream is None:
        stream = torch.cuda.current_stream(like.device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def cache_desc(k_cache: torch.Tensor, v_cache: torch.Tensor) -> PkvdCache:
    """Describe [num_blocks, block_size, Hkv, D] views (e.g. kv_cache[0, layer])."""
    if k_cache.shape != v_cache.shape or k_cache.stride() != v_cache.stride():
        raise ValueError("K and V caches must share shape and strides")
    if k_cache.dim() != 4 or k_cache.stride(3) != 1:
        raise ValueError("cache views must be [num_blocks, block_size, Hkv, D] with D contiguous")
    nb, bs, H, D = k_cache.shape
    c = PkvdCache()
    c.k_base = ptr(k_cache)
    c.v_base = ptr(v_cache)
    c.dtype = dtype_code(k_cache.dtype)
    c.block_size = bs
    c.num_blocks = nb
    c.num_kv_heads = H
    c.head_dim = D
    c.block_stride = k_cache.stride(0)
    c.token_stride = k_cache.stride(1)
    c.head_stride = k_cache.stride(2)
    return c

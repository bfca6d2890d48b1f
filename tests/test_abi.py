"""The C-ABI library loads, exports every symbol pkvd.h declares, and its
host-side checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pkvd.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_decode_store_gb300 as pk
    return pk.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkvd_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    from paged_kv_decode_store_gb300 import _capi
    assert set(_capi.SIGNATURES) == set(names)


def test_status_strings_and_version(L):
    assert L.pkvd_status_string(0) == b"ok"
    assert L.pkvd_status_string(4) == b"workspace too small"
    assert L.pkvd_version() >= 100


def _cache(**kw):
    from paged_kv_decode_store_gb300._capi import PkvdCache
    c = PkvdCache()
    c.k_base, c.v_base = 1 << 20, 2 << 20          # fake, aligned, never dereferenced
    c.dtype, c.block_size, c.num_blocks, c.num_kv_heads, c.head_dim = 2, 16, 64, 8, 128
    c.block_stride, c.token_stride, c.head_stride = 16 * 8 * 128, 8 * 128, 128
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def _attn(L, cache, hq=48, ws=1 << 20, path=0, num_seqs=4, scale=0.088):
    return L.pkvd_paged_decode_attention_ex(1 << 21, 1 << 22, ctypes.byref(cache), 1 << 23, 8, 1 << 24,
                                            128, num_seqs, hq, ctypes.c_float(scale), 1 << 25, ws, None,
                                            None, path)


def test_attention_host_checks(L):
    assert _attn(L, _cache(), hq=44) == 3                    # 44 % 8 != 0
    assert _attn(L, _cache(), hq=8 * 9) == 3                 # group 9 > 8
    assert _attn(L, _cache(head_dim=96)) == 3
    assert _attn(L, _cache(block_size=24)) == 3              # not a power of two
    assert _attn(L, _cache(block_size=8)) == 3               # below one 16-token chunk
    assert _attn(L, _cache(dtype=7)) == 2
    assert _attn(L, _cache(k_base=0)) == 1
    assert _attn(L, _cache(token_stride=8 * 128 + 3)) == 3   # 16-byte rule
    assert _attn(L, _cache(), scale=float("nan")) == 1
    assert _attn(L, _cache(dtype=0), path=2) == 3             # no tensor-core path for fp32
    assert _attn(L, _cache(num_kv_heads=4, block_stride=16 * 4 * 128, token_stride=4 * 128), hq=16,
                 path=2) == 3
    assert _attn(L, _cache(), path=9) == 1
    assert _attn(L, _cache(), num_seqs=0) == 0               # nothing to do, nothing launched


def test_workspace_query_is_host_only(L):
    n = ctypes.c_size_t(0)
    assert L.pkvd_decode_workspace_bytes(32, 48, 128, 2048, 152, ctypes.byref(n)) == 0
    grid = min(152, 32 * 128)
    assert n.value == grid * 2 * 48 * 132 * 4                # partial records [grid][2][Hq][D + 4] fp32
    assert L.pkvd_decode_workspace_bytes(4, 4, 64, 50, 152, ctypes.byref(n)) == 0
    assert n.value == min(152, 4 * 4) * 2 * 4 * 68 * 4
    assert L.pkvd_decode_workspace_bytes(4, 4, 64, 0, 152, ctypes.byref(n)) == 0
    assert n.value == 0                                      # no context: nothing to combine
    assert L.pkvd_decode_workspace_bytes(-1, 4, 64, 50, 152, ctypes.byref(n)) == 1


def test_store_slot_and_sample_host_checks(L):
    c = _cache()
    assert L.pkvd_kv_store(1 << 20, 1 << 21, 1 << 22, -1, ctypes.byref(c), None, None) == 1
    assert L.pkvd_kv_store(1 << 20, 1 << 21, 1 << 22, 0, ctypes.byref(c), None, None) == 0
    assert L.pkvd_kv_store(1 << 20, (1 << 21) + 8, 1 << 22, 3, ctypes.byref(c), None, None) == 3
    assert L.pkvd_kv_store(1 << 20, 1 << 21, 1 << 22, 3, ctypes.byref(_cache(head_dim=32)), None, None) == 3
    paged = lambda k, v, tab, nmax, ctx, n, cc: L.pkvd_kv_store_paged(k, v, tab, nmax, ctx, n, None, ctypes.byref(cc),
                                                                    None, None)
    assert paged(1 << 20, 1 << 21, 1 << 22, 4, 1 << 23, -1, c) == 1
    assert paged(1 << 20, 1 << 21, 1 << 22, 4, 1 << 23, 0, c) == 0
    assert paged(1 << 20, 1 << 21, None, 4, 1 << 23, 3, c) == 1
    assert paged(1 << 20, 1 << 21, 1 << 22, 0, 1 << 23, 3, c) == 1
    assert paged(1 << 20, (1 << 21) + 8, 1 << 22, 4, 1 << 23, 3, c) == 3
    assert L.pkvd_slot_mapping(1 << 20, 1 << 21, 4, 1 << 22, 0, 16, 64, None, None) == 0
    assert L.pkvd_slot_mapping(1 << 20, 1 << 21, 4, 1 << 22, 2, 0, 64, None, None) == 1
    args = [1 << 20, 1 << 21]
    tail = [1 << 22] * 5 + [None, 0, None]
    assert L.pkvd_sample(*args, 3, 4, 100, 100, *tail) == 2           # dtype
    assert L.pkvd_sample(*args, 2, 4, 100, 99, *tail) == 1            # row_stride < vocab
    assert L.pkvd_sample(*args, 2, 4, (1 << 23) + 1, (1 << 23) + 1, *tail) == 3
    assert L.pkvd_sample(*args, 2, 0, 100, 100, *tail) == 0
    n = ctypes.c_size_t(7)
    assert L.pkvd_sample_workspace_bytes(4, 100, ctypes.byref(n)) == 0 and n.value == 4 * 32     # extras' row cuts


def test_prefill_host_checks(L):
    def attn(cache, hq=48, q=1 << 22, out=1 << 21, seqs=4, total=100, maxq=64, scale=0.088, window=0):
        return L.pkvd_prefill_attention(out, q, ctypes.byref(cache), 1 << 23, 8, 1 << 24, 1 << 25, seqs, total,
                                        maxq, hq, ctypes.c_float(scale), window, None, None)
    def attn_ex(cache, path, hq=48):
        return L.pkvd_prefill_attention_ex(1 << 21, 1 << 22, ctypes.byref(cache), 1 << 23, 8, 1 << 24, 1 << 25, 4,
                                           100, 64, hq, ctypes.c_float(0.088), 0, None, None, path)
    # every call below is rejected on the host (the pointers are fake)
    assert attn_ex(_cache(dtype=0), path=2) == 2                # no fp32 tensor-core prefill
    assert attn_ex(_cache(dtype=0), path=3) == 2
    assert attn_ex(_cache(dtype=0), path=0, hq=8 * 17) == 3    # fp32 goes to the CUDA-core path: group <= 16
    assert attn_ex(_cache(), path=1, hq=8 * 17) == 3
    assert attn_ex(_cache(), path=9) == 1
    assert attn(_cache(), hq=44) == 3                          # 44 % 8 != 0
    assert attn(_cache(num_kv_heads=1, block_stride=16 * 128, token_stride=128), hq=129) == 3   # group > 128
    assert attn(_cache(head_dim=96)) == 3
    assert attn(_cache(), window=-1) == 1
    assert attn(_cache(), scale=float("inf")) == 1
    assert attn(_cache(), q=(1 << 22) + 8) == 3                # q must be 16-byte aligned
    assert attn(_cache(), out=(1 << 21) + 2) == 3              # out 4-byte aligned
    assert attn(_cache(), seqs=70000) == 3                     # grid y limit
    assert attn(_cache(), maxq=65536 * 21 + 1) == 3            # grid z limit (21 tokens per tile at group 6)
    assert attn(_cache(), seqs=0) == 0
    assert attn(_cache(), total=0) == 0
    assert attn(_cache(), seqs=-1) == 1
    store = lambda k, v, total, cc, tab=1 << 22: L.pkvd_kv_store_prefill(k, v, tab, 8, 1 << 23, 1 << 24, 4, total,
                                                                         None, ctypes.byref(cc), None, None)
    assert store(1 << 20, 1 << 21, -1, _cache()) == 1
    assert store(1 << 20, 1 << 21, 0, _cache()) == 0
    assert store(None, 1 << 21, 5, _cache()) == 1
    assert store(1 << 20, 1 << 21, 5, _cache(), tab=None) == 1
    assert store(1 << 20, (1 << 21) + 8, 5, _cache()) == 3

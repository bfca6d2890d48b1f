"""Python handle on the native host block manager (include/pkvd.h, pkvd_bm_*).

Argument marshalling only: every decision is made by the C++ object.  Block
tables are plain lists of physical block ids.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _capi


def _arr(values, extra=0):
    """int32 host array (numpy) with `extra` spare slots; returns (array, pointer).
    A contiguous int32 numpy array with no spare slots is passed as it is."""
    if extra == 0 and isinstance(values, np.ndarray) and values.dtype == np.int32 and values.flags.c_contiguous \
            and values.size > 0:
        return values, values.ctypes.data_as(ctypes.c_void_p)
    a = np.zeros(len(values) + extra + 1, dtype=np.int32)
    a[:len(values)] = np.asarray(values, dtype=np.int64)
    return a, a.ctypes.data_as(ctypes.c_void_p)


class BlockManager:
    """Physical KV-cache blocks for sequences: exact prefix sharing, clone-N
    (fork) and copy-on-write of a shared partial block."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = _capi.lib()
        h = ctypes.c_void_p()
        _capi.check(self._lib.pkvd_bm_create(num_blocks, block_size, ctypes.byref(h)))
        self._h = h
        self.nb, self.bs = int(num_blocks), int(block_size)

    def close(self) -> None:
        if self._h:
            self._lib.pkvd_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free(self) -> int:
        return int(self._lib.pkvd_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(self._lib.pkvd_bm_ref_count(self._h, block))

    def allocate(self, tokens):
        """(block table, cached token count) for a new prompt, or None when no space."""
        nblk = -(-len(tokens) // self.bs)
        toks, tp = _arr(tokens)
        table, tbp = _arr([], nblk)
        n, cached = ctypes.c_int32(0), ctypes.c_int32(0)
        st = self._lib.pkvd_bm_allocate(self._h, tp, len(tokens), tbp, nblk, ctypes.byref(n), ctypes.byref(cached))
        if st == _capi.NO_SPACE:
            return None
        _capi.check(st)
        return table[:n.value].tolist(), int(cached.value)

    def append(self, tokens, table):
        """The sequence now holds `tokens`: (new table, (src, dst, rows) or None),
        or (None, None) when no block is free."""
        cap = len(table) + 1
        t, tptr = _arr(table, 1)
        toks, tp = _arr(tokens)
        n = ctypes.c_int32(len(table))
        cs, cd, cr = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
        st = self._lib.pkvd_bm_append(self._h, tp, len(tokens), tptr, ctypes.byref(n), cap,
                                      ctypes.byref(cs), ctypes.byref(cd), ctypes.byref(cr))
        if st == _capi.NO_SPACE:
            return None, None
        _capi.check(st)
        copy = (cs.value, cd.value, cr.value) if cs.value >= 0 else None
        return t[:n.value].tolist(), copy

    def fork(self, table):
        t, tp = _arr(table)
        _capi.check(self._lib.pkvd_bm_fork(self._h, tp, len(table)))
        return list(table)

    def release(self, table) -> None:
        t, tp = _arr(table)
        _capi.check(self._lib.pkvd_bm_release(self._h, tp, len(table)))


def shared_prefix_len(block_tables, context_lens, block_size: int) -> int:
    """Tokens a decode batch shares at the start of every row (whole blocks
    that are the same physical block in every table and full before each
    row's newest token), for the shared-prefix attention call.  Host arrays."""
    t = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    c = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    out = ctypes.c_int32(0)
    _capi.check(_capi.lib().pkvd_bm_shared_prefix(t.ctypes.data_as(ctypes.c_void_p), t.shape[0], t.shape[1],
                                                  c.ctypes.data_as(ctypes.c_void_p), block_size, ctypes.byref(out)))
    return int(out.value)

"""Python binding of the host block manager in libpa.so (pa_bm_* in
include/pa.h): the pool's allocator and prefix cache.  Thin ctypes
marshalling; every operation runs in the library's C++ code."""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import _check, lib

_i32 = C.c_int32


def block_hash(token_ids, prefix: int | None = None) -> int:
    """Chained hash of one block: XXH64 over [prefix as 8 LE bytes] + tokens as int64 LE."""
    t = np.ascontiguousarray(token_ids, dtype=np.int64)
    return int(lib().pa_bm_block_hash(t.ctypes.data_as(C.c_void_p), t.size, 0 if prefix is None else 1,
                                      0 if prefix is None else prefix))


def xxh64(data: bytes, seed: int = 0) -> int:
    buf = C.create_string_buffer(data, len(data))
    return int(lib().pa_bm_xxh64(buf if data else None, len(data), seed))


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        self._L = lib()
        h = C.c_void_p()
        _check(self._L.pa_bm_create(num_blocks, block_size, C.byref(h)), "pa_bm_create")
        self._h = h
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if getattr(self, "_h", None):
            self._L.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    # sequences
    def add_sequence(self, token_ids) -> int:
        t = np.ascontiguousarray(token_ids, dtype=np.int64)
        sid = _i32(0)
        _check(self._L.pa_bm_seq_add(self._h, t.ctypes.data_as(C.c_void_p), t.size, C.byref(sid)), "pa_bm_seq_add")
        return sid.value

    def append_token(self, seq: int, token_id: int):
        _check(self._L.pa_bm_seq_append_token(self._h, seq, int(token_id)), "pa_bm_seq_append_token")

    def set_num_cached_tokens(self, seq: int, n: int):
        _check(self._L.pa_bm_seq_set_num_cached_tokens(self._h, seq, n), "pa_bm_seq_set_num_cached_tokens")

    def seq_info(self, seq: int):
        a, b, c = _i32(0), _i32(0), _i32(0)
        _check(self._L.pa_bm_seq_info(self._h, seq, C.byref(a), C.byref(b), C.byref(c)), "pa_bm_seq_info")
        return {"num_tokens": a.value, "num_cached_tokens": b.value, "num_table_blocks": c.value}

    # the pages' operations
    def can_allocate(self, seq: int) -> int:
        r = self._L.pa_bm_can_allocate(self._h, seq)
        if r < -1:
            _check(3, "pa_bm_can_allocate")
        return r

    def allocate(self, seq: int, num_cached_blocks: int):
        _check(self._L.pa_bm_allocate(self._h, seq, num_cached_blocks), "pa_bm_allocate")

    def deallocate(self, seq: int):
        _check(self._L.pa_bm_deallocate(self._h, seq), "pa_bm_deallocate")

    def can_append(self, seq: int) -> bool:
        r = self._L.pa_bm_can_append(self._h, seq)
        if r < 0:
            _check(3, "pa_bm_can_append")
        return bool(r)

    def may_append(self, seq: int):
        _check(self._L.pa_bm_may_append(self._h, seq), "pa_bm_may_append")

    def hash_blocks(self, seq: int, num_scheduled_tokens: int):
        _check(self._L.pa_bm_hash_blocks(self._h, seq, num_scheduled_tokens), "pa_bm_hash_blocks")

    # views
    def block_table(self, seq: int) -> list:
        n = self._L.pa_bm_seq_block_table(self._h, seq, None, 0)
        out = np.empty(max(n, 1), dtype=np.int32)
        self._L.pa_bm_seq_block_table(self._h, seq, out.ctypes.data_as(C.c_void_p), n)
        return out[:n].tolist()

    def block_tables(self, seqs, max_blocks_per_seq: int) -> np.ndarray:
        ids = np.ascontiguousarray(seqs, dtype=np.int32)
        out = np.empty((ids.size, max_blocks_per_seq), dtype=np.int32)
        _check(self._L.pa_bm_block_tables(self._h, ids.ctypes.data_as(C.c_void_p), ids.size,
                                          out.ctypes.data_as(C.c_void_p), max_blocks_per_seq), "pa_bm_block_tables")
        return out

    def free_block_ids(self) -> list:
        n = self._L.pa_bm_free_block_ids(self._h, None, 0)
        out = np.empty(max(n, 1), dtype=np.int32)
        self._L.pa_bm_free_block_ids(self._h, out.ctypes.data_as(C.c_void_p), n)
        return out[:n].tolist()

    def block(self, block_id: int):
        rc, hh, nt = _i32(0), _i32(0), _i32(0)
        hv = C.c_uint64(0)
        _check(self._L.pa_bm_block_info(self._h, block_id, C.byref(rc), C.byref(hh), C.byref(hv), C.byref(nt)),
               "pa_bm_block_info")
        return {"ref_count": rc.value, "hash": hv.value if hh.value else None, "num_token_ids": nt.value}

    def lookup(self, h: int) -> int:
        return int(self._L.pa_bm_lookup_hash(self._h, h))

    def num_hashes(self) -> int:
        return int(self._L.pa_bm_num_hashes(self._h))

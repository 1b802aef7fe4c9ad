"""CPU oracle for paged-KV attention (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product library never loads it, and the two share
no code.  The attention and store arithmetic lives in ``pa_oracle.c``
(plain C, double precision); this module compiles it with gcc and marshals
numpy arrays.  The sampler, whose page fixes fp32, is ``sampler.py`` (numpy
float32).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libpa_oracle.so")
_LIB = None
_LOCK = threading.Lock()

OK, EINVAL, EDUP = 0, -1, -2


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libpa_oracle.so (gcc, no SIMD flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = load(build())
    return _LIB


def load(path: str):
    """Load an oracle shared object and declare its signatures."""
    L = C.CDLL(path)
    i32, i64, dbl, vp = C.c_int32, C.c_int64, C.c_double, C.c_void_p
    L.pa_oracle_version.restype = C.c_int
    L.pa_oracle_slot_mapping.argtypes = [vp, i32, i32, i32, i32, vp]
    L.pa_oracle_slot_mapping.restype = C.c_int
    L.pa_oracle_decode_slot.argtypes = [vp, i32, i32, i32]
    L.pa_oracle_decode_slot.restype = i32
    L.pa_oracle_store_kvcache.argtypes = [vp, i64, vp, i64, vp, vp, vp, i32, i32, i32, i64]
    L.pa_oracle_store_kvcache.restype = C.c_int
    L.pa_oracle_decode.argtypes = [vp, vp, i64, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32,
                                   dbl, vp, i64]
    L.pa_oracle_decode.restype = C.c_int
    L.pa_oracle_prefill.argtypes = [vp, vp, i64, vp, vp, i64, vp, i32, vp, vp, i32, i32, i32, i32,
                                    i32, i32, dbl, i32, vp, i64]
    L.pa_oracle_prefill.restype = C.c_int
    return L


class OracleError(RuntimeError):
    pass


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def slot_mapping(block_table_row, block_size: int, start: int, end: int, L=None) -> np.ndarray:
    """Slots of positions [start, end) of one sequence (block-by-block form)."""
    L = L or lib()
    bt = _c(block_table_row, np.int32)
    out = np.zeros(max(0, end - start), dtype=np.int32)
    n = L.pa_oracle_slot_mapping(_p(bt), len(bt), block_size, start, end, _p(out))
    if n < 0:
        raise OracleError(f"slot_mapping rc={n}")
    return out[:n]


def decode_slot(block_table_row, block_size: int, context_len: int, L=None) -> int:
    """Slot of the newest token of a sequence of length context_len (-1 if 0)."""
    L = L or lib()
    bt = _c(block_table_row, np.int32)
    s = L.pa_oracle_decode_slot(_p(bt), len(bt), block_size, context_len)
    if s == -(2 ** 31):
        raise OracleError("decode_slot: invalid arguments")
    return int(s)


def store_kvcache(key, value, k_cache, v_cache, slot_mapping_, L=None) -> None:
    """In-place scatter into caches [num_blocks, B, Hkv, D] (uint16 bf16 bits).

    key/value are [N, Hkv, D] or [N, row_stride] (row_stride >= Hkv*D, only
    the first Hkv*D entries of a row belong to the token)."""
    L = L or lib()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    _, _, hkv, d = k_cache.shape
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    n = key.shape[0]
    ks = int(np.prod(key.shape[1:])) if key.ndim > 1 else 0
    vs = int(np.prod(value.shape[1:])) if value.ndim > 1 else 0
    sm = _c(slot_mapping_, np.int32)
    num_slots = k_cache.shape[0] * k_cache.shape[1]
    rc = L.pa_oracle_store_kvcache(_p(key), ks, _p(value), vs, _p(k_cache), _p(v_cache),
                                   _p(sm), n, hkv, d, num_slots)
    if rc != OK:
        raise OracleError(f"store_kvcache rc={rc}")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, rows=None,
           L=None) -> np.ndarray:
    """Paged decode attention in float64.  q [batch, Hq, D]; caches
    [num_blocks, B, Hkv, D]; returns [batch, Hq, D] (rows=None) or
    [len(rows), D] for rows = b*Hq + h."""
    L = L or lib()
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    batch, hq, d = q.shape
    nb, B, hkv, _ = k_cache.shape
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    r = None if rows is None else _c(rows, np.int64)
    n = batch * hq if r is None else len(r)
    out = np.zeros((n, d), dtype=np.float64)
    rc = L.pa_oracle_decode(_p(out), _p(q), hq * d, _p(k_cache), _p(v_cache), _p(bt), bt.shape[1],
                            _p(cl), batch, hq, hkv, d, B, nb, float(scale), _p(r),
                            0 if r is None else len(r))
    if rc != OK:
        raise OracleError(f"decode rc={rc}")
    return out.reshape(batch, hq, d) if r is None else out


def prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, block_tables=None,
            causal: bool = True, rows=None, L=None) -> np.ndarray:
    """Varlen prefill attention in float64.  q [total_q, Hq, D].  With
    block_tables, k/v are caches [num_blocks, B, Hkv, D]; without, k/v are
    contiguous [total_k, Hkv, D].  Returns [total_q, Hq, D] or [len(rows), D]
    for rows = token*Hq + h."""
    L = L or lib()
    q = _c(q, np.uint16)
    cq = _c(cu_seqlens_q, np.int32)
    ck = _c(cu_seqlens_k, np.int32)
    tq, hq, d = q.shape
    assert k.flags.c_contiguous and v.flags.c_contiguous
    if block_tables is not None:
        bt = _c(block_tables, np.int32)
        nb, B, hkv, _ = k.shape
        mb, rs = bt.shape[1], 0
    else:
        bt = None
        _, hkv, _ = k.shape
        nb, B, mb, rs = 0, 1, 0, hkv * d
    r = None if rows is None else _c(rows, np.int64)
    n = tq * hq if r is None else len(r)
    out = np.zeros((n, d), dtype=np.float64)
    rc = L.pa_oracle_prefill(_p(out), _p(q), hq * d, _p(k), _p(v), rs, _p(bt), mb, _p(cq), _p(ck),
                             len(cq) - 1, hq, hkv, d, B, nb, float(scale), 1 if causal else 0, _p(r),
                             0 if r is None else len(r))
    if rc != OK:
        raise OracleError(f"prefill rc={rc}")
    return out.reshape(tq, hq, d) if r is None else out

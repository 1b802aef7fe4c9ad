"""The oracle's decode and prefill run over disjoint row sets on several host
threads (test infrastructure, like the rest of this package).

Nothing here computes attention: every row is still produced by one call of
the unchanged C oracle (``pa_oracle_decode`` / ``pa_oracle_prefill``), with
exactly the float64 arithmetic of a single-threaded call.  The C code keeps
no global state, and ctypes releases the GIL for the duration of a foreign
call, so the threads run the oracle's loops in parallel.  Rows are dealt out
round-robin in small chunks, which balances causal prefill rows (row i of a
sequence sees c + i + 1 keys).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import decode as _decode
from . import lib as _lib
from . import prefill as _prefill


def host_threads() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def _map_rows(call, n_rows: int, threads: int, d: int, chunks_per_thread: int = 16) -> np.ndarray:
    out = np.zeros((n_rows, d), dtype=np.float64)
    if n_rows == 0:
        return out
    nchunks = max(1, min(n_rows, threads * chunks_per_thread))
    parts = [np.arange(c, n_rows, nchunks, dtype=np.int64) for c in range(nchunks)]
    _lib()  # compile / load once, before the threads start

    def run(idx):
        return idx, call(idx)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for idx, res in ex.map(run, parts):
            out[idx] = res
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, rows=None, threads=None):
    """``oracle.decode`` computed on `threads` host threads (default: all
    cores); same result, same layout."""
    threads = threads or host_threads()
    batch, hq, d = q.shape
    sel = np.arange(batch * hq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    res = _map_rows(lambda idx: _decode(q, k_cache, v_cache, block_tables, context_lens, scale, rows=sel[idx]),
                    len(sel), threads, d)
    return res.reshape(batch, hq, d) if rows is None else res


def prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, block_tables=None, causal: bool = True,
            rows=None, threads=None):
    """``oracle.prefill`` computed on `threads` host threads (default: all
    cores); same result, same layout."""
    threads = threads or host_threads()
    tq, hq, d = q.shape
    sel = np.arange(tq * hq, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    res = _map_rows(lambda idx: _prefill(q, k, v, cu_seqlens_q, cu_seqlens_k, scale, block_tables=block_tables,
                                         causal=causal, rows=sel[idx]), len(sel), threads, d)
    return res.reshape(tq, hq, d) if rows is None else res

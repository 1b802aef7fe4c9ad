"""The multi-threaded driver of the oracle (oracle/parallel.py) gives, row for
row, exactly the single-threaded oracle's float64 result: it only splits the
rows between threads.  Row order, duplicated rows and the thread count do
not change a bit."""
import numpy as np

import oracle as O
from oracle import parallel as OP
from paged_kv_cache_store_gb300.workloads import make_decode, make_prefill


def test_parallel_decode_equals_serial():
    inp = make_decode("par", 71, 6, 16, 8, [1, 300, 513, 20, 1024, 7], num_blocks=40)
    want = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    for t in (1, 3, 8):
        got = OP.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, threads=t)
        assert np.array_equal(got, want)
    rows = np.array([95, 3, 3, 40, 0], np.int64)
    got = OP.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, rows=rows,
                    threads=4)
    assert np.array_equal(got, want.reshape(-1, 128)[rows])


def test_parallel_prefill_equals_serial():
    p = make_prefill("par", 72, [300, 129, 600], None, 16, 8, cached_tokens=[256, 0, 100])
    for causal in (True, False):
        want = O.prefill(p.q, p.k_cache, p.v_cache, p.cu_seqlens_q, p.cu_seqlens_k, p.scale,
                         block_tables=p.block_tables, causal=causal)
        got = OP.prefill(p.q, p.k_cache, p.v_cache, p.cu_seqlens_q, p.cu_seqlens_k, p.scale,
                         block_tables=p.block_tables, causal=causal, threads=5)
        assert np.array_equal(got, want)

"""GPU parity: pa_prefill_varlen (after the suffix is stored through
pa_slot_mapping_prefill + pa_store_kvcache) against the float64 oracle,
max-abs <= 2e-2 and mean-abs <= 2e-3 on bf16 outputs.  Cases cover several
query and key tiles with ragged tails, prefixes that end mid-block (chunked
prefill), all GQA group sizes, block sizes from 16 to 512, the contiguous
(no block table) path, non-causal attention, and the full prefill workload
(every row)."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import parallel as OP
import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300.workloads import make_prefill, prefill_config
from gpu_util import assert_close, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu


def gpu_prefill(p, causal=True):
    """store the uncached suffix, then prefill through the block tables."""
    kc, vc = dev_bf16(p.k_cache), dev_bf16(p.v_cache)
    bt, cq, ck = dev_i32(p.block_tables), dev_i32(p.cu_seqlens_q), dev_i32(p.cu_seqlens_k)
    slots = pa.slot_mapping_prefill(bt, cq, ck, p.block_size, total_q=p.total_q)
    pa.store_kvcache(dev_bf16(p.new_k), dev_bf16(p.new_v), kc, vc, slots)
    out = pa.prefill_varlen(dev_bf16(p.q), kc, vc, cq, ck, int(p.seqlens_q.max()), int(p.seqlens_k.max()),
                            p.scale, block_tables=bt, causal=causal)
    code, where = pa.get_device_error()
    assert code == 0, (code, where)
    return out, kc, vc


def oracle_caches(p):
    kc, vc = p.k_cache.copy(), p.v_cache.copy()
    slots = np.concatenate([O.slot_mapping(p.block_tables[s], p.block_size,
                                           int(p.seqlens_k[s] - p.seqlens_q[s]), int(p.seqlens_k[s]))
                            for s in range(p.num_seqs)])
    O.store_kvcache(p.new_k, p.new_v, kc, vc, slots)
    return kc, vc


def oracle_prefill(p, rows=None, causal=True):
    kc, vc = oracle_caches(p)
    return O.prefill(p.q, kc, vc, p.cu_seqlens_q, p.cu_seqlens_k, p.scale, block_tables=p.block_tables,
                     causal=causal, rows=rows), kc, vc


CASES = {
    # name: (Lk list, cached tokens list)
    "one-tile": ([5, 128, 1], [0, 0, 0]),
    "ragged": ([129, 255, 300, 513], [0, 0, 0, 0]),
    "prefix-blocks": ([700, 520, 1100], [256, 512, 768]),
    "prefix-mid-block": ([450, 301, 999, 130], [3, 255, 777, 129]),
    "long-suffix": ([1500, 1025], [0, 256]),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_paged_cases(case):
    lk, c = CASES[case]
    p = make_prefill(case, 300 + len(case), lk, None, 32, 8, cached_tokens=c)
    out, kc, vc = gpu_prefill(p)
    want, okc, ovc = oracle_prefill(p)
    assert np.array_equal(host_bits(kc), okc) and np.array_equal(host_bits(vc), ovc)
    assert_close(host_f64(out), want, case)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (4, 1)])
def test_prefill_gqa_groups(hq, hkv):
    p = make_prefill("gqa", 400 + hq, [333, 200], None, hq, hkv, cached_tokens=[100, 0])
    out, _, _ = gpu_prefill(p)
    want, _, _ = oracle_prefill(p)
    assert_close(host_f64(out), want, f"gqa {hq}/{hkv}")


@pytest.mark.parametrize("B", [16, 32, 48, 64, 128, 512])
def test_prefill_block_sizes(B):
    lk = [3 * B + 5, B, 260]
    c = [B + 1, 0, 17]
    p = make_prefill("bs", 500 + B, lk, None, 16, 8, block_size=B, cached_tokens=c)
    out, _, _ = gpu_prefill(p)
    want, _, _ = oracle_prefill(p)
    assert_close(host_f64(out), want, f"block_size {B}")


def test_prefill_non_causal():
    p = make_prefill("nc", 600, [200, 129, 64], None, 16, 8, cached_tokens=[50, 0, 0])
    out, _, _ = gpu_prefill(p, causal=False)
    want, _, _ = oracle_prefill(p, causal=False)
    assert_close(host_f64(out), want, "non-causal")


def test_prefill_contiguous_path():
    """No block table: contiguous k/v rows indexed by cu_seqlens_k (with and
    without extra leading keys)."""
    lens_k = [300, 17, 140]
    lens_q = [300, 10, 1]
    hq, hkv = 16, 8
    from paged_kv_cache_store_gb300.workloads import normal_bf16
    tq, tk = sum(lens_q), sum(lens_k)
    q = normal_bf16(700, 1, (tq, hq, 128))
    k = normal_bf16(700, 2, (tk, hkv, 128))
    v = normal_bf16(700, 3, (tk, hkv, 128))
    cq = np.cumsum([0] + lens_q).astype(np.int32)
    ck = np.cumsum([0] + lens_k).astype(np.int32)
    out = pa.prefill_varlen(dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_i32(cq), dev_i32(ck), max(lens_q),
                            max(lens_k), 128 ** -0.5)
    assert pa.get_device_error() == (0, 0)
    want = O.prefill(q, k, v, cq, ck, 128 ** -0.5)
    assert_close(host_f64(out), want, "contiguous")


def test_prefill_last_row_matches_decode():
    """The last query row of each sequence equals decode over the same pool."""
    p = make_prefill("x", 800, [900, 257, 1300], None, 32, 8, cached_tokens=[256, 0, 1000])
    out, kc, vc = gpu_prefill(p)
    last = p.cu_seqlens_q[1:] - 1
    q_last = dev_bf16(p.q[last])
    dec = pa.decode(q_last, kc, vc, dev_i32(p.block_tables), dev_i32(p.seqlens_k), p.scale)
    a, b = host_f64(out)[last], host_f64(dec)
    assert np.abs(a - b).max() <= 2e-2


def test_prefill_workload_full_size():
    """The 16-sequence prefill workload (prefix hits of 0..3 blocks) in the
    launch configuration the benchmark times: every (token, head) row against
    the oracle (run on all host cores by oracle.parallel, each row by the
    unchanged oracle), and the stored suffix bit-exact."""
    p = prefill_config(5)
    out, kc, vc = gpu_prefill(p)
    okc, ovc = oracle_caches(p)
    assert np.array_equal(host_bits(kc), okc) and np.array_equal(host_bits(vc), ovc)
    want = OP.prefill(p.q, okc, ovc, p.cu_seqlens_q, p.cu_seqlens_k, p.scale, block_tables=p.block_tables)
    assert_close(host_f64(out), want, "prefill workload, all rows")


def test_prefill_repeat_runs_bitwise_identical():
    """Each output tile is computed by one CTA in a fixed order, so repeated
    runs agree bit for bit.  A missed wait between the tensor-core pipeline
    and the softmax/epilogue warps (reading O or a staged tile too early)
    shows up here as a run that differs; the runs alternate cold and warm L2
    to vary the timing."""
    p = prefill_config(5)
    kc, vc = dev_bf16(p.k_cache), dev_bf16(p.v_cache)
    bt, cq, ck = dev_i32(p.block_tables), dev_i32(p.cu_seqlens_q), dev_i32(p.cu_seqlens_k)
    q = dev_bf16(p.q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ref = None
    for it in range(12):
        if it % 2:
            flush.zero_()
        out = pa.prefill_varlen(q, kc, vc, cq, ck, int(p.seqlens_q.max()), int(p.seqlens_k.max()), p.scale,
                                block_tables=bt)
        bits = out.view(torch.int16).cpu()
        if ref is None:
            ref = bits
        else:
            assert torch.equal(bits, ref), f"run {it} differs"
    assert pa.get_device_error() == (0, 0)


def test_prefill_schedules_agree():
    """Up to 512 (query tile, sequence) groups the kernel deals units out
    longest first; above that, in query-tile order.  A larger max_seqlen_q
    hint (allowed: it only bounds the lengths) switches to the second order
    on the same inputs: the outputs must be bit-identical, and match the
    oracle."""
    lk = [130, 700, 260, 1025, 77, 513, 300, 900, 128, 640, 999, 20, 400, 256, 1300, 90]
    c = [0, 256, 3, 512, 0, 129, 44, 0, 0, 300, 768, 0, 17, 0, 256, 0]
    p = make_prefill("sched", 31, lk, None, 16, 8, cached_tokens=c)
    kc, vc = dev_bf16(p.k_cache), dev_bf16(p.v_cache)
    bt, cq, ck = dev_i32(p.block_tables), dev_i32(p.cu_seqlens_q), dev_i32(p.cu_seqlens_k)
    slots = pa.slot_mapping_prefill(bt, cq, ck, p.block_size, total_q=p.total_q)
    pa.store_kvcache(dev_bf16(p.new_k), dev_bf16(p.new_v), kc, vc, slots)
    q = dev_bf16(p.q)
    mq, mk = int(p.seqlens_q.max()), int(p.seqlens_k.max())
    assert -(-mq // 128) * p.num_seqs <= 512 < 40 * p.num_seqs
    sorted_out = pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, p.scale, block_tables=bt)
    plain_out = pa.prefill_varlen(q, kc, vc, cq, ck, 40 * 128, mk, p.scale, block_tables=bt)
    assert pa.get_device_error() == (0, 0)
    assert torch.equal(sorted_out, plain_out)
    want, _, _ = oracle_prefill(p)
    assert_close(host_f64(sorted_out), want)


def fused_vs_unfused(p, ws=None, causal=True):
    """The fused store + prefill against slot mapping + store + prefill on
    copies of the same pool: identical outputs and identical caches."""
    bt, cq, ck = dev_i32(p.block_tables), dev_i32(p.cu_seqlens_q), dev_i32(p.cu_seqlens_k)
    q, nk, nv = dev_bf16(p.q), dev_bf16(p.new_k), dev_bf16(p.new_v)
    mq, mk = int(p.seqlens_q.max()), int(p.seqlens_k.max())
    kc1, vc1 = dev_bf16(p.k_cache), dev_bf16(p.v_cache)
    slots = pa.slot_mapping_prefill(bt, cq, ck, p.block_size, total_q=p.total_q)
    pa.store_kvcache(nk, nv, kc1, vc1, slots)
    ref = pa.prefill_varlen(q, kc1, vc1, cq, ck, mq, mk, p.scale, block_tables=bt, causal=causal)
    kc2, vc2 = dev_bf16(p.k_cache), dev_bf16(p.v_cache)
    got = pa.prefill_varlen(q, kc2, vc2, cq, ck, mq, mk, p.scale, block_tables=bt, new_k=nk, new_v=nv, workspace=ws,
                            causal=causal)
    assert pa.get_device_error() == (0, 0)
    assert torch.equal(got, ref)
    assert torch.equal(kc2, kc1) and torch.equal(vc2, vc1)
    return got


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_fused_store_equals_store_then_prefill(case):
    lk, c = CASES[case]
    p = make_prefill(case, 41, lk, None, 16, 8, cached_tokens=c)
    got = fused_vs_unfused(p)
    want, _, _ = oracle_prefill(p)
    assert_close(host_f64(got), want)


@pytest.mark.parametrize("B", [16, 48, 512])
def test_prefill_fused_store_block_sizes(B):
    """Blocks smaller than a 128-key tile (several boxes per tile) and larger."""
    p = make_prefill("fbs", 700 + B, [3 * B + 5, B, 260], None, 16, 8, block_size=B, cached_tokens=[B + 1, 0, 17])
    got = fused_vs_unfused(p)
    want, _, _ = oracle_prefill(p)
    assert_close(host_f64(got), want, f"fused, block_size {B}")


def test_prefill_fused_store_non_causal():
    p = make_prefill("fnc", 601, [200, 129, 64], None, 16, 8, cached_tokens=[50, 0, 0])
    got = fused_vs_unfused(p, causal=False)
    want, _, _ = oracle_prefill(p, causal=False)
    assert_close(host_f64(got), want, "fused, non-causal")


def test_prefill_fused_store_workspace_reused():
    """One workspace serves consecutive calls: the grid barrier leaves its
    counter at zero and only moves its generation on."""
    ws = pa.prefill_store_workspace()
    for seed, lk, c in ((5, [300, 40, 700], [0, 0, 256]), (6, [129, 1025], [17, 512]), (7, [64], [0])):
        p = make_prefill("ws", seed, lk, None, 8, 2, cached_tokens=c)
        fused_vs_unfused(p, ws)
    words = ws.view(torch.int32).cpu().tolist()
    assert words[0] == 0 and words[1] > 0


def test_prefill_fused_store_bad_block_recorded_not_written():
    p = make_prefill("bad", 9, [300, 200], None, 16, 8, cached_tokens=[0, 0])
    bt = p.block_tables.copy()
    bt[1, 0] = p.k_cache.shape[0] + 3  # sequence 1's first block id is outside the pool
    kc, vc = dev_bf16(p.k_cache), dev_bf16(p.v_cache)
    pa.get_device_error()
    pa.prefill_varlen(dev_bf16(p.q), kc, vc, dev_i32(p.cu_seqlens_q), dev_i32(p.cu_seqlens_k), 300, 300, p.scale,
                      block_tables=dev_i32(bt), new_k=dev_bf16(p.new_k), new_v=dev_bf16(p.new_v))
    code, where = pa.get_device_error()
    assert code == pa.PA_DEV_BAD_SLOT and 300 <= where < 300 + p.block_size  # a token of sequence 1
    # Sequence 0's rows are stored; sequence 1's are not; nothing else changed.
    for cache, new, orig in ((kc, p.new_k, p.k_cache), (vc, p.new_v, p.v_cache)):
        want = orig.copy().reshape(-1, 8 * 128)
        want[O.slot_mapping(p.block_tables[0], p.block_size, 0, 300)] = new[:300].reshape(300, -1)
        assert np.array_equal(host_bits(cache).reshape(-1, 8 * 128), want)


def test_prefill_fused_store_workload_full_size():
    fused_vs_unfused(prefill_config(5))


def test_prefill_fused_store_barrier_timeout_is_recorded():
    """Failure detection without a fault: with the workspace's arrival count
    seeded far from the grid size no CTA is ever the last to arrive, so every
    CTA's bounded wait at the grid barrier runs out (after ~1 s), records
    PA_DEV_TIMEOUT at site 440 and skips its units.  The context stays
    usable: after zeroing the workspace the same call gives the right
    answer."""
    p = make_prefill("timeout", 12, [300, 129], None, 8, 2, cached_tokens=[0, 17])
    ws = pa.prefill_store_workspace()
    ws.view(torch.int32)[0] = 1 << 30
    kc, vc = dev_bf16(p.k_cache), dev_bf16(p.v_cache)
    bt, cq, ck = dev_i32(p.block_tables), dev_i32(p.cu_seqlens_q), dev_i32(p.cu_seqlens_k)
    q, nk, nv = dev_bf16(p.q), dev_bf16(p.new_k), dev_bf16(p.new_v)
    pa.get_device_error()
    pa.prefill_varlen(q, kc, vc, cq, ck, 300, 300, p.scale, block_tables=bt, new_k=nk, new_v=nv, workspace=ws)
    assert pa.get_device_error() == (pa.PA_DEV_TIMEOUT, 440)
    ws.zero_()
    fused_vs_unfused(p, ws)

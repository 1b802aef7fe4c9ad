"""GPU parity: pa_decode (after pa_store_kvcache of the decoded token)
against the float64 oracle, max-abs <= 2e-2 and mean-abs <= 2e-3 on bf16
outputs.  Small odd shapes span several tiles, chunks and ragged tails; the
four decode workloads run at full size in the launch configuration the
benchmark times."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300.workloads import decode_config, make_decode
from gpu_util import assert_close, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu


def run_gpu_step(inp):
    """store the decoded token's K/V at its slot, then decode; returns (out, caches)."""
    kc, vc = dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx = dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    slots = pa.slot_mapping_decode(bt, ctx, inp.block_size)
    pa.store_kvcache(dev_bf16(inp.new_k), dev_bf16(inp.new_v), kc, vc, slots)
    out = pa.decode(dev_bf16(inp.q), kc, vc, bt, ctx, inp.scale)
    code, where = pa.get_device_error()
    assert code == 0, (code, where)
    return out, kc, vc


def run_oracle_step(inp, rows=None):
    kc, vc = inp.k_cache.copy(), inp.v_cache.copy()
    slots = np.array([O.decode_slot(inp.block_tables[b], inp.block_size, int(inp.context_lens[b]))
                      for b in range(inp.batch)], np.int32)
    O.store_kvcache(inp.new_k, inp.new_v, kc, vc, slots)
    return O.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale, rows=rows), kc, vc


EDGE_CTX = [1, 2, 15, 16, 17, 63, 64, 65, 255, 256, 257, 511, 512, 513, 1000, 1537]


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8), (64, 8)])
def test_decode_edge_lengths(hq, hkv):
    inp = make_decode(f"edge {hq}/{hkv}", 100 + hq, len(EDGE_CTX), hq, hkv, EDGE_CTX)
    out, kc, vc = run_gpu_step(inp)
    want, okc, ovc = run_oracle_step(inp)
    assert np.array_equal(host_bits(kc), okc)
    assert_close(host_f64(out), want, f"decode {hq}/{hkv}")


@pytest.mark.parametrize("B", [16, 32, 48, 64, 128, 256, 512])
def test_decode_block_sizes(B):
    ctx = [1, B - 1, B, B + 1, 3 * B + 7, 700]
    inp = make_decode(f"B={B}", 200 + B, len(ctx), 32, 8, ctx, block_size=B)
    out, _, _ = run_gpu_step(inp)
    want, _, _ = run_oracle_step(inp)
    assert_close(host_f64(out), want, f"block_size {B}")


def test_decode_zero_context_rows_and_padded_tables():
    ctx = [0, 300, 0, 1, 4097]
    inp = make_decode("zero rows", 7, len(ctx), 16, 8, [max(c, 1) for c in ctx], extra_table_cols=3)
    inp.context_lens[:] = ctx
    inp.block_tables[[0, 2], :] = -1
    kc, vc = dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    out = torch.full((len(ctx), 16, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    pa.decode(dev_bf16(inp.q), kc, vc, dev_i32(inp.block_tables), dev_i32(inp.context_lens), inp.scale, out=out)
    assert pa.get_device_error() == (0, 0)
    want = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    got = host_f64(out)
    assert np.all(got[[0, 2]] == 0.0)
    assert_close(got, want, "zero rows")


def test_decode_shared_prefix_blocks():
    ctx = [1025, 1300, 2048, 4000, 1100, 600]
    inp = make_decode("shared", 8, len(ctx), 32, 8, ctx, shared_prefix_seqs=4, shared_prefix_blocks=4)
    out, _, _ = run_gpu_step(inp)
    want, _, _ = run_oracle_step(inp)
    assert_close(host_f64(out), want, "shared prefix")


def test_decode_strided_q_rows():
    ctx = [100, 2000, 3]
    inp = make_decode("strided q", 9, 3, 16, 8, ctx)
    qkv = torch.zeros(3, (16 + 16) * 128, dtype=torch.bfloat16, device="cuda")
    qkv[:, :16 * 128] = dev_bf16(inp.q).view(3, -1)
    q = qkv[:, :16 * 128].view(3, 16, 128)
    out = pa.decode(q, dev_bf16(inp.k_cache), dev_bf16(inp.v_cache), dev_i32(inp.block_tables),
                    dev_i32(inp.context_lens), inp.scale)
    want = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    assert_close(host_f64(out), want, "strided q")


def test_decode_pairs_cut_across_many_ctas():
    """One long sequence: its 8 (sequence, kv head) pairs of 157 tiles are cut
    into ranges of ~8 tiles, so every pair is merged from ~20 CTA partials,
    most of them a CTA's only segment."""
    inp = make_decode("long", 10, 1, 32, 8, [10000])
    out, _, _ = run_gpu_step(inp)
    want, _, _ = run_oracle_step(inp)
    assert_close(host_f64(out), want, "long")


def test_decode_fewer_tiles_than_ctas():
    """Fewer tiles than CTAs: most CTAs get no work, the rest one tile, and a
    pair of several tiles is merged from one-tile partials.  (The grid is
    sized from the table width, so the tables get padding columns to keep it
    at one CTA per SM.)"""
    for hq, hkv, ctx in [(8, 8, [1]), (16, 8, [130, 5]), (8, 1, [64 * 40 + 3])]:
        inp = make_decode(f"few {hq}/{hkv}", 14, len(ctx), hq, hkv, ctx, extra_table_cols=320)
        out, _, _ = run_gpu_step(inp)
        want, _, _ = run_oracle_step(inp)
        assert_close(host_f64(out), want, f"few tiles {hq}/{hkv} {ctx}")


def test_decode_small_grid_from_narrow_tables():
    """Narrow tables bound the work, so the grid shrinks (here to a few CTAs,
    each with several tiles): same results, fused store included."""
    for hq, hkv, ctx in [(16, 8, [600, 1, 257, 90]), (32, 8, [5, 64]), (8, 2, [1000])]:
        inp = make_decode(f"narrow {hq}/{hkv}", 15, len(ctx), hq, hkv, ctx)
        out, _, _ = run_gpu_step(inp)
        want, _, _ = run_oracle_step(inp)
        assert_close(host_f64(out), want, f"narrow {hq}/{hkv} {ctx}")
        fout, fkc, fvc = run_gpu_fused(inp)
        assert torch.equal(fout, out)


def test_decode_repeated_calls_reuse_workspace():
    """Many calls on one workspace give identical results: each call leaves
    its counters zeroed for the next."""
    ctx = [3000, 5000, 257, 1]
    inp = make_decode("repeat", 11, 4, 16, 8, ctx)
    kc, vc = dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    q, bt, cl = dev_bf16(inp.q), dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    ws = pa.decode_workspace(16, 8, 128)
    outs = [pa.decode(q, kc, vc, bt, cl, inp.scale, workspace=ws) for _ in range(5)]
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    want = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    assert_close(host_f64(outs[0]), want, "repeat")


def test_decode_bad_context_is_recorded():
    inp = make_decode("bad ctx", 12, 2, 16, 8, [10, 10])
    cl = inp.context_lens.copy()
    cl[1] = inp.max_blocks * inp.block_size + 1
    pa.get_device_error()
    pa.decode(dev_bf16(inp.q), dev_bf16(inp.k_cache), dev_bf16(inp.v_cache), dev_i32(inp.block_tables),
              dev_i32(cl), inp.scale)
    code, where = pa.get_device_error()
    assert code == pa.PA_DEV_BAD_CONTEXT and where == 1


def test_decode_checked_mode_records_bad_block():
    inp = make_decode("bad block", 13, 2, 16, 8, [300, 10])
    bt = inp.block_tables.copy()
    bt[0, 1] = inp.num_blocks + 3
    pa.get_device_error()
    pa.set_checked(True)
    try:
        out = pa.decode(dev_bf16(inp.q), dev_bf16(inp.k_cache), dev_bf16(inp.v_cache), dev_i32(bt),
                        dev_i32(inp.context_lens), inp.scale)
        code, where = pa.get_device_error()
    finally:
        pa.set_checked(False)
    assert code == pa.PA_DEV_BAD_BLOCK and where == 1
    # Sequence 1 is unaffected.
    want = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
    assert_close(host_f64(out)[1], want[1], "unaffected row")


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_decode_workloads_full_size(cfg):
    """The four decode workloads at full size (store + decode, the benchmark's
    step), every output row against the oracle."""
    inp = decode_config(cfg)
    out, kc, vc = run_gpu_step(inp)
    want, okc, ovc = run_oracle_step(inp)
    # The store touched exactly the decoded tokens' slots.
    assert np.array_equal(host_bits(kc), okc) and np.array_equal(host_bits(vc), ovc)
    assert_close(host_f64(out), want, f"workload {cfg}")


def test_decode_one_workspace_serves_every_gqa_group():
    """A workspace sized for the largest group is reused by calls of other
    groups in turn; its counters stay zeroed between them (they sit at offsets
    that do not depend on the group)."""
    ws = pa.decode_workspace(64, 8, 128)
    for hq, ctx in [(32, [4000, 77, 1300]), (16, [1, 17, 200, 255, 256]), (64, [2500, 9]), (8, [700] * 6),
                    (16, [5000, 5000])]:
        inp = make_decode(f"ws {hq}", 20 + hq, len(ctx), hq, 8, ctx)
        out = pa.decode(dev_bf16(inp.q), dev_bf16(inp.k_cache), dev_bf16(inp.v_cache), dev_i32(inp.block_tables),
                        dev_i32(inp.context_lens), inp.scale, workspace=ws)
        assert pa.get_device_error() == (0, 0)
        want = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale)
        assert_close(host_f64(out), want, f"shared workspace {hq}/8")


def run_gpu_fused(inp, strided=False):
    """pa_decode_store: the kernel stores the token's K/V itself, then decodes."""
    kc, vc = dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx = dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    nk, nv = dev_bf16(inp.new_k), dev_bf16(inp.new_v)
    if strided:  # K and V as column slices of one fused [batch, 2*Hkv*D] tensor
        both = torch.cat([nk.reshape(inp.batch, -1), nv.reshape(inp.batch, -1)], dim=1)
        half = nk[0].numel()
        nk = both[:, :half].view(inp.batch, inp.num_kv_heads, inp.head_dim)
        nv = both[:, half:].view(inp.batch, inp.num_kv_heads, inp.head_dim)
    out = pa.decode(dev_bf16(inp.q), kc, vc, bt, ctx, inp.scale, new_k=nk, new_v=nv)
    code, where = pa.get_device_error()
    assert code == 0, (code, where)
    return out, kc, vc


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8), (64, 8)])
def test_decode_store_fused_edge_lengths(hq, hkv):
    """The fused store leaves the caches exactly as store_kvcache would, and the
    attention sees the new token."""
    inp = make_decode(f"fused {hq}/{hkv}", 300 + hq, len(EDGE_CTX), hq, hkv, EDGE_CTX)
    out, kc, vc = run_gpu_fused(inp, strided=(hq == 32))
    want, okc, ovc = run_oracle_step(inp)
    assert np.array_equal(host_bits(kc), okc) and np.array_equal(host_bits(vc), ovc)
    assert_close(host_f64(out), want, f"fused decode {hq}/{hkv}")


@pytest.mark.parametrize("B", [16, 64, 256])
def test_decode_store_fused_block_sizes_and_zero_rows(B):
    ctx = [1, B - 1, B, B + 1, 0, 3 * B + 7]
    inp = make_decode(f"fused B={B}", 400 + B, len(ctx), 32, 8, [max(c, 1) for c in ctx], block_size=B)
    inp.context_lens[:] = ctx
    out, kc, vc = run_gpu_fused(inp)
    # ctx == 0 rows store nothing (as a -1 slot would), the others one row.
    okc, ovc = inp.k_cache.copy(), inp.v_cache.copy()
    slots = np.array([O.decode_slot(inp.block_tables[b], B, c) if c > 0 else -1 for b, c in enumerate(ctx)], np.int32)
    O.store_kvcache(inp.new_k, inp.new_v, okc, ovc, slots)
    assert np.array_equal(host_bits(kc), okc) and np.array_equal(host_bits(vc), ovc)
    want = O.decode(inp.q, okc, ovc, inp.block_tables, inp.context_lens, inp.scale)
    assert_close(host_f64(out), want, f"fused B={B}")


def test_decode_store_fused_workload_full_size():
    """The qwen3-0.6b decode workload through the fused path: caches bit-exact,
    sampled rows against the oracle, and the same output as the unfused step."""
    inp = decode_config(2)
    out, kc, vc = run_gpu_fused(inp)
    out2, kc2, vc2 = run_gpu_step(inp)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(out, out2)
    rows = np.arange(0, inp.batch * inp.num_q_heads, 37)
    want, _, _ = run_oracle_step(inp, rows=rows)
    assert_close(host_f64(out).reshape(-1, 128)[rows], want, "fused workload")

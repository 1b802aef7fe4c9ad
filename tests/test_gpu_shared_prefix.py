"""GPU parity of pa_decode_shared_prefix: batches in which sequences share
prefix-cache blocks ([NV12 §12.8]: the same physical blocks at the start of
several block tables).  The shared prefix is attended once per kv head for
all members and merged into each member's suffix attention, so the result
must equal the plain definition (the float64 oracle) within the attention
tolerance, and the new token's K/V rows must land in the caches bit-exactly.
Cases: the Qwen3-8B-shaped workload at full size (every row), interleaved
groups whose members diverge after different numbers of blocks, block sizes
that do not divide the 64-row tile, every GQA group, a prefix that ends one
token before the newest, a group larger than one work chunk, and a batch
with no sharing (bit-identical to pa_decode)."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import parallel as OP
import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300.workloads import decode_config, make_decode
from gpu_util import assert_close, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu


def oracle_step(inp):
    kc, vc = inp.k_cache.copy(), inp.v_cache.copy()
    slots = np.array([O.decode_slot(inp.block_tables[b], inp.block_size, int(inp.context_lens[b]))
                      for b in range(inp.batch)], np.int32)
    O.store_kvcache(inp.new_k, inp.new_v, kc, vc, slots)
    return OP.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale), kc, vc


def gpu_step(inp, store=True, ws=None):
    kc, vc = dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx = dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    if store:
        out = pa.decode(dev_bf16(inp.q), kc, vc, bt, ctx, inp.scale, new_k=dev_bf16(inp.new_k),
                        new_v=dev_bf16(inp.new_v), shared_prefix=True, workspace=ws)
    else:
        slots = pa.slot_mapping_decode(bt, ctx, inp.block_size)
        pa.store_kvcache(dev_bf16(inp.new_k), dev_bf16(inp.new_v), kc, vc, slots)
        out = pa.decode(dev_bf16(inp.q), kc, vc, bt, ctx, inp.scale, shared_prefix=True, workspace=ws)
    code, where = pa.get_device_error()
    assert code == 0, (code, where)
    return out, kc, vc


def share(inp, groups):
    """Rewrite block tables so that each (leader, members, nblocks) group's
    members use the leader's first nblocks physical blocks (their own blocks
    there are simply no longer referenced)."""
    bt = inp.block_tables
    for leader, members, n in groups:
        for m in members:
            assert (int(inp.context_lens[m]) - 1) // inp.block_size >= n, "only full blocks before the last"
            bt[m, :n] = bt[leader, :n]
    return inp


def check(inp, store=True):
    out, kc, vc = gpu_step(inp, store=store)
    want, okc, ovc = oracle_step(inp)
    assert np.array_equal(host_bits(kc), okc) and np.array_equal(host_bits(vc), ovc)
    assert_close(host_f64(out), want, inp.name)
    return out


def test_shared_prefix_qwen3_8b_workload_full_size():
    """The headline workload: 128 of 256 sequences share their first 4 blocks."""
    check(decode_config(3))


@pytest.mark.parametrize("store", [True, False])
def test_shared_prefix_interleaved_groups(store):
    ctx = [1100, 900, 1300, 700, 1025, 2000, 1500, 513, 300, 800]
    inp = make_decode("groups", 41, len(ctx), 32, 8, ctx)
    # group A: 0, 2, 4 share 3 blocks, but 6 agrees only on block 0, so A shares 1 block;
    # group B: 1, 3 share 2 blocks; 7 shares block 0 with 9 (2 members); 5 and 8 alone.
    share(inp, [(0, [2, 4], 4), (0, [6], 1), (1, [3], 2), (7, [9], 1)])
    inp.block_tables[4, 3] = inp.block_tables[0, 3]  # 4 agrees with the leader longer than 6 does
    check(inp, store=store)


@pytest.mark.parametrize("B", [16, 48, 64, 128, 256, 512])
def test_shared_prefix_block_sizes(B):
    ctx = [9 * B + 5, 6 * B + 1, 7 * B + 30, 4 * B + 2, 12 * B]
    inp = make_decode(f"B={B}", 42 + B, len(ctx), 16, 8, ctx, block_size=B)
    share(inp, [(0, [1, 2, 4], 5), (3, [], 0)])
    check(inp)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8)])
def test_shared_prefix_gqa_groups(hq, hkv):
    ctx = [1300, 1025, 1500, 257, 800]
    inp = make_decode(f"gqa {hq}/{hkv}", 43 + hq, len(ctx), hq, hkv, ctx)
    share(inp, [(0, [1, 2], 4), (4, [3], 1)])
    check(inp)


def test_shared_prefix_up_to_the_newest_token():
    """Members whose whole context but the newest token is the shared prefix."""
    ctx = [4 * 256 + 1, 4 * 256 + 1, 5 * 256, 4 * 256 + 1]
    inp = make_decode("tight", 44, len(ctx), 32, 8, ctx)
    share(inp, [(0, [1, 2, 3], 4)])
    check(inp)


def test_shared_prefix_large_group():
    """40 members of one group (several 16-member work chunks per kv head) and
    a second group, with ragged suffixes."""
    rng = np.random.default_rng(45)
    ctx = list(rng.integers(3 * 256 + 1, 2500, size=48))
    inp = make_decode("large", 45, len(ctx), 32, 8, ctx, shared_prefix_seqs=40, shared_prefix_blocks=3)
    share(inp, [(40, list(range(41, 48)), 2)])
    check(inp)


def test_shared_prefix_one_block_of_64():
    """A shared prefix of one 64-key tile: three of the four key splits have
    no tile and leave empty partials."""
    ctx = [200, 65, 130, 300]
    inp = make_decode("one tile", 46, len(ctx), 32, 8, ctx, block_size=64)
    share(inp, [(0, [1, 2, 3], 1)])
    check(inp)


def test_shared_prefix_two_chunks_gqa1():
    """GQA group 1: 128 members per work item, so 140 members need two."""
    rng = np.random.default_rng(47)
    ctx = list(rng.integers(2 * 256 + 1, 1200, size=140))
    inp = make_decode("gqa1 140", 47, len(ctx), 8, 8, ctx, shared_prefix_seqs=140, shared_prefix_blocks=2)
    check(inp)


def test_shared_prefix_members_past_the_partial_rows():
    """64 q heads: 8192 partial rows hold 128 members; the other 12 members of
    the group read the shared prefix themselves."""
    rng = np.random.default_rng(48)
    ctx = list(rng.integers(2 * 256 + 1, 900, size=140))
    inp = make_decode("cap", 48, len(ctx), 64, 8, ctx, shared_prefix_seqs=140, shared_prefix_blocks=2)
    check(inp)


def test_shared_prefix_without_sharing_equals_pa_decode():
    inp = decode_config(2)  # no shared blocks
    kc, vc = dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx, q = dev_i32(inp.block_tables), dev_i32(inp.context_lens), dev_bf16(inp.q)
    ref = pa.decode(q, kc, vc, bt, ctx, inp.scale)
    got = pa.decode(q, kc, vc, bt, ctx, inp.scale, shared_prefix=True)
    assert pa.get_device_error() == (0, 0)
    assert torch.equal(got, ref)


def test_shared_prefix_workspace_reused():
    """Two calls on one workspace agree bit for bit (the workspace's counters
    are left zeroed; the prefix partials are rewritten)."""
    inp = decode_config(3)
    ws = pa.decode_workspace(inp.num_q_heads, inp.num_kv_heads, inp.head_dim, shared_prefix=True)
    outs = []
    for _ in range(2):
        out, _, _ = gpu_step(inp, store=False, ws=ws)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])

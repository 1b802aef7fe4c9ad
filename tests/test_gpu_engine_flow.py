"""GPU integration of the host block manager with the kernels, the way an
engine step uses them [NV12 §12.8 BlockManager; VS §1.2.4-1.2.5]: the C++
block manager (pa_bm_*) allocates blocks, finds prefix-cache hits and hands
out block tables; the kernels store the uncached suffix, run the varlen
prefill through those tables, then run fused decode steps (store of the new
token + attention) while the manager appends blocks and hashes full ones.
Every attention output is compared with the float64 oracle run on a host
mirror of the caches, which the oracle's own store updates; the caches must
end bit-identical to the mirror, and the blocks shared through the prefix
cache must never be rewritten.

K and V rows depend only on (token id, position), as a model's would, so a
prefix-cache hit holds exactly what recomputation would have produced."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300.block_manager import BlockManager
from paged_kv_cache_store_gb300.workloads import f32_to_bf16_bits
from gpu_util import assert_close, dev_bf16, dev_i32, host_bits, host_f64

pytestmark = pytest.mark.gpu

B, HQ, HKV, D, NB, MAXB = 16, 8, 4, 128, 48, 12
SCALE = 1.0 / math.sqrt(D)


def rows(tokens, positions, kind, heads):
    """bf16 bits [n, heads, D]: one row per (token id, position); kind 0 = K,
    1 = V, 2 = q."""
    out = np.empty((len(tokens), heads, D), dtype=np.uint16)
    for i, (t, p) in enumerate(zip(tokens, positions)):
        rng = np.random.default_rng([int(t), int(p), kind])
        out[i] = f32_to_bf16_bits(rng.standard_normal((heads, D)).astype(np.float32))
    return out


class Engine:
    def __init__(self):
        self.bm = BlockManager(NB, B)
        rng = np.random.default_rng(77)
        stale = lambda: f32_to_bf16_bits(rng.standard_normal((NB, B, HKV, D)).astype(np.float32))
        self.kc_h, self.vc_h = stale(), stale()  # host mirror (stale pool contents)
        self.kc, self.vc = dev_bf16(self.kc_h), dev_bf16(self.vc_h)
        self.tokens = {}
        self.ws = pa.decode_workspace(HQ, HKV, D, torch.device("cuda"))

    def tables(self, sids):
        return self.bm.block_tables(sids, MAXB)

    def prefill(self, seqs):
        """seqs: {sid: token list}; allocates (with prefix hits) and runs the
        uncached suffixes.  Returns the number of cached blocks per sid."""
        cached = {}
        for sid in seqs:
            n = self.bm.can_allocate(sid)
            assert n >= 0
            self.bm.allocate(sid, n)
            cached[sid] = n
        sids = list(seqs)
        bt = self.tables(sids)
        cq, ck, q, nk, nv, slots_h = [0], [0], [], [], [], []
        for i, sid in enumerate(sids):
            toks = seqs[sid]
            c = cached[sid] * B
            pos = list(range(c, len(toks)))
            suf = toks[c:]
            q.append(rows(suf, pos, 2, HQ))
            nk.append(rows(suf, pos, 0, HKV))
            nv.append(rows(suf, pos, 1, HKV))
            cq.append(cq[-1] + len(suf))
            ck.append(ck[-1] + len(toks))
            slots_h.append(O.slot_mapping(bt[i], B, c, len(toks)))
        q, nk, nv = np.concatenate(q), np.concatenate(nk), np.concatenate(nv)
        cq, ck = np.asarray(cq, np.int32), np.asarray(ck, np.int32)
        # device: slot mapping, store, prefill
        bt_d, cq_d, ck_d = dev_i32(bt), dev_i32(cq), dev_i32(ck)
        slots = pa.slot_mapping_prefill(bt_d, cq_d, ck_d, B, total_q=int(cq[-1]))
        pa.store_kvcache(dev_bf16(nk), dev_bf16(nv), self.kc, self.vc, slots)
        mq, mk = int(np.diff(cq).max()), int(np.diff(ck).max())
        out = pa.prefill_varlen(dev_bf16(q), self.kc, self.vc, cq_d, ck_d, mq, mk, SCALE, block_tables=bt_d)
        assert pa.get_device_error() == (0, 0)
        # host mirror
        slots_h = np.concatenate(slots_h)
        assert slots.cpu().numpy().tolist() == slots_h.tolist()
        O.store_kvcache(nk, nv, self.kc_h, self.vc_h, slots_h)
        want = O.prefill(q, self.kc_h, self.vc_h, cq, ck, SCALE, block_tables=bt)
        assert_close(host_f64(out), want, "prefill")
        for sid in sids:
            self.bm.hash_blocks(sid, len(seqs[sid]) - cached[sid] * B)
            self.bm.set_num_cached_tokens(sid, len(seqs[sid]))
            self.tokens[sid] = list(seqs[sid])
        return cached

    def decode_step(self, sids, new_tokens):
        for sid, t in zip(sids, new_tokens):
            self.tokens[sid].append(t)
            self.bm.append_token(sid, t)
            assert self.bm.can_append(sid)
            self.bm.may_append(sid)
        ctx = np.asarray([len(self.tokens[s]) for s in sids], np.int32)
        bt = self.tables(sids)
        pos = ctx - 1
        q = rows(new_tokens, pos, 2, HQ)
        nk, nv = rows(new_tokens, pos, 0, HKV), rows(new_tokens, pos, 1, HKV)
        out = pa.decode(dev_bf16(q), self.kc, self.vc, dev_i32(bt), dev_i32(ctx), SCALE, workspace=self.ws,
                        new_k=dev_bf16(nk), new_v=dev_bf16(nv))
        assert pa.get_device_error() == (0, 0)
        slots_h = np.asarray([O.decode_slot(bt[i], B, int(ctx[i])) for i in range(len(sids))], np.int64)
        O.store_kvcache(nk, nv, self.kc_h, self.vc_h, slots_h)
        want = O.decode(q, self.kc_h, self.vc_h, bt, ctx, SCALE)
        assert_close(host_f64(out), want, "decode")
        for sid in sids:  # a block that just filled joins the prefix index
            n = len(self.tokens[sid])
            self.bm.set_num_cached_tokens(sid, n - 1)
            self.bm.hash_blocks(sid, 1)
            self.bm.set_num_cached_tokens(sid, n)

    def caches_match_mirror(self):
        return (np.array_equal(host_bits(self.kc), self.kc_h) and np.array_equal(host_bits(self.vc), self.vc_h))


def test_block_manager_tables_drive_store_prefill_and_decode():
    e = Engine()
    prompt = list(range(1000, 1040))                 # 40 shared tokens: two full blocks and 8 more
    a_toks = prompt + list(range(2000, 2010))        # 50
    c_toks = prompt + list(range(3000, 3020))        # 60
    sid_a = e.bm.add_sequence(a_toks)
    assert e.prefill({sid_a: a_toks}) == {sid_a: 0}
    shared = e.bm.block_table(sid_a)[:2]
    snapshot = (host_bits(e.kc)[shared].copy(), host_bits(e.vc)[shared].copy())

    # The second prompt hits the first two blocks (the third differs after token 40).
    sid_c = e.bm.add_sequence(c_toks)
    assert e.prefill({sid_c: c_toks}) == {sid_c: 2}
    assert e.bm.block_table(sid_c)[:2] == shared
    assert [e.bm.block(b)["ref_count"] for b in shared] == [2, 2]

    # Fused decode steps for both; A crosses the 64-token block boundary, C 64 and 80.
    for step in range(24):
        e.decode_step([sid_a, sid_c], [5000 + 2 * step, 6000 + 2 * step])
    assert len(e.bm.block_table(sid_a)) == math.ceil(74 / B)
    assert len(e.bm.block_table(sid_c)) == math.ceil(84 / B)
    assert e.caches_match_mirror()
    # The shared blocks were never rewritten.
    assert np.array_equal(host_bits(e.kc)[shared], snapshot[0])
    assert np.array_equal(host_bits(e.vc)[shared], snapshot[1])

    # A finishes; a third prompt with the same 40 tokens still hits the shared
    # blocks (held by C), and its prefill and decode read them.
    e.bm.deallocate(sid_a)
    assert [e.bm.block(b)["ref_count"] for b in shared] == [1, 1]
    d_toks = prompt + list(range(4000, 4005))
    sid_d = e.bm.add_sequence(d_toks)
    assert e.prefill({sid_d: d_toks}) == {sid_d: 2}
    for step in range(4):
        e.decode_step([sid_c, sid_d], [7000 + step, 8000 + step])
    assert e.caches_match_mirror()

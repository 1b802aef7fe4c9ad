"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes a loaded oracle library and raises
AssertionError if the oracle disagrees with:
  * values the pages print for worked examples (tests/golden/*.txt),
  * closed forms (one valid key => that value row; equal keys => mean of V;
    a two-key softmax written out by hand),
  * a library routine on cases that reduce to it (torch's
    scaled_dot_product_attention in float64 on dense, unpaged tensors),
  * invariants (block permutation, shared vs private prefix blocks, GQA
    replication, cached-prefix prefill vs full prefill, batch independence).
The pytest wrappers live in test_oracle_pins.py; test_oracle_mutants.py runs
the same pins against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle as O
from paged_kv_cache_store_gb300.workloads import (bf16_bits_to_f32, f32_to_bf16_bits, make_decode,
                                                  make_prefill, normal_bf16)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


def _ints(s):
    return [int(x) for x in s.split()]


def bf(x):
    """float array -> bf16 bits (values chosen to be exact in bf16)."""
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def widen(h):
    return bf16_bits_to_f32(h).astype(np.float64)


# ----------------------------------------------------------------------------
# Slot mapping and addressing: printed and hand-worked examples.
# ----------------------------------------------------------------------------

def pin_slot_mapping_examples(L):
    for B, bt, start, end, exp, _where in golden_rows("slot_mapping_examples.txt"):
        got = O.slot_mapping(_ints(bt), int(B), int(start), int(end), L=L)
        assert got.tolist() == _ints(exp), (bt, start, end, got)


def pin_two_level_mapping(L):
    bt = [7, 12, 3]
    rows = golden_rows("two_level_mapping.txt")
    for B, p, slot in rows:
        got = O.slot_mapping(bt, int(B), int(p), int(p) + 1, L=L)
        assert got.tolist() == [int(slot)], (B, p, got)
    # One call over the whole table agrees with the single positions.
    for B in (4, 256):
        allp = O.slot_mapping(bt, B, 0, 3 * B, L=L)
        for b2, p, slot in rows:
            if int(b2) == B:
                assert allp[int(p)] == int(slot)


def pin_decode_slot(L):
    for B, bt, ctx, slot in golden_rows("decode_slot_examples.txt"):
        got = O.decode_slot(_ints(bt), int(B), int(ctx), L=L)
        assert got == int(slot), (B, ctx, got)


# ----------------------------------------------------------------------------
# store_kvcache.
# ----------------------------------------------------------------------------

def pin_store_by_hand(L):
    # Pool of 3 blocks x 4 slots, 1 kv head of 2 values; sentinel 0xFFFF.
    kc = np.full((3, 4, 1, 2), 0xFFFF, dtype=np.uint16)
    vc = kc.copy()
    # Rows are 3 elements apart (a fused projection view); the third is not the token's.
    key = bf([[1, 2, 99], [3, 4, 99], [5, 6, 99]])
    val = bf([[10, 20, 99], [30, 40, 99], [50, 60, 99]])
    O.store_kvcache(key, val, kc, vc, np.array([5, -1, 2], np.int32), L=L)
    ek = np.full((12, 2), 0xFFFF, dtype=np.uint16)
    ev = ek.copy()
    ek[5] = bf([1, 2]); ev[5] = bf([10, 20])
    ek[2] = bf([5, 6]); ev[2] = bf([50, 60])
    assert np.array_equal(kc.reshape(12, 2), ek)
    assert np.array_equal(vc.reshape(12, 2), ev)


def pin_store_rejects_bad_slots(L):
    kc = np.zeros((2, 4, 1, 2), dtype=np.uint16)
    vc = kc.copy()
    key = bf([[1, 2], [3, 4]]).reshape(2, 1, 2)
    for sm, code in (([3, 3], O.EDUP), ([8, 0], O.EINVAL)):
        try:
            O.store_kvcache(key, key, kc, vc, np.array(sm, np.int32), L=L)
        except O.OracleError as e:
            assert f"rc={code}" in str(e)
        else:
            raise AssertionError(f"slot_mapping {sm} accepted")


def pin_store_random_rows(L):
    """Scatter of seeded rows, checked row by row against where they were sent."""
    rng = np.random.default_rng(7)
    nb, B, hkv, d = 5, 16, 2, 8
    kc = normal_bf16(11, 1, (nb, B, hkv, d))
    vc = normal_bf16(11, 2, (nb, B, hkv, d))
    k0, v0 = kc.copy(), vc.copy()
    n = 20
    slots = rng.permutation(nb * B)[:n].astype(np.int32)
    slots[[3, 11]] = -1
    key = normal_bf16(11, 3, (n, hkv, d))
    val = normal_bf16(11, 4, (n, hkv, d))
    O.store_kvcache(key, val, kc, vc, slots, L=L)
    fk, fv, fk0, fv0 = (a.reshape(nb * B, hkv, d) for a in (kc, vc, k0, v0))
    written = set()
    for i, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(fk[s], key[i]) and np.array_equal(fv[s], val[i])
            written.add(int(s))
    for s in range(nb * B):
        if s not in written:
            assert np.array_equal(fk[s], fk0[s]) and np.array_equal(fv[s], fv0[s])


# ----------------------------------------------------------------------------
# Decode attention.
# ----------------------------------------------------------------------------

def _contiguous_tables(ctx, B, first_block=1):
    """Each sequence owns a run of consecutive blocks, so its rows are one
    contiguous range of the pool: the test can slice them with no paging
    arithmetic.  Returns (block_tables, first_slot per sequence, blocks used)."""
    nbs = [max(1, -(-c // B)) for c in ctx]
    mb = max(nbs)
    bt = np.full((len(ctx), mb), -1, np.int32)
    first, nxt = [], first_block
    for b, n in enumerate(nbs):
        bt[b, :n] = np.arange(nxt, nxt + n)
        first.append(nxt * B)
        nxt += n
    return bt, first, nxt


def _sdpa(q, k, v, scale, causal=False, mask=None):
    """torch SDPA in float64; q [Hq, Lq, D], k/v [Hkv, Lk, D]; GQA by torch."""
    gq = q.shape[0] != k.shape[0]
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=None if mask is None else torch.from_numpy(mask)[None, None],
        is_causal=causal, scale=scale, enable_gqa=gq)
    return o[0].numpy()


def pin_decode_reads_paged_address(L):
    """With one spiked key, attention returns that key's value row; the value
    rows encode their own slot, so the output names the slot the oracle read
    for position p, which must be the slot the pages' mapping gives."""
    B, hkv, hq, d = 256, 2, 4, 6
    nb = 13
    bt = np.array([[7, 12, 3]], np.int32)
    kc = np.zeros((nb, B, hkv, d), np.uint16)
    vc = np.zeros((nb, B, hkv, d), np.float32)
    slot_ids = np.arange(nb * B)
    for digit in range(4):
        vc.reshape(nb * B, hkv, d)[:, :, digit] = ((slot_ids >> (4 * digit)) & 15)[:, None]
    vc[:, :, :, 4] = np.arange(hkv)[None, None, :]
    vc[:, :, :, 5] = 1.0
    vc = bf(vc)
    q = np.zeros((1, hq, d), np.float32)
    q[0, :, 0] = 1.0
    q = bf(q)
    for Bg, p, slot in golden_rows("two_level_mapping.txt"):
        if int(Bg) != B:
            continue
        p, slot = int(p), int(slot)
        for g in range(hkv):
            k = np.zeros((nb * B, hkv, d), np.float32)
            k[slot, g, 0] = 64.0
            k = bf(k).reshape(nb, B, hkv, d)
            out = O.decode(q, k, vc, bt, np.array([p + 1], np.int32), 1.0, L=L)
            h = 2 * g  # a q head of kv group g (2 q heads per kv head)
            read = sum(int(round(out[0, h, digit])) << (4 * digit) for digit in range(4))
            assert read == slot, (p, g, read, slot)
            assert abs(out[0, h, 4] - g) < 1e-9


def pin_decode_ctx1_is_v0(L):
    inp = make_decode("t", 21, 3, 4, 2, [1, 1, 1], head_dim=16, block_size=16)
    out = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, L=L)
    for b in range(3):
        blk = inp.block_tables[b, 0]
        for h in range(4):
            assert np.array_equal(out[b, h], widen(inp.v_cache[blk, 0, h // 2]))


def pin_decode_equal_keys_mean(L):
    B, hkv, hq, d = 8, 1, 2, 16
    ctx = [19, 5]
    bt, first, nbu = _contiguous_tables(ctx, B)
    kc = normal_bf16(31, 1, (nbu + 1, B, hkv, d))
    vc = normal_bf16(31, 2, (nbu + 1, B, hkv, d))
    flat = kc.reshape(-1, hkv, d)
    row = normal_bf16(31, 3, (hkv, d))
    for b, c in enumerate(ctx):
        flat[first[b]:first[b] + c] = row
    q = normal_bf16(31, 4, (2, hq, d))
    out = O.decode(q, kc, vc, bt, np.array(ctx, np.int32), 0.3, L=L)
    vflat = widen(vc.reshape(-1, hkv, d))
    for b, c in enumerate(ctx):
        mean = vflat[first[b]:first[b] + c, 0].mean(axis=0)
        for h in range(hq):
            assert np.allclose(out[b, h], mean, rtol=0, atol=1e-13)


def pin_decode_two_token_closed_form(L):
    # q = [1, 0], K0 = [0, 0], K1 = [3, 0], scale 0.5 -> scores 0 and 1.5.
    kc = np.zeros((1, 4, 1, 2), np.float32)
    kc[0, 1, 0] = [3.0, 0.0]
    vc = np.zeros((1, 4, 1, 2), np.float32)
    vc[0, 0, 0] = [1.0, 2.0]
    vc[0, 1, 0] = [-3.0, 0.5]
    out = O.decode(bf([[[1.0, 0.0]]]), bf(kc), bf(vc), np.array([[0]], np.int32),
                   np.array([2], np.int32), 0.5, L=L)
    e = math.exp(1.5)
    want = [(1.0 + e * -3.0) / (1.0 + e), (2.0 + e * 0.5) / (1.0 + e)]
    assert np.allclose(out[0, 0], want, rtol=1e-14, atol=0)


def pin_decode_matches_sdpa(L):
    B, hkv, hq, d = 16, 2, 6, 32
    ctx = [1, 15, 16, 17, 40, 0, 33]
    bt, first, nbu = _contiguous_tables(ctx, B)
    kc = normal_bf16(41, 1, (nbu + 2, B, hkv, d))
    vc = normal_bf16(41, 2, (nbu + 2, B, hkv, d))
    q = normal_bf16(41, 3, (len(ctx), hq, d))
    scale = 1 / math.sqrt(d)
    out = O.decode(q, kc, vc, bt, np.array(ctx, np.int32), scale, L=L)
    kf, vf = widen(kc.reshape(-1, hkv, d)), widen(vc.reshape(-1, hkv, d))
    for b, c in enumerate(ctx):
        if c == 0:
            assert np.all(out[b] == 0.0)
            continue
        kk = kf[first[b]:first[b] + c].transpose(1, 0, 2).copy()
        vv = vf[first[b]:first[b] + c].transpose(1, 0, 2).copy()
        ref = _sdpa(widen(q[b])[:, None, :], kk, vv, scale)[:, 0, :]
        assert np.allclose(out[b], ref, rtol=0, atol=1e-12), np.abs(out[b] - ref).max()


def _permute_blocks(kc, vc, bt, seed):
    perm = np.random.default_rng(seed).permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    return kc2, vc2, bt2


def pin_decode_block_permutation_invariance(L):
    inp = make_decode("t", 51, 5, 8, 2, [1, 30, 64, 65, 200], head_dim=16, block_size=32)
    a = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, L=L)
    kc2, vc2, bt2 = _permute_blocks(inp.k_cache, inp.v_cache, inp.block_tables, 5)
    b = O.decode(inp.q, kc2, vc2, bt2, inp.context_lens, inp.scale, L=L)
    assert np.array_equal(a, b)


def pin_decode_shared_prefix_equals_private(L):
    B = 16
    ctx = [70, 49, 100, 20]
    inp = make_decode("t", 61, 4, 4, 2, ctx, head_dim=16, block_size=B,
                      shared_prefix_seqs=3, shared_prefix_blocks=2)
    a = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, L=L)
    # Give every sharing sequence its own copy of the shared blocks.
    kc, vc, bt = inp.k_cache, inp.v_cache, inp.block_tables.copy()
    extra_k, extra_v = [], []
    nxt = kc.shape[0]
    for b in range(3):
        for j in range(2):
            src = bt[b, j]
            extra_k.append(kc[src]); extra_v.append(vc[src])
            bt[b, j] = nxt
            nxt += 1
    kc2 = np.concatenate([kc, np.stack(extra_k)])
    vc2 = np.concatenate([vc, np.stack(extra_v)])
    b2 = O.decode(inp.q, kc2, vc2, bt, inp.context_lens, inp.scale, L=L)
    assert np.array_equal(a, b2)


def pin_decode_gqa_replication(L):
    inp = make_decode("t", 71, 3, 8, 2, [5, 77, 128], head_dim=16, block_size=16)
    a = O.decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, L=L)
    g = 4
    kc = np.ascontiguousarray(np.repeat(inp.k_cache, g, axis=2))
    vc = np.ascontiguousarray(np.repeat(inp.v_cache, g, axis=2))
    b = O.decode(inp.q, kc, vc, inp.block_tables, inp.context_lens, inp.scale, L=L)
    assert np.array_equal(a, b)


def pin_decode_zero_context(L):
    inp = make_decode("t", 81, 3, 4, 2, [9, 1, 9], head_dim=16, block_size=16)
    bt = inp.block_tables.copy()
    bt[1, :] = -1
    ctx = inp.context_lens.copy()
    ctx[1] = 0
    out = O.decode(inp.q, inp.k_cache, inp.v_cache, bt, ctx, inp.scale, L=L)
    assert np.all(out[1] == 0.0) and np.any(out[0] != 0.0)


# ----------------------------------------------------------------------------
# Prefill attention.
# ----------------------------------------------------------------------------

def _golden_cu():
    (lens, cu), = golden_rows("cu_seqlens_example.txt")
    return _ints(lens), _ints(cu)


def pin_prefill_no_cache_sdpa(L):
    lens, cu = _golden_cu()
    hq, hkv, d = 4, 2, 16
    tot = cu[-1]
    q = normal_bf16(91, 1, (tot, hq, d))
    k = normal_bf16(91, 2, (tot, hkv, d))
    v = normal_bf16(91, 3, (tot, hkv, d))
    cu = np.array(cu, np.int32)
    out = O.prefill(q, k, v, cu, cu, 0.25, L=L)
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        ref = _sdpa(widen(q[a:e]).transpose(1, 0, 2).copy(), widen(k[a:e]).transpose(1, 0, 2).copy(),
                    widen(v[a:e]).transpose(1, 0, 2).copy(), 0.25, causal=True)
        assert np.allclose(out[a:e], ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def pin_prefill_non_causal_sdpa(L):
    lens, cu = _golden_cu()
    hq, hkv, d = 2, 2, 8
    tot = cu[-1]
    q = normal_bf16(92, 1, (tot, hq, d))
    k = normal_bf16(92, 2, (tot, hkv, d))
    v = normal_bf16(92, 3, (tot, hkv, d))
    cu = np.array(cu, np.int32)
    out = O.prefill(q, k, v, cu, cu, 0.3, causal=False, L=L)
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        ref = _sdpa(widen(q[a:e]).transpose(1, 0, 2).copy(), widen(k[a:e]).transpose(1, 0, 2).copy(),
                    widen(v[a:e]).transpose(1, 0, 2).copy(), 0.3)
        assert np.allclose(out[a:e], ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def pin_prefill_batch_independence(L):
    """cu_seqlens marks independent sequences: the packed batch equals each
    sequence run alone."""
    lens, cu = _golden_cu()
    hq, hkv, d = 4, 1, 8
    tot = cu[-1]
    q = normal_bf16(93, 1, (tot, hq, d))
    k = normal_bf16(93, 2, (tot, hkv, d))
    v = normal_bf16(93, 3, (tot, hkv, d))
    cu = np.array(cu, np.int32)
    out = O.prefill(q, k, v, cu, cu, 0.35, L=L)
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        one = np.array([0, e - a], np.int32)
        alone = O.prefill(q[a:e], k[a:e].copy(), v[a:e].copy(), one, one, 0.35, L=L)
        assert np.array_equal(out[a:e], alone)


def _prefill_case(seed, lk, cached_tokens, hq=4, hkv=2, d=16, B=16):
    return make_prefill("t", seed, lk, None, hq, hkv, head_dim=d, block_size=B,
                        cached_tokens=cached_tokens)


def pin_prefill_cached_prefix_matches_full(L):
    """Rows of a prefill that starts after c cached tokens equal the last
    rows of a prefill of the whole sequence over the same keys, which in turn
    is textbook causal attention (checked against torch SDPA)."""
    lk, c = [45, 33, 16], [32, 7, 0]
    p = _prefill_case(94, lk, c)
    # Full-sequence query rows: reuse the suffix q rows at the suffix positions;
    # the leading rows get their own draws.
    extra = normal_bf16(94, 9, (sum(c), p.num_q_heads, p.head_dim))
    full_q, pos = [], 0
    for s in range(3):
        full_q.append(extra[pos:pos + c[s]]); pos += c[s]
        full_q.append(p.q[p.cu_seqlens_q[s]:p.cu_seqlens_q[s + 1]])
    full_q = np.concatenate(full_q)
    cu_full = p.cu_seqlens_k
    part = O.prefill(p.q, p.k_cache, p.v_cache, p.cu_seqlens_q, p.cu_seqlens_k, p.scale,
                     block_tables=p.block_tables, L=L)
    full = O.prefill(full_q, p.k_cache, p.v_cache, cu_full, cu_full, p.scale,
                     block_tables=p.block_tables, L=L)
    for s in range(3):
        a, e = p.cu_seqlens_q[s], p.cu_seqlens_q[s + 1]
        fe = cu_full[s + 1]
        assert np.array_equal(part[a:e], full[fe - (e - a):fe])
    # The full prefill with contiguous tables is SDPA causal.
    bt, first, nbu = _contiguous_tables(lk, p.block_size)
    kc = normal_bf16(95, 1, (nbu, p.block_size, p.num_kv_heads, p.head_dim))
    vc = normal_bf16(95, 2, (nbu, p.block_size, p.num_kv_heads, p.head_dim))
    full2 = O.prefill(full_q, kc, vc, cu_full, cu_full, p.scale, block_tables=bt, L=L)
    kf = widen(kc.reshape(-1, p.num_kv_heads, p.head_dim))
    vf = widen(vc.reshape(-1, p.num_kv_heads, p.head_dim))
    for s in range(3):
        a, e = cu_full[s], cu_full[s + 1]
        kk = kf[first[s]:first[s] + lk[s]].transpose(1, 0, 2).copy()
        vv = vf[first[s]:first[s] + lk[s]].transpose(1, 0, 2).copy()
        ref = _sdpa(widen(full_q[a:e]).transpose(1, 0, 2).copy(), kk, vv, p.scale, causal=True)
        assert np.allclose(full2[a:e], ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def pin_prefill_paged_equals_contiguous(L):
    lk, c = [40, 17], [16, 5]
    p = _prefill_case(96, lk, c, B=8)
    paged = O.prefill(p.q, p.k_cache, p.v_cache, p.cu_seqlens_q, p.cu_seqlens_k, p.scale,
                      block_tables=p.block_tables, L=L)
    # Gather the same rows into contiguous [total_k, Hkv, D] by walking each
    # sequence's blocks in order (block-level copies, no per-token arithmetic).
    ks, vs = [], []
    for s in range(2):
        n = -(-lk[s] // p.block_size)
        blk = p.block_tables[s, :n]
        ks.append(p.k_cache[blk].reshape(-1, p.num_kv_heads, p.head_dim)[:lk[s]])
        vs.append(p.v_cache[blk].reshape(-1, p.num_kv_heads, p.head_dim)[:lk[s]])
    k = np.ascontiguousarray(np.concatenate(ks))
    v = np.ascontiguousarray(np.concatenate(vs))
    cont = O.prefill(p.q, k, v, p.cu_seqlens_q, p.cu_seqlens_k, p.scale, L=L)
    assert np.array_equal(paged, cont)


def pin_prefill_last_row_equals_decode(L):
    lk, c = [37, 64, 9], [16, 48, 0]
    p = _prefill_case(97, lk, c)
    pre = O.prefill(p.q, p.k_cache, p.v_cache, p.cu_seqlens_q, p.cu_seqlens_k, p.scale,
                    block_tables=p.block_tables, L=L)
    last = p.cu_seqlens_q[1:] - 1
    dec = O.decode(p.q[last], p.k_cache, p.v_cache, p.block_tables, np.array(lk, np.int32),
                   p.scale, L=L)
    assert np.array_equal(pre[last], dec)


def pin_prefill_first_query_is_v0(L):
    p = _prefill_case(98, [20, 9], [0, 0])
    out = O.prefill(p.q, p.k_cache, p.v_cache, p.cu_seqlens_q, p.cu_seqlens_k, p.scale,
                    block_tables=p.block_tables, L=L)
    for s in range(2):
        t = p.cu_seqlens_q[s]
        blk = p.block_tables[s, 0]
        for h in range(p.num_q_heads):
            assert np.array_equal(out[t, h], widen(p.v_cache[blk, 0, h // 2]))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

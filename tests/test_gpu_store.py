"""GPU parity: pa_store_kvcache and the slot-mapping builders against the
oracle, bit-exact.  Calls go through the C ABI (ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle as O
import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300.workloads import decode_config, make_decode, make_prefill, normal_bf16
from gpu_util import dev_bf16, dev_i32, host_bits
from oracle_pins import golden_rows, _ints

pytestmark = pytest.mark.gpu


def _sentinel_pool(nb, B, hkv, d):
    return np.full((nb, B, hkv, d), 0xFFFF, dtype=np.uint16)  # a NaN pattern


@pytest.mark.parametrize("hkv,n,nb,B", [(8, 64, 40, 256), (8, 1, 4, 256), (2, 333, 30, 16), (4, 2000, 70, 32)])
def test_store_bit_exact(hkv, n, nb, B):
    rng = np.random.default_rng(n)
    slots = rng.permutation(nb * B)[:n].astype(np.int32)
    slots[rng.random(n) < 0.15] = -1   # padding
    key = normal_bf16(n, 1, (n, hkv, 128))
    val = normal_bf16(n, 2, (n, hkv, 128))
    kc, vc = _sentinel_pool(nb, B, hkv, 128), _sentinel_pool(nb, B, hkv, 128)
    dk, dv = dev_bf16(kc), dev_bf16(vc)
    pa.store_kvcache(dev_bf16(key), dev_bf16(val), dk, dv, dev_i32(slots))
    O.store_kvcache(key, val, kc, vc, slots)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dk), kc)
    assert np.array_equal(host_bits(dv), vc)
    assert pa.get_device_error() == (0, 0)


def test_store_strided_fused_qkv_rows():
    """key/value are column slices of a fused [N, (Hq+2*Hkv)*D] projection."""
    n, hq, hkv, d, nb, B = 50, 16, 8, 128, 8, 256
    qkv = normal_bf16(5, 1, (n, (hq + 2 * hkv) * d))
    slots = np.random.default_rng(5).permutation(nb * B)[:n].astype(np.int32)
    t = dev_bf16(qkv)
    key = t[:, hq * d:(hq + hkv) * d].view(n, hkv, d)
    val = t[:, (hq + hkv) * d:].view(n, hkv, d)
    kc, vc = np.zeros((nb, B, hkv, d), np.uint16), np.zeros((nb, B, hkv, d), np.uint16)
    dk, dv = dev_bf16(kc), dev_bf16(vc)
    pa.store_kvcache(key, val, dk, dv, dev_i32(slots))
    O.store_kvcache(qkv[:, hq * d:(hq + hkv) * d], qkv[:, (hq + hkv) * d:], kc, vc, slots)
    assert np.array_equal(host_bits(dk), kc) and np.array_equal(host_bits(dv), vc)


def test_store_out_of_range_slot_is_recorded_not_written():
    n, hkv, nb, B = 4, 8, 2, 16
    key = normal_bf16(9, 1, (n, hkv, 128))
    slots = np.array([3, nb * B + 5, -1, 7], np.int32)
    kc = _sentinel_pool(nb, B, hkv, 128)
    dk, dv = dev_bf16(kc), dev_bf16(kc)
    pa.get_device_error()
    pa.store_kvcache(dev_bf16(key), dev_bf16(key), dk, dv, dev_i32(slots))
    code, where = pa.get_device_error()
    assert code == pa.PA_DEV_BAD_SLOT and where == 1
    good = slots.copy()
    good[1] = -1
    O.store_kvcache(key, key, kc, kc.copy(), good)
    assert np.array_equal(host_bits(dk), kc)


def test_slot_mapping_worked_examples_on_gpu():
    """The pages' prefill examples through the device builder (positions [start, end))."""
    for B, bt, start, end, exp, _ in golden_rows("slot_mapping_examples.txt"):
        bt, start, end = _ints(bt), int(start), int(end)
        cu_q = dev_i32([0, end - start])
        cu_k = dev_i32([0, end])
        got = pa.slot_mapping_prefill(dev_i32([bt]), cu_q, cu_k, int(B)).cpu().numpy()
        assert got.tolist() == _ints(exp)
    for B, bt, ctx, slot in golden_rows("decode_slot_examples.txt"):
        got = pa.slot_mapping_decode(dev_i32([_ints(bt)]), dev_i32([int(ctx)]), int(B)).cpu().numpy()
        assert got.tolist() == [int(slot)]


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_slot_mapping_decode_matches_oracle(cfg):
    inp = decode_config(cfg)
    got = pa.slot_mapping_decode(dev_i32(inp.block_tables), dev_i32(inp.context_lens), inp.block_size)
    want = [O.decode_slot(inp.block_tables[b], inp.block_size, int(inp.context_lens[b]))
            for b in range(inp.batch)]
    assert got.cpu().numpy().tolist() == want


def test_slot_mapping_prefill_chunked_matches_oracle():
    """Cached prefixes that end mid-block (chunked prefill) and at block edges."""
    lk = [6, 300, 513, 1024, 77, 256]
    c = [3, 255, 256, 1000, 0, 255]
    p = make_prefill("t", 3, lk, None, 4, 2, block_size=256, cached_tokens=c)
    got = pa.slot_mapping_prefill(dev_i32(p.block_tables), dev_i32(p.cu_seqlens_q), dev_i32(p.cu_seqlens_k),
                                  p.block_size).cpu().numpy()
    want = np.concatenate([O.slot_mapping(p.block_tables[s], p.block_size, c[s], lk[s]) for s in range(len(lk))])
    assert np.array_equal(got, want)
    # block_size 4 with the [1, 6] table of the pages, three sequences packed.
    bt = np.array([[1, 6], [2, 5], [0, 3]], np.int32)
    lk2, c2 = [6, 8, 5], [3, 4, 0]
    cu_q = np.cumsum([0] + [a - b for a, b in zip(lk2, c2)]).astype(np.int32)
    cu_k = np.cumsum([0] + lk2).astype(np.int32)
    got = pa.slot_mapping_prefill(dev_i32(bt), dev_i32(cu_q), dev_i32(cu_k), 4).cpu().numpy()
    want = np.concatenate([O.slot_mapping(bt[s], 4, c2[s], lk2[s]) for s in range(3)])
    assert np.array_equal(got, want)
    assert got[:3].tolist() == [7, 24, 25]

"""The calls are CUDA-graph capturable (no host reads of device data, grids
fixed by host arguments, counters reset in the kernels), as an engine that
replays a captured decode step needs [NV12 §12.7 CUDA graphs: static input
buffers, replay after copying the step's inputs in].  Captured steps replayed
with new inputs must give exactly what the same calls give eagerly."""
import numpy as np
import pytest
import torch

import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300.workloads import make_decode, make_prefill, normal_bf16
from gpu_util import dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_fused_decode_step_replays():
    """One captured fused decode step (store of the new token + attention),
    replayed for successive steps: the context grows by one each time and the
    new token's rows change; caches and outputs equal eager calls."""
    # Every sequence stays inside its allocated blocks for the 4 steps.
    base = make_decode("graph", 21, 6, 16, 8, [300, 1, 500, 200, 2000, 77], extra_table_cols=2)
    steps = 4

    class Rows:
        def __init__(self, i):
            self.q = normal_bf16(100 + i, 1, (6, 16, 128))
            self.new_k = normal_bf16(100 + i, 2, (6, 8, 128))
            self.new_v = normal_bf16(100 + i, 3, (6, 8, 128))
    news = [Rows(i) for i in range(steps)]
    kc_g, vc_g = dev_bf16(base.k_cache), dev_bf16(base.v_cache)
    kc_e, vc_e = dev_bf16(base.k_cache), dev_bf16(base.v_cache)
    bt = dev_i32(base.block_tables)
    ctx = dev_i32(base.context_lens)
    q, nk, nv = dev_bf16(news[0].q), dev_bf16(news[0].new_k), dev_bf16(news[0].new_v)
    out = torch.empty(6, 16, 128, dtype=torch.bfloat16, device="cuda")
    ws_g = pa.decode_workspace(16, 8, 128)
    ws_e = pa.decode_workspace(16, 8, 128)
    g = capture(lambda: pa.decode(q, kc_g, vc_g, bt, ctx, base.scale, workspace=ws_g, out=out, new_k=nk, new_v=nv))
    # The warm-up stored rows at the first step's positions: redo the eager side the same way.
    pa.decode(q, kc_e, vc_e, bt, ctx, base.scale, workspace=ws_e, new_k=nk, new_v=nv)
    lens = base.context_lens.copy()
    for i in range(steps):
        lens = lens + 1 if i else lens
        ctx.copy_(torch.from_numpy(lens.astype(np.int32)))
        q.copy_(dev_bf16(news[i].q))
        nk.copy_(dev_bf16(news[i].new_k))
        nv.copy_(dev_bf16(news[i].new_v))
        g.replay()
        want = pa.decode(q, kc_e, vc_e, bt, ctx, base.scale, workspace=ws_e, new_k=nk, new_v=nv)
        torch.cuda.synchronize()
        assert pa.get_device_error() == (0, 0)
        assert torch.equal(out, want), f"step {i}"
        assert torch.equal(kc_g, kc_e) and torch.equal(vc_g, vc_e), f"step {i}"


def test_shared_prefix_decode_step_replays():
    """The shared-prefix decode step (grouping + prefix kernel + decode kernel
    with the fused store), captured once and replayed for successive steps
    with new query and new-token rows and growing contexts: equal to eager
    calls."""
    ctx0 = [1100, 1030, 1500, 300, 2000, 1025]
    base = make_decode("graph-sp", 23, 6, 32, 8, ctx0, shared_prefix_seqs=3, shared_prefix_blocks=4,
                       extra_table_cols=1)
    steps = 3

    class Rows:
        def __init__(self, i):
            self.q = normal_bf16(200 + i, 1, (6, 32, 128))
            self.new_k = normal_bf16(200 + i, 2, (6, 8, 128))
            self.new_v = normal_bf16(200 + i, 3, (6, 8, 128))
    news = [Rows(i) for i in range(steps)]
    kc_g, vc_g = dev_bf16(base.k_cache), dev_bf16(base.v_cache)
    kc_e, vc_e = dev_bf16(base.k_cache), dev_bf16(base.v_cache)
    bt, ctx = dev_i32(base.block_tables), dev_i32(base.context_lens)
    q, nk, nv = dev_bf16(news[0].q), dev_bf16(news[0].new_k), dev_bf16(news[0].new_v)
    out = torch.empty(6, 32, 128, dtype=torch.bfloat16, device="cuda")
    ws_g = pa.decode_workspace(32, 8, 128, shared_prefix=True)
    ws_e = pa.decode_workspace(32, 8, 128, shared_prefix=True)
    g = capture(lambda: pa.decode(q, kc_g, vc_g, bt, ctx, base.scale, workspace=ws_g, out=out, new_k=nk, new_v=nv,
                                  shared_prefix=True))
    pa.decode(q, kc_e, vc_e, bt, ctx, base.scale, workspace=ws_e, new_k=nk, new_v=nv, shared_prefix=True)
    lens = base.context_lens.copy()
    for i in range(steps):
        lens = lens + 1 if i else lens
        ctx.copy_(torch.from_numpy(lens.astype(np.int32)))
        q.copy_(dev_bf16(news[i].q))
        nk.copy_(dev_bf16(news[i].new_k))
        nv.copy_(dev_bf16(news[i].new_v))
        g.replay()
        want = pa.decode(q, kc_e, vc_e, bt, ctx, base.scale, workspace=ws_e, new_k=nk, new_v=nv, shared_prefix=True)
        torch.cuda.synchronize()
        assert pa.get_device_error() == (0, 0)
        assert torch.equal(out, want), f"step {i}"
        assert torch.equal(kc_g, kc_e) and torch.equal(vc_g, vc_e), f"step {i}"


@pytest.mark.parametrize("fused", [False, True])
def test_prefill_step_replays(fused):
    """Slot mapping + store + prefill (three launches), or the fused store +
    prefill (one cooperative launch), captured once and replayed for a second
    batch of prompts with the same shapes."""
    pa_ = make_prefill("g1", 31, [300, 700, 129], None, 16, 8, cached_tokens=[0, 256, 17])
    pb_ = make_prefill("g2", 32, [300, 700, 129], None, 16, 8, cached_tokens=[0, 256, 17])
    kc, vc = dev_bf16(pa_.k_cache), dev_bf16(pa_.v_cache)
    bt, cq, ck = dev_i32(pa_.block_tables), dev_i32(pa_.cu_seqlens_q), dev_i32(pa_.cu_seqlens_k)
    q, nk, nv = dev_bf16(pa_.q), dev_bf16(pa_.new_k), dev_bf16(pa_.new_v)
    out = torch.empty_like(q)
    slots = torch.empty(pa_.total_q, dtype=torch.int32, device="cuda")
    mq, mk = int(pa_.seqlens_q.max()), int(pa_.seqlens_k.max())
    ws = pa.prefill_store_workspace()

    def step():
        if fused:
            pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, pa_.scale, block_tables=bt, out=out, new_k=nk, new_v=nv,
                              workspace=ws)
        else:
            pa.slot_mapping_prefill(bt, cq, ck, pa_.block_size, total_q=pa_.total_q, out=slots)
            pa.store_kvcache(nk, nv, kc, vc, slots)
            pa.prefill_varlen(q, kc, vc, cq, ck, mq, mk, pa_.scale, block_tables=bt, out=out)

    g = capture(step)
    # Second batch: same tables and lengths, new rows and queries.
    kc.copy_(dev_bf16(pb_.k_cache))
    vc.copy_(dev_bf16(pb_.v_cache))
    q.copy_(dev_bf16(pb_.q))
    nk.copy_(dev_bf16(pb_.new_k))
    nv.copy_(dev_bf16(pb_.new_v))
    g.replay()
    torch.cuda.synchronize()
    assert pa.get_device_error() == (0, 0)
    kc_e, vc_e = dev_bf16(pb_.k_cache), dev_bf16(pb_.v_cache)
    s_e = pa.slot_mapping_prefill(bt, cq, ck, pb_.block_size, total_q=pb_.total_q)
    pa.store_kvcache(dev_bf16(pb_.new_k), dev_bf16(pb_.new_v), kc_e, vc_e, s_e)
    want = pa.prefill_varlen(dev_bf16(pb_.q), kc_e, vc_e, cq, ck, mq, mk, pb_.scale, block_tables=bt)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    assert torch.equal(kc, kc_e) and torch.equal(vc, vc_e)

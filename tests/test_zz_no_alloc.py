"""pa_decode_static: decode attention for callers that cannot allocate device
memory (a framework's memory pool they must not bypass, a plugin barred from
the allocator, a host that forbids allocation after start-up).  Its split
scratch is an array built into the library instead of a caller workspace.

The entry point is called through the C ABI twice in a row per shape and
compared with pa_decode (caller workspace) at the attention tolerance; the
device's free memory and torch's allocator are unchanged across the calls;
and a call after the array's work counters were left non-zero (as a call
that stopped on a device error can leave them) is still correct, because
every call clears them first.  This file is collected last so a failure here
comes after every other test has run; it also passes when run alone in a
fresh process."""
import ctypes as C

import numpy as np
import pytest
import torch

import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300.workloads import decode_config, make_decode
from gpu_util import MAX_ABS, MEAN_ABS, dev_bf16, dev_i32, host_f64

pytestmark = pytest.mark.gpu


def _static_call(q, kc, vc, bt, ctx, scale, out):
    batch, hq, d = q.shape
    nb, B, hkv, _ = kc.shape
    return pa.lib().pa_decode_static(
        C.c_void_p(out.data_ptr()), C.c_void_p(q.data_ptr()), q.stride(0), C.c_void_p(kc.data_ptr()),
        C.c_void_p(vc.data_ptr()), C.c_void_p(bt.data_ptr()), bt.shape[1], C.c_void_p(ctx.data_ptr()),
        batch, hq, hkv, d, B, nb, float(scale),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("case", ["qwen3-0.6b", "gqa4-long", "single-chunk"])
def test_static_scratch_matches_workspace_entry_point(case):
    if case == "qwen3-0.6b":
        inp = decode_config(2)                      # G = 2
    elif case == "gqa4-long":
        inp = make_decode("static", 31, 3, 32, 8, [9000, 4097, 300])   # G = 4, pairs cut across CTAs
    else:
        inp = make_decode("static1", 32, 5, 16, 8, [1, 17, 200, 255, 256])
    q, kc, vc = dev_bf16(inp.q), dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx = dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    ref = pa.decode(q, kc, vc, bt, ctx, inp.scale)
    want = host_f64(ref)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        st = _static_call(q, kc, vc, bt, ctx, inp.scale, out)
        assert st == pa.PA_OK, pa.lib().pa_last_error_message()
        torch.cuda.synchronize()
        got = host_f64(out)
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        err = np.abs(got - want)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (call, err.max(), err.mean())
    assert pa.get_device_error() == (0, 0)


def test_static_scratch_holds_the_largest_shapes():
    """The scratch does not grow with batch or context: 256 sequences x 32 q
    heads with contexts up to ~7.6k tokens run through it."""
    inp = decode_config(3)
    q, kc, vc = dev_bf16(inp.q), dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx = dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    ref = pa.decode(q, kc, vc, bt, ctx, inp.scale)
    out = torch.full_like(ref, float("nan"))
    assert _static_call(q, kc, vc, bt, ctx, inp.scale, out) == pa.PA_OK
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert pa.get_device_error() == (0, 0)


def _scratch():
    ptr, nbytes = C.c_void_p(), C.c_size_t()
    assert pa.lib().pa_decode_static_scratch(C.byref(ptr), C.byref(nbytes)) == pa.PA_OK
    return ptr.value, nbytes.value


class _DevBytes:
    """A view of device bytes for torch.as_tensor (no copy, no allocation)."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (ptr, False),
                                        "strides": None, "version": 3}


def test_static_allocates_nothing():
    """Free device memory (cudaMemGetInfo) and torch's allocation counters do
    not move across two calls made after the outputs exist (one call before
    the measured window does the once-per-device set-up)."""
    inp = decode_config(2)
    q, kc, vc = dev_bf16(inp.q), dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx = dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    ref = pa.decode(q, kc, vc, bt, ctx, inp.scale)
    outs = [torch.empty_like(ref) for _ in range(2)]
    assert _static_call(q, kc, vc, bt, ctx, inp.scale, outs[0]) == pa.PA_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    n_alloc0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    for out in outs:
        assert _static_call(q, kc, vc, bt, ctx, inp.scale, out) == pa.PA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == n_alloc0
    for out in outs:
        assert torch.equal(out, ref)
    assert pa.get_device_error() == (0, 0)


def test_static_call_after_counters_left_dirty():
    """The array's leading work counters (tail counter, done counter, one
    arrival counter per range) are set non-zero, as a call that stopped on a
    device error can leave them; the next two calls still equal pa_decode
    (the counters would otherwise skip tail ranges and merge split pairs
    early, leaving wrong or unwritten rows)."""
    inp = make_decode("static-dirty", 33, 5, 32, 8, [7000, 3000, 257, 9000, 1200])   # many split pairs
    q, kc, vc = dev_bf16(inp.q), dev_bf16(inp.k_cache), dev_bf16(inp.v_cache)
    bt, ctx = dev_i32(inp.block_tables), dev_i32(inp.context_lens)
    ref = pa.decode(q, kc, vc, bt, ctx, inp.scale)
    ptr, nbytes = _scratch()
    assert ptr and nbytes == 8 << 20
    counters = torch.as_tensor(_DevBytes(ptr, 4096), device="cuda").view(torch.int32)
    for call in range(2):
        counters.fill_(3)   # every counter non-zero
        torch.cuda.synchronize()
        out = torch.full_like(ref, float("nan"))
        assert _static_call(q, kc, vc, bt, ctx, inp.scale, out) == pa.PA_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}"
        # A completed call leaves its counters at zero.
        assert int(counters[:64 + 512].abs().sum()) == 0
    assert pa.get_device_error() == (0, 0)

"""Paged-KV attention for GB300 (sm_103a): Python binding of libpa.so.

Thin ctypes marshalling over the C ABI declared in include/pa.h: every
function here checks tensor dtypes/devices, passes raw pointers, sizes and
the current CUDA stream to the library, and raises PagedAttentionError on a
non-OK status.  All computation happens in the library's CUDA kernels; there
is no CPU or PyTorch fallback, and importing the binding fails loudly when
libpa.so has not been built (see build.py).

Entry points (same names as the C ABI without the ``pa_`` prefix):
  store_kvcache, slot_mapping_decode, slot_mapping_prefill,
  decode_workspace_size, decode, decode_static, prefill_varlen,
  sample_gumbel, set_checked, get_device_error;
  block_manager.BlockManager wraps the host block manager (pa_bm_*).
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA, PA_ERR_DEVICE_CHECK = range(6)
(PA_DEV_TIMEOUT, PA_DEV_BAD_SLOT, PA_DEV_BAD_CONTEXT, PA_DEV_BAD_BLOCK, PA_DEV_BAD_SEQLENS, PA_DEV_SMEM_ALIGN,
 PA_DEV_BAD_TEMPERATURE) = range(1, 8)

# Every symbol include/pa.h declares, with its ctypes signature.
_i32, _i64, _sz, _f32, _vp = C.c_int32, C.c_int64, C.c_size_t, C.c_float, C.c_void_p
SIGNATURES = {
    "pa_version": (C.c_int, []),
    "pa_status_str": (C.c_char_p, [C.c_int]),
    "pa_last_error_message": (C.c_char_p, []),
    "pa_store_kvcache": (C.c_int, [_vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _vp]),
    "pa_slot_mapping_decode": (C.c_int, [_vp, _vp, _i32, _vp, _i32, _i32, _vp]),
    "pa_slot_mapping_prefill": (C.c_int, [_vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _vp]),
    "pa_decode_workspace_size": (_sz, [_i32, _i32, _i32]),
    "pa_decode": (C.c_int, [_vp, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                            _i32, _f32, _vp, _sz, _vp]),
    "pa_decode_static": (C.c_int, [_vp, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                   _i32, _f32, _vp]),
    "pa_decode_static_scratch": (C.c_int, [C.POINTER(_vp), C.POINTER(_sz)]),
    "pa_decode_shared_prefix_workspace_size": (_sz, [_i32, _i32, _i32]),
    "pa_decode_shared_prefix": (C.c_int, [_vp, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                                          _i32, _i32, _i32, _i32, _f32, _vp, _sz, _vp]),
    "pa_decode_store": (C.c_int, [_vp, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                                  _i32, _i32, _i32, _i32, _f32, _vp, _sz, _vp]),
    "pa_prefill_varlen": (C.c_int, [_vp, _vp, _i64, _i32, _vp, _vp, _i64, _i32, _vp, _i32, _vp, _vp, _i32,
                                    _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp]),
    "pa_prefill_store_workspace_size": (C.c_size_t, []),
    "pa_prefill_store_varlen": (C.c_int, [_vp, _vp, _i64, _i32, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _vp,
                                          _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _vp,
                                          C.c_size_t, _vp]),
    "pa_sample_gumbel": (C.c_int, [_vp, _vp, _i64, _i32, _vp, _vp, _i64, _i32, _i32, _vp]),
    "pa_set_checked": (C.c_int, [_i32]),
    # host block manager
    "pa_bm_create": (C.c_int, [_i32, _i32, C.POINTER(_vp)]),
    "pa_bm_destroy": (None, [_vp]),
    "pa_bm_seq_add": (C.c_int, [_vp, _vp, _i32, C.POINTER(_i32)]),
    "pa_bm_seq_append_token": (C.c_int, [_vp, _i32, _i64]),
    "pa_bm_seq_set_num_cached_tokens": (C.c_int, [_vp, _i32, _i32]),
    "pa_bm_seq_info": (C.c_int, [_vp, _i32, C.POINTER(_i32), C.POINTER(_i32), C.POINTER(_i32)]),
    "pa_bm_can_allocate": (_i32, [_vp, _i32]),
    "pa_bm_allocate": (C.c_int, [_vp, _i32, _i32]),
    "pa_bm_deallocate": (C.c_int, [_vp, _i32]),
    "pa_bm_can_append": (_i32, [_vp, _i32]),
    "pa_bm_may_append": (C.c_int, [_vp, _i32]),
    "pa_bm_hash_blocks": (C.c_int, [_vp, _i32, _i32]),
    "pa_bm_seq_block_table": (_i32, [_vp, _i32, _vp, _i32]),
    "pa_bm_block_tables": (C.c_int, [_vp, _vp, _i32, _vp, _i32]),
    "pa_bm_free_block_ids": (_i32, [_vp, _vp, _i32]),
    "pa_bm_block_info": (C.c_int, [_vp, _i32, C.POINTER(_i32), C.POINTER(_i32), C.POINTER(C.c_uint64),
                                   C.POINTER(_i32)]),
    "pa_bm_lookup_hash": (_i32, [_vp, C.c_uint64]),
    "pa_bm_num_hashes": (_i32, [_vp]),
    "pa_bm_block_hash": (C.c_uint64, [_vp, _i32, _i32, C.c_uint64]),
    "pa_bm_xxh64": (C.c_uint64, [_vp, _sz, C.c_uint64]),
    "pa_get_device_error": (C.c_int, [_vp, C.POINTER(_i32), C.POINTER(_i64)]),
}

_LIB = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [status {status}]")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Load libpa.so and declare its signatures (no GPU needed)."""
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with paged_kv_cache_store_gb300.build.build()")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def lib():
    global _LIB
    if _LIB is None:
        _LIB = load_library()
    return _LIB


def _check(status: int, what: str):
    if status != PA_OK:
        L = lib()
        msg = (L.pa_last_error_message() or b"").decode(errors="replace")
        name = (L.pa_status_str(status) or b"").decode()
        raise PagedAttentionError(status, f"{what}: {name}: {msg}")


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _row_stride(t, name):
    """Elements between rows of a [N, ...] tensor whose trailing dims are contiguous."""
    inner = 1
    for d in t.shape[1:]:
        inner *= d
    if t.shape[0] == 0:
        return inner
    if t.dim() > 1 and not t[0].is_contiguous():
        raise ValueError(f"{name}: each row must be contiguous")
    return t.stride(0) if t.shape[0] > 1 else inner


def store_kvcache(key, value, k_cache, v_cache, slot_mapping, stream=None):
    """Scatter key/value [N, Hkv, D] (bf16, rows may be strided) into the pool
    [num_blocks, B, Hkv, D] at slot_mapping (int32 [N], negatives skipped)."""
    for t, n in ((key, "key"), (value, "value"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(slot_mapping, torch.int32, "slot_mapping")
    nb, B, hkv, d = k_cache.shape
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    n = key.shape[0]
    if slot_mapping.numel() != n or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous with one entry per token")
    _check(lib().pa_store_kvcache(_ptr(key), _row_stride(key, "key"), _ptr(value),
                                  _row_stride(value, "value"), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(slot_mapping), n, hkv, d, nb * B, _stream(stream)),
           "pa_store_kvcache")


def slot_mapping_decode(block_tables, context_lens, block_size, out=None, stream=None):
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    batch = context_lens.numel()
    if out is None:
        out = torch.empty(batch, dtype=torch.int32, device=context_lens.device)
    _check(lib().pa_slot_mapping_decode(_ptr(out), _ptr(block_tables.contiguous()), block_tables.shape[1],
                                        _ptr(context_lens), batch, block_size, _stream(stream)),
           "pa_slot_mapping_decode")
    return out


def slot_mapping_prefill(block_tables, cu_seqlens_q, cu_seqlens_k, block_size, total_q=None,
                         out=None, stream=None):
    _need(block_tables, torch.int32, "block_tables")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    num_seqs = cu_seqlens_q.numel() - 1
    if total_q is None:
        total_q = int(cu_seqlens_q[-1].item())
    if out is None:
        out = torch.empty(total_q, dtype=torch.int32, device=cu_seqlens_q.device)
    _check(lib().pa_slot_mapping_prefill(_ptr(out), _ptr(block_tables.contiguous()), block_tables.shape[1],
                                         _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), num_seqs, total_q,
                                         block_size, _stream(stream)),
           "pa_slot_mapping_prefill")
    return out


def decode_workspace_size(num_q_heads, num_kv_heads, head_dim) -> int:
    return int(lib().pa_decode_workspace_size(num_q_heads, num_kv_heads, head_dim))


def decode_workspace(num_q_heads, num_kv_heads, head_dim, device="cuda", shared_prefix=False):
    """Allocate (with torch) a zero-filled workspace for pa_decode (at most
    about 6.4 MB; it depends only on the GQA group), or, with shared_prefix,
    for pa_decode_shared_prefix (about 8.6 MB more).  The calls leave it
    zeroed, so it can be reused by any number of calls on one stream."""
    n = (int(lib().pa_decode_shared_prefix_workspace_size(num_q_heads, num_kv_heads, head_dim)) if shared_prefix
         else decode_workspace_size(num_q_heads, num_kv_heads, head_dim))
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


def decode(q, k_cache, v_cache, block_tables, context_lens, softmax_scale=None, workspace=None, out=None,
           stream=None, new_k=None, new_v=None, shared_prefix=False):
    """Paged decode attention.  q [batch, Hq, D] bf16 (rows may be strided);
    caches [num_blocks, B, Hkv, D]; block_tables int32 [batch, max_blocks];
    context_lens int32 [batch].  Returns out [batch, Hq, D] bf16.  With
    new_k / new_v ([batch, Hkv, D] bf16, rows may be strided) the kernel first
    stores them at position context_lens-1 (pa_decode_store).  With
    shared_prefix, sequences that share leading blocks read them once
    (pa_decode_shared_prefix; its workspace is larger)."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    batch, hq, d = q.shape
    nb, B, hkv, _ = k_cache.shape
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and block_tables.is_contiguous()):
        raise ValueError("caches and block_tables must be contiguous")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    mb = block_tables.shape[1]
    if workspace is None:
        workspace = decode_workspace(hq, hkv, d, q.device, shared_prefix=shared_prefix)
    if out is None:
        out = torch.empty(batch, hq, d, dtype=torch.bfloat16, device=q.device)
    if shared_prefix:
        if new_k is not None or new_v is not None:
            _need(new_k, torch.bfloat16, "new_k")
            _need(new_v, torch.bfloat16, "new_v")
        nk_args = ((_ptr(new_k), _row_stride(new_k, "new_k"), _ptr(new_v), _row_stride(new_v, "new_v"))
                   if new_k is not None else (None, 0, None, 0))
        _check(lib().pa_decode_shared_prefix(_ptr(out), _ptr(q), _row_stride(q, "q"), *nk_args, _ptr(k_cache),
                                             _ptr(v_cache), _ptr(block_tables), mb, _ptr(context_lens), batch, hq, hkv,
                                             d, B, nb, float(softmax_scale), _ptr(workspace), workspace.numel(),
                                             _stream(stream)),
               "pa_decode_shared_prefix")
        return out
    if new_k is not None or new_v is not None:
        _need(new_k, torch.bfloat16, "new_k")
        _need(new_v, torch.bfloat16, "new_v")
        _check(lib().pa_decode_store(_ptr(out), _ptr(q), _row_stride(q, "q"), _ptr(new_k), _row_stride(new_k, "new_k"),
                                     _ptr(new_v), _row_stride(new_v, "new_v"), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_tables), mb, _ptr(context_lens), batch, hq, hkv, d, B, nb,
                                     float(softmax_scale), _ptr(workspace), workspace.numel(), _stream(stream)),
               "pa_decode_store")
        return out
    _check(lib().pa_decode(_ptr(out), _ptr(q), _row_stride(q, "q"), _ptr(k_cache), _ptr(v_cache),
                           _ptr(block_tables), mb, _ptr(context_lens), batch, hq, hkv, d, B, nb,
                           float(softmax_scale), _ptr(workspace), workspace.numel(), _stream(stream)),
           "pa_decode")
    return out


def decode_static(q, k_cache, v_cache, block_tables, context_lens, softmax_scale=None, out=None, stream=None):
    """pa_decode without a workspace: for callers that must not allocate device
    memory.  The split scratch is an 8 MiB array built into the library (shared
    by all calls, so calls that may overlap on the GPU must be serialised).
    Only `out` is allocated here, and only when the caller passes none."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    batch, hq, d = q.shape
    nb, B, hkv, _ = k_cache.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(batch, hq, d, dtype=torch.bfloat16, device=q.device)
    _check(lib().pa_decode_static(_ptr(out), _ptr(q), _row_stride(q, "q"), _ptr(k_cache), _ptr(v_cache),
                                  _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), batch, hq, hkv,
                                  d, B, nb, float(softmax_scale), _stream(stream)),
           "pa_decode_static")
    return out


def prefill_store_workspace(device="cuda"):
    """Zero-filled workspace for prefill_varlen(..., new_k=, new_v=) (a grid
    barrier's counter; the call leaves it as found, reusable on one stream)."""
    n = int(lib().pa_prefill_store_workspace_size())
    return torch.zeros(n, dtype=torch.uint8, device=device)


def prefill_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, softmax_scale=None,
                   block_tables=None, causal=True, out=None, stream=None, new_k=None, new_v=None, workspace=None):
    """Varlen prefill attention.  q [total_q, Hq, D]; with block_tables, k/v are
    the caches [num_blocks, B, Hkv, D]; without, contiguous [total_k, Hkv, D].
    With new_k / new_v ([total_q, Hkv, D], the uncached suffix in q's order;
    block_tables required) the same launch first stores them into the caches
    (pa_prefill_store_varlen)."""
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    tq, hq, d = q.shape
    if block_tables is not None:
        _need(block_tables, torch.int32, "block_tables")
        nb, B, hkv, _ = k.shape
        mb, kv_stride, tk = block_tables.shape[1], 0, 0
    else:
        tk, hkv, _ = k.shape
        nb, B, mb, kv_stride = 0, 16, 0, _row_stride(k, "k")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(tq, hq, d, dtype=torch.bfloat16, device=q.device)
    if new_k is not None or new_v is not None:
        if new_k is None or new_v is None or block_tables is None:
            raise ValueError("the fused store needs new_k, new_v and block_tables")
        _need(new_k, torch.bfloat16, "new_k")
        _need(new_v, torch.bfloat16, "new_v")
        if new_k.shape[0] != tq or new_v.shape[0] != tq:
            raise ValueError("new_k / new_v need one row per query token")
        if workspace is None:
            workspace = prefill_store_workspace(q.device)
        _check(lib().pa_prefill_store_varlen(
            _ptr(out), _ptr(q), _row_stride(q, "q"), tq, _ptr(new_k), _row_stride(new_k, "new_k"), _ptr(new_v),
            _row_stride(new_v, "new_v"), _ptr(k), _ptr(v), _ptr(block_tables), mb, _ptr(cu_seqlens_q),
            _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, int(max_seqlen_q), int(max_seqlen_k), hq, hkv, d, B, nb,
            float(softmax_scale), 1 if causal else 0, _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream)), "pa_prefill_store_varlen")
        return out
    _check(lib().pa_prefill_varlen(_ptr(out), _ptr(q), _row_stride(q, "q"), tq, _ptr(k), _ptr(v), kv_stride, tk,
                                   _ptr(block_tables), mb, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                   cu_seqlens_q.numel() - 1, int(max_seqlen_q), int(max_seqlen_k), hq, hkv,
                                   d, B, nb, float(softmax_scale), 1 if causal else 0, _stream(stream)),
           "pa_prefill_varlen")
    return out


def sample_gumbel(logits, temperatures, exp_noise, out=None, stream=None):
    """One token per row: argmax softmax(logits / T) / max(E, 1e-10) (Gumbel-max).
    logits [batch, vocab] bf16 or fp32 (rows may be strided); temperatures
    fp32 [batch]; exp_noise fp32 [batch, vocab] of Exp(1) draws (the caller's
    random state).  Returns int32 [batch]."""
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("logits must be bfloat16 or float32")
    _need(temperatures, torch.float32, "temperatures")
    _need(exp_noise, torch.float32, "exp_noise")
    batch, vocab = logits.shape
    if tuple(exp_noise.shape) != (batch, vocab) or tuple(temperatures.shape) != (batch,):
        raise ValueError("exp_noise must be [batch, vocab] and temperatures [batch]")
    if logits.stride(1) != 1 or exp_noise.stride(1) != 1 or not temperatures.is_contiguous():
        raise ValueError("rows must be contiguous")
    if out is None:
        out = torch.empty(batch, dtype=torch.int32, device=logits.device)
    _check(lib().pa_sample_gumbel(_ptr(out), _ptr(logits), logits.stride(0), 1 if logits.dtype == torch.float32 else 0,
                                  _ptr(temperatures), _ptr(exp_noise), exp_noise.stride(0), batch, vocab,
                                  _stream(stream)),
           "pa_sample_gumbel")
    return out


def set_checked(enabled: bool):
    _check(lib().pa_set_checked(1 if enabled else 0), "pa_set_checked")


def get_device_error(stream=None):
    """Synchronise the stream; return (code, where) of the first device-side
    error since the last call ((0, 0) if none) and clear it."""
    code, where = _i32(0), _i64(0)
    st = lib().pa_get_device_error(_stream(stream), C.byref(code), C.byref(where))
    if st not in (PA_OK, PA_ERR_DEVICE_CHECK):
        _check(st, "pa_get_device_error")
    return int(code.value), int(where.value)

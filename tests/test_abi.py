"""The C ABI library loads and exports every symbol include/pa.h declares;
host-side argument checks reject bad calls before anything reaches a GPU.
CPU only: no call here launches a kernel."""
import ctypes as C
import os
import re

import pytest

import paged_kv_cache_store_gb300 as pa
from paged_kv_cache_store_gb300 import build as pabuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")


@pytest.fixture(scope="module")
def L():
    pabuild.build()
    return pa.load_library()


def declared_symbols():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", text)))


def test_header_symbols_are_exported(L):
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), f"{n} declared in pa.h but not exported"
    assert set(names) == set(pa.SIGNATURES), "binding signatures and header disagree"


def test_only_api_symbols_exported():
    out = os.popen(f"nm -D --defined-only {pa.LIB_PATH}").read()
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_symbols())


def test_status_strings(L):
    assert L.pa_status_str(0) == b"PA_OK"
    assert L.pa_status_str(3) == b"PA_ERR_WORKSPACE"
    assert L.pa_status_str(99) == b"PA_ERR_UNKNOWN"
    assert L.pa_version() >= 10000


def test_workspace_size_host_math(L):
    # Two partial slots of G heads per range (a head and a tail range per CTA of
    # the largest grid, 256 CTAs), plus counters: independent of batch and context length.
    ranges = 2 * 256
    for hq, hkv in [(16, 8), (32, 8), (8, 8), (64, 8)]:
        g = hq // hkv
        n = L.pa_decode_workspace_size(hq, hkv, 128)
        assert 2 * ranges * g * (128 * 4 + 8) <= n <= 2 * ranges * g * (128 * 4 + 8) + ranges * 4 + 2048
    assert L.pa_decode_workspace_size(64, 8, 128) <= 8 << 20       # fits the static scratch
    # Unsupported shapes give 0.
    assert L.pa_decode_workspace_size(16, 8, 64) == 0
    assert L.pa_decode_workspace_size(24, 8, 128) == 0
    assert L.pa_decode_workspace_size(12, 8, 128) == 0


def _msg(L):
    return L.pa_last_error_message().decode()


def test_store_argument_checks(L):
    p = C.c_void_p(16)
    assert L.pa_store_kvcache(None, 1024, p, 1024, p, p, p, 4, 8, 128, 1024, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_store_kvcache(p, 1024, p, 1024, p, p, p, 4, 8, 64, 1024, None) == pa.PA_ERR_UNSUPPORTED
    assert L.pa_store_kvcache(p, 1020, p, 1024, p, p, p, 4, 8, 128, 1 << 20, None) == pa.PA_ERR_INVALID_ARG
    assert "stride" in _msg(L)
    assert L.pa_store_kvcache(p, 1028, p, 1028, p, p, p, 4, 8, 128, 1 << 20, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_store_kvcache(C.c_void_p(18), 1024, p, 1024, p, p, p, 4, 8, 128, 1 << 20, None) == \
        pa.PA_ERR_INVALID_ARG
    assert "aligned" in _msg(L)
    assert L.pa_store_kvcache(p, 1024, p, 1024, p, p, p, 0, 8, 128, 1024, None) == pa.PA_OK  # no-op


def _decode(L, **kw):
    p = C.c_void_p(256)
    a = dict(out=p, q=p, q_row_stride=2048, k=p, v=p, bt=p, mb=16, ctx=p, batch=4, hq=16, hkv=8, d=128,
             B=256, nb=64, scale=0.088, ws=p, wsb=1 << 30, stream=None)
    a.update(kw)
    return L.pa_decode(a["out"], a["q"], a["q_row_stride"], a["k"], a["v"], a["bt"], a["mb"], a["ctx"],
                       a["batch"], a["hq"], a["hkv"], a["d"], a["B"], a["nb"], a["scale"],
                       a["ws"], a["wsb"], a["stream"])


def test_decode_argument_checks(L):
    assert _decode(L, batch=0) == pa.PA_OK
    assert _decode(L, q=None) == pa.PA_ERR_INVALID_ARG
    assert _decode(L, hq=12, hkv=8) == pa.PA_ERR_INVALID_ARG
    assert _decode(L, hq=24, hkv=8) == pa.PA_ERR_UNSUPPORTED     # group of 3
    assert _decode(L, d=64) == pa.PA_ERR_UNSUPPORTED
    assert _decode(L, B=24) == pa.PA_ERR_UNSUPPORTED
    assert _decode(L, q_row_stride=2047) == pa.PA_ERR_INVALID_ARG
    assert _decode(L, q_row_stride=1024) == pa.PA_ERR_INVALID_ARG
    assert _decode(L, scale=0.0) == pa.PA_ERR_INVALID_ARG
    assert _decode(L, batch=5000) == pa.PA_ERR_UNSUPPORTED
    assert _decode(L, ws=None, wsb=0) == pa.PA_ERR_WORKSPACE
    assert _decode(L, wsb=100) == pa.PA_ERR_WORKSPACE
    assert "workspace" in _msg(L)
    assert _decode(L, k=C.c_void_p(258)) == pa.PA_ERR_INVALID_ARG
    assert _decode(L, ws=C.c_void_p(264)) == pa.PA_ERR_INVALID_ARG      # unaligned workspace
    assert _decode(L, nb=1 << 24) == pa.PA_ERR_UNSUPPORTED       # slots overflow int32
    assert _decode(L, batch=2048, mb=1 << 20, nb=1024, B=1024) == pa.PA_ERR_UNSUPPORTED  # tile prefix overflows


def test_slot_mapping_argument_checks(L):
    p = C.c_void_p(256)
    assert L.pa_slot_mapping_decode(p, p, 4, p, 0, 256, None) == pa.PA_OK
    assert L.pa_slot_mapping_decode(None, p, 4, p, 3, 256, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_slot_mapping_decode(p, p, 4, p, 3, 0, None) == pa.PA_ERR_INVALID_ARG
    assert L.pa_slot_mapping_prefill(p, p, 4, p, p, 2, 0, 256, None) == pa.PA_OK
    assert L.pa_slot_mapping_prefill(p, p, 4, p, p, -1, 3, 256, None) == pa.PA_ERR_INVALID_ARG


def _prefill(L, **kw):
    p = C.c_void_p(256)
    a = dict(out=p, q=p, qs=32 * 128, tq=100, k=p, v=p, kvs=0, tk=0, bt=p, mb=8, cq=p, ck=p, ns=2, mq=64, mk=900,
             hq=32, hkv=8, d=128, B=256, nb=64, scale=0.088, causal=1, stream=None)
    a.update(kw)
    return L.pa_prefill_varlen(a["out"], a["q"], a["qs"], a["tq"], a["k"], a["v"], a["kvs"], a["tk"], a["bt"],
                               a["mb"], a["cq"], a["ck"], a["ns"], a["mq"], a["mk"], a["hq"], a["hkv"], a["d"],
                               a["B"], a["nb"], a["scale"], a["causal"], a["stream"])


def test_prefill_argument_checks(L):
    assert _prefill(L, ns=0) == pa.PA_OK                      # nothing to do
    assert _prefill(L, tq=0) == pa.PA_OK
    assert _prefill(L, ns=-1) == pa.PA_ERR_INVALID_ARG
    assert _prefill(L, q=None) == pa.PA_ERR_INVALID_ARG
    assert _prefill(L, hq=12) == pa.PA_ERR_INVALID_ARG        # not a multiple of Hkv
    assert _prefill(L, d=64) == pa.PA_ERR_UNSUPPORTED
    assert _prefill(L, qs=32 * 128 - 8) == pa.PA_ERR_INVALID_ARG
    assert _prefill(L, out=C.c_void_p(264)) == pa.PA_ERR_INVALID_ARG   # unaligned output
    assert _prefill(L, scale=-1.0) == pa.PA_ERR_INVALID_ARG
    assert _prefill(L, B=24) == pa.PA_ERR_UNSUPPORTED                # block size not a multiple of 16
    assert _prefill(L, nb=0) == pa.PA_ERR_INVALID_ARG
    assert _prefill(L, bt=None, tk=0) == pa.PA_ERR_INVALID_ARG        # contiguous k/v without total_k
    assert _prefill(L, bt=None, tk=100, kvs=8 * 128 - 8) == pa.PA_ERR_INVALID_ARG
    assert _prefill(L, ns=1 << 20, mq=1 << 20) == pa.PA_ERR_UNSUPPORTED  # tiles overflow int32


def _sample(L, **kw):
    p = C.c_void_p(256)
    a = dict(out=p, lg=p, ls=1024, fp32=0, t=p, e=p, es=1024, b=4, v=1000, stream=None)
    a.update(kw)
    return L.pa_sample_gumbel(a["out"], a["lg"], a["ls"], a["fp32"], a["t"], a["e"], a["es"], a["b"], a["v"],
                              a["stream"])


def test_sample_argument_checks(L):
    assert _sample(L, b=0) == pa.PA_OK
    assert _sample(L, b=-1) == pa.PA_ERR_INVALID_ARG
    assert _sample(L, v=0) == pa.PA_ERR_INVALID_ARG
    assert _sample(L, out=None) == pa.PA_ERR_INVALID_ARG
    assert _sample(L, fp32=2) == pa.PA_ERR_INVALID_ARG
    assert _sample(L, ls=999) == pa.PA_ERR_INVALID_ARG       # stride below vocab
    assert _sample(L, ls=1004) == pa.PA_ERR_INVALID_ARG      # bf16 rows must stay 16-byte aligned
    assert _sample(L, es=1002) == pa.PA_ERR_INVALID_ARG
    assert _sample(L, lg=C.c_void_p(258)) == pa.PA_ERR_INVALID_ARG
    assert _sample(L, b=70000) == pa.PA_ERR_UNSUPPORTED


def test_decode_store_argument_checks(L):
    p = C.c_void_p(256)

    def call(**kw):
        a = dict(out=p, q=p, qs=2048, nk=p, nks=1024, nv=p, nvs=1024, k=p, v=p, bt=p, mb=16, ctx=p, batch=4,
                 hq=16, hkv=8, d=128, B=256, nb=64, scale=0.088, ws=p, wsb=1 << 30, stream=None)
        a.update(kw)
        return L.pa_decode_store(a["out"], a["q"], a["qs"], a["nk"], a["nks"], a["nv"], a["nvs"], a["k"], a["v"],
                                 a["bt"], a["mb"], a["ctx"], a["batch"], a["hq"], a["hkv"], a["d"], a["B"], a["nb"],
                                 a["scale"], a["ws"], a["wsb"], a["stream"])

    assert call(batch=0) == pa.PA_OK
    assert call(nk=None) == pa.PA_ERR_INVALID_ARG
    assert call(nv=C.c_void_p(264)) == pa.PA_ERR_INVALID_ARG      # unaligned
    assert call(nks=1000) == pa.PA_ERR_INVALID_ARG                # stride below Hkv*D
    assert call(nvs=1028) == pa.PA_ERR_INVALID_ARG                # not a multiple of 8
    assert call(hq=24) == pa.PA_ERR_UNSUPPORTED                   # decode's own checks still apply
    assert call(ws=None, wsb=0) == pa.PA_ERR_WORKSPACE


def _prefill_store(L, **kw):
    p = C.c_void_p(256)
    a = dict(out=p, q=p, qs=32 * 128, tq=100, nk=p, nks=8 * 128, nv=p, nvs=8 * 128, kc=p, vc=p, bt=p, mb=8,
             cq=p, ck=p, ns=2, mq=64, mk=512, hq=32, hkv=8, d=128, B=256, nb=16, scale=0.088, causal=1,
             ws=p, wsb=256, stream=None)
    a.update(kw)
    return L.pa_prefill_store_varlen(a["out"], a["q"], a["qs"], a["tq"], a["nk"], a["nks"], a["nv"], a["nvs"],
                                     a["kc"], a["vc"], a["bt"], a["mb"], a["cq"], a["ck"], a["ns"], a["mq"],
                                     a["mk"], a["hq"], a["hkv"], a["d"], a["B"], a["nb"], a["scale"],
                                     a["causal"], a["ws"], a["wsb"], a["stream"])


def test_prefill_store_argument_checks(L):
    """Every case fails (or has nothing to do) before any launch."""
    assert L.pa_prefill_store_workspace_size() >= 8
    assert _prefill_store(L, ns=0) == pa.PA_OK
    assert _prefill_store(L, tq=0) == pa.PA_OK
    assert _prefill_store(L, bt=None) == pa.PA_ERR_INVALID_ARG     # the fused store needs a paged pool
    assert _prefill_store(L, nk=None) == pa.PA_ERR_INVALID_ARG
    assert _prefill_store(L, nvs=8 * 128 - 8) == pa.PA_ERR_INVALID_ARG  # shorter than a row
    assert _prefill_store(L, nks=8 * 128 + 4) == pa.PA_ERR_INVALID_ARG  # not a multiple of 8
    assert _prefill_store(L, nv=C.c_void_p(264)) == pa.PA_ERR_INVALID_ARG  # unaligned
    assert _prefill_store(L, ws=None) == pa.PA_ERR_WORKSPACE
    assert _prefill_store(L, wsb=4) == pa.PA_ERR_WORKSPACE
    assert _prefill_store(L, ws=C.c_void_p(260)) == pa.PA_ERR_INVALID_ARG  # workspace not 8-byte aligned
    assert _prefill_store(L, hq=12) == pa.PA_ERR_INVALID_ARG   # the prefill's own checks follow
    assert _prefill_store(L, d=64) == pa.PA_ERR_UNSUPPORTED
    assert _prefill_store(L, B=24) == pa.PA_ERR_UNSUPPORTED


def test_shared_prefix_argument_checks(L):
    """pa_decode_shared_prefix: its own checks (new rows both or neither,
    batch <= 1024, the larger workspace), then pa_decode's; every case fails
    (or has nothing to do) before any launch."""
    p = C.c_void_p(256)
    base = L.pa_decode_workspace_size(32, 8, 128)
    full = L.pa_decode_shared_prefix_workspace_size(32, 8, 128)
    # the groups and 8192 (member, head) rows of prefix partials in two splits, after the decode workspace
    assert full >= base + 2 * 8192 * (128 * 4 + 8)
    assert full <= base + 2 * 8192 * (128 * 4 + 8) + 2 * 1024 * 4 + 1024
    assert L.pa_decode_shared_prefix_workspace_size(24, 8, 128) == 0

    def call(**kw):
        a = dict(out=p, q=p, qs=4096, nk=p, nks=1024, nv=p, nvs=1024, k=p, v=p, bt=p, mb=16, ctx=p, batch=4,
                 hq=32, hkv=8, d=128, B=256, nb=64, scale=0.088, ws=p, wsb=full, stream=None)
        a.update(kw)
        return L.pa_decode_shared_prefix(a["out"], a["q"], a["qs"], a["nk"], a["nks"], a["nv"], a["nvs"], a["k"],
                                         a["v"], a["bt"], a["mb"], a["ctx"], a["batch"], a["hq"], a["hkv"], a["d"],
                                         a["B"], a["nb"], a["scale"], a["ws"], a["wsb"], a["stream"])

    assert call(batch=0) == pa.PA_OK
    assert call(nv=None) == pa.PA_ERR_INVALID_ARG                  # new K without new V
    assert call(nk=None) == pa.PA_ERR_INVALID_ARG
    assert call(nk=C.c_void_p(264)) == pa.PA_ERR_INVALID_ARG       # unaligned
    assert call(nks=1000) == pa.PA_ERR_INVALID_ARG                 # stride below Hkv*D
    assert call(batch=1025) == pa.PA_ERR_UNSUPPORTED               # beyond the grouping's batch
    assert call(wsb=base) == pa.PA_ERR_WORKSPACE                   # the plain decode workspace is too small
    assert "workspace" in _msg(L)
    assert call(hq=24) == pa.PA_ERR_UNSUPPORTED                    # pa_decode's own checks still apply
    assert call(scale=-1.0) == pa.PA_ERR_INVALID_ARG

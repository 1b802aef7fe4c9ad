"""Plants plausible mistakes in copies of the oracle source and checks that
every one of them fails at least one pin.  This shows the pins constrain
each step of the oracle (addressing, head mapping, scaling, masking,
normalisation, slot arithmetic, the store).  CPU only: the mutants are
compiled with gcc into a temporary directory."""
import os
import subprocess

import pytest

import oracle as O
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(O.__file__), "pa_oracle.c")

MUTANTS = {
    "page index uses p % B": ("int32_t block = block_table[p / B];",
                              "int32_t block = block_table[p % B];"),
    "in-block offset dropped": ("int64_t slot = (int64_t)block * B + p % B;",
                                "int64_t slot = (int64_t)block * B;"),
    "kv head offset dropped": ("return cache + (slot * Hkv + g) * D;",
                               "return cache + (slot * Hkv) * D;"),
    "interleaved GQA in decode": ("int32_t g = h / group;\n        int32_t ctx",
                                  "int32_t g = h % num_kv_heads;\n        int32_t ctx"),
    "interleaved GQA in prefill": ("int32_t h = (int32_t)(row % num_q_heads), g = h / group;",
                                   "int32_t h = (int32_t)(row % num_q_heads), g = h % num_kv_heads;"),
    "softmax scale dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "normalisation dropped": ("for (int32_t d = 0; d < D; ++d) out[d] /= denom;", ""),
    "max not subtracted consistently": ("double w = exp(s[j] - m);", "double w = exp(s[j] - m) + 1e-3;"),
    "top-left causal alignment": ("int64_t pos = (lk - lq) + i;", "int64_t pos = i;"),
    "query excludes itself": ("int64_t nkeys = causal ? pos + 1 : lk;",
                              "int64_t nkeys = causal ? pos : lk;"),
    "decode drops newest token": ("V_rows, ctx, head_dim, softmax_scale, s);",
                                  "V_rows, ctx - 1, head_dim, softmax_scale, s);"),
    "first-block offset dropped": ("if (i == start_block) slot_start += start % block_size;", ""),
    "last-block end off by one": ("slot_end = first + (int64_t)end - (int64_t)i * block_size;",
                                  "slot_end = first + (int64_t)end - (int64_t)i * block_size - 1;"),
    "decode slot off by one": ("return block_table[num_blocks - 1] * block_size + last_block_num_tokens - 1;",
                               "return block_table[num_blocks - 1] * block_size + last_block_num_tokens;"),
    "store ignores row stride": ("k_cache[(int64_t)slot * D + j] = key[(int64_t)i * key_row_stride + j];",
                                 "k_cache[(int64_t)slot * D + j] = key[(int64_t)i * D + j];"),
    "store ignores padding": ("if (slot < 0) continue; /* padding */",
                              "if (slot < 0) slot = 0; /* padding */"),
    "contiguous prefill ignores cu_seqlens_k": ("int64_t kr = cu_seqlens_k[s] + j;",
                                                "int64_t kr = cu_seqlens_q[s] + j;"),
    "q row stride ignored in decode": ("q + (int64_t)b * q_row_stride + (int64_t)h * head_dim",
                                       "q + (int64_t)h * head_dim"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) == 1, f"mutation site not unique/found: {old!r}"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new), encoding="utf-8")
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC",
                           "-o", str(so), str(mut), "-lm"])
    L = O.load(str(so))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(L)
        except (AssertionError, O.OracleError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutant '{name}'"

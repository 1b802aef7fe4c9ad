"""Host block manager: the C++ library (pa_bm_*) and the Python oracle, each
checked against what the pages print (tests/golden/block_manager_trace.txt:
the 7-round trace with 11 blocks, the R7 prefix hit, the 8-block structure
example), against published XXH64 reference values, against each other
on random operation sequences, and on the behaviours the pages spell out
(stale hashes dropped on reuse, released blocks taken back by a prefix hit,
decode needing a block exactly at len % B == 1).  CPU only."""
import os
import random

import numpy as np
import pytest

from oracle import block_manager as OB
from paged_kv_cache_store_gb300 import build as pabuild

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_manager_trace.txt")


@pytest.fixture(scope="module")
def PB():
    pabuild.build()
    from paged_kv_cache_store_gb300 import block_manager
    return block_manager


# ---------------------------------------------------------------- adapters
class Prod:
    def __init__(self, PB, num_blocks, B):
        self.m, self.B = PB.BlockManager(num_blocks, B), B

    def add(self, toks):
        return self.m.add_sequence(toks)

    def can_allocate(self, s):
        return self.m.can_allocate(s)

    def allocate(self, s, n):
        self.m.allocate(s, n)

    def deallocate(self, s):
        self.m.deallocate(s)

    def can_append(self, s):
        return self.m.can_append(s)

    def may_append(self, s):
        self.m.may_append(s)

    def hash_blocks(self, s, n):
        self.m.hash_blocks(s, n)

    def cached(self, s):
        return self.m.seq_info(s)["num_cached_tokens"]

    def length(self, s):
        return self.m.seq_info(s)["num_tokens"]

    def set_cached(self, s, n):
        self.m.set_num_cached_tokens(s, n)

    def append(self, s, t):
        self.m.append_token(s, t)

    def table(self, s):
        return self.m.block_table(s)

    def free(self):
        return self.m.free_block_ids()

    def hashed(self):
        return [b for b in range(self.m.num_blocks) if self.m.block(b)["hash"] is not None]

    def ref(self, b):
        return self.m.block(b)["ref_count"]

    def hash_of(self, b):
        return self.m.block(b)["hash"]

    def num_hashes(self):
        return self.m.num_hashes()


class Orc:
    def __init__(self, num_blocks, B):
        self.m, self.B, self.seqs = OB.BlockManager(num_blocks, B), B, []

    def add(self, toks):
        self.seqs.append(OB.Sequence(toks, self.B))
        return len(self.seqs) - 1

    def can_allocate(self, s):
        return self.m.can_allocate(self.seqs[s])

    def allocate(self, s, n):
        self.m.allocate(self.seqs[s], n)

    def deallocate(self, s):
        self.m.deallocate(self.seqs[s])

    def can_append(self, s):
        return self.m.can_append(self.seqs[s])

    def may_append(self, s):
        self.m.may_append(self.seqs[s])

    def hash_blocks(self, s, n):
        self.m.hash_blocks(self.seqs[s], n)

    def cached(self, s):
        return self.seqs[s].num_cached_tokens

    def length(self, s):
        return len(self.seqs[s])

    def set_cached(self, s, n):
        self.seqs[s].num_cached_tokens = n

    def append(self, s, t):
        self.seqs[s].token_ids.append(t)

    def table(self, s):
        return list(self.seqs[s].block_table)

    def free(self):
        return list(self.m.free)

    def hashed(self):
        return [b for b, h in enumerate(self.m.block_hash) if h is not None]

    def ref(self, b):
        return self.m.ref_count[b]

    def hash_of(self, b):
        return self.m.block_hash[b]

    def num_hashes(self):
        return len(self.m.index)


def both(PB, num_blocks, B):
    return [("product", Prod(PB, num_blocks, B)), ("oracle", Orc(num_blocks, B))]


# ---------------------------------------------------------------- golden fixture
def golden():
    rounds, extra = {}, {}
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kind, rest = line.split(" ", 1)
        fields = [f.strip() for f in rest.split("|")]
        if kind == "trace" and fields[0].startswith("round="):
            r = int(fields[0].split("=")[1])
            free = fields[1].split("=")[1]
            tables = {}
            for t in fields[2].split():
                name, ids = t.split("=")
                tables[name] = [int(x) for x in ids.split(",")] if ids else []
            rounds[r] = {"free": [] if free == "-" else [int(x) for x in free.split(",")], "tables": tables,
                         "hashed": [int(x) for x in fields[3].split("=")[1].split(",")]}
        else:
            extra[kind] = dict(f.split("=", 1) for f in fields if "=" in f)
    return rounds, extra


def _ints(s):
    return [int(x) for x in s.split(",")] if s else []


# ---------------------------------------------------------------- pins
def test_xxh64_reference_values(PB):
    # XXH64 with seed 0: the published reference values for "" and "abc".
    for f in (PB.xxh64, OB.xxh64):
        assert f(b"") == 0xEF46DB3751D8E999
        assert f(b"abc") == 0x44BC2CF5AD770999


def test_xxh64_product_equals_oracle_on_random_inputs(PB):
    rng = random.Random(3)
    for n in list(range(0, 80)) + [255, 256, 1024, 2056, 4099]:
        data = bytes(rng.getrandbits(8) for _ in range(n))
        seed = rng.getrandbits(64) if n % 3 else 0
        assert PB.xxh64(data, seed) == OB.xxh64(data, seed), n


def test_chained_block_hash(PB):
    toks = list(range(100, 356))
    h0 = PB.block_hash(toks)
    assert h0 == OB.prefix_hash(toks, None) == OB.xxh64(np.array(toks, np.int64).tobytes())
    h1 = PB.block_hash(toks, h0)
    assert h1 == OB.prefix_hash(toks, h0) == OB.xxh64(h0.to_bytes(8, "little") + np.array(toks, np.int64).tobytes())
    assert h1 != h0  # same tokens after a different prefix: a different key


def _prompts():
    lens = {"R1": 300, "R2": 400, "R3": 255, "R4": 1200, "R5": 200}
    return {k: [1000 * (i + 1) + j for j in range(n)] for i, (k, n) in enumerate(lens.items())}


def _finish_step(bm, s, scheduled, tok):
    """What follows a model step for one sequence: register the blocks the
    step filled, count its tokens as computed, append the sampled token once
    the prompt is fully computed (a chunk of a prompt appends nothing)."""
    bm.hash_blocks(s, scheduled)
    bm.set_cached(s, bm.cached(s) + scheduled)
    if bm.cached(s) == bm.length(s):
        bm.append(s, tok)


def _check_round(bm, seqs, want, who, r):
    assert bm.free() == want["free"], (who, r)
    for name, ids in want["tables"].items():
        assert bm.table(seqs[name]) == ids, (who, r, name)
    assert bm.hashed() == want["hashed"], (who, r)


@pytest.mark.parametrize("who", ["product", "oracle"])
def test_seven_round_trace(PB, who):
    rounds, extra = golden()
    bm = dict(both(PB, 11, 256))[who]
    p = _prompts()
    s = {k: bm.add(v) for k, v in p.items() if k != "R5"}
    tok = iter(range(900000, 901000))
    # Round 1: prefill R1, R2, R3 (R4 does not fit the remaining token budget).
    for k in ("R1", "R2", "R3"):
        assert bm.can_allocate(s[k]) == 0
        bm.allocate(s[k], 0)
    for k in ("R1", "R2", "R3"):
        _finish_step(bm, s[k], len(p[k]), next(tok))
    _check_round(bm, s, rounds[1], who, 1)
    # Round 2: R4's first 1024 tokens; all 5 of its blocks are taken at once.
    assert bm.can_allocate(s["R4"]) == 0
    bm.allocate(s["R4"], 0)
    _finish_step(bm, s["R4"], 1024, next(tok))
    _check_round(bm, s, rounds[2], who, 2)
    # Round 3: the remaining 176 tokens of R4.
    _finish_step(bm, s["R4"], 176, next(tok))
    _check_round(bm, s, rounds[3], who, 3)
    # Round 4: one decode step each for R1..R4; R3's first block fills.
    for k in ("R1", "R2", "R3", "R4"):
        assert bm.can_append(s[k])
        bm.may_append(s[k])
    for k in ("R1", "R2", "R3", "R4"):
        _finish_step(bm, s[k], 1, next(tok))
    _check_round(bm, s, rounds[4], who, 4)
    # Round 5: R5 arrives and is prefilled (decode skipped this round).
    s["R5"] = bm.add(p["R5"])
    assert bm.can_allocate(s["R5"]) == 0
    bm.allocate(s["R5"], 0)
    _finish_step(bm, s["R5"], len(p["R5"]), next(tok))
    _check_round(bm, s, rounds[5], who, 5)
    # Round 6: decode; R3 (length 257) needs a block, none is free: the last
    # running sequence, R5, is preempted (its blocks released) and R3 takes
    # the freed block.
    assert bm.length(s["R3"]) == 257 and bm.length(s["R1"]) == 302 and bm.length(s["R2"]) == 402
    for k in ("R1", "R2"):
        assert bm.can_append(s[k])
        bm.may_append(s[k])
    assert not bm.can_append(s["R3"])
    bm.deallocate(s["R5"])
    assert bm.free() == [10] and bm.hash_of(10) is None  # R5's block was never full
    assert bm.can_append(s["R3"])
    bm.may_append(s["R3"])
    assert bm.can_append(s["R4"])
    bm.may_append(s["R4"])
    for k in ("R1", "R2", "R3", "R4"):
        _finish_step(bm, s[k], 1, next(tok))
    _check_round(bm, s, rounds[6], who, 6)
    # Round 7: R5 cannot come back (no free block); decode R1..R4.
    assert bm.can_allocate(s["R5"]) == int(extra["trace"]["can_allocate_R5_round7"])
    for k in ("R1", "R2", "R3", "R4"):
        assert bm.can_append(s[k])
        bm.may_append(s[k])
        _finish_step(bm, s[k], 1, next(tok))
    _check_round(bm, s, rounds[7], who, 7)


@pytest.mark.parametrize("who", ["product", "oracle"])
def test_prefix_hit_r7(PB, who):
    rounds, extra = golden()
    want = extra["r7"]
    bm = dict(both(PB, 11, 256))[who]
    p = _prompts()
    s = {k: bm.add(p[k]) for k in ("R1", "R2", "R3")}
    for k in ("R1", "R2", "R3"):
        bm.allocate(s[k], bm.can_allocate(s[k]))
        _finish_step(bm, s[k], len(p[k]), 7)
    _check_round(bm, s, rounds[1], who, 1)
    r7 = bm.add(p["R1"][:256] + [77000 + j for j in range(344)])
    n = bm.can_allocate(r7)
    assert n == int(want["can_allocate"])
    bm.allocate(r7, n)
    assert bm.table(r7) == _ints(want["table"])
    assert bm.ref(0) == int(want["ref0"])
    assert bm.cached(r7) == int(want["num_cached_tokens"])


@pytest.mark.parametrize("who", ["product", "oracle"])
def test_prefix_hit_r7_with_exactly_enough_free_blocks(PB, who):
    """The page's R7 arithmetic: 3 blocks, block 0 cached and in use, so R7
    fits when 2 blocks are free; with only 1 free it does not."""
    bm = dict(both(PB, 11, 256))[who]
    p = _prompts()
    s = {k: bm.add(p[k]) for k in ("R1", "R2", "R3")}
    for k in ("R1", "R2", "R3"):
        bm.allocate(s[k], bm.can_allocate(s[k]))
        _finish_step(bm, s[k], len(p[k]), 7)
    filler = bm.add(list(range(5000, 5000 + 4 * 256)))  # takes 4 of the 6 free blocks
    bm.allocate(filler, bm.can_allocate(filler))
    assert len(bm.free()) == 2
    r7 = bm.add(p["R1"][:256] + [77000 + j for j in range(344)])
    assert bm.can_allocate(r7) == 1
    other = bm.add(list(range(8000, 8000 + 256)))
    bm.allocate(other, bm.can_allocate(other))
    assert len(bm.free()) == 1 and bm.can_allocate(r7) == -1


@pytest.mark.parametrize("who", ["product", "oracle"])
def test_last_block_never_counts_as_cached(PB, who):
    """Even a full, cached last block is not looked up (the page: the last
    block may be partial, so it is always computed)."""
    bm = dict(both(PB, 8, 4))[who]
    a = bm.add(list(range(1, 9)))  # two full blocks
    bm.allocate(a, bm.can_allocate(a))
    _finish_step(bm, a, 8, 0)
    assert bm.hashed() == bm.table(a)  # both blocks hashed
    b = bm.add(list(range(1, 9)))
    assert bm.can_allocate(b) == 1


@pytest.mark.parametrize("who", ["product", "oracle"])
def test_structure_example_nv12(PB, who):
    want = golden()[1]["nv12"]
    B = 4
    bm = dict(both(PB, 8, B))[who]
    a = bm.add(list(range(1, 13)))                      # three full blocks
    b = bm.add(list(range(1, 9)) + [50, 51, 52, 53])    # same first two blocks
    bm.allocate(a, bm.can_allocate(a))
    _finish_step(bm, a, 12, 0)
    n = bm.can_allocate(b)
    assert n == 2
    bm.allocate(b, n)
    _finish_step(bm, b, 12 - bm.cached(b), 0)
    assert bm.table(a) == _ints(want["tableA"]) and bm.table(b) == _ints(want["tableB"])
    assert [bm.ref(i) for i in range(4)] == _ints(want["ref"])
    assert bm.free() == _ints(want["free"])
    assert bm.num_hashes() == int(want["hashes"])


@pytest.mark.parametrize("who", ["product", "oracle"])
def test_stale_hash_dropped_on_reuse_and_kept_on_release(PB, who):
    """A released block keeps its hash (a later identical prefix takes it
    back); once the block is handed out fresh, its old index entry goes."""
    bm = dict(both(PB, 3, 4))[who]
    x = bm.add([1, 2, 3, 4, 9])
    bm.allocate(x, bm.can_allocate(x))
    _finish_step(bm, x, 5, 0)
    h = bm.hash_of(0)
    assert h is not None and bm.num_hashes() == 1
    bm.deallocate(x)
    assert bm.free() == [2, 1, 0] and bm.hash_of(0) == h and bm.num_hashes() == 1  # last block first
    y = bm.add([1, 2, 3, 4, 5, 6])            # same first block: taken back from the free queue
    assert bm.can_allocate(y) == 1
    bm.allocate(y, 1)
    assert bm.table(y) == [0, 2] and bm.ref(0) == 1 and bm.free() == [1]
    bm.deallocate(y)
    z = bm.add([7] * 12)                      # three fresh blocks: block 0's entry must go
    assert bm.can_allocate(z) == 0
    bm.allocate(z, 0)
    assert bm.num_hashes() == 0 and bm.hash_of(0) is None


@pytest.mark.parametrize("who", ["product", "oracle"])
def test_decode_needs_a_block_at_len_mod_b_equal_1(PB, who):
    bm = dict(both(PB, 3, 4))[who]
    s = bm.add([1, 2, 3, 4])
    bm.allocate(s, bm.can_allocate(s))
    assert len(bm.table(s)) == 1
    bm.append(s, 5)                      # length 5 = 1 mod 4: one more block
    assert bm.can_append(s)
    bm.may_append(s)
    assert len(bm.table(s)) == 2
    bm.append(s, 6)                      # length 6: none
    bm.may_append(s)
    assert len(bm.table(s)) == 2


def test_block_tables_for_the_kernels(PB):
    m = PB.BlockManager(8, 4)
    a = m.add_sequence(range(9))
    b = m.add_sequence(range(100, 104))
    m.allocate(a, m.can_allocate(a))
    m.allocate(b, m.can_allocate(b))
    t = m.block_tables([a, b], 4)
    assert t.tolist() == [[0, 1, 2, -1], [3, -1, -1, -1]]


def test_product_matches_oracle_on_random_operations(PB):
    """Random admissions, decode steps, chunked prefills, preemptions and
    finishes, with shared prefixes: after every operation both managers hold
    the same free queue, tables, reference counts and hashes."""
    rng = random.Random(11)
    B, nblk = 4, 24
    pm, om = Prod(PB, nblk, B), Orc(nblk, B)
    prefixes = [[rng.randrange(50) for _ in range(rng.randrange(1, 13))] for _ in range(4)]
    live = []  # (handle in product, handle in oracle)

    def same():
        assert pm.free() == om.free()
        for i in range(nblk):
            assert pm.ref(i) == om.ref(i) and pm.hash_of(i) == om.hash_of(i), i
        for hp, ho in live:
            assert pm.table(hp) == om.table(ho) and pm.cached(hp) == om.cached(ho)
        assert pm.num_hashes() == om.num_hashes()

    for step in range(600):
        op = rng.random()
        if op < 0.35 or not live:
            toks = rng.choice(prefixes) + [rng.randrange(50) for _ in range(rng.randrange(0, 9))]
            hp, ho = pm.add(toks), om.add(toks)
            n = pm.can_allocate(hp)
            assert n == om.can_allocate(ho)
            if n < 0:
                continue
            pm.allocate(hp, n)
            om.allocate(ho, n)
            live.append((hp, ho))
            # prefill the uncached part, in one or two chunks
            rest = pm.length(hp) - pm.cached(hp)
            first = rest if rng.random() < 0.7 else rng.randrange(0, rest + 1)
            for chunk in (first, rest - first):
                if chunk == 0:
                    continue
                t = rng.randrange(50)
                _finish_step(pm, hp, chunk, t)
                _finish_step(om, ho, chunk, t)
        elif op < 0.8:
            hp, ho = rng.choice(live)
            if pm.cached(hp) != pm.length(hp) - 1:
                continue  # still prefilling
            ok = pm.can_append(hp)
            assert ok == om.can_append(ho)
            if not ok:
                continue
            pm.may_append(hp)
            om.may_append(ho)
            t = rng.randrange(50)
            _finish_step(pm, hp, 1, t)
            _finish_step(om, ho, 1, t)
        else:
            k = rng.randrange(len(live))
            hp, ho = live.pop(k)
            pm.deallocate(hp)
            om.deallocate(ho)
        same()


# Plausible mistakes planted in copies of the oracle: each must fail a pin.
BM_MUTANTS = {
    "free queue used as a stack": ("b = self.free.popleft()", "b = self.free.pop()"),
    "stale index entry kept": ("            del self.index[old]\n", "            pass\n"),
    "hash dropped on release": ("        self.used.remove(b)\n        self.free.append(b)",
                                "        self.used.remove(b)\n        self.free.append(b)\n"
                                "        self.block_hash[b] = None"),
    "last block looked up too": ("for i in range(seq.num_blocks - 1):", "for i in range(seq.num_blocks):"),
    "hash not chained": ("prev = prefix_hash(toks, prev)\n            b = self.index.get(prev)",
                         "prev = prefix_hash(toks, None)\n            b = self.index.get(prev)"),
    "cached block in use still counted as needed": (
        "need = seq.num_blocks - sum(1 for _, in_use in hits if in_use)", "need = seq.num_blocks"),
    "decode block at len % B == 0": ("needs_block = len(seq) % self.block_size == 1",
                                     "needs_block = len(seq) % self.block_size == 0"),
    "released in allocation order": ("for b in reversed(seq.block_table):", "for b in seq.block_table:"),
}


@pytest.mark.parametrize("name", sorted(BM_MUTANTS))
def test_every_block_manager_mutant_fails_a_pin(PB, name, monkeypatch):
    import types
    src = open(OB.__file__, encoding="utf-8").read()
    old, new = BM_MUTANTS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("bm_mutant")
    exec(compile(src.replace(old, new), "bm_mutant.py", "exec"), mod.__dict__)
    monkeypatch.setattr(__import__(__name__), "OB", mod)
    pins = [lambda: test_seven_round_trace(PB, "oracle"), lambda: test_prefix_hit_r7(PB, "oracle"),
            lambda: test_structure_example_nv12(PB, "oracle"),
            lambda: test_stale_hash_dropped_on_reuse_and_kept_on_release(PB, "oracle"),
            lambda: test_decode_needs_a_block_at_len_mod_b_equal_1(PB, "oracle"),
            lambda: test_prefix_hit_r7_with_exactly_enough_free_blocks(PB, "oracle"),
            lambda: test_last_block_never_counts_as_cached(PB, "oracle")]
    failed = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, KeyError, IndexError, ValueError):
            failed += 1
    assert failed > 0, f"mutant '{name}' passes every pin"

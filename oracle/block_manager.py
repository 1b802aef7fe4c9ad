"""Block manager oracle (test infrastructure: only the tests use it; the product
library never loads it and shares no code with it).

A plain Python restatement of the pages' BlockManager
[NV12 §12.8 "BlockManager: 分页 KV Cache + Prefix Caching"; VS §1.1, §1.2.4,
§1.2.5], written from what each operation does:

* state: per block a reference count, the prefix hash (None when unhashed)
  and the token ids; a FIFO of free ids (collections.deque: take left, give
  back right), a set of used ids, a dict prefix-hash -> block id;
* prefix hash of block i = XXH64(seed 0) of the previous block's hash as 8
  little-endian bytes (absent for block 0) then the block's tokens as int64
  little-endian; XXH64 itself is restated below from its published
  specification;
* the operations can_allocate, allocate, deallocate, can_append, may_append
  and hash_blocks as the pages describe them (see each docstring).

Sequences are plain objects with token ids, a block table and the number of
tokens whose K/V is already computed (num_cached_tokens).
"""
from __future__ import annotations

from collections import deque

_M = (1 << 64) - 1
_P1, _P2, _P3 = 0x9E3779B185EBCA87, 0xC2B2AE3D27D4EB4F, 0x165667B19E3779F9
_P4, _P5 = 0x85EBCA77C2B2AE63, 0x27D4EB2F165667C5


def _rotl(x: int, r: int) -> int:
    return ((x << r) | (x >> (64 - r))) & _M


def _lane(acc: int, word: int) -> int:
    return (_rotl((acc + word * _P2) & _M, 31) * _P1) & _M


def xxh64(data: bytes, seed: int = 0) -> int:
    """XXH64 of `data`: 32-byte stripes through four accumulators, then the
    remaining 8-, 4- and 1-byte pieces, then the final avalanche."""
    n = len(data)
    pos = 0
    if n >= 32:
        acc = [(seed + _P1 + _P2) & _M, (seed + _P2) & _M, seed & _M, (seed - _P1) & _M]
        while pos + 32 <= n:
            for j in range(4):
                acc[j] = _lane(acc[j], int.from_bytes(data[pos + 8 * j:pos + 8 * j + 8], "little"))
            pos += 32
        h = (_rotl(acc[0], 1) + _rotl(acc[1], 7) + _rotl(acc[2], 12) + _rotl(acc[3], 18)) & _M
        for a in acc:
            h = ((h ^ _lane(0, a)) * _P1 + _P4) & _M
    else:
        h = (seed + _P5) & _M
    h = (h + n) & _M
    while pos + 8 <= n:
        h ^= _lane(0, int.from_bytes(data[pos:pos + 8], "little"))
        h = (_rotl(h, 27) * _P1 + _P4) & _M
        pos += 8
    if pos + 4 <= n:
        h ^= (int.from_bytes(data[pos:pos + 4], "little") * _P1) & _M
        h = (_rotl(h, 23) * _P2 + _P3) & _M
        pos += 4
    while pos < n:
        h ^= (data[pos] * _P5) & _M
        h = (_rotl(h, 11) * _P1) & _M
        pos += 1
    h ^= h >> 33
    h = (h * _P2) & _M
    h ^= h >> 29
    h = (h * _P3) & _M
    h ^= h >> 32
    return h


def prefix_hash(tokens, prev: int | None) -> int:
    """Hash of a block given the hash of the block before it (None: first block)."""
    head = b"" if prev is None else prev.to_bytes(8, "little")
    return xxh64(head + b"".join(int(t).to_bytes(8, "little", signed=True) for t in tokens))


class Sequence:
    def __init__(self, token_ids, block_size: int):
        self.token_ids = list(token_ids)
        self.block_size = block_size
        self.block_table: list[int] = []
        self.num_cached_tokens = 0

    def __len__(self):
        return len(self.token_ids)

    @property
    def num_blocks(self) -> int:
        return -(-len(self.token_ids) // self.block_size)

    def block(self, i: int) -> list:
        return self.token_ids[i * self.block_size:(i + 1) * self.block_size]


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.ref_count = [0] * num_blocks
        self.block_hash: list[int | None] = [None] * num_blocks
        self.block_tokens: list[list] = [[] for _ in range(num_blocks)]
        self.free = deque(range(num_blocks))
        self.used: set[int] = set()
        self.index: dict[int, int] = {}  # prefix hash -> block id

    # -- single blocks ---------------------------------------------------
    def _take_fresh(self) -> int:
        """Front of the free queue; its old index entry goes (the content is
        about to be overwritten); reference count 1, no hash, no tokens."""
        b = self.free.popleft()
        assert self.ref_count[b] == 0
        old = self.block_hash[b]
        if old is not None and self.index.get(old) == b:
            del self.index[old]
        self.ref_count[b], self.block_hash[b], self.block_tokens[b] = 1, None, []
        self.used.add(b)
        return b

    def _release(self, b: int) -> None:
        """Back of the free queue; the hash and tokens stay for later hits."""
        assert self.ref_count[b] == 0
        self.used.remove(b)
        self.free.append(b)

    def _cache_hits(self, seq: Sequence):
        """(block id, in use) for the leading full blocks of seq found in the
        index with the same tokens; never the last block."""
        hits, prev = [], None
        for i in range(seq.num_blocks - 1):
            toks = seq.block(i)
            prev = prefix_hash(toks, prev)
            b = self.index.get(prev)
            if b is None or self.block_tokens[b] != toks:
                break
            hits.append((b, b in self.used))
        return hits

    # -- the pages' operations -------------------------------------------
    def can_allocate(self, seq: Sequence) -> int:
        """Cached block count, or -1 if the free queue is shorter than the
        blocks still needed (a cached block in use needs none)."""
        hits = self._cache_hits(seq)
        need = seq.num_blocks - sum(1 for _, in_use in hits if in_use)
        return -1 if len(self.free) < need else len(hits)

    def allocate(self, seq: Sequence, num_cached_blocks: int) -> None:
        assert not seq.block_table
        hits = self._cache_hits(seq)
        assert num_cached_blocks <= len(hits)
        for b, _ in hits[:num_cached_blocks]:
            if b in self.used:
                self.ref_count[b] += 1
            else:  # released earlier, content intact
                self.ref_count[b] = 1
                self.free.remove(b)
                self.used.add(b)
            seq.block_table.append(b)
        while len(seq.block_table) < seq.num_blocks:
            seq.block_table.append(self._take_fresh())
        seq.num_cached_tokens = num_cached_blocks * self.block_size

    def deallocate(self, seq: Sequence) -> None:
        for b in reversed(seq.block_table):
            self.ref_count[b] -= 1
            if self.ref_count[b] == 0:
                self._release(b)
        seq.num_cached_tokens = 0
        seq.block_table = []

    def can_append(self, seq: Sequence) -> bool:
        needs_block = len(seq) % self.block_size == 1
        return len(self.free) >= (1 if needs_block else 0)

    def may_append(self, seq: Sequence) -> None:
        if len(seq) % self.block_size == 1:
            seq.block_table.append(self._take_fresh())

    def hash_blocks(self, seq: Sequence, num_scheduled_tokens: int) -> None:
        """Register the blocks this step filled, chained from the block before."""
        first = seq.num_cached_tokens // self.block_size
        last = (seq.num_cached_tokens + num_scheduled_tokens) // self.block_size
        prev = self.block_hash[seq.block_table[first - 1]] if first > 0 else None
        for i in range(first, last):
            b = seq.block_table[i]
            toks = seq.block(i)
            prev = prefix_hash(toks, prev)
            self.block_hash[b], self.block_tokens[b] = prev, toks
            self.index[prev] = b

    # -- snapshot for comparisons ----------------------------------------
    def state(self):
        return {"free": list(self.free), "used": sorted(self.used), "ref": list(self.ref_count),
                "hash": list(self.block_hash), "index": dict(self.index)}

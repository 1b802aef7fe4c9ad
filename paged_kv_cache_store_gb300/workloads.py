"""Seeded synthetic inputs for the paged-KV attention path.

This module only draws numbers: context lengths, which physical blocks a
sequence owns, and N(0,1) bf16 tensors.  It holds none of the method's
arithmetic (no slot computation, no attention); both the CUDA path and the
CPU oracle consume what it returns, so they see identical bytes.

Recipes (the workloads the five named configurations describe):

* tiny decode       : batch 4, 16 q / 8 kv heads, pool of 64 blocks,
                      context_lens ~ U{1..600}, disjoint random blocks.
* qwen3-0.6b decode : batch 64, 16 q / 8 kv heads, context_lens ~ U{1..4096},
                      pool = ceil(1.2 * blocks needed), random permutation.
* qwen3-8b decode   : batch 256, 32 q / 8 kv heads, context_lens =
                      clamp(round(1024 * exp(Z)), 1, 8192) (lognormal, median
                      1024, unit log-std); sequences 0..127 share the same 4
                      physical blocks as their logical blocks 0..3 (so their
                      context is at least 4*256+1), 128..255 are private.
* long-context      : batch 8, 32 q / 8 kv heads, context_lens 32768 each,
                      scattered blocks, pool = ceil(1.2 * blocks needed).
* prefill           : 16 sequences, 32 q / 8 kv heads, total lengths
                      Lk ~ U{128..2048}, k ~ U{0..3} leading whole blocks
                      already cached (k clipped so the last block is always
                      computed), only the Lq = Lk - 256k suffix is new.

All value tensors are N(0,1) float32 rounded to bf16 (round to nearest even)
and returned as uint16 bit patterns.  Every tensor is drawn from streams keyed
by (seed, tensor tag, chunk index), so a seed fixes every byte.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math
import numpy as np

HEAD_DIM = 128
BLOCK_SIZE = 256


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK = 1 << 22
_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        import os
        from concurrent.futures import ThreadPoolExecutor
        _POOL = ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))
    return _POOL


def normal_bf16(seed: int, tag: int, shape) -> np.ndarray:
    """N(0,1) samples rounded to bf16.

    The tensor is cut into fixed chunks of 2**22 elements; chunk j is drawn
    from its own PCG64 stream keyed by (seed, tag, j), so the bytes do not
    depend on how many threads draw them.
    """
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)

    def fill(j):
        s, e = j * _CHUNK, min(n, (j + 1) * _CHUNK)
        ss = np.random.SeedSequence(entropy=seed, spawn_key=(tag, j))
        g = np.random.Generator(np.random.PCG64(ss))
        out[s:e] = f32_to_bf16_bits(g.standard_normal(e - s, dtype=np.float32))

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for j in range(nchunks):
            fill(j)
    else:
        list(_pool().map(fill, range(nchunks)))
    return out.reshape(shape)


@dataclass
class DecodeInputs:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray      # int32 [batch]
    block_tables: np.ndarray      # int32 [batch, max_blocks], -1 padded
    q: np.ndarray                 # uint16 (bf16) [batch, Hq, D]
    new_k: np.ndarray             # uint16 [batch, Hkv, D]; K of the token being decoded
    new_v: np.ndarray             # uint16 [batch, Hkv, D]
    k_cache: np.ndarray           # uint16 [num_blocks, B, Hkv, D]
    v_cache: np.ndarray           # uint16 [num_blocks, B, Hkv, D]
    shared_blocks: list = field(default_factory=list)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]


@dataclass
class PrefillInputs:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    seqlens_k: np.ndarray         # int32 [num_seqs]   total length incl. cached
    seqlens_q: np.ndarray         # int32 [num_seqs]   uncached suffix length
    cu_seqlens_q: np.ndarray      # int32 [num_seqs+1]
    cu_seqlens_k: np.ndarray      # int32 [num_seqs+1]
    block_tables: np.ndarray      # int32 [num_seqs, max_blocks], -1 padded
    q: np.ndarray                 # uint16 [total_q, Hq, D]
    new_k: np.ndarray             # uint16 [total_q, Hkv, D]  suffix K, stored before attention
    new_v: np.ndarray             # uint16 [total_q, Hkv, D]
    k_cache: np.ndarray           # uint16 [num_blocks, B, Hkv, D]
    v_cache: np.ndarray

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])


def _cumsum0(x) -> np.ndarray:
    out = np.zeros(len(x) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(x, dtype=np.int64))
    return out.astype(np.int32)


def _tables(owned: list, max_blocks: int | None = None) -> np.ndarray:
    mb = max(1, max((len(o) for o in owned), default=1)) if max_blocks is None else max_blocks
    bt = np.full((len(owned), mb), -1, dtype=np.int32)
    for i, o in enumerate(owned):
        bt[i, :len(o)] = o
    return bt


def make_decode(name: str, seed: int, batch: int, num_q_heads: int, num_kv_heads: int,
                context_lens, head_dim: int = HEAD_DIM, block_size: int = BLOCK_SIZE,
                num_blocks: int | None = None, pool_slack: float = 1.2,
                shared_prefix_seqs: int = 0, shared_prefix_blocks: int = 0,
                extra_table_cols: int = 0) -> DecodeInputs:
    """Decode inputs for explicit context lengths.

    The block permutation comes from default_rng(seed); each value tensor
    has its own stream (tags 1..5: q, new_k, new_v, k pool, v pool).  Sequences [0, shared_prefix_seqs) use the same
    `shared_prefix_blocks` physical blocks as their first logical blocks.
    """
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    assert ctx.shape == (batch,)
    nb = [(int(c) + block_size - 1) // block_size for c in ctx]
    shared_n = shared_prefix_blocks if shared_prefix_seqs > 0 else 0
    for b in range(shared_prefix_seqs):
        assert nb[b] > shared_n, "a sharing sequence must own blocks past the shared prefix"
    need = shared_n + sum(n - (shared_n if b < shared_prefix_seqs else 0) for b, n in enumerate(nb))
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_slack * need))
    assert need <= num_blocks, "pool too small"
    perm = rng.permutation(num_blocks).astype(np.int32)
    shared = [int(x) for x in perm[:shared_n]]
    pos = shared_n
    owned = []
    for b in range(batch):
        own = list(shared) if b < shared_prefix_seqs else []
        k = nb[b] - len(own)
        own += [int(x) for x in perm[pos:pos + k]]
        pos += k
        owned.append(own)
    bt = _tables(owned, max(1, max(nb)) + extra_table_cols)
    q = normal_bf16(seed, 1, (batch, num_q_heads, head_dim))
    new_k = normal_bf16(seed, 2, (batch, num_kv_heads, head_dim))
    new_v = normal_bf16(seed, 3, (batch, num_kv_heads, head_dim))
    kc = normal_bf16(seed, 4, (num_blocks, block_size, num_kv_heads, head_dim))
    vc = normal_bf16(seed, 5, (num_blocks, block_size, num_kv_heads, head_dim))
    return DecodeInputs(name, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                        ctx.astype(np.int32), bt, q, new_k, new_v, kc, vc, shared)


def decode_config(idx: int) -> DecodeInputs:
    """The four decode workloads (1..4); seed = the workload number."""
    rng = np.random.default_rng(1000 + idx)   # context-length draws
    if idx == 1:
        ctx = rng.integers(1, 601, size=4)
        return make_decode("tiny decode b4 h16/8 pool64 ctx~U[1,600]", 1, 4, 16, 8, ctx,
                           num_blocks=64)
    if idx == 2:
        ctx = rng.integers(1, 4097, size=64)
        return make_decode("qwen3-0.6b decode b64 h16/8 ctx~U[1,4096]", 2, 64, 16, 8, ctx)
    if idx == 3:
        z = rng.standard_normal(256)
        ctx = np.clip(np.round(1024.0 * np.exp(z)), 1, 8192).astype(np.int64)
        ctx[:128] = np.maximum(ctx[:128], 4 * BLOCK_SIZE + 1)
        return make_decode("qwen3-8b decode b256 h32/8 ctx~lognormal(1024) 128 seqs share 4 blocks",
                           3, 256, 32, 8, ctx, shared_prefix_seqs=128, shared_prefix_blocks=4)
    if idx == 4:
        ctx = np.full(8, 32768)
        return make_decode("long-context decode b8 h32/8 ctx=32768", 4, 8, 32, 8, ctx)
    raise ValueError(idx)


def make_prefill(name: str, seed: int, seqlens_k, cached_blocks, num_q_heads: int,
                 num_kv_heads: int, head_dim: int = HEAD_DIM, block_size: int = BLOCK_SIZE,
                 num_blocks: int | None = None, pool_slack: float = 1.2,
                 cached_tokens=None) -> PrefillInputs:
    """Prefill inputs.  `cached_blocks[s]` whole blocks (or `cached_tokens[s]`
    tokens, if given) of sequence s are already in the pool; the rest is new.

    The block permutation comes from default_rng(seed); value tensors use
    tags 1..5 (q, new_k, new_v, k pool, v pool).
    """
    rng = np.random.default_rng(seed)
    lk = np.asarray(seqlens_k, dtype=np.int64)
    if cached_tokens is None:
        cached_tokens = np.asarray(cached_blocks, dtype=np.int64) * block_size
    c = np.asarray(cached_tokens, dtype=np.int64)
    assert np.all(c < lk) and np.all(c >= 0)
    lq = lk - c
    nb = [(int(x) + block_size - 1) // block_size for x in lk]
    need = sum(nb)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_slack * need))
    perm = rng.permutation(num_blocks).astype(np.int32)
    owned, pos = [], 0
    for n in nb:
        owned.append([int(x) for x in perm[pos:pos + n]])
        pos += n
    bt = _tables(owned)
    total_q = int(lq.sum())
    q = normal_bf16(seed, 1, (total_q, num_q_heads, head_dim))
    new_k = normal_bf16(seed, 2, (total_q, num_kv_heads, head_dim))
    new_v = normal_bf16(seed, 3, (total_q, num_kv_heads, head_dim))
    kc = normal_bf16(seed, 4, (num_blocks, block_size, num_kv_heads, head_dim))
    vc = normal_bf16(seed, 5, (num_blocks, block_size, num_kv_heads, head_dim))
    return PrefillInputs(name, len(lk), num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         lk.astype(np.int32), lq.astype(np.int32), _cumsum0(lq), _cumsum0(lk), bt,
                         q, new_k, new_v, kc, vc)


def prefill_config(idx: int = 5) -> PrefillInputs:
    """The varlen prefill workload with prefix-cache hits (seed 5)."""
    assert idx == 5
    rng = np.random.default_rng(1005)
    lk = rng.integers(128, 2049, size=16)
    k = rng.integers(0, 4, size=16)
    k = np.minimum(k, (lk + BLOCK_SIZE - 1) // BLOCK_SIZE - 1)
    return make_prefill("varlen prefill 16 seqs h32/8 Lk~U[128,2048] 0..3 cached blocks",
                        5, lk, k, 32, 8)


# ----------------------------------------------------------------------------
# Sampler inputs: logits of one decode step and the Exp(1) draws of the
# Gumbel-max sampler.  Vocabulary 151936 (the Qwen3 vocabulary), logits
# N(0, 2^2) rounded to bf16, temperatures ~ U[0.5, 1.2], one Exp(1) draw per
# (row, token) in fp32 (the caller's random state in the sampler's contract).

QWEN3_VOCAB = 151936


def exponential_f32(seed: int, tag: int, shape) -> np.ndarray:
    """Exp(1) samples in float32, drawn in fixed chunks from PCG64 streams
    keyed by (seed, tag, chunk) like normal_bf16."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)

    def fill(j):
        s, e = j * _CHUNK, min(n, (j + 1) * _CHUNK)
        ss = np.random.SeedSequence(entropy=seed, spawn_key=(tag, j))
        g = np.random.Generator(np.random.PCG64(ss))
        out[s:e] = g.standard_exponential(e - s, dtype=np.float32)

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for j in range(nchunks):
            fill(j)
    else:
        list(_pool().map(fill, range(nchunks)))
    return out.reshape(shape)


@dataclass
class SamplerInputs:
    name: str
    batch: int
    vocab: int
    logits: np.ndarray        # uint16 bf16 bits [batch, vocab]
    temperatures: np.ndarray  # float32 [batch]
    exp_noise: np.ndarray     # float32 [batch, vocab], Exp(1)


def make_sampler(name: str, seed: int, batch: int, vocab: int, logit_std: float = 2.0) -> SamplerInputs:
    z = normal_bf16(seed, 20, (batch, vocab))
    logits = f32_to_bf16_bits(bf16_bits_to_f32(z) * np.float32(logit_std))
    rng = np.random.default_rng(seed + 1000)
    temps = rng.uniform(0.5, 1.2, size=batch).astype(np.float32)
    return SamplerInputs(name, batch, vocab, logits, temps, exponential_f32(seed, 21, (batch, vocab)))


def sampler_config(batch: int = 64) -> SamplerInputs:
    """Sampling after a decode step: `batch` rows over the Qwen3 vocabulary."""
    return make_sampler(f"gumbel-max sampler, batch {batch}, vocab {QWEN3_VOCAB}, bf16 logits", 6 + batch,
                        batch, QWEN3_VOCAB)

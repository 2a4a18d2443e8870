"""Seeded synthetic inputs for paged attention (shared by the CUDA path's
tests, the oracle's tests and the benchmark).

This module only *draws and places data*: sequence lengths, block tables,
KV pools, queries and the new tokens' K/V.  It contains none of the attention
arithmetic and never performs the slot scatter (the new tokens' K/V are
handed over separately, with the slots they must land in).

The shapes follow the paged-KV problem statement:

* KV pool ``[num_blocks, block_size=16, kv_heads, head_dim]`` bf16, blocks of
  16 tokens reached through a per-sequence block table ("03 - Engines
  Papers", section 2 PagedAttention (vLLM), Key trick).
* ``block_tables`` int32 ``[num_seqs, max_blocks_per_seq]`` (unused entries
  hold -1), ``seq_lens`` int32 (the length *after* this step's new token),
  ``slot_mapping`` int64 with ``slot = block * 16 + offset``.
* Copy-on-write sharing with refcounts (same section, What to extract) for
  the prefix-sharing mix: groups of sequences alias one physical prefix; a
  member whose new token would land in a shared block gets a private copy
  first (listed in ``cow_pairs``; block tables are already repointed).

Random draws: ``numpy.random.default_rng(seed)`` (PCG64); configuration i of
the five named workloads uses seed 1000 + i.  Draw order: sequence lengths,
block placement, K pool, V pool, queries, new keys, new values.  Normals are
drawn as float32 N(0, 1) (in seeded chunks, see ``normal_bf16``) and rounded
to bf16 to nearest-even.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Optional

import numpy as np

BLOCK_SIZE = 16
BF16_NAN = np.uint16(0x7FC0)
_CHUNK = 1 << 22


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_chunk(base: int, i: int, n: int) -> np.ndarray:
    return f32_to_bf16_bits(np.random.default_rng([base, i]).standard_normal(n, dtype=np.float32))


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) float32 draws rounded to bf16 bits.

    One 63-bit integer ``base`` is drawn from ``rng``; the array is then filled
    in chunks of 2**22 elements, chunk i from ``default_rng([base, i])``, so
    the result does not depend on how many threads fill it.
    """
    n = int(np.prod(shape))
    base = int(rng.integers(0, 2**63 - 1))
    out = np.empty(n, dtype=np.uint16)
    bounds = [(lo, min(n, lo + _CHUNK)) for lo in range(0, n, _CHUNK)]

    def fill(i):
        lo, hi = bounds[i]
        out[lo:hi] = _normal_chunk(base, i, hi - lo)

    if len(bounds) <= 1:
        for i in range(len(bounds)):
            fill(i)
    else:
        workers = min(len(bounds), os.cpu_count() or 1)
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(len(bounds))))
    return out.reshape(shape)


@dataclasses.dataclass
class Workload:
    """One batch of paged-attention inputs (all numpy, bf16 as uint16 bits)."""

    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    block_size: int
    k_cache: np.ndarray          # [nb, bs, Hkv, D] uint16, state before this step
    v_cache: np.ndarray
    block_tables: np.ndarray     # [S_all, max_blocks] int32 (-1 = unused)
    seq_lens: np.ndarray         # [S_all] int32, length after the new tokens
    q: np.ndarray                # [Tq, Hq, D] uint16 (chunk rows first, then decode rows)
    key: np.ndarray              # [T_new, Hkv, D] uint16, this step's new tokens
    value: np.ndarray
    slot_mapping: np.ndarray     # [T_new] int64
    refcount: np.ndarray         # [nb] int32 (after copy-on-write)
    cow_pairs: np.ndarray        # [n, 2] int64 (src, dst) block copies before the scatter
    # decode part: sequences decode_seq0 .. S_all-1, queries at rows q_decode_row0 ..
    decode_seq0: int = 0
    q_decode_row0: int = 0
    # prefill-chunk part (hybrid batch): chunk c is sequence c (c < num_chunks)
    num_chunks: int = 0
    cu_q_lens: Optional[np.ndarray] = None    # [C + 1] int32
    q_start_pos: Optional[np.ndarray] = None  # [C] int32
    partition_tokens: int = 0
    token_budget: int = 0

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_decode_seqs(self) -> int:
        return int(self.seq_lens.shape[0]) - self.decode_seq0

    @property
    def decode_seq_lens(self) -> np.ndarray:
        return self.seq_lens[self.decode_seq0:]

    @property
    def decode_block_tables(self) -> np.ndarray:
        return self.block_tables[self.decode_seq0:]

    @property
    def decode_q(self) -> np.ndarray:
        return self.q[self.q_decode_row0:self.q_decode_row0 + self.num_decode_seqs]

    @property
    def chunk_q(self) -> np.ndarray:
        return self.q[:self.q_decode_row0]


def _blocks_for(n: int, bs: int = BLOCK_SIZE) -> int:
    return (int(n) + bs - 1) // bs


def _place(rng, lens, bs, pool_factor, max_blocks, pool_blocks=None):
    """Assign each sequence ceil(len / bs) distinct physical blocks drawn at
    random (without replacement) from a pool ``pool_factor`` times the need."""
    need = [_blocks_for(n, bs) for n in lens]
    total = int(sum(need))
    nb = pool_blocks if pool_blocks is not None else int(math.ceil(pool_factor * total))
    chosen = rng.choice(nb, size=total, replace=False).astype(np.int32)
    bt = np.full((len(lens), max_blocks), -1, dtype=np.int32)
    pos = 0
    for s, k in enumerate(need):
        bt[s, :k] = chosen[pos:pos + k]
        pos += k
    refcount = np.zeros(nb, dtype=np.int32)
    refcount[chosen] = 1
    return bt, nb, refcount


def _decode_slots(bt, lens, bs):
    slots = np.empty(len(lens), dtype=np.int64)
    for s, n in enumerate(lens):
        p = int(n) - 1
        slots[s] = np.int64(bt[s, p // bs]) * bs + p % bs
    return slots


def _poison_unused(k_cache, v_cache, bt, lens, bs):
    """Fill every slot that holds no valid token of any sequence with NaN."""
    nb = k_cache.shape[0]
    valid = np.zeros((nb, bs), dtype=bool)
    for s, n in enumerate(lens):
        n = int(n)
        for j in range(_blocks_for(n, bs)):
            blk = int(bt[s, j])
            valid[blk, : min(bs, n - j * bs)] = True
    k_cache[~valid] = BF16_NAN
    v_cache[~valid] = BF16_NAN


def _finish(name, seed, rng, lens, bt, nb, refcount, Hq, Hkv, D, scale, poison,
            cow_pairs=None, **extra):
    bs = BLOCK_SIZE
    k_cache = normal_bf16(rng, (nb, bs, Hkv, D))
    v_cache = normal_bf16(rng, (nb, bs, Hkv, D))
    S = len(lens)
    q = normal_bf16(rng, (S, Hq, D))
    key = normal_bf16(rng, (S, Hkv, D))
    value = normal_bf16(rng, (S, Hkv, D))
    slots = _decode_slots(bt, lens, bs)
    if poison:
        _poison_unused(k_cache, v_cache, bt, lens, bs)
    if cow_pairs is None:
        cow_pairs = np.zeros((0, 2), dtype=np.int64)
    return Workload(name=name, seed=seed, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                    scale=scale, block_size=bs, k_cache=k_cache, v_cache=v_cache,
                    block_tables=bt, seq_lens=np.asarray(lens, dtype=np.int32), q=q,
                    key=key, value=value, slot_mapping=slots, refcount=refcount,
                    cow_pairs=cow_pairs, **extra)


def tiny(seed: int = 1001, poison: bool = False) -> Workload:
    """4 sequences, lengths {5, 16, 17, 40}, 4 q / 2 kv heads, head_dim 64,
    a 16-block pool with a seeded random block-table permutation, scale 1/8,
    one new token per sequence."""
    rng = np.random.default_rng(seed)
    lens = np.array([5, 16, 17, 40], dtype=np.int32)
    perm = rng.permutation(16).astype(np.int32)
    bt = np.full((4, 3), -1, dtype=np.int32)
    pos = 0
    refcount = np.zeros(16, dtype=np.int32)
    for s, n in enumerate(lens):
        k = _blocks_for(n)
        bt[s, :k] = perm[pos:pos + k]
        refcount[perm[pos:pos + k]] = 1
        pos += k
    return _finish("tiny", seed, rng, lens, bt, 16, refcount, 4, 2, 64, 1.0 / 8.0, poison)


def decode_batch(num_seqs: int, len_lo: int, len_hi: int, Hq: int, Hkv: int, D: int,
                 seed: int, name: str = "decode", poison: bool = False,
                 pool_factor: float = 1.25, partition_tokens: int = 0,
                 max_len: Optional[int] = None, lens=None) -> Workload:
    """Uniform-length decode batch: lengths uniform[len_lo, len_hi] (inclusive),
    blocks drawn at random from a pool ``pool_factor`` times the need."""
    rng = np.random.default_rng(seed)
    if lens is None:
        lens = rng.integers(len_lo, len_hi, size=num_seqs, endpoint=True).astype(np.int32)
    else:
        lens = np.asarray(lens, dtype=np.int32)
    max_blocks = _blocks_for(max_len if max_len is not None else max(len_hi, int(lens.max())))
    bt, nb, refcount = _place(rng, lens, BLOCK_SIZE, pool_factor, max_blocks)
    return _finish(name, seed, rng, lens, bt, nb, refcount, Hq, Hkv, D,
                   1.0 / math.sqrt(D), poison, partition_tokens=partition_tokens)


def llama3_8b_layer(seed: int = 1002, poison: bool = False) -> Workload:
    """64 sequences, lengths uniform[128, 2048], 32 q / 8 kv heads, head_dim 128."""
    return decode_batch(64, 128, 2048, 32, 8, 128, seed, "llama3_8b_decode_layer", poison)


def long_context_split(seed: int = 1003, poison: bool = False,
                       partition_tokens: int = 512) -> Workload:
    """8 sequences, lengths uniform[32768, 131072], 32 q / 8 kv heads, head_dim
    128, KV partitions of 512 tokens merged by log-sum-exp."""
    return decode_batch(8, 32768, 131072, 32, 8, 128, seed, "long_context_split_kv", poison,
                        partition_tokens=partition_tokens)


def cow_mix(seed: int = 1004, poison: bool = False, num_seqs: int = 256,
            group: int = 4, prefix_tokens: int = 256, Hq: int = 64, Hkv: int = 8,
            D: int = 128, max_len: int = 8192, median: float = 512.0, len_offset: int = 0,
            name: str = "cow_prefix_mix") -> Workload:
    """Continuous-batching mix with copy-on-write prefix sharing.

    Lengths ``len_offset`` + lognormal(median ``median``, sigma 1), rounded
    half-to-even and clipped to [1, max_len].  Consecutive groups of ``group`` sequences alias the same
    physical prefix blocks (``prefix_tokens`` tokens); a shared block's
    refcount is the number of members that reference it.  A member whose new
    token lands in a shared block with refcount > 1 first receives a private
    copy of that block (``cow_pairs``) and its table entry is repointed.
    """
    rng = np.random.default_rng(seed)
    bs = BLOCK_SIZE
    z = rng.standard_normal(num_seqs)
    lens = np.clip(len_offset + np.rint(np.exp(math.log(median) + z)), 1, max_len).astype(np.int32)
    max_blocks = _blocks_for(max_len)
    pb = prefix_tokens // bs
    # logical block lists: ('shared', group, j) or ('private', seq, j)
    logical = []
    for s, n in enumerate(lens):
        k = _blocks_for(n)
        g = s // group
        logical.append([("shared", g, j) if j < pb else ("private", s, j) for j in range(k)])
    keys = []
    seen = set()
    for rows in logical:
        for key in rows:
            if key not in seen:
                seen.add(key)
                keys.append(key)
    # copy-on-write: a member whose last (written) block is shared and still
    # referenced by others gets a fresh private block
    refs = {}
    for rows in logical:
        for key in rows:
            refs[key] = refs.get(key, 0) + 1
    cow = []  # (seq, j, shared key)
    for s, n in enumerate(lens):
        j = (int(n) - 1) // bs
        key = logical[s][j]
        if key[0] == "shared" and refs[key] > 1:
            refs[key] -= 1
            new_key = ("cow", s, j)
            logical[s][j] = new_key
            refs[new_key] = 1
            keys.append(new_key)
            cow.append((s, j, key))
    total = len(keys)
    nb = int(math.ceil(1.25 * total))
    chosen = rng.choice(nb, size=total, replace=False).astype(np.int32)
    phys = {key: int(chosen[i]) for i, key in enumerate(keys)}
    bt = np.full((num_seqs, max_blocks), -1, dtype=np.int32)
    for s, rows in enumerate(logical):
        for j, key in enumerate(rows):
            bt[s, j] = phys[key]
    refcount = np.zeros(nb, dtype=np.int32)
    for key, r in refs.items():
        refcount[phys[key]] = r
    cow_pairs = np.array([(phys[shared], phys[("cow", s, j)]) for s, j, shared in cow],
                         dtype=np.int64).reshape(-1, 2)
    w = _finish(name, seed, rng, lens, bt, nb, refcount, Hq, Hkv, D,
                1.0 / math.sqrt(D), False, cow_pairs=cow_pairs)
    if poison:
        # poison what no sequence reads, judged on the post-copy tables.  A
        # shared prefix block holds the whole common prefix, so all its slots
        # stay valid (copies taken from it need them); copy destinations hold
        # garbage until the copy runs.
        valid = np.zeros((nb, bs), dtype=bool)
        for s, n in enumerate(lens):
            n = int(n)
            for j in range(_blocks_for(n, bs)):
                valid[int(bt[s, j]), : min(bs, n - j * bs)] = True
        for key, blk in phys.items():
            if key[0] == "shared":
                valid[blk, :] = True
        w.k_cache[~valid] = BF16_NAN
        w.v_cache[~valid] = BF16_NAN
        for src, dst in cow_pairs:
            w.k_cache[dst] = BF16_NAN
            w.v_cache[dst] = BF16_NAN
    return w


def shared_prompt_batch(seed: int = 1006, poison: bool = False) -> Workload:
    """A long system prompt shared by groups of requests (the case cascade
    attention is for): 128 sequences in 16 groups of 8, each group aliasing one
    2048-token prompt (128 blocks) followed by a private suffix of
    lognormal(median 256, sigma 1) tokens; Llama-3-8B heads (32 q / 8 kv,
    head_dim 128).  No member writes into the shared prompt, so there are no
    copy-on-write pairs."""
    return cow_mix(seed=seed, poison=poison, num_seqs=128, group=8, prefix_tokens=2048, Hq=32,
                   Hkv=8, D=128, max_len=8192, median=256.0, len_offset=2048,
                   name="shared_prompt_batch")


def sarathi_hybrid(seed: int = 1005, poison: bool = False, chunk_tokens: int = 512,
                   chunk_start: int = 1536, num_decode: int = 128, dec_lo: int = 256,
                   dec_hi: int = 4096, Hq: int = 32, Hkv: int = 8, D: int = 128) -> Workload:
    """Sarathi hybrid batch: one prefill chunk of ``chunk_tokens`` query tokens
    at positions chunk_start .. chunk_start + chunk_tokens - 1 attending
    causally over its own paged KV, plus ``num_decode`` decode sequences with
    lengths uniform[dec_lo, dec_hi]; token budget chunk_tokens + num_decode.

    Sequence 0 is the chunk's sequence (its positions < chunk_start stand in
    for earlier chunks); sequences 1.. are the decodes.  Query rows 0 ..
    chunk_tokens - 1 belong to the chunk, the next ``num_decode`` rows to the
    decodes; new tokens are ordered the same way.
    """
    rng = np.random.default_rng(seed)
    bs = BLOCK_SIZE
    dec = rng.integers(dec_lo, dec_hi, size=num_decode, endpoint=True).astype(np.int32)
    chunk_len = chunk_start + chunk_tokens
    lens = np.concatenate([[chunk_len], dec]).astype(np.int32)
    max_blocks = _blocks_for(max(chunk_len, dec_hi))
    bt, nb, refcount = _place(rng, lens, bs, 1.25, max_blocks)
    k_cache = normal_bf16(rng, (nb, bs, Hkv, D))
    v_cache = normal_bf16(rng, (nb, bs, Hkv, D))
    T = chunk_tokens + num_decode
    q = normal_bf16(rng, (T, Hq, D))
    key = normal_bf16(rng, (T, Hkv, D))
    value = normal_bf16(rng, (T, Hkv, D))
    slots = np.empty(T, dtype=np.int64)
    for i in range(chunk_tokens):
        p = chunk_start + i
        slots[i] = np.int64(bt[0, p // bs]) * bs + p % bs
    slots[chunk_tokens:] = _decode_slots(bt[1:], dec, bs)
    if poison:
        _poison_unused(k_cache, v_cache, bt, lens, bs)
    return Workload(name="sarathi_hybrid", seed=seed, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim=D, scale=1.0 / math.sqrt(D), block_size=bs, k_cache=k_cache,
                    v_cache=v_cache, block_tables=bt, seq_lens=lens, q=q, key=key,
                    value=value, slot_mapping=slots, refcount=refcount,
                    cow_pairs=np.zeros((0, 2), dtype=np.int64), decode_seq0=1,
                    q_decode_row0=chunk_tokens, num_chunks=1,
                    cu_q_lens=np.array([0, chunk_tokens], dtype=np.int32),
                    q_start_pos=np.array([chunk_start], dtype=np.int32),
                    token_budget=T)


def prefill_batch(chunks, Hq: int, Hkv: int, D: int, seed: int, poison: bool = False,
                  pool_factor: float = 1.25) -> Workload:
    """Several causal prefill chunks (no decodes): ``chunks`` is a list of
    (q_start_pos, q_len); each chunk's sequence holds q_start_pos + q_len tokens."""
    rng = np.random.default_rng(seed)
    bs = BLOCK_SIZE
    lens = np.array([p + n for p, n in chunks], dtype=np.int32)
    max_blocks = _blocks_for(int(lens.max()))
    bt, nb, refcount = _place(rng, lens, bs, pool_factor, max_blocks)
    k_cache = normal_bf16(rng, (nb, bs, Hkv, D))
    v_cache = normal_bf16(rng, (nb, bs, Hkv, D))
    T = int(sum(n for _, n in chunks))
    q = normal_bf16(rng, (T, Hq, D))
    key = normal_bf16(rng, (T, Hkv, D))
    value = normal_bf16(rng, (T, Hkv, D))
    slots = np.empty(T, dtype=np.int64)
    cu = np.zeros(len(chunks) + 1, dtype=np.int32)
    r = 0
    for c, (p0, n) in enumerate(chunks):
        for i in range(n):
            p = p0 + i
            slots[r + i] = np.int64(bt[c, p // bs]) * bs + p % bs
        r += n
        cu[c + 1] = r
    if poison:
        _poison_unused(k_cache, v_cache, bt, lens, bs)
    return Workload(name="prefill_chunks", seed=seed, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim=D, scale=1.0 / math.sqrt(D), block_size=bs, k_cache=k_cache,
                    v_cache=v_cache, block_tables=bt, seq_lens=lens, q=q, key=key,
                    value=value, slot_mapping=slots, refcount=refcount,
                    cow_pairs=np.zeros((0, 2), dtype=np.int64), decode_seq0=len(chunks),
                    q_decode_row0=T, num_chunks=len(chunks), cu_q_lens=cu,
                    q_start_pos=np.array([p for p, _ in chunks], dtype=np.int32))


CONFIGS = {
    "tiny": tiny,
    "llama3_8b_decode_layer": llama3_8b_layer,
    "long_context_split_kv": long_context_split,
    "cow_prefix_mix": cow_mix,
    "sarathi_hybrid": sarathi_hybrid,
    "shared_prompt_batch": shared_prompt_batch,
}


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """KV bytes per token of context: 2 (K and V) x layers x heads x head_dim x
    bytes per element ("The LLM inference engine playbook", Theme 11, Stage 0)."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def logical_kv_bytes(seq_lens, kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K+V bytes one attention layer reads for these sequences (every token once)."""
    return int(np.asarray(seq_lens, dtype=np.int64).sum()) * kv_bytes_per_token(
        1, kv_heads, head_dim, elem_bytes)


def unique_kv_bytes(block_tables, seq_lens, kv_heads: int, head_dim: int,
                    block_size: int = BLOCK_SIZE, elem_bytes: int = 2) -> int:
    """K+V bytes of distinct physical slots read (shared prefix slots count once)."""
    best = {}
    for s, n in enumerate(np.asarray(seq_lens)):
        n = int(n)
        for j in range(_blocks_for(n, block_size)):
            blk = int(block_tables[s, j])
            best[blk] = max(best.get(blk, 0), min(block_size, n - j * block_size))
    return int(sum(best.values())) * kv_bytes_per_token(1, kv_heads, head_dim, elem_bytes)


def cascade_groups(w: "Workload", group: int):
    """Cascade metadata for a batch whose consecutive sequences form groups of
    ``group`` sharing prefix blocks (the copy-on-write mix): the group's
    prefix table is, at each block index, the physical block most members of
    the group hold there (ties: the lowest id), as long as at least two
    members agree (a lone member's block is not shared); a sequence's
    shared-block count is the length of the leading run of its table that
    equals the prefix table.  Returns (group_offsets int32 [G + 1],
    prefix_tables int32 [G, P], shared_blocks int32 [S])."""
    bt = w.decode_block_tables
    lens = w.decode_seq_lens
    S = bt.shape[0]
    G = -(-S // group)
    offsets = np.minimum(np.arange(G + 1) * group, S).astype(np.int32)
    rows = []
    for g in range(G):
        members = range(offsets[g], offsets[g + 1])
        pref = []
        for j in range(bt.shape[1]):
            ids = [int(bt[s, j]) for s in members if j < _blocks_for(int(lens[s]))]
            if len(ids) < 2:
                break
            vals, counts = np.unique(ids, return_counts=True)
            if counts.max() < 2:
                break
            pref.append(int(vals[np.argmax(counts)]))
        rows.append(pref)
    P = max(1, max(len(r) for r in rows))
    prefix = np.full((G, P), -1, dtype=np.int32)
    for g, r in enumerate(rows):
        prefix[g, :len(r)] = r
    shared = np.zeros(S, dtype=np.int32)
    for g in range(G):
        r = rows[g]
        for s in range(offsets[g], offsets[g + 1]):
            k = 0
            while k < len(r) and k < _blocks_for(int(lens[s])) and bt[s, k] == r[k]:
                k += 1
            shared[s] = k
    return offsets, prefix, shared

"""Host block manager (include/pa_block_manager.h) against its oracle.

Pins of the oracle itself, independent of the C++ code:
  * hand-worked scripts whose expected block ids, slots, copy pairs and
    counters follow from the stated policy step by step (comments give the
    reasoning);
  * a policy-free invariant on random scripts: a simulated pool of token ids
    that receives each step's copy pairs and then its slot writes must read
    back every live sequence's tokens through its block table; refcounts
    equal the references held; blocks are conserved; no slot is handed out
    twice in a step; a step's copy pairs never reuse a block;
  * a planted mistake (an oracle that forgets the copy pair of a copy on
    write) that the invariant catches.
Then the C++ manager, called through the C ABI, must return exactly what the
oracle returns on seeded random scripts (statuses, slots, cached counts,
copy pairs, block tables, counters).  No GPU is involved.
"""
import random

import numpy as np
import pytest

from oracle.block_manager import BlockManagerOracle, INVALID, NO_BLOCKS, OK, STEP


# ------------------------------------------------------------------ pins

def test_pin_refcounts_fork_and_copy_on_write():
    o = BlockManagerOracle(num_blocks=4, block_size=4, prefix_caching=False)
    # 6 tokens need 2 blocks: the free queue's head, 0 then 1
    assert o.add_sequence(1, [1, 2, 3, 4, 5, 6]) == (OK, [0, 1, 2, 3, 4, 5], 0)
    # 3 tokens: block 2, slots 8..10
    assert o.add_sequence(2, [7, 8, 9]) == (OK, [8, 9, 10], 0)
    # position 6 lies in block 1 at offset 2
    assert o.append_token(1, 10) == (OK, 6)
    assert o.fork(1, 3) == OK and o.ref[0] == 2 and o.ref[1] == 2
    # seq 3 would write into shared block 1, which got a slot this step
    assert o.append_token(3, 11) == (STEP, None)
    assert o.end_step() == []
    # next step: copy on write of block 1 into block 3 (the last free one)
    assert o.append_token(3, 11) == (OK, 3 * 4 + 3)
    # block 1 is now seq 1's alone: no copy
    assert o.append_token(1, 12) == (OK, 1 * 4 + 3)
    assert o.ref[1] == 1 and o.ref[3] == 1
    # freeing seq 2 parks block 2 until the step ends
    assert o.free_sequence(2) == OK and o.counters() == (0, 1, 0, 0)
    assert o.add_sequence(4, [5]) == (NO_BLOCKS, None, 0)
    assert o.end_step() == [(1, 3)]
    assert o.add_sequence(4, [5]) == (OK, [8], 0)
    assert o.build_tables([1, 3, 4], 3) == (OK, [[0, 1, -1], [0, 3, -1], [2, -1, -1]], [8, 8, 1])
    assert o.free_sequence(99) == INVALID and o.fork(99, 5) == INVALID


def test_pin_prefix_reuse():
    o = BlockManagerOracle(num_blocks=6, block_size=2, prefix_caching=True)
    # 5 tokens -> blocks 0,1,2; the full blocks 0 (1,2) and 1 (1,2,3,4) are cached
    assert o.add_sequence(1, [1, 2, 3, 4, 5]) == (OK, [0, 1, 2, 3, 4], 0)
    assert o.counters() == (3, 0, 2, 0)
    o.end_step()
    # release last block first: 2, 1, 0 parked; at the step's end block 2
    # (uncached) joins the free queue's tail, 1 then 0 the eviction order
    assert o.free_sequence(1) == OK
    o.end_step()
    assert list(o.free) == [3, 4, 5, 2] and o.lru == [1, 0]
    # the prompt's first two blocks match; the fifth token needs one new block
    assert o.add_sequence(2, [1, 2, 3, 4, 9]) == (OK, [-1, -1, -1, -1, 6], 4)
    assert o.lru == [] and o.ref[0] == 1 and o.ref[1] == 1
    # a 4-token prompt may reuse only floor(3/2) = 1 block; its second block
    # (1,2,3,4) is cached already (block 1), so block 4 stays uncached
    assert o.add_sequence(3, [1, 2, 3, 4]) == (OK, [-1, -1, 8, 9], 2)
    assert o.ref[0] == 2 and 4 not in o.prefix_of
    # a different first block matches nothing
    assert o.add_sequence(4, [2, 1, 3, 4, 5])[2] == 0


def test_pin_eviction_order():
    o = BlockManagerOracle(num_blocks=3, block_size=2, prefix_caching=True)
    assert o.add_sequence(1, [1, 2, 3, 4])[0] == OK  # blocks 0, 1, both cached
    o.end_step()
    o.free_sequence(1)
    o.end_step()
    assert list(o.free) == [2] and o.lru == [1, 0]
    # two blocks needed: block 2 from the free queue, then the least recently
    # released cached block, 1, is evicted
    assert o.add_sequence(2, [7, 8, 9]) == (OK, [4, 5, 2], 0)
    assert (1, 2, 3, 4) not in o.cache and o.cache[(1, 2)] == 0 and o.cache[(7, 8)] == 2
    # three more blocks cannot be had (only block 0 is evictable)
    assert o.add_sequence(3, [5, 6, 5, 6, 5]) == (NO_BLOCKS, None, 0)
    assert o.counters() == (0, 0, 2, 1)


def test_pin_eviction_drops_descendants():
    o = BlockManagerOracle(num_blocks=4, block_size=2, prefix_caching=True)
    o.add_sequence(1, [1, 2, 3, 4, 5, 6])  # blocks 0,1,2 cached as a chain
    o.end_step()
    o.free_sequence(1)
    o.end_step()
    assert o.lru == [2, 1, 0]
    # evicting the chain's head drops the cached prefixes that extend it;
    # those nobody holds go to the free queue in ascending id
    o._evict(0)
    assert o.cache == {} and o.lru == [] and list(o.free) == [3, 1, 2]


# ------------------------------------------------------------------ random scripts

def random_script(seed, n_ops, block_size):
    """A seeded list of operations over a small vocabulary with a few shared
    prompt prefixes, so that prefix reuse, forks and copies on write occur."""
    rng = random.Random(seed)
    systems = [[rng.randrange(50) for _ in range(rng.randrange(1, 4 * block_size))]
               for _ in range(3)]
    ops, next_id, live = [], 0, []
    for _ in range(n_ops):
        r = rng.random()
        if r < 0.25 or not live:
            prompt = list(rng.choice(systems)) if rng.random() < 0.7 else []
            prompt += [rng.randrange(50) for _ in range(rng.randrange(1, 3 * block_size))]
            ops.append(("add", next_id, prompt))
            live.append(next_id)
            next_id += 1
        elif r < 0.65:
            ops.append(("append", rng.choice(live), rng.randrange(50)))
        elif r < 0.72:
            ops.append(("fork", rng.choice(live), next_id))
            live.append(next_id)
            next_id += 1
        elif r < 0.85:
            sid = rng.choice(live)
            live.remove(sid)
            ops.append(("free", sid))
        else:
            ops.append(("end",))
    ops.append(("end",))
    return ops


def run_oracle_with_pool(o, ops):
    """Run a script on the oracle, keeping a simulated pool of token ids, and
    check the invariants after every step."""
    B, N = o.B, o.N
    pool = [None] * (N * B)
    writes = {}
    for op in ops:
        if op[0] == "add":
            st, slots, cached = o.add_sequence(op[1], op[2])
            if st == OK:
                for p, s in enumerate(slots):
                    if s >= 0:
                        assert s not in writes, "slot handed out twice in one step"
                        writes[s] = op[2][p]
        elif op[0] == "append":
            st, slot = o.append_token(op[1], op[2])
            if st == OK:
                assert slot not in writes, "slot handed out twice in one step"
                writes[slot] = op[2]
        elif op[0] == "fork":
            o.fork(op[1], op[2])
        elif op[0] == "free":
            o.free_sequence(op[1])
        else:
            pairs = o.end_step()
            srcs = [a for a, _ in pairs]
            dsts = [b for _, b in pairs]
            assert len(set(dsts)) == len(dsts) and not set(srcs) & set(dsts)
            old = {a: pool[a * B:(a + 1) * B] for a in srcs}
            for a, b in pairs:
                pool[b * B:(b + 1) * B] = old[a]
            for s, t in writes.items():
                pool[s] = t
            writes = {}
            # every live sequence reads back its own tokens
            for sid, s in o.seqs.items():
                for p, t in enumerate(s["tokens"]):
                    assert pool[s["blocks"][p // B] * B + p % B] == t, (sid, p)
            # refcounts equal the references held; blocks are conserved
            held = [0] * N
            for s in o.seqs.values():
                for b in s["blocks"]:
                    held[b] += 1
            assert held == o.ref
            in_use = sum(1 for r in o.ref if r > 0)
            free, parked, cached, evictable = o.counters()
            assert parked == 0
            assert free + evictable + in_use == N
            assert set(o.free).isdisjoint(o.lru)
            assert all(o.ref[b] == 0 for b in list(o.free) + o.lru)
            assert all(o.prefix_of[b] == k for k, b in o.cache.items())


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("caching", [True, False])
def test_oracle_readback_invariant(seed, caching):
    o = BlockManagerOracle(num_blocks=24, block_size=4, prefix_caching=caching)
    run_oracle_with_pool(o, random_script(seed, 400, 4))


def test_invariant_catches_a_forgotten_copy():
    class Broken(BlockManagerOracle):
        def append_token(self, seq_id, token):
            st, slot = super().append_token(seq_id, token)
            self.copies = []  # planted mistake: the copy pairs are lost
            return st, slot

    caught = 0
    for seed in range(6):
        try:
            run_oracle_with_pool(Broken(24, 4, True), random_script(seed, 400, 4))
        except AssertionError:
            caught += 1
    assert caught > 0


# ------------------------------------------------------------------ C++ vs oracle

@pytest.fixture(scope="module")
def bmmod():
    import os
    from paged_kv_cache_218_gb300 import build
    if not os.path.exists(build.LIB):
        build.build()
    from paged_kv_cache_218_gb300 import block_manager
    return block_manager


def _status(fn, *a):
    from paged_kv_cache_218_gb300.block_manager import BlockManagerError
    try:
        return OK, fn(*a)
    except BlockManagerError as e:
        return e.status, None


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("caching", [True, False])
def test_cpp_manager_matches_oracle(bmmod, seed, caching):
    N, B = 32, 4
    o = BlockManagerOracle(N, B, caching)
    m = bmmod.BlockManager(N, B, caching)
    for op in random_script(1000 + seed, 600, B):
        if op[0] == "add":
            st, slots, cached = o.add_sequence(op[1], op[2])
            st2, r = _status(m.add_sequence, op[1], op[2])
            assert st == st2, op
            if st == OK:
                assert list(r[0]) == slots and r[1] == cached
        elif op[0] == "append":
            st, slot = o.append_token(op[1], op[2])
            st2, slot2 = _status(m.append_token, op[1], op[2])
            assert st == st2 and (st != OK or slot == slot2), op
        elif op[0] == "fork":
            assert o.fork(op[1], op[2]) == _status(m.fork, op[1], op[2])[0]
        elif op[0] == "free":
            assert o.free_sequence(op[1]) == _status(m.free_sequence, op[1])[0]
        else:
            pairs = o.end_step()
            assert [tuple(p) for p in m.end_step().tolist()] == pairs
            ids = sorted(o.seqs)
            st, rows, lens = o.build_tables(ids, 64)
            t2, l2 = m.build_tables(ids, 64)
            assert st == OK and t2.tolist() == rows and l2.tolist() == lens
        assert (m.num_free_blocks(), m.num_parked_blocks(), m.num_cached_blocks(),
                m.num_evictable_blocks()) == o.counters(), op
        assert [m.refcount(b) for b in range(N)] == o.ref
    m.close()


def test_cpp_manager_argument_checks(bmmod):
    with pytest.raises(ValueError):
        bmmod.BlockManager(0, 16)
    m = bmmod.BlockManager(4, 16)
    m.add_sequence(7, [1, 2, 3])
    for fn, args in ((m.add_sequence, (7, [1])), (m.append_token, (8, 1)), (m.fork, (8, 9)),
                     (m.fork, (7, 7)), (m.free_sequence, (8,))):
        with pytest.raises(bmmod.BlockManagerError) as e:
            fn(*args)
        assert e.value.status == bmmod.PA_ERR_INVALID
    with pytest.raises(bmmod.BlockManagerError):
        m.build_tables([7], 0)  # one block does not fit in a zero-wide table
    assert m.refcount(-1) == -1 and m.refcount(4) == -1 and m.seq_len(7) == 3
    assert m.seq_len(8) == -1


def test_cpp_batched_appends_match_single_appends(bmmod):
    N, B = 40, 4
    o = BlockManagerOracle(N, B, True)
    m = bmmod.BlockManager(N, B, True)
    rng = random.Random(5)
    for i in range(6):
        prompt = [rng.randrange(9) for _ in range(rng.randrange(1, 10))]
        assert o.add_sequence(i, prompt)[0] == OK
        m.add_sequence(i, prompt)
    o.fork(0, 6)
    m.fork(0, 6)
    o.end_step()
    m.end_step()
    for step in range(12):
        ids = [rng.randrange(7) for _ in range(9)]  # repeats: later ones may hit STEP
        toks = [rng.randrange(9) for _ in ids]
        want, status = [], OK
        for i, t in zip(ids, toks):
            st, slot = o.append_token(i, t)
            if st != OK:
                status = st
                break
            want.append(slot)
        if status == OK:
            assert m.append_tokens(ids, toks).tolist() == want
        else:
            with pytest.raises(bmmod.BlockManagerError) as e:
                m.append_tokens(ids, toks)
            assert e.value.status == status and e.value.done == len(want)
        assert [tuple(p) for p in m.end_step().tolist()] == o.end_step()
        assert [m.refcount(b) for b in range(N)] == o.ref

"""Pins of the cascade oracle (prefix pass + suffix pass + log-sum-exp merge,
"03 - Engines Papers" section 12): the two-level attention must reproduce the
plain decode definition (already pinned) whenever the shared-prefix metadata
describes the tables truthfully, for any split point; with no shared blocks
it is the plain decode; and a sequence's shared part is read through the
group's prefix table (a wrong table there changes exactly those outputs)."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_218_gb300 import workload as W


def scattered(w):
    kc, vc = oracle.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs)
    return oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping)


@pytest.mark.parametrize("kw", [dict(num_seqs=24, group=4, prefix_tokens=64, Hq=16, Hkv=2, D=32,
                                     max_len=400),
                                dict(num_seqs=15, group=3, prefix_tokens=96, Hq=8, Hkv=8, D=16,
                                     max_len=300, poison=True)])
def test_cascade_equals_plain_decode(kw):
    w = W.cow_mix(**kw)
    kc, vc = scattered(w)
    go, pt, sb = W.cascade_groups(w, kw["group"])
    assert sb.max() > 0  # something is shared
    ref, ref_lse = oracle.decode(w.decode_q, kc, vc, w.decode_block_tables, w.decode_seq_lens,
                                 w.scale)
    out, lse = oracle.cascade_decode(w.decode_q, kc, vc, w.decode_block_tables,
                                     w.decode_seq_lens, go, pt, sb, w.scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    # any smaller shared count is also a valid split
    rng = np.random.default_rng(0)
    sb2 = (sb * rng.random(sb.shape)).astype(np.int32)
    out2, _ = oracle.cascade_decode(w.decode_q, kc, vc, w.decode_block_tables,
                                    w.decode_seq_lens, go, pt, sb2, w.scale)
    np.testing.assert_allclose(out2, ref, rtol=1e-12, atol=1e-12)


def test_cascade_without_sharing_is_plain_decode():
    w = W.decode_batch(6, 1, 70, 8, 2, 32, seed=4)
    kc, vc = scattered(w)
    S = w.num_decode_seqs
    go = np.arange(S + 1, dtype=np.int32)
    pt = np.full((S, 1), -1, np.int32)
    out, lse = oracle.cascade_decode(w.decode_q, kc, vc, w.decode_block_tables,
                                     w.decode_seq_lens, go, pt, np.zeros(S, np.int32), w.scale)
    ref, ref_lse = oracle.decode(w.decode_q, kc, vc, w.decode_block_tables, w.decode_seq_lens,
                                 w.scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_shared_part_is_read_through_the_prefix_table():
    w = W.cow_mix(num_seqs=8, group=4, prefix_tokens=64, Hq=8, Hkv=2, D=16, max_len=200, seed=9)
    kc, vc = scattered(w)
    go, pt, sb = W.cascade_groups(w, 4)
    pt2 = pt.copy()
    g = 0
    k = int(sb[go[g]:go[g + 1]].max())
    assert k >= 2
    spare = [b for b in range(kc.shape[0]) if b not in set(w.block_tables.ravel().tolist())]
    pt2[g, 1] = spare[0]  # the prefix table now names another block at index 1
    out, _ = oracle.cascade_decode(w.decode_q, kc, vc, w.decode_block_tables, w.decode_seq_lens,
                                   go, pt2, sb, w.scale)
    # the same as a plain decode whose affected rows name that block
    bt = w.decode_block_tables.copy()
    for s in range(go[g], go[g + 1]):
        if sb[s] > 1:
            bt[s, 1] = spare[0]
    ref, _ = oracle.decode(w.decode_q, kc, vc, bt, w.decode_seq_lens, w.scale)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)

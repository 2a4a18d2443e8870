"""Pins for the fp64 oracle, checked against things other than itself:
closed forms, invariants the paged method must satisfy, brute force in numpy
and mpmath, and torch's fp64 attention.  CPU only.

Where each property comes from:
* gathering from non-contiguous blocks must equal attention over the
  contiguous sequence ("03 - Engines Papers", section 2 PagedAttention,
  Key trick and What to extract) -> placement, aliasing and contiguity pins;
* copy-on-write blocks shared through refcounts (same section) -> the
  aliasing + copy pin;
* partial attentions combine by log-sum-exp ("03 - Engines Papers",
  section 12 Cascade Inference; split-K softmax reduction, "The LLM inference
  engine playbook", Theme 4) -> split/merge pins;
* a prefill chunk's query at position p sees keys 0..p ("03 - Engines
  Papers", section 3 Sarathi) -> causal pins;
* GQA head sharing ("References", GQA) -> group-mapping pin.
"""
import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_218_gb300 import workload as W
from tests import _indep as ind


def _scattered(w):
    kc, vc = oracle.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs)
    return oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping)


# ---------------------------------------------------------------- scatter

def test_scatter_writes_exact_bits_and_nothing_else():
    w = W.tiny()
    kc, vc = oracle.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, w.slot_mapping)
    touched = np.zeros(w.k_cache.shape[:2], dtype=bool)
    for t, slot in enumerate(w.slot_mapping):
        b, o = divmod(int(slot), 16)
        assert np.array_equal(kc[b, o], w.key[t])
        assert np.array_equal(vc[b, o], w.value[t])
        touched[b, o] = True
    assert np.array_equal(kc[~touched], w.k_cache[~touched])
    assert np.array_equal(vc[~touched], w.v_cache[~touched])


def test_scatter_skips_negative_slots_and_rejects_out_of_range():
    w = W.tiny()
    slots = w.slot_mapping.copy()
    slots[1] = -1
    kc, _ = oracle.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots)
    b, o = divmod(int(w.slot_mapping[1]), 16)
    assert np.array_equal(kc[b, o], w.k_cache[b, o])
    slots[1] = 16 * 16
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots)


def test_copy_blocks_exact():
    w = W.tiny()
    kc, vc = oracle.copy_blocks(w.k_cache, w.v_cache, [[3, 9], [0, 2]])
    assert np.array_equal(kc[9], w.k_cache[3]) and np.array_equal(vc[2], w.v_cache[0])
    keep = [i for i in range(16) if i not in (9, 2)]
    assert np.array_equal(kc[keep], w.k_cache[keep])


# ---------------------------------------------------------------- closed forms

def test_seq_len_one_returns_that_v_row_and_its_score():
    w = W.tiny()
    lens = np.ones(4, dtype=np.int32)
    out, lse = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale)
    for s in range(4):
        for h in range(4):
            kvh = h // 2
            v = ind.to_f64(w.v_cache[w.block_tables[s, 0], 0, kvh])
            k = ind.to_f64(w.k_cache[w.block_tables[s, 0], 0, kvh])
            assert np.array_equal(out[s, h], v)
            assert lse[s, h] == pytest.approx(w.scale * float(ind.to_f64(w.q[s, h]) @ k),
                                              rel=1e-14, abs=1e-14)


def test_constant_v_returns_v():
    w = W.tiny()
    vc = w.v_cache.copy()
    const = W.f32_to_bf16_bits(np.linspace(-3, 3, 64, dtype=np.float32))
    vc[:] = const
    out, _ = oracle.decode(w.q, w.k_cache, vc, w.block_tables, w.seq_lens, w.scale)
    np.testing.assert_allclose(out, np.broadcast_to(ind.to_f64(const), out.shape),
                               rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("zero", ["q", "k"])
def test_zero_scores_give_mean_of_v(zero):
    w = W.tiny()
    q = np.zeros_like(w.q) if zero == "q" else w.q
    kc = np.zeros_like(w.k_cache) if zero == "k" else w.k_cache
    out, lse = oracle.decode(q, kc, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    for s in range(4):
        n = int(w.seq_lens[s])
        for h in range(4):
            V = ind.gather(w.v_cache, w.block_tables[s], h // 2, n)
            np.testing.assert_allclose(out[s, h], V.mean(axis=0), rtol=1e-13, atol=1e-14)
            assert lse[s, h] == pytest.approx(math.log(n), rel=1e-14)


def test_dominant_score_selects_its_row():
    w = W.tiny()
    kc = w.k_cache.copy()
    s, h, j = 3, 1, 21
    qv = ind.to_f64(w.q[s, h])
    blk, off = w.block_tables[s, j // 16], j % 16
    # a key parallel to q with scale * q.k about 400 above any other score
    kc[blk, off, h // 2] = W.f32_to_bf16_bits((qv * (400.0 / (w.scale * qv @ qv)))
                                              .astype(np.float32))
    out, _ = oracle.decode(w.q, kc, w.v_cache, w.block_tables, w.seq_lens, w.scale)
    np.testing.assert_allclose(out[s, h], ind.to_f64(w.v_cache[blk, off, h // 2]),
                               rtol=0, atol=1e-12)


def test_two_keys_closed_form_pins_the_scale():
    w = W.tiny()
    lens = np.full(4, 2, dtype=np.int32)
    out, _ = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale)
    for s in range(4):
        for h in range(4):
            K = ind.gather(w.k_cache, w.block_tables[s], h // 2, 2)
            V = ind.gather(w.v_cache, w.block_tables[s], h // 2, 2)
            d = w.scale * float(ind.to_f64(w.q[s, h]) @ (K[0] - K[1]))
            sig = 1.0 / (1.0 + math.exp(-d))
            np.testing.assert_allclose(out[s, h], sig * V[0] + (1 - sig) * V[1],
                                       rtol=1e-13, atol=1e-14)


def test_output_within_convex_hull_of_v():
    w = W.llama3_8b_layer()
    kc, vc = _scattered(w)
    sel = [(0, 0), (5, 17), (63, 31), (20, 8)]
    out, _ = oracle.decode_pairs(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale, sel)
    for i, (s, h) in enumerate(sel):
        V = ind.gather(vc, w.block_tables[s], h // 4, int(w.seq_lens[s]))
        assert np.all(out[i] <= V.max(axis=0) + 1e-12)
        assert np.all(out[i] >= V.min(axis=0) - 1e-12)


def test_gqa_mapping_uses_contiguous_groups():
    w = W.tiny()  # 4 q heads over 2 kv heads
    vc = w.v_cache.copy()
    vc[:, :, 0, :] = W.f32_to_bf16_bits(np.float32(1.0))
    vc[:, :, 1, :] = W.f32_to_bf16_bits(np.float32(-2.0))
    out, _ = oracle.decode(w.q, w.k_cache, vc, w.block_tables, w.seq_lens, w.scale)
    assert np.all(out[:, 0:2] == 1.0) and np.all(out[:, 2:4] == -2.0)


def test_empty_sequence_gives_zero_output_and_minus_inf_lse():
    w = W.tiny()
    lens = w.seq_lens.copy()
    lens[2] = 0
    out, lse = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale)
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))


def test_invalid_metadata_is_rejected():
    w = W.tiny()
    bt = w.block_tables.copy()
    bt[3, 2] = 99
    with pytest.raises(ValueError):
        oracle.decode(w.q, w.k_cache, w.v_cache, bt, w.seq_lens, w.scale)
    lens = w.seq_lens.copy()
    lens[0] = 3 * 16 + 1
    with pytest.raises(ValueError):
        oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale)


# ---------------------------------------------------------------- invariants

def _replace_blocks(w, rng, kc, vc):
    """Move every referenced block to a new random physical location."""
    nb = w.num_blocks
    perm = rng.permutation(nb).astype(np.int32)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    return kc2, vc2, bt2


@pytest.mark.parametrize("make", [W.tiny, W.llama3_8b_layer])
def test_block_placement_permutation_invariance(make):
    w = make()
    kc, vc = _scattered(w)
    out, lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    kc2, vc2, bt2 = _replace_blocks(w, np.random.default_rng(7), kc, vc)
    out2, lse2 = oracle.decode(w.q, kc2, vc2, bt2, w.seq_lens, w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_paged_equals_contiguous_layout():
    w = W.tiny()
    kc, vc = _scattered(w)
    out, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    # contiguous: sequence s owns blocks [3s, 3s + 3) in order (identity-like table)
    S, mb = w.block_tables.shape
    kc2 = np.zeros((S * mb,) + kc.shape[1:], dtype=np.uint16)
    vc2 = np.zeros_like(kc2)
    bt2 = np.arange(S * mb, dtype=np.int32).reshape(S, mb)
    for s in range(S):
        n = int(w.seq_lens[s])
        for kvh in range(2):
            rows_k = ind.gather(kc, w.block_tables[s], kvh, n)
            rows_v = ind.gather(vc, w.block_tables[s], kvh, n)
            for j in range(n):
                kc2[bt2[s, j // 16], j % 16, kvh] = W.f32_to_bf16_bits(rows_k[j].astype(np.float32))
                vc2[bt2[s, j // 16], j % 16, kvh] = W.f32_to_bf16_bits(rows_v[j].astype(np.float32))
    out2, _ = oracle.decode(w.q, kc2, vc2, bt2, w.seq_lens, w.scale)
    assert np.array_equal(out, out2)


def test_aliasing_with_copy_on_write_equals_private_copies():
    """The whole copy-on-write batch through oracle.decode (the function every
    GPU parity test compares against): outputs and lse are bit for bit those
    of the same batch with every aliased block replaced by a private copy."""
    w = W.cow_mix()
    assert len(w.cow_pairs) > 0 and w.refcount.max() > 1
    kc, vc = _scattered(w)
    out, lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    # de-alias: give every (sequence, logical block) its own physical block
    S, mb = w.block_tables.shape
    need = [(int(n) + 15) // 16 for n in w.seq_lens]
    total = sum(need)
    kc2 = np.empty((total,) + kc.shape[1:], dtype=np.uint16)
    vc2 = np.empty_like(kc2)
    bt2 = np.full((S, mb), -1, dtype=np.int32)
    r = 0
    for s in range(S):
        for j in range(need[s]):
            kc2[r] = kc[w.block_tables[s, j]]
            vc2[r] = vc[w.block_tables[s, j]]
            bt2[s, j] = r
            r += 1
    # the batch really shares blocks: fewer physical blocks than logical ones
    assert len(np.unique(w.block_tables[w.block_tables >= 0])) < total
    out2, lse2 = oracle.decode(w.q, kc2, vc2, bt2, w.seq_lens, w.scale)
    assert np.array_equal(out, out2)
    assert np.array_equal(lse, lse2)


def test_cow_copy_protects_the_other_members():
    """Without the copy, a member's scatter into a shared block would change
    what the other members of its group read (whole batch, oracle.decode)."""
    w = W.cow_mix()
    kc, vc = _scattered(w)
    good, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    # what would happen without copy-on-write: write through the shared blocks
    bt_bad = w.block_tables.copy()
    for src, dst in w.cow_pairs:
        bt_bad[bt_bad == dst] = src
    slots_bad = w.slot_mapping.copy()
    writers = []
    for s, n in enumerate(w.seq_lens):
        j = (int(n) - 1) // 16
        if any(int(w.block_tables[s, j]) == int(d) for _, d in w.cow_pairs):
            slots_bad[s] = int(bt_bad[s, j]) * 16 + (int(n) - 1) % 16
            writers.append(s)
    assert writers
    kb, vb = oracle.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots_bad)
    bad, _ = oracle.decode(w.q, kb, vb, bt_bad, w.seq_lens, w.scale)
    # a group member that reads the slot a writer overwrote sees other data
    readers = set()
    for s_w in writers:
        n = int(w.seq_lens[s_w])
        blk = int(bt_bad[s_w, (n - 1) // 16])
        g0 = (s_w // 4) * 4
        for s in range(g0, g0 + 4):
            if s != s_w and int(w.seq_lens[s]) > n - 1 and int(bt_bad[s, (n - 1) // 16]) == blk:
                readers.add(s)
    assert readers
    for s in readers:
        assert not np.array_equal(good[s], bad[s])
    # members whose blocks no writer touched read the same as with the copies
    touched = {int(bt_bad[s_w, (int(w.seq_lens[s_w]) - 1) // 16]) for s_w in writers}
    for s in range(len(w.seq_lens)):
        nb = (int(w.seq_lens[s]) + 15) // 16
        if s not in writers and not touched & set(int(b) for b in bt_bad[s, :nb]):
            assert np.array_equal(good[s], bad[s])


@pytest.mark.parametrize("make", [W.llama3_8b_layer, W.cow_mix])
def test_decode_pairs_equals_decode_rows(make):
    """oracle.decode_pairs (the sampled form used at full size) returns, bit for
    bit, the rows of oracle.decode for each listed (sequence, q head): pins its
    kv-head mapping and its output row.  Pairs include both sides of every
    group boundary, duplicates and an unsorted order."""
    w = make()
    kc, vc = _scattered(w)
    out, lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    S, Hq = w.q.shape[:2]
    G = Hq // w.k_cache.shape[2]
    rng = np.random.default_rng(7)
    sel = [(int(s), g * G + d) for s in rng.choice(S, 24, replace=False)
           for g in range(Hq // G) for d in (0, G - 1)]
    sel += [(int(s), int(h)) for s, h in zip(rng.integers(0, S, 200), rng.integers(0, Hq, 200))]
    sel += sel[:10]
    sel = [sel[i] for i in rng.permutation(len(sel))]
    assert len(sel) >= 400
    po, pl = oracle.decode_pairs(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale, sel)
    for i, (s, h) in enumerate(sel):
        assert np.array_equal(po[i], out[s, h]), (s, h)
        assert pl[i] == lse[s, h], (s, h)


def test_decode_pairs_brute_force_at_group_boundaries():
    """decode_pairs against a numpy full-matrix restatement at group 8 (the
    copy-on-write mix), for the first and last q head of several kv heads."""
    w = W.cow_mix()
    kc, vc = _scattered(w)
    G = w.q.shape[1] // w.k_cache.shape[2]
    sel = [(s, h) for s in (0, 3, 101, 255) for h in (0, G - 1, G, 3 * G + 7, 63)]
    po, pl = oracle.decode_pairs(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale, sel)
    for i, (s, h) in enumerate(sel):
        n = int(w.seq_lens[s])
        K = ind.gather(kc, w.block_tables[s], h // G, n)
        V = ind.gather(vc, w.block_tables[s], h // G, n)
        ref, ref_lse = ind.softmax_attention_np(ind.to_f64(w.q[s, h]), K, V, w.scale)
        np.testing.assert_allclose(po[i], ref, rtol=1e-11, atol=1e-12)
        assert abs(pl[i] - ref_lse) < 1e-11


# ---------------------------------------------------------------- split + merge

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_split_at_arbitrary_points_then_merge_equals_full(seed):
    rng = np.random.default_rng(seed)
    w = W.decode_batch(6, 1, 300, 8, 2, 64, seed=100 + seed)
    kc, vc = _scattered(w)
    full, full_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    S, Hq, D = w.q.shape
    P = 5
    part_o = np.zeros((S, Hq, P, D))
    part_lse = np.full((S, Hq, P), -np.inf)
    nparts = np.zeros(S, dtype=np.int32)
    for s in range(S):
        n = int(w.seq_lens[s])
        k = int(rng.integers(1, P + 1))
        cuts = np.sort(rng.integers(0, n + 1, size=k - 1))
        edges = [0, *cuts.tolist(), n]
        nparts[s] = k
        for h in range(Hq):
            for p in range(k):
                part_o[s, h, p], part_lse[s, h, p] = oracle.attend_range(
                    w.q, kc, vc, w.block_tables, s, h, edges[p], edges[p + 1], w.scale)
    merged, merged_lse = oracle.merge(part_o, part_lse, nparts)
    np.testing.assert_allclose(merged, full, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(merged_lse, full_lse, rtol=1e-12, atol=1e-13)


def test_merge_special_cases():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((1, 1, 3, 8))
    lse = np.array([[[0.7, 0.7, -np.inf]]])
    out, l = oracle.merge(o[:, :, :1], lse[:, :, :1], [1])
    np.testing.assert_array_equal(out[0, 0], o[0, 0, 0])
    assert l[0, 0] == 0.7
    same = np.repeat(o[:, :, :1], 2, axis=2)
    out, l = oracle.merge(same, lse[:, :, :2], [2])
    np.testing.assert_allclose(out[0, 0], o[0, 0, 0], rtol=1e-15)
    assert l[0, 0] == pytest.approx(0.7 + math.log(2.0), rel=1e-15)
    out, l = oracle.merge(o, lse, [3])  # the -inf part carries no weight
    np.testing.assert_allclose(out[0, 0], 0.5 * (o[0, 0, 0] + o[0, 0, 1]), rtol=1e-14)
    out, l = oracle.merge(o, np.full((1, 1, 3), -np.inf), [3])
    assert np.all(out == 0) and np.isneginf(l[0, 0])


def test_merge_of_two_singletons_is_two_key_softmax():
    a, b = 1.25, -0.5
    va, vb = np.array([1.0, 2.0]), np.array([-3.0, 4.0])
    out, l = oracle.merge(np.array([[[va, vb]]]), np.array([[[a, b]]]), [2])
    wa = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(out[0, 0], wa * va + (1 - wa) * vb, rtol=1e-15)
    assert l[0, 0] == pytest.approx(math.log(math.exp(a) + math.exp(b)), rel=1e-15)


# ---------------------------------------------------------------- brute force

def test_tiny_matches_numpy_full_matrix():
    w = W.tiny()
    kc, vc = _scattered(w)
    out, lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    ref, ref_lse = ind.decode_np(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-14)


def test_tiny_matches_mpmath_50_digits():
    w = W.tiny()
    kc, vc = _scattered(w)
    out, lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    for s in range(4):
        n = int(w.seq_lens[s])
        for h in (0, 3):
            K = ind.gather(kc, w.block_tables[s], h // 2, n)
            V = ind.gather(vc, w.block_tables[s], h // 2, n)
            ref, ref_lse = ind.attention_mpmath(ind.to_f64(w.q[s, h]), K, V, w.scale)
            np.testing.assert_allclose(out[s, h], ref, rtol=1e-12, atol=1e-13)
            assert lse[s, h] == pytest.approx(ref_lse, rel=1e-12)


def test_matches_torch_sdpa_fp64():
    torch = pytest.importorskip("torch")
    w = W.decode_batch(5, 1, 200, 8, 2, 128, seed=55)
    kc, vc = _scattered(w)
    out, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    for s in range(5):
        n = int(w.seq_lens[s])
        K = np.stack([ind.gather(kc, w.block_tables[s], g, n) for g in range(2)])  # [2, n, D]
        V = np.stack([ind.gather(vc, w.block_tables[s], g, n) for g in range(2)])
        q = torch.from_numpy(ind.to_f64(w.q[s]))[:, None, :]                      # [8, 1, D]
        Kt = torch.from_numpy(K).repeat_interleave(4, dim=0)
        Vt = torch.from_numpy(V).repeat_interleave(4, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(q, Kt, Vt, scale=w.scale)
        np.testing.assert_allclose(out[s], ref[:, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_random_small_shapes_match_numpy():
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=25, deadline=None)
    @hyp.given(S=st.integers(1, 4), Hkv=st.sampled_from([1, 2]), G=st.sampled_from([1, 2, 4, 8]),
               D=st.sampled_from([64, 128]), hi=st.integers(1, 300), seed=st.integers(0, 10**6))
    def check(S, Hkv, G, D, hi, seed):
        w = W.decode_batch(S, 1, hi, Hkv * G, Hkv, D, seed=seed)
        kc, vc = _scattered(w)
        out, lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
        ref, ref_lse = ind.decode_np(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-13)

    check()


# ---------------------------------------------------------------- prefill (causal)

def _chunks_workload():
    return W.prefill_batch([(0, 37), (40, 25), (7, 1)], Hq=8, Hkv=2, D=64, seed=77)


def test_prefill_query_equals_decode_over_its_prefix():
    w = _chunks_workload()
    kc, vc = _scattered(w)
    out, lse = oracle.prefill(w.q, kc, vc, w.block_tables, w.cu_q_lens, w.q_start_pos,
                              w.seq_lens, w.scale)
    for c in range(w.num_chunks):
        for i in range(int(w.cu_q_lens[c + 1] - w.cu_q_lens[c])):
            t = int(w.cu_q_lens[c]) + i
            p = int(w.q_start_pos[c]) + i
            dec, dlse = oracle.decode(w.q[t:t + 1], kc, vc, w.block_tables[c:c + 1],
                                      np.array([p + 1], dtype=np.int32), w.scale)
            assert np.array_equal(out[t], dec[0]) and np.array_equal(lse[t], dlse[0])


def test_prefill_matches_numpy_causal_brute_force():
    w = _chunks_workload()
    kc, vc = _scattered(w)
    out, _ = oracle.prefill(w.q, kc, vc, w.block_tables, w.cu_q_lens, w.q_start_pos,
                            w.seq_lens, w.scale)
    for c in range(w.num_chunks):
        q0, q1 = int(w.cu_q_lens[c]), int(w.cu_q_lens[c + 1])
        n = int(w.seq_lens[c])
        p0 = int(w.q_start_pos[c])
        for h in range(8):
            K = ind.gather(kc, w.block_tables[c], h // 4, n)
            V = ind.gather(vc, w.block_tables[c], h // 4, n)
            Q = ind.to_f64(w.q[q0:q1, h])
            x = w.scale * Q @ K.T
            pos_q = p0 + np.arange(q1 - q0)[:, None]
            x = np.where(np.arange(n)[None, :] <= pos_q, x, -np.inf)
            P = np.exp(x - x.max(axis=1, keepdims=True))
            ref = (P @ V) / P.sum(axis=1, keepdims=True)
            np.testing.assert_allclose(out[q0:q1, h], ref, rtol=1e-12, atol=1e-13)


def test_prefill_is_causal_and_first_position_returns_v0():
    w = _chunks_workload()
    kc, vc = _scattered(w)
    out, _ = oracle.prefill(w.q, kc, vc, w.block_tables, w.cu_q_lens, w.q_start_pos,
                            w.seq_lens, w.scale)
    # chunk 0 starts at position 0: its first query sees only key 0
    for h in range(8):
        assert np.array_equal(out[0, h], ind.to_f64(vc[w.block_tables[0, 0], 0, h // 4]))
    # changing K/V at positions after p leaves query p unchanged
    kc2, vc2 = kc.copy(), vc.copy()
    p = 20  # chunk 0, query row 20 sits at position 20
    for j in range(p + 1, int(w.seq_lens[0])):
        kc2[w.block_tables[0, j // 16], j % 16] = W.f32_to_bf16_bits(np.float32(9.0))
        vc2[w.block_tables[0, j // 16], j % 16] = W.f32_to_bf16_bits(np.float32(-9.0))
    out2, _ = oracle.prefill(w.q, kc2, vc2, w.block_tables, w.cu_q_lens, w.q_start_pos,
                             w.seq_lens, w.scale)
    assert np.array_equal(out[:p + 1], out2[:p + 1])
    assert not np.array_equal(out[p + 1:37], out2[p + 1:37])


def test_prefill_dominant_key_selects_its_value_from_its_position_on():
    """Queries all 1 and one key all 16 (scaled score 2048 / sqrt(128), about
    177 above any other in natural-log units): every query row at or after
    the key's position returns the key's value (the other weights, below
    e^-170, vanish against the 1e-12 tolerance); the rows before it are
    exactly those of the batch without that key."""
    def run(kpos):
        w = W.prefill_batch([(256, 32)], Hq=8, Hkv=2, D=128, seed=910)
        w.q[:] = W.f32_to_bf16_bits(np.float32(1.0))
        base_w = W.prefill_batch([(256, 32)], Hq=8, Hkv=2, D=128, seed=910)
        base_w.q[:] = w.q
        big = W.f32_to_bf16_bits(np.float32(16.0))
        if kpos < 256:
            w.k_cache[w.block_tables[0, kpos // 16], kpos % 16] = big
        else:
            w.key[kpos - 256] = big
        outs = []
        for ww in (w, base_w):
            kc, vc = _scattered(ww)
            outs.append(oracle.prefill(ww.q, kc, vc, ww.block_tables, ww.cu_q_lens,
                                       ww.q_start_pos, ww.seq_lens, ww.scale)[0])
        return w, outs[0], outs[1]
    for kpos in (0, 127, 200, 261):
        w, out, base = run(kpos)
        kc, vc = _scattered(w)
        blk, off = w.block_tables[0, kpos // 16], kpos % 16
        first = max(0, kpos - 256)  # first query row (position 256 + i) that sees the key
        for h in range(8):
            v = ind.to_f64(vc[blk, off, h // 4])
            for i in range(first, 32):
                np.testing.assert_allclose(out[i, h], v, rtol=0, atol=1e-12)
        assert np.array_equal(out[:first], base[:first])


# ---------------------------------------------------------------- KV byte formula

def test_kv_byte_formula_golden():
    """tests/golden/kv_bytes.txt: values of the KV-bytes-per-token formula."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "kv_bytes.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert rows
    for layers, heads, dim, elem, expect in rows:
        assert W.kv_bytes_per_token(int(layers), int(heads), int(dim), int(elem)) == int(expect)

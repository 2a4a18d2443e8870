"""The seeded generators: determinism and the structure each workload promises."""
import numpy as np
import pytest

from paged_kv_cache_218_gb300 import workload as W


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    torch = pytest.importorskip("torch")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(W.f32_to_bf16_bits(x), ref)
    assert np.array_equal(W.bf16_bits_to_f32(ref), torch.from_numpy(ref.view(np.int16))
                          .view(torch.bfloat16).float().numpy())


def test_generation_is_deterministic():
    a, b = W.tiny(), W.tiny()
    for f in ("k_cache", "v_cache", "q", "key", "value", "block_tables", "slot_mapping"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    c = W.tiny(seed=5)
    assert not np.array_equal(a.q, c.q)


def test_tiny_structure():
    w = W.tiny()
    assert list(w.seq_lens) == [5, 16, 17, 40]
    assert w.num_blocks == 16 and w.head_dim == 64 and w.num_q_heads == 4
    assert w.scale == 1.0 / 8.0
    used = w.block_tables[w.block_tables >= 0]
    assert len(used) == 7 and len(set(used.tolist())) == 7


def _check_slots(w):
    nb = w.num_blocks
    assert np.all((w.slot_mapping >= 0) & (w.slot_mapping < nb * 16))
    assert len(set(w.slot_mapping.tolist())) == len(w.slot_mapping)


@pytest.mark.parametrize("make", [W.llama3_8b_layer, W.sarathi_hybrid])
def test_random_placement_structure(make):
    w = make()
    need = sum((int(n) + 15) // 16 for n in w.seq_lens)
    assert w.num_blocks == int(np.ceil(1.25 * need))
    used = w.block_tables[w.block_tables >= 0]
    assert len(used) == need and len(np.unique(used)) == need
    _check_slots(w)


def test_llama_layer_lengths():
    w = W.llama3_8b_layer()
    assert len(w.seq_lens) == 64 and w.seq_lens.min() >= 128 and w.seq_lens.max() <= 2048
    assert w.num_q_heads == 32 and w.num_kv_heads == 8 and w.head_dim == 128


def test_cow_mix_aliasing_and_refcounts():
    w = W.cow_mix()
    assert len(w.seq_lens) == 256 and w.seq_lens.min() >= 1 and w.seq_lens.max() <= 8192
    counts = {}
    for s, n in enumerate(w.seq_lens):
        for j in range((int(n) + 15) // 16):
            b = int(w.block_tables[s, j])
            counts[b] = counts.get(b, 0) + 1
    for b, c in counts.items():
        assert w.refcount[b] == c
    # shared blocks stay within a group of 4 and cover only the 256-token prefix
    owners = {}
    for s, n in enumerate(w.seq_lens):
        for j in range((int(n) + 15) // 16):
            owners.setdefault(int(w.block_tables[s, j]), set()).add((s // 4, j))
    shared = [b for b, c in counts.items() if c > 1]
    assert shared
    for b in shared:
        assert len({g for g, _ in owners[b]}) == 1 and all(j < 16 for _, j in owners[b])
    # no sequence writes its new token into a block another sequence reads
    for slot in w.slot_mapping:
        assert w.refcount[int(slot) // 16] == 1
    # every copy destination is referenced once, every source is shared or was
    for src, dst in w.cow_pairs:
        assert w.refcount[dst] == 1 and w.refcount[src] >= 1


def test_shared_prompt_batch_groups_share_exactly_the_prompt():
    w = W.shared_prompt_batch()
    assert len(w.seq_lens) == 128 and w.seq_lens.min() > 2048 and len(w.cow_pairs) == 0
    for g in range(16):
        rows = w.block_tables[8 * g:8 * g + 8]
        # the 128 prompt blocks are the same physical blocks for all 8 members ...
        assert (rows[:, :128] == rows[0, :128]).all()
        assert (w.refcount[rows[0, :128]] == 8).all()
        # ... and no block after the prompt is shared
        for s in range(8 * g, 8 * g + 8):
            own = w.block_tables[s, 128:(int(w.seq_lens[s]) + 15) // 16]
            assert (w.refcount[own] == 1).all()
    go, pt, sb = W.cascade_groups(w, 8)
    assert (sb == 128).all() and pt.shape == (16, 128)
    assert (pt == w.block_tables[::8, :128]).all()


def test_hybrid_layout():
    w = W.sarathi_hybrid()
    assert w.num_chunks == 1 and list(w.cu_q_lens) == [0, 512]
    assert w.q_start_pos[0] == 1536 and w.seq_lens[0] == 2048
    assert w.num_decode_seqs == 128 and w.q.shape[0] == 640 == w.token_budget
    assert w.decode_seq_lens.min() >= 256 and w.decode_seq_lens.max() <= 4096


def test_poison_marks_only_unused_slots():
    w = W.tiny(poison=True)
    for s, n in enumerate(w.seq_lens):
        for j in range(int(n)):
            assert w.k_cache[w.block_tables[s, j // 16], j % 16, 0, 0] != W.BF16_NAN
    n_nan = int((w.k_cache[:, :, 0, 0] == W.BF16_NAN).sum())
    assert n_nan == 16 * 16 - 78


def test_kv_byte_accounting():
    w = W.llama3_8b_layer()
    assert W.logical_kv_bytes(w.seq_lens, 8, 128) == int(w.seq_lens.sum()) * 4096
    c4 = W.cow_mix()
    assert W.unique_kv_bytes(c4.block_tables, c4.seq_lens, 8, 128) < \
        W.logical_kv_bytes(c4.seq_lens, 8, 128)

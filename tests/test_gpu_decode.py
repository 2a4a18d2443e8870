"""GPU parity of the slot scatter, block copy, decode (all three split modes)
and the LSE merge against the fp64 oracle, through the C ABI."""
import functools
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_218_gb300 import workload as W
from tests.gpu_common import (DeviceWorkload, assert_close, bits_to_dev, dev_to_bits,
                              oracle_scattered)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa(cuda_device):
    from paged_kv_cache_218_gb300 import binding
    binding.pa_device_error_flags(reset=True)
    return binding


@functools.lru_cache(maxsize=None)
def _workload(name, poison=False):
    return {"tiny": W.tiny, "c2": W.llama3_8b_layer, "c3": W.long_context_split,
            "c4": W.cow_mix, "c5": W.sarathi_hybrid}[name](poison=poison)


@functools.lru_cache(maxsize=None)
def _oracle_decode(name, poison=False):
    w = _workload(name, poison)
    kc, vc = oracle_scattered(w)
    out, lse = oracle.decode(w.decode_q, kc, vc, w.decode_block_tables, w.decode_seq_lens,
                             w.scale)
    return kc, vc, out, lse


def _decode(pa, dw, partition_tokens, with_lse=True):
    w = dw.w
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=dw.q.device)
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dw.q.device) \
        if with_lse else None
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(
        S, Hq, w.num_kv_heads, D, w.max_blocks_per_seq, 16, partition_tokens), dw.q.device)
    pa.pa_decode(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                 partition_tokens=partition_tokens, out_lse=lse, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, ws


# ------------------------------------------------------------------ scatter

@pytest.mark.parametrize("name", ["tiny", "c2", "c4", "c5"])
def test_scatter_and_copy_on_write_bit_exact(pa, cuda_device, name):
    w = _workload(name)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    torch.cuda.synchronize()
    kc, vc = oracle_scattered(w)
    assert np.array_equal(dev_to_bits(dw.k_cache), kc)
    assert np.array_equal(dev_to_bits(dw.v_cache), vc)
    assert pa.pa_device_error_flags() == 0


def test_scatter_skips_padding_and_flags_out_of_range(pa, cuda_device):
    w = _workload("tiny")
    dw = DeviceWorkload(w, cuda_device)
    slots = w.slot_mapping.copy()
    slots[0] = -1
    slots[2] = 16 * 16 + 5  # beyond the pool: skipped and flagged
    dw.slot_mapping = torch.from_numpy(slots).to(cuda_device)
    dw.scatter(pa)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags() == pa.PA_DEVERR_SLOT
    slots_ok = slots.copy()
    slots_ok[2] = -1
    kc, vc = oracle.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots_ok)
    assert np.array_equal(dev_to_bits(dw.k_cache), kc)
    assert np.array_equal(dev_to_bits(dw.v_cache), vc)


def test_scatter_strided_rows(pa, cuda_device):
    """key/value rows taken from a wider fused buffer (row stride > Hkv*D)."""
    w = _workload("tiny")
    dw = DeviceWorkload(w, cuda_device)
    T, Hkv, D = w.key.shape
    fused = torch.zeros((T, 3 * Hkv, D), dtype=torch.bfloat16, device=cuda_device)
    fused[:, Hkv:2 * Hkv] = dw.key
    fused[:, 2 * Hkv:] = dw.value
    pa.pa_reshape_and_cache(fused[:, Hkv:2 * Hkv], fused[:, 2 * Hkv:], dw.k_cache, dw.v_cache,
                            dw.slot_mapping)
    torch.cuda.synchronize()
    kc, vc = oracle_scattered(w)
    assert np.array_equal(dev_to_bits(dw.k_cache), kc)
    assert np.array_equal(dev_to_bits(dw.v_cache), vc)


# ------------------------------------------------------------------ decode parity

CASES = [
    ("tiny", -1), ("tiny", 0), ("tiny", 16), ("tiny", 32),
    ("c2", -1), ("c2", 0), ("c2", 256), ("c2", 512),
    ("c4", 0), ("c4", -1), ("c4", 1024),
    ("c5", 0),
]


@pytest.mark.parametrize("name,partition", CASES)
def test_decode_matches_oracle(pa, cuda_device, name, partition):
    w = _workload(name)
    kc, vc, ref, ref_lse = _oracle_decode(name)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse, _ = _decode(pa, dw, partition)
    assert_close(out, ref, f"{name} P={partition} out")
    assert_close(lse.cpu().numpy(), ref_lse, f"{name} P={partition} lse")
    assert pa.pa_device_error_flags() == 0


@pytest.mark.slow
@pytest.mark.parametrize("partition", [512, 0])
def test_long_context_split_kv_matches_oracle(pa, cuda_device, partition):
    w = _workload("c3")
    kc, vc, ref, ref_lse = _oracle_decode("c3")
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse, _ = _decode(pa, dw, partition)
    assert_close(out, ref, f"c3 P={partition}")
    assert_close(lse.cpu().numpy(), ref_lse, f"c3 P={partition} lse")
    assert pa.pa_device_error_flags() == 0


@pytest.mark.parametrize("name", ["tiny", "c2", "c4"])
@pytest.mark.parametrize("partition", [0, -1, 64])
def test_decode_ignores_nan_in_unused_slots(pa, cuda_device, name, partition):
    w = _workload(name, poison=True)
    kc, vc, ref, _ = _oracle_decode(name, poison=True)
    assert np.isfinite(ref).all()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, _, _ = _decode(pa, dw, partition, with_lse=False)
    assert torch.isfinite(out).all()
    assert_close(out, ref, f"{name} poisoned P={partition}")


def test_balanced_workspace_is_left_zeroed_and_reusable(pa, cuda_device):
    w = _workload("c2")
    _, _, ref, _ = _oracle_decode("c2")
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, _, ws = _decode(pa, dw, 0, with_lse=False)
    counters = ws[: 4 * torch.cuda.get_device_properties(0).multi_processor_count]
    assert int(counters.sum()) == 0
    for _ in range(3):
        pa.pa_decode(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                     partition_tokens=0, workspace=ws)
    torch.cuda.synchronize()
    assert_close(out, ref, "c2 balanced, repeated")


# ------------------------------------------------------------------ edge cases

EDGE = [
    # (num_seqs, lo, hi, Hq, Hkv, D, seed)
    (7, 1, 1, 8, 8, 128, 1),       # seq_len 1 everywhere, group 1
    (5, 16, 16, 8, 4, 64, 2),      # exactly one full block, group 2
    (5, 17, 17, 16, 2, 128, 3),    # one token into the second block, group 8
    (9, 1, 300, 12, 4, 128, 4),    # group 3 (padded MMA columns)
    (3, 1, 40, 7, 1, 64, 5),       # group 7, one kv head
    (33, 500, 3000, 32, 8, 128, 6),
    (6, 1, 100, 6, 3, 128, 7),     # three kv heads: two warps per head, two warps idle
    (4, 20, 90, 10, 5, 64, 8),     # five kv heads: one warp per head, three idle
]


@pytest.mark.parametrize("S,lo,hi,Hq,Hkv,D,seed", EDGE)
@pytest.mark.parametrize("partition", [-1, 0, 48])
def test_decode_edge_shapes(pa, cuda_device, S, lo, hi, Hq, Hkv, D, seed, partition):
    w = W.decode_batch(S, lo, hi, Hq, Hkv, D, seed=300 + seed, poison=True)
    kc, vc = oracle_scattered(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse, _ = _decode(pa, dw, partition)
    assert_close(out, ref, f"edge S={S} G={Hq // Hkv} D={D} P={partition}")
    assert_close(lse.cpu().numpy(), ref_lse, "edge lse")


@pytest.mark.parametrize("partition", [-1, 0, 256])
def test_decode_scores_climbing_along_the_sequence(pa, cuda_device, partition):
    """Queries all 1 and every key of positions 128 t .. 128 t + 127 equal to
    0.75 t (bf16-exact): scores climb by about 12 log2 units per 128 keys,
    so the running maximum moves at almost every block and the pieces of a
    split sequence carry log-sum-exps hundreds of units apart for the merge."""
    w = W.decode_batch(6, 100, 3000, 32, 8, 128, seed=940)
    w.q[:] = W.f32_to_bf16_bits(np.float32(1.0))
    for s_ in range(w.num_decode_seqs):
        n = int(w.seq_lens[s_])
        for pos in range(n - 1):
            w.k_cache[w.block_tables[s_, pos // 16], pos % 16] = \
                W.f32_to_bf16_bits(np.float32(0.75 * (pos // 128)))
        w.key[s_] = W.f32_to_bf16_bits(np.float32(0.75 * ((n - 1) // 128)))
    kc, vc = oracle_scattered(w)
    ref, ref_lse = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse, _ = _decode(pa, dw, partition)
    assert torch.isfinite(out).all()
    assert_close(out, ref, f"climbing scores P={partition}")
    assert_close(lse.cpu().numpy(), ref_lse, f"climbing scores P={partition}: lse")
    assert pa.pa_device_error_flags() == 0


@pytest.mark.parametrize("partition", [-1, 0, 32])
def test_decode_empty_sequences_give_zero(pa, cuda_device, partition):
    w = W.decode_batch(6, 1, 70, 8, 2, 128, seed=91)
    lens = w.seq_lens.copy()
    lens[[1, 4]] = 0
    w.seq_lens = lens
    dw = DeviceWorkload(w, cuda_device)
    out, lse, _ = _decode(pa, dw, partition)
    ref, ref_lse = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, lens, w.scale)
    assert_close(out, ref, "empty seqs")
    got_lse = lse.cpu().numpy()
    assert np.all(np.isneginf(got_lse[[1, 4]]))
    assert_close(got_lse[[0, 2, 3, 5]], ref_lse[[0, 2, 3, 5]], "empty seqs lse")


def test_decode_zero_batch_is_a_no_op(pa, cuda_device):
    w = _workload("tiny")
    dw = DeviceWorkload(w, cuda_device)
    out = torch.empty((0, 4, 64), dtype=torch.bfloat16, device=cuda_device)
    pa.pa_decode(out, dw.q[:0], dw.k_cache, dw.v_cache, dw.block_tables[:0], dw.seq_lens[:0],
                 w.scale, partition_tokens=-1)
    torch.cuda.synchronize()


def test_decode_flags_bad_metadata_without_faulting(pa, cuda_device):
    w = _workload("tiny")
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    bt = w.block_tables.copy()
    bt[3, 1] = 10_000  # outside the 16-block pool
    lens = w.seq_lens.copy()
    lens[0] = 999      # beyond the 3-entry table
    out = torch.empty((4, 4, 64), dtype=torch.bfloat16, device=cuda_device)
    pa.pa_decode(out, dw.q, dw.k_cache, dw.v_cache, torch.from_numpy(bt).to(cuda_device),
                 torch.from_numpy(lens).to(cuda_device), w.scale, partition_tokens=-1)
    flags = pa.pa_device_error_flags()
    assert flags & pa.PA_DEVERR_BLOCK_ID and flags & pa.PA_DEVERR_SEQ_LEN
    # untouched sequences are still right
    kc, vc = oracle_scattered(w)
    ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    assert_close(out[1:3], ref[1:3], "good rows next to bad ones")


def test_host_rejects_bad_arguments(pa, cuda_device):
    w = _workload("tiny")
    dw = DeviceWorkload(w, cuda_device)
    out = torch.empty((4, 4, 64), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens, w.scale,
                     partition_tokens=0, workspace=None)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens, w.scale,
                     partition_tokens=24)
    assert e.value.status == pa.PA_ERR_INVALID


# ------------------------------------------------------------------ merge

@pytest.mark.parametrize("D", [64, 128])
def test_merge_partials_matches_oracle(pa, cuda_device, D):
    rng = np.random.default_rng(8)
    S, Hq, P = 5, 6, 9
    part_o = rng.standard_normal((S, Hq, P, D)).astype(np.float32)
    part_lse = (3 * rng.standard_normal((S, Hq, P))).astype(np.float32)
    part_lse[0, 0, :] = -np.inf
    part_lse[1, 2, 3] = -np.inf
    nparts = np.array([3, 1, 9, 0, 5], dtype=np.int32)
    ref, ref_lse = oracle.merge(part_o.astype(np.float64), part_lse.astype(np.float64), nparts)
    out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=cuda_device)
    lse = torch.empty((S, Hq), dtype=torch.float32, device=cuda_device)
    pa.pa_merge_partials(out, torch.from_numpy(part_o).to(cuda_device),
                         torch.from_numpy(part_lse).to(cuda_device),
                         torch.from_numpy(nparts).to(cuda_device), out_lse=lse)
    torch.cuda.synchronize()
    assert_close(out, ref, "merge")
    got = lse.cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isneginf(got), ~fin)
    assert_close(got[fin], ref_lse[fin], "merge lse")


def test_split_partials_merge_to_single_pass(pa, cuda_device):
    """Decode with fixed partitions, keep the partials, merge them again with
    the public merge call: same as the single-pass result."""
    w = _workload("c2")
    _, _, ref, _ = _oracle_decode("c2")
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    P = 256
    out, _, ws = _decode(pa, dw, P, with_lse=False)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    mp = (w.max_blocks_per_seq * 16 + P - 1) // P
    rows = S * Hq * mp
    part_o = ws[: rows * D * 4].view(torch.float32).view(S, Hq, mp, D)
    off = (rows * D * 4 + 255) // 256 * 256
    part_lse = ws[off: off + rows * 4].view(torch.float32).view(S, Hq, mp)
    nparts = torch.from_numpy(np.maximum(1, -(-w.seq_lens // P)).astype(np.int32)).to(cuda_device)
    single = nparts.cpu().numpy() == 1
    out2 = torch.empty_like(out)
    pa.pa_merge_partials(out2, part_o, part_lse, nparts)
    torch.cuda.synchronize()
    assert_close(out2[torch.from_numpy(~single)], ref[~single], "re-merged partials")


@pytest.mark.parametrize("partition", [-1, 16, 0])
def test_decode_is_bitwise_deterministic_on_one_block_pieces(pa, cuda_device, partition):
    """Many one-block pieces at 64 q heads stress the query staging ring: the
    outputs of repeated launches must be identical bit for bit."""
    w = W.decode_batch(600, 1, 16, 64, 8, 128, seed=3)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, 8, D, w.max_blocks_per_seq, 16,
                                                        partition), cuda_device)
    outs = []
    for _ in range(12):
        out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=cuda_device)
        pa.pa_decode(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                     partition_tokens=partition, workspace=ws)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_decode_lengths_written_by_the_previous_kernel(pa, cuda_device):
    """The balanced decode plans its split from the lengths before it waits on
    the previous kernel, then checks them again; here the previous kernel on
    the stream (a scatter, launched as the decode's programmatic primary)
    writes new lengths into the very buffer the decode reads them from.
    Every decode must follow the new lengths."""
    w = W.decode_batch(64, 1, 900, 32, 8, 128, seed=41)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    kc, vc = oracle_scattered(w)
    rng = np.random.default_rng(5)
    full = w.seq_lens.astype(np.int32)  # the tables hold blocks up to these lengths
    lens_sets = [full, rng.integers(1, full + 1).astype(np.int32),
                 np.maximum(1, full // 3).astype(np.int32)]
    refs = [oracle.decode(w.q, kc, vc, w.block_tables, ls, w.scale)[0] for ls in lens_sets]
    # the lengths live in a scatter destination: 16-byte slots of a pool with
    # one kv head of 8 columns, so slot j holds lengths 4j .. 4j+3
    nslot = S // 4
    meta_k = torch.zeros((nslot // 16 + 1, 16, 1, 8), dtype=torch.bfloat16, device=cuda_device)
    meta_v = torch.zeros_like(meta_k)
    lens_dev = meta_k.view(torch.int32).view(-1)[:S]
    rows = [torch.from_numpy(ls.view(np.int16).reshape(nslot, 1, 8).copy()).view(torch.bfloat16)
            .to(cuda_device) for ls in lens_sets]
    slots = torch.arange(nslot, dtype=torch.int64, device=cuda_device)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, 8, D, w.max_blocks_per_seq, 16, 0),
                            cuda_device)
    outs = []
    for i in range(24):
        k = i % 3
        pa.pa_reshape_and_cache(rows[k], rows[k], meta_k, meta_v, slots)
        out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=cuda_device)
        pa.pa_decode(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, lens_dev, w.scale,
                     partition_tokens=0, workspace=ws)
        outs.append((k, out))
    torch.cuda.synchronize()
    for k, out in outs:
        assert_close(out, refs[k], f"lengths set {k}")
    assert pa.pa_device_error_flags() == 0

"""pa_decode_append: the slot scatter fused into the decode.

Each sequence's new token (row s of key / value) goes into the slot of
position seq_len - 1 named by its block table, and the decode attends over
[0, seq_len) with it in place ("03 - Engines Papers", section 2
PagedAttention).  Checked against the fp64 oracle's scatter (every byte of
both pools, bit for bit) and decode (elementwise), and bit for bit against
pa_reshape_and_cache followed by pa_decode, in every split mode.  The pools'
copy of the new token's slot is poisoned with NaN beforehand, so the kernel
must attend the token it was given, not what the pool held."""
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


def _poison_new_slots(w):
    """The slots the step writes hold NaN before it (a stale token would show)."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    for s, n in enumerate(w.seq_lens):
        if n > 0:
            b, o = divmod(int(w.slot_mapping[s]), 16)
            kc[b, o] = W.BF16_NAN
            vc[b, o] = W.BF16_NAN
    return kc, vc


def _expected_slots(w):
    """Slot of position seq_len - 1 through the table (the append's target)."""
    out = np.full(len(w.seq_lens), -1, dtype=np.int64)
    for s, n in enumerate(w.seq_lens):
        if n > 0:
            out[s] = int(w.block_tables[s, (n - 1) // 16]) * 16 + (n - 1) % 16
    return out


def _run_append(pa, w, kc_bits, vc_bits, device, partition, key=None, value=None):
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    kc, vc = bits_to_dev(kc_bits, device), bits_to_dev(vc_bits, device)
    q = bits_to_dev(w.q, device)
    key = bits_to_dev(w.key, device) if key is None else key
    value = bits_to_dev(w.value, device) if value is None else value
    bt = torch.from_numpy(w.block_tables).to(device)
    sl = torch.from_numpy(w.seq_lens).to(device)
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=device)
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=device)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                        w.max_blocks_per_seq, 16, partition),
                            device)
    pa.pa_decode_append(out, q, key, value, kc, vc, bt, sl, w.scale, partition_tokens=partition,
                        out_lse=lse, workspace=ws)
    torch.cuda.synchronize()
    return out, lse, kc, vc


CASES = [
    (lambda: W.tiny(poison=True), (0, -1, 16)),
    (lambda: W.llama3_8b_layer(poison=True), (0, -1, 512)),
    (lambda: W.decode_batch(40, 1, 300, 16, 8, 64, seed=81, poison=True), (0, -1, 64)),
    (lambda: W.decode_batch(24, 1, 200, 12, 3, 128, seed=82, poison=True), (0, -1, 32)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_append_matches_oracle_scatter_and_decode(pa, cuda_device, case):
    make, partitions = CASES[case]
    w = make()
    assert np.array_equal(w.slot_mapping, _expected_slots(w))
    kc0, vc0 = _poison_new_slots(w)
    okc, ovc = oracle.reshape_and_cache(w.key, w.value, kc0, vc0, w.slot_mapping)
    ref, ref_lse = oracle.decode(w.q, okc, ovc, w.block_tables, w.seq_lens, w.scale)
    for part in partitions:
        out, lse, kc, vc = _run_append(pa, w, kc0, vc0, cuda_device, part)
        assert np.array_equal(dev_to_bits(kc), okc), f"K pool (partition_tokens={part})"
        assert np.array_equal(dev_to_bits(vc), ovc), f"V pool (partition_tokens={part})"
        assert_close(out, ref, f"append decode (partition_tokens={part})")
        assert_close(lse.cpu().numpy(), ref_lse, f"append lse (partition_tokens={part})")
    assert pa.pa_device_error_flags() == 0


@pytest.mark.parametrize("partition", [0, -1, 512])
def test_append_equals_scatter_then_decode_bitwise(pa, cuda_device, partition):
    w = W.llama3_8b_layer(poison=True)
    out, lse, kc, vc = _run_append(pa, w, w.k_cache, w.v_cache, cuda_device, partition)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                        w.max_blocks_per_seq, 16, partition),
                            cuda_device)
    pa.pa_decode(out2, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                 partition_tokens=partition, out_lse=lse2, workspace=ws)
    torch.cuda.synchronize()
    # bit patterns (the pools hold NaN poison, which compares unequal as a value)
    assert np.array_equal(dev_to_bits(kc), dev_to_bits(dw.k_cache))
    assert np.array_equal(dev_to_bits(vc), dev_to_bits(dw.v_cache))
    assert np.array_equal(dev_to_bits(out), dev_to_bits(out2))
    assert torch.equal(lse, lse2)


def test_append_full_size_long_context(pa, cuda_device):
    """The long-context batch (8 x 32K-131K tokens), fixed 512-token partitions
    merged by log-sum-exp, every output checked."""
    w = W.long_context_split()
    okc, ovc = oracle.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, w.slot_mapping)
    ref, _ = oracle.decode(w.q, okc, ovc, w.block_tables, w.seq_lens, w.scale)
    out, _, kc, vc = _run_append(pa, w, w.k_cache, w.v_cache, cuda_device, 512)
    assert_close(out, ref, "append long context")
    rows = [int(w.slot_mapping[s]) for s in range(8)]
    kcb = dev_to_bits(kc).reshape(-1, *okc.shape[2:])
    assert np.array_equal(kcb[rows], okc.reshape(-1, *okc.shape[2:])[rows])


def test_append_strided_rows_and_empty_sequences(pa, cuda_device):
    """key / value rows with a token stride above Hkv * D; sequences of
    length 0 write nothing and output zeros."""
    lens = [0, 17, 1, 0, 33, 16]
    w = W.decode_batch(6, 0, 0, 8, 2, 128, seed=83, lens=lens, max_len=64)
    dev = cuda_device
    S, Hkv, D = 6, 2, 128
    wide_k = torch.zeros((S, Hkv * D + 64), dtype=torch.bfloat16, device=dev)
    wide_v = torch.zeros_like(wide_k)
    wide_k[:, :Hkv * D] = bits_to_dev(w.key, dev).view(S, Hkv * D)
    wide_v[:, :Hkv * D] = bits_to_dev(w.value, dev).view(S, Hkv * D)
    key = wide_k.as_strided((S, Hkv, D), (Hkv * D + 64, D, 1))
    value = wide_v.as_strided((S, Hkv, D), (Hkv * D + 64, D, 1))
    assert all(w.slot_mapping[s] == -1 for s, n in enumerate(lens) if n == 0)
    okc, ovc = oracle.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, w.slot_mapping)
    ref, _ = oracle.decode(w.q, okc, ovc, w.block_tables, w.seq_lens, w.scale)
    for part in (0, -1, 16):
        out, _, kc, vc = _run_append(pa, w, w.k_cache, w.v_cache, dev, part, key=key,
                                     value=value)
        assert np.array_equal(dev_to_bits(kc), okc) and np.array_equal(dev_to_bits(vc), ovc)
        assert_close(out, ref, f"strided / empty (partition_tokens={part})")
    assert pa.pa_device_error_flags() == 0

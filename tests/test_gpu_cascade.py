"""Cascade decode on the GPU (prefix pass + suffix decode started from it),
through the C ABI, against the oracle's plain decode definition: the same
outputs and lse within the parity tolerance, on the copy-on-write mix at
full size (groups of 4 sharing 256 tokens, group 8) in all split modes, on
other group shapes (up to 32 query rows per kv head), with NaN poison in
unused slots, with sequences whose whole length lies in the shared prefix,
without any sharing, and with bad metadata flagged instead of faulting."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_218_gb300 import workload as W
from tests.gpu_common import DeviceWorkload, assert_close, oracle_scattered

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa(cuda_device):
    from paged_kv_cache_218_gb300 import binding
    return binding


def run(pa, dev, w, group, partition, go=None, pt=None, sb=None, expect_flags=0):
    if go is None:
        go, pt, sb = W.cascade_groups(w, group)
    dw = DeviceWorkload(w, dev)
    dw.scatter(pa)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dev)
    ws = pa.alloc_workspace(pa.pa_cascade_workspace_size(S, Hq, w.num_kv_heads, D,
                                                         w.max_blocks_per_seq, 16, partition), dev)
    pa.pa_cascade_decode(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens,
                         torch.from_numpy(go).to(dev), group, torch.from_numpy(pt).to(dev),
                         torch.from_numpy(sb).to(dev), w.scale, partition_tokens=partition,
                         out_lse=lse, workspace=ws)
    torch.cuda.synchronize()
    kc, vc = oracle_scattered(w)
    ref, ref_lse = oracle.decode(w.decode_q, kc, vc, w.decode_block_tables, w.decode_seq_lens,
                                 w.scale)
    assert_close(out, ref, f"{w.name} cascade, partition {partition}")
    assert_close(lse.cpu().numpy(), ref_lse, f"{w.name} cascade lse, partition {partition}")
    assert pa.pa_device_error_flags() == expect_flags
    return go, pt, sb


@pytest.mark.parametrize("partition", [0, 512, -1])
def test_cascade_cow_mix_full_size(pa, cuda_device, partition):
    go, pt, sb = run(pa, cuda_device, W.cow_mix(), 4, partition)
    assert sb.max() == 16 and (sb == 16).sum() > 150


@pytest.mark.parametrize("partition", [0, -1])
def test_cascade_shared_prompt_batch_full_size(pa, cuda_device, partition):
    """Groups of 8 sharing a 2048-token prompt (32 member x head rows per kv
    head, the most one prefix CTA takes), at full size."""
    go, pt, sb = run(pa, cuda_device, W.shared_prompt_batch(), 8, partition)
    assert (sb == 128).all()


@pytest.mark.parametrize("partition", [0, -1])
def test_cascade_scores_climbing_along_the_sequence(pa, cuda_device, partition):
    """Queries all 1 and every key at position p equal to 0.75 (p // 128)
    (bf16-exact), groups of 8 sharing 512 tokens: scores climb by about 12
    log2 units per 128 keys, so a member's suffix carries a running maximum
    far above its prefix's and the suffix decode starts from a prefix (o, lse)
    whose weight is e^-100 or less."""
    w = W.cow_mix(num_seqs=40, group=8, prefix_tokens=512, Hq=32, Hkv=8, D=128,
                  max_len=2048, seed=950)
    w.q[:] = W.f32_to_bf16_bits(np.float32(1.0))
    for s_ in range(w.num_decode_seqs):
        n = int(w.seq_lens[s_])
        for pos in range(n - 1):
            w.k_cache[w.block_tables[s_, pos // 16], pos % 16] = \
                W.f32_to_bf16_bits(np.float32(0.75 * (pos // 128)))
        w.key[s_] = W.f32_to_bf16_bits(np.float32(0.75 * ((n - 1) // 128)))
    run(pa, cuda_device, w, 8, partition)


SHAPES = [  # num_seqs, group, prefix_tokens, Hq, Hkv, max_len
    (40, 8, 512, 32, 8, 2048),   # 8 members x group 4 = 32 rows
    (30, 3, 96, 16, 2, 600),     # 24 rows, two kv heads
    (16, 4, 160, 8, 1, 900),     # one kv head
    (48, 16, 256, 32, 16 // 2, 1500),  # group 4, 16 members -> 64 rows: too many
    (36, 6, 64, 16, 8, 400),     # group 2, 6 members = 12 rows (one warp per kv head)
]


@pytest.mark.parametrize("n,group,prefix,Hq,Hkv,max_len", SHAPES)
@pytest.mark.parametrize("partition", [0, 64])
def test_cascade_group_shapes_with_poison(pa, cuda_device, n, group, prefix, Hq, Hkv, max_len,
                                          partition):
    w = W.cow_mix(num_seqs=n, group=group, prefix_tokens=prefix, Hq=Hq, Hkv=Hkv, D=128,
                  max_len=max_len, poison=True, seed=100 + n)
    if group * (Hq // Hkv) > 32:
        with pytest.raises(pa.PAError) as e:
            run(pa, cuda_device, w, group, partition)
        assert e.value.status == pa.PA_ERR_UNSUPPORTED
        return
    run(pa, cuda_device, w, group, partition)


@pytest.mark.parametrize("partition", [0, -1])
def test_cascade_whole_sequence_in_the_prefix(pa, cuda_device, partition):
    """Members no longer than the shared prefix: the suffix pass has nothing
    to attend, and the prefix pass's result is the output.  Two groups of
    four whose members name the first four blocks of the group's longest
    member; no new tokens this step (all slots are padding)."""
    w = W.decode_batch(8, 1, 200, 32, 8, 128, seed=77,
                       lens=[200, 30, 64, 100, 150, 16, 48, 90], poison=True)
    bt = w.block_tables
    for g in (0, 1):
        for m in range(1, 4):
            bt[4 * g + m, :4] = bt[4 * g, :4]
    w.slot_mapping[:] = -1
    go = np.array([0, 4, 8], np.int32)
    pt = bt[[0, 4], :4].copy()
    sb = np.array([min(4, -(-int(n) // 16)) for n in w.seq_lens], np.int32)
    assert np.sum(16 * sb >= w.seq_lens) >= 4
    run(pa, cuda_device, w, 4, partition, go, pt, sb)


@pytest.mark.parametrize("partition", [0, 512])
def test_cascade_without_sharing_equals_decode(pa, cuda_device, partition):
    w = W.llama3_8b_layer()
    S = w.num_decode_seqs
    go = np.arange(0, S + 1, 2, dtype=np.int32)
    pt = np.full((S // 2, 1), -1, np.int32)
    run(pa, cuda_device, w, 2, partition, go, pt, np.zeros(S, np.int32))


def test_cascade_flags_bad_shared_blocks(pa, cuda_device):
    w = W.cow_mix(num_seqs=8, group=4, prefix_tokens=64, Hq=16, Hkv=4, D=128, max_len=200,
                  seed=5)
    go, pt, sb = W.cascade_groups(w, 4)
    sb = sb.copy()
    sb[1] = -3  # negative: clamped to 0 (nothing shared) and flagged
    run(pa, cuda_device, w, 4, 0, go, pt, sb, expect_flags=pa.PA_DEVERR_GROUP)
    pa.pa_device_error_flags(reset=True)


@pytest.mark.parametrize("partition", [512, 0])
def test_cascade_is_bitwise_deterministic(pa, cuda_device, partition):
    """The suffix pass of the copy-on-write mix is mostly one-block pieces:
    repeated launches must agree bit for bit."""
    w = W.cow_mix()
    go, pt, sb = W.cascade_groups(w, 4)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    args = [torch.from_numpy(x).to(cuda_device) for x in (go, pt, sb)]
    outs = []
    for _ in range(12):
        out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=cuda_device)
        ws = pa.alloc_workspace(pa.pa_cascade_workspace_size(S, Hq, 8, D, w.max_blocks_per_seq,
                                                             16, partition), cuda_device)
        pa.pa_cascade_decode(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, args[0], 4,
                             args[1], args[2], w.scale, partition_tokens=partition, workspace=ws)
        outs.append(out)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))

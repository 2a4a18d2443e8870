"""Metadata from the host block manager driving the GPU path.

A serving-style batch: groups of four requests share a 256-token system
prompt, so the prefix cache hands later members the first member's blocks;
one member per group is forked (parallel sampling), so the decode step's
appends copy the forked partial blocks on write.  The Python oracle manager
and the C++ manager run the same script and must agree exactly; the oracle's
metadata feeds the fp64 oracle, the C++ manager's identical metadata feeds
the kernels.  On the GPU: the prompt step's scatter, then the decode step's
pa_copy_blocks + scatter + pa_decode.  The pools must equal the oracle's bit
for bit, the outputs within the parity tolerance.  Pool slots nobody wrote
hold bf16 NaN, so a read of any of them would show.
"""
import numpy as np
import pytest
import torch

from oracle.block_manager import BlockManagerOracle, OK
from paged_kv_cache_218_gb300 import workload as W
from tests.gpu_common import assert_close, bits_to_dev, dev_to_bits

pytestmark = pytest.mark.gpu

B = 16
NAN_BF16 = np.uint16(0x7FC0)


def run_script(seed, groups=16, members=4, system_tokens=256, num_blocks=2048):
    from paged_kv_cache_218_gb300.block_manager import BlockManager
    rng = np.random.default_rng(seed)
    o = BlockManagerOracle(num_blocks, B, True)
    m = BlockManager(num_blocks, B, True)
    systems = [rng.integers(0, 32000, system_tokens).tolist() for _ in range(groups)]
    prompt_slots, cached_total = [], 0
    ids = []
    for g in range(groups):
        for k in range(members):
            sid = g * members + k
            n = int(np.clip(np.rint(np.exp(np.log(128.0) + rng.standard_normal())), 1, 1200))
            prompt = systems[g] + rng.integers(0, 32000, n).tolist()
            st, slots, cached = o.add_sequence(sid, prompt)
            slots2, cached2 = m.add_sequence(sid, prompt)
            assert st == OK and list(slots2) == slots and cached2 == cached
            prompt_slots += [s for s in slots if s >= 0]
            cached_total += cached
            ids.append(sid)
        fork_id = 10_000 + g
        assert o.fork(g * members, fork_id) == OK
        m.fork(g * members, fork_id)
        ids.append(fork_id)
    assert o.end_step() == [] and len(m.end_step()) == 0
    decode_slots = []
    for sid in ids:
        tok = int(rng.integers(0, 32000))
        st, slot = o.append_token(sid, tok)
        assert st == OK and m.append_token(sid, tok) == slot
        decode_slots.append(slot)
    pairs = o.end_step()
    pairs2 = m.end_step()
    assert [tuple(p) for p in pairs2.tolist()] == pairs
    max_blocks = max(len(o.seqs[i]["blocks"]) for i in ids)
    st, rows, lens = o.build_tables(ids, max_blocks)
    t2, l2 = m.build_tables(ids, max_blocks)
    assert st == OK and t2.tolist() == rows and l2.tolist() == lens
    m.close()
    return dict(ids=ids, prompt_slots=np.array(prompt_slots, np.int64),
                decode_slots=np.array(decode_slots, np.int64),
                pairs=np.array(pairs, np.int64).reshape(-1, 2),
                tables=np.array(rows, np.int32), lens=np.array(lens, np.int32),
                cached_total=cached_total, num_blocks=num_blocks)


@pytest.mark.parametrize("partition_tokens", [0, 512])
def test_block_manager_metadata_on_gpu(cuda_device, partition_tokens):
    import oracle
    from paged_kv_cache_218_gb300 import binding as pa
    md = run_script(seed=2024)
    # the script must really share prefixes (three members per group reuse the
    # 16 system-prompt blocks) and copy on write (a forked partial block)
    assert md["cached_total"] == 16 * 3 * 256 and md["pairs"].shape[0] >= 8
    Hq, Hkv, D = 32, 8, 128
    scale = 1.0 / np.sqrt(D)
    rng = np.random.default_rng(7)
    nb = md["num_blocks"]
    pool_k = np.full((nb, B, Hkv, D), NAN_BF16, np.uint16)
    pool_v = np.full((nb, B, Hkv, D), NAN_BF16, np.uint16)
    T0, S = md["prompt_slots"].shape[0], len(md["ids"])
    k0, v0 = W.normal_bf16(rng, (T0, Hkv, D)), W.normal_bf16(rng, (T0, Hkv, D))
    k1, v1 = W.normal_bf16(rng, (S, Hkv, D)), W.normal_bf16(rng, (S, Hkv, D))
    q = W.normal_bf16(rng, (S, Hq, D))

    # oracle: prompt step's scatter, then the decode step
    kc, vc = oracle.reshape_and_cache(k0, v0, pool_k, pool_v, md["prompt_slots"])
    kc, vc = oracle.copy_blocks(kc, vc, md["pairs"])
    kc, vc = oracle.reshape_and_cache(k1, v1, kc, vc, md["decode_slots"])
    ref, _ = oracle.decode(q, kc, vc, md["tables"], md["lens"], scale)

    dev = cuda_device
    dk, dv = bits_to_dev(pool_k, dev), bits_to_dev(pool_v, dev)
    pa.pa_reshape_and_cache(bits_to_dev(k0, dev), bits_to_dev(v0, dev), dk, dv,
                            torch.from_numpy(md["prompt_slots"]).to(dev))
    pa.pa_copy_blocks(dk, dv, torch.from_numpy(md["pairs"]).to(dev))
    pa.pa_reshape_and_cache(bits_to_dev(k1, dev), bits_to_dev(v1, dev), dk, dv,
                            torch.from_numpy(md["decode_slots"]).to(dev))
    tables = torch.from_numpy(md["tables"]).to(dev)
    lens = torch.from_numpy(md["lens"]).to(dev)
    out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, Hkv, D, tables.shape[1], B,
                                                        partition_tokens), dev)
    pa.pa_decode(out, bits_to_dev(q, dev), dk, dv, tables, lens, scale,
                 partition_tokens=partition_tokens, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(dev_to_bits(dk), kc) and np.array_equal(dev_to_bits(dv), vc)
    assert_close(out, ref, "decode over block-manager metadata")
    assert pa.pa_device_error_flags() == 0

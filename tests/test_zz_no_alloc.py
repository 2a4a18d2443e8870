"""pa_decode_noalloc: the balanced decode for callers that cannot allocate
device memory (a serving loop that must not call cudaMalloc on its hot path,
an engine whose memory is all reserved for the KV pool, a plain-C caller
without a framework allocator).  It draws its scratch from a static array
inside libpa.so instead of a caller workspace.

This file is collected last on purpose.  Through the C ABI it checks that two
calls in a row match the fp64 oracle within the tolerance the other parity
tests use, and give bit for bit what pa_decode gives with a workspace (the
same kernel and split); that a shape needing more than the static scratch is
refused before anything runs; and that a call refused for a bad argument
enqueues nothing that would disturb the next call.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_218_gb300 import workload as W
from tests.gpu_common import DeviceWorkload, assert_close, dev_to_bits, oracle_scattered

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa(cuda_device):
    from paged_kv_cache_218_gb300 import binding
    return binding


def _workspace_decode(pa, dw, device):
    w = dw.w
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    ref = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=device)
    ref_lse = torch.empty((S, Hq), dtype=torch.float32, device=device)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                        w.max_blocks_per_seq, 16, 0), device)
    pa.pa_decode(ref, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                 partition_tokens=0, out_lse=ref_lse, workspace=ws)
    return ref, ref_lse


@pytest.mark.parametrize("make", [W.llama3_8b_layer, W.tiny])
def test_noalloc_decode_matches_oracle_twice(pa, cuda_device, make):
    w = make()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    kc, vc = oracle_scattered(w)
    ref, ref_lse = oracle.decode(w.q[w.q_decode_row0:w.q_decode_row0 + w.num_decode_seqs], kc,
                                 vc, w.block_tables[w.decode_seq0:], w.seq_lens[w.decode_seq0:],
                                 w.scale)
    ws_out, ws_lse = _workspace_decode(pa, dw, cuda_device)
    for call in range(2):
        out = torch.full_like(ws_out, float("nan"))
        lse = torch.full_like(ws_lse, float("nan"))
        pa.pa_decode_noalloc(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                             out_lse=lse)
        torch.cuda.synchronize()
        assert_close(out, ref, f"no-alloc decode, call {call + 1}")
        assert_close(lse.cpu().numpy(), ref_lse, f"no-alloc lse, call {call + 1}")
        # the same kernel and split as pa_decode with a workspace: the same bits
        assert np.array_equal(dev_to_bits(out), dev_to_bits(ws_out))
        assert torch.equal(lse, ws_lse)
    assert pa.pa_device_error_flags() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch(pa, cuda_device):
    w = W.decode_batch(4, 16, 64, 64, 8, 128, seed=5)  # 64 q heads need more than 8 MiB
    dw = DeviceWorkload(w, cuda_device)
    out = torch.empty((4, 64, 128), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_noalloc(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens,
                             w.scale)
    assert e.value.status == pa.PA_ERR_SCRATCH_LIMIT


def test_noalloc_rejected_call_leaves_the_next_call_exact(pa, cuda_device):
    """A call refused for a bad argument (a non-finite scale, a too-long batch
    for the balanced split) returns its status before anything is enqueued;
    the valid call after it still matches the oracle."""
    w = W.tiny()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    kc, vc = oracle_scattered(w)
    ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    out = torch.full((4, 4, 64), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    for bad_scale in (float("nan"), float("inf"), -0.125):
        with pytest.raises(pa.PAError) as e:
            pa.pa_decode_noalloc(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                 dw.seq_lens, bad_scale)
        assert e.value.status == pa.PA_ERR_INVALID
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()  # nothing ran
    pa.pa_decode_noalloc(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens,
                         w.scale)
    torch.cuda.synchronize()
    assert_close(out, ref, "no-alloc decode after refused calls")
    assert pa.pa_device_error_flags() == 0

"""The kernels' bounded waits, run out on a GPU without a fault or a hang.

Every mbarrier wait in the decode and prefill kernels gives up after a time
limit, sets PA_DEVERR_TIMEOUT and lets the CTA skip the rest of its waits
and return.  pa_test_decode_stalled / pa_test_prefill_stalled make one launch
whose loaders issue no load at all, with a limit of a millisecond: every wait
then runs out with no copy in flight.  Each test checks that the error word
reads exactly PA_DEVERR_TIMEOUT, then that the next normal call on the same
stream (and, for the decode, the same workspace) matches the fp64 oracle.
"""
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
    binding.pa_device_error_flags(reset=True)
    return binding


@pytest.mark.parametrize("partition_tokens", [0, -1, 512])
def test_decode_wait_runs_out_then_next_call_exact(pa, cuda_device, partition_tokens):
    w = W.llama3_8b_layer()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags(reset=True) == 0
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                        w.max_blocks_per_seq, 16,
                                                        partition_tokens), cuda_device)
    out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=cuda_device)
    pa.pa_test_decode_stalled(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                              partition_tokens=partition_tokens, workspace=ws,
                              wait_limit_us=1000)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags(reset=True) == pa.PA_DEVERR_TIMEOUT
    # the same stream and workspace: the next call is exact
    out.fill_(float("nan"))
    pa.pa_decode(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                 partition_tokens=partition_tokens, workspace=ws)
    torch.cuda.synchronize()
    kc, vc = oracle_scattered(w)
    ref, _ = oracle.decode(w.q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    assert_close(out, ref, f"decode after a stalled launch (partition_tokens={partition_tokens})")
    assert pa.pa_device_error_flags() == 0


def test_prefill_wait_runs_out_then_next_call_exact(pa, cuda_device):
    w = W.prefill_batch([(0, 40), (100, 300)], Hq=16, Hkv=4, D=128, seed=71, poison=True)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags(reset=True) == 0
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    max_q = int(np.max(np.diff(w.cu_q_lens)))
    cu = torch.from_numpy(w.cu_q_lens).to(cuda_device)
    qs = torch.from_numpy(w.q_start_pos).to(cuda_device)
    out = torch.empty((T, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=cuda_device)
    pa.pa_test_prefill_stalled(out, dw.q[:T], dw.k_cache, dw.v_cache, dw.block_tables[:C], cu,
                               qs, dw.seq_lens[:C], max_q, w.scale, wait_limit_us=1000)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags(reset=True) == pa.PA_DEVERR_TIMEOUT
    out.fill_(float("nan"))
    pa.pa_prefill_chunk(out, dw.q[:T], dw.k_cache, dw.v_cache, dw.block_tables[:C], cu, qs,
                        dw.seq_lens[:C], max_q, w.scale)
    torch.cuda.synchronize()
    kc, vc = oracle_scattered(w)
    ref, _ = oracle.prefill(w.q[:T], kc, vc, w.block_tables[:C], w.cu_q_lens, w.q_start_pos,
                            w.seq_lens[:C], w.scale)
    assert_close(out, ref, "prefill after a stalled launch")
    assert pa.pa_device_error_flags() == 0


def test_stalled_launch_limit_is_checked(pa, cuda_device):
    w = W.tiny()
    dw = DeviceWorkload(w, cuda_device)
    out = torch.empty((4, 4, 64), dtype=torch.bfloat16, device=cuda_device)
    for bad in (0, 2_000_001):
        with pytest.raises(pa.PAError) as e:
            pa.pa_test_decode_stalled(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables,
                                      dw.seq_lens, w.scale, partition_tokens=-1,
                                      wait_limit_us=bad)
        assert e.value.status == pa.PA_ERR_INVALID

"""pa_decode_noalloc: the balanced decode for callers that cannot allocate
device memory (a serving loop that must not call cudaMalloc on its hot path,
an engine whose memory is all reserved for the KV pool, a plain-C caller
without a framework allocator).  It draws its scratch from a static array
inside libpa.so instead of a caller workspace.

This file is collected last on purpose.  It checks, through the C ABI, that
two calls in a row give the same result as pa_decode with a workspace, within
the tolerance the other parity tests use, and that a shape needing more than
the static scratch is refused before anything runs.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_218_gb300 import workload as W
from tests.gpu_common import DeviceWorkload, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa(cuda_device):
    from paged_kv_cache_218_gb300 import binding
    return binding


@pytest.mark.parametrize("make", [W.llama3_8b_layer, W.tiny])
def test_noalloc_decode_matches_workspace_decode_twice(pa, cuda_device, make):
    w = make()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    ref = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=cuda_device)
    ref_lse = torch.empty((S, Hq), dtype=torch.float32, device=cuda_device)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                        w.max_blocks_per_seq, 16, 0), cuda_device)
    pa.pa_decode(ref, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                 partition_tokens=0, out_lse=ref_lse, workspace=ws)
    torch.cuda.synchronize()
    ref64 = ref.float().cpu().numpy().astype(np.float64)
    ref_lse64 = ref_lse.cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        pa.pa_decode_noalloc(out, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                             out_lse=lse)
        torch.cuda.synchronize()
        assert_close(out, ref64, f"no-alloc decode, call {call + 1}")
        assert_close(lse.cpu().numpy(), ref_lse64, f"no-alloc lse, call {call + 1}")
    assert pa.pa_device_error_flags() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch(pa, cuda_device):
    w = W.decode_batch(4, 16, 64, 64, 8, 128, seed=5)  # 64 q heads need more than 8 MiB
    dw = DeviceWorkload(w, cuda_device)
    out = torch.empty((4, 64, 128), dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_noalloc(out, dw.q, dw.k_cache, dw.v_cache, dw.block_tables, dw.seq_lens,
                             w.scale)
    assert e.value.status == pa.PA_ERR_SCRATCH_LIMIT

"""GPU parity of the tcgen05 causal prefill chunk and of the Sarathi hybrid
step (chunk + decodes under one token budget) against the fp64 oracle."""
import functools

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


def _prefill(pa, dw, with_lse=True, stream=None):
    w = dw.w
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    q = dw.q[:T]
    out = torch.full((T, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16,
                     device=q.device)
    lse = torch.full((T, w.num_q_heads), float("nan"), dtype=torch.float32, device=q.device) \
        if with_lse else None
    max_q = int(np.max(np.diff(w.cu_q_lens)))
    dev = q.device
    pa.pa_prefill_chunk(out, q, dw.k_cache, dw.v_cache, dw.block_tables[:C],
                        torch.from_numpy(w.cu_q_lens).to(dev),
                        torch.from_numpy(w.q_start_pos).to(dev), dw.seq_lens[:C], max_q,
                        w.scale, out_lse=lse, stream=stream)
    return out, lse


def _oracle_prefill(w):
    kc, vc = oracle_scattered(w)
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    return oracle.prefill(w.q[:T], kc, vc, w.block_tables[:C], w.cu_q_lens, w.q_start_pos,
                          w.seq_lens[:C], w.scale)


CHUNKS = [
    # (chunks [(start, len)], Hq, Hkv, seed)
    ([(0, 40)], 8, 2, 1),                                # one chunk from position 0, group 4
    ([(0, 37), (40, 25), (7, 1), (100, 130)], 8, 2, 2),  # ragged starts and lengths
    ([(0, 128), (128, 128)], 8, 8, 3),                   # group 1: 128 tokens per tile
    ([(5, 77), (300, 19)], 16, 8, 4),                    # group 2
    ([(33, 200), (0, 16), (250, 3)], 32, 4, 5),          # group 8: 16 tokens per tile
    ([(1000, 300)], 16, 4, 6),                           # long prefix, several key tiles
]


@pytest.mark.parametrize("chunks,Hq,Hkv,seed", CHUNKS)
def test_prefill_chunks_match_oracle(pa, cuda_device, chunks, Hq, Hkv, seed):
    w = W.prefill_batch(chunks, Hq=Hq, Hkv=Hkv, D=128, seed=700 + seed, poison=True)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse = _prefill(pa, dw)
    torch.cuda.synchronize()
    ref, ref_lse = _oracle_prefill(w)
    assert torch.isfinite(out).all()
    assert_close(out, ref, f"prefill {chunks} G={Hq // Hkv}")
    assert_close(lse.cpu().numpy(), ref_lse, "prefill lse")
    assert pa.pa_device_error_flags() == 0


# Positions of a planted dominant key: both ends of every 32-column group of
# both 64-column halves of key tiles 0 and 1, which every query row of the
# chunk sees whole (the row maximum comes from the tensor-memory load there),
# and one key of the chunk itself on the causal diagonal (a masked half,
# hidden from the chunk's first five rows).
DOMINANT_KEYS = [0, 31, 32, 63, 64, 95, 96, 127, 128, 159, 160, 191, 192, 223, 224, 255, 261]


def _dominant_workload(kpos):
    """Queries all 1 and one key all 16: its scaled score, 2048 / sqrt(128)
    (about 261 in log2 units), exceeds every other score of a row by more
    than 128 in log2 units, so its 2^(s - m) overflows fp32 unless the row
    maximum m includes it."""
    w = W.prefill_batch([(256, 32)], Hq=8, Hkv=2, D=128, seed=910)
    w.q[:] = W.f32_to_bf16_bits(np.float32(1.0))
    big = W.f32_to_bf16_bits(np.float32(16.0))
    if kpos < 256:
        w.k_cache[w.block_tables[0, kpos // 16], kpos % 16] = big
    else:
        w.key[kpos - 256] = big
    return w


@pytest.mark.parametrize("kpos", DOMINANT_KEYS)
def test_prefill_dominant_key_in_every_column(pa, cuda_device, kpos):
    w = _dominant_workload(kpos)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse = _prefill(pa, dw)
    torch.cuda.synchronize()
    ref, ref_lse = _oracle_prefill(w)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    assert_close(out, ref, f"dominant key at position {kpos}")
    assert_close(lse.cpu().numpy(), ref_lse, f"dominant key at position {kpos}: lse")
    assert pa.pa_device_error_flags() == 0


@pytest.mark.parametrize("chunk,Hq,Hkv", [((1536, 64), 8, 2), ((200, 333), 16, 2)])
def test_prefill_row_maximum_moving_at_every_tile(pa, cuda_device, chunk, Hq, Hkv):
    """Queries all 1 and every key of key tile t equal to 0.75 t (bf16-exact):
    a key of tile t scores 128 * 0.75 t / sqrt(128), about 12.2 t in log2
    units, so each tile's scores exceed the previous tile's by more than the
    kernel's rescale threshold and the running maximum, the sum and O are
    rescaled at every tile."""
    w = W.prefill_batch([chunk], Hq=Hq, Hkv=Hkv, D=128, seed=930)
    w.q[:] = W.f32_to_bf16_bits(np.float32(1.0))
    p0, n = chunk
    for pos in range(p0 + n):
        val = W.f32_to_bf16_bits(np.float32(0.75 * (pos // 128)))
        if pos < p0:
            w.k_cache[w.block_tables[0, pos // 16], pos % 16] = val
        else:
            w.key[pos - p0] = val
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse = _prefill(pa, dw)
    torch.cuda.synchronize()
    ref, ref_lse = _oracle_prefill(w)
    assert torch.isfinite(out).all()
    assert_close(out, ref, f"maximum moving every tile {chunk}")
    assert_close(lse.cpu().numpy(), ref_lse, "maximum moving every tile: lse")
    assert pa.pa_device_error_flags() == 0


@functools.lru_cache(maxsize=None)
def _hybrid():
    w = W.sarathi_hybrid()
    kc, vc = oracle_scattered(w)
    ref_c, ref_c_lse = oracle.prefill(w.chunk_q, kc, vc, w.block_tables[:1], w.cu_q_lens,
                                      w.q_start_pos, w.seq_lens[:1], w.scale)
    ref_d, _ = oracle.decode(w.decode_q, kc, vc, w.decode_block_tables, w.decode_seq_lens,
                             w.scale)
    return w, ref_c, ref_c_lse, ref_d


def test_sarathi_chunk_matches_oracle(pa, cuda_device):
    w, ref_c, ref_c_lse, _ = _hybrid()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, lse = _prefill(pa, dw)
    torch.cuda.synchronize()
    assert_close(out, ref_c, "sarathi chunk")
    assert_close(lse.cpu().numpy(), ref_c_lse, "sarathi chunk lse")


def test_sarathi_hybrid_step_on_two_streams(pa, cuda_device):
    """Scatter the 640 new tokens, then run the chunk and the 128 decodes
    concurrently on two streams; both results match the oracle."""
    w, ref_c, _, ref_d = _hybrid()
    dw = DeviceWorkload(w, cuda_device)
    main = torch.cuda.current_stream()
    s_chunk, s_dec = torch.cuda.Stream(), torch.cuda.Stream()
    dw.scatter(pa)
    ready = torch.cuda.Event()
    ready.record(main)
    s_chunk.wait_event(ready)
    s_dec.wait_event(ready)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    out_d = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=cuda_device)
    ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                        w.max_blocks_per_seq, 16, 0),
                            cuda_device)
    with torch.cuda.stream(s_chunk):
        out_c, _ = _prefill(pa, dw, with_lse=False, stream=s_chunk)
    with torch.cuda.stream(s_dec):
        pa.pa_decode(out_d, dw.dq, dw.k_cache, dw.v_cache, dw.dtables, dw.dlens, w.scale,
                     partition_tokens=0, workspace=ws, stream=s_dec)
    main.wait_stream(s_chunk)
    main.wait_stream(s_dec)
    torch.cuda.synchronize()
    assert_close(out_c, ref_c, "hybrid chunk")
    assert_close(out_d, ref_d, "hybrid decode")
    assert pa.pa_device_error_flags() == 0


def test_prefill_query_equals_decode_of_its_prefix(pa, cuda_device):
    """The chunk's query at position p and a decode with seq_len p + 1 over the
    same cache agree (two different kernels)."""
    w = W.prefill_batch([(50, 60)], Hq=8, Hkv=2, D=128, seed=41)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    out, _ = _prefill(pa, dw, with_lse=False)
    rows = [0, 17, 59]
    q = dw.q[rows]
    lens = torch.tensor([50 + r + 1 for r in rows], dtype=torch.int32, device=cuda_device)
    tables = dw.block_tables[[0, 0, 0]]
    out_d = torch.empty((3, 8, 128), dtype=torch.bfloat16, device=cuda_device)
    pa.pa_decode(out_d, q, dw.k_cache, dw.v_cache, tables, lens, w.scale, partition_tokens=-1)
    torch.cuda.synchronize()
    diff = (out[rows].float() - out_d.float()).abs().max().item()
    assert diff <= 2e-2


def test_prefill_flags_inconsistent_chunks(pa, cuda_device):
    w = W.prefill_batch([(0, 20), (10, 20)], Hq=8, Hkv=2, D=128, seed=9)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    bad_start = w.q_start_pos.copy()
    bad_start[1] = 25  # 25 + 20 > seq_len 30
    w2 = W.Workload(**{**w.__dict__, "q_start_pos": bad_start})
    dw.w = w2
    out, _ = _prefill(pa, dw, with_lse=False)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags() & pa.PA_DEVERR_CHUNK
    ref, _ = _oracle_prefill(w)
    assert_close(out[:20], ref[:20], "good chunk beside a bad one")


def test_prefill_flags_block_ids_outside_the_pool(pa, cuda_device):
    # chunk 0: an id past the pool in its first K/V tile (ids read ahead of
    # the set-up); chunk 1: a negative id in its third tile (ids read with the
    # tile); chunk 2 is clean and must stay exact.  Bad ids read as zeros.
    w = W.prefill_batch([(0, 40), (300, 20), (100, 50)], Hq=8, Hkv=2, D=128, seed=11)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    nb = dw.k_cache.shape[0]
    bt = w.block_tables[:C].copy()
    bt[0, 1] = nb + 5
    bt[1, 17] = -7
    out = torch.full((T, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16,
                     device=cuda_device)
    pa.pa_device_error_flags(reset=True)
    pa.pa_prefill_chunk(out, dw.q[:T], dw.k_cache, dw.v_cache, torch.from_numpy(bt).to(cuda_device),
                        torch.from_numpy(w.cu_q_lens).to(cuda_device),
                        torch.from_numpy(w.q_start_pos).to(cuda_device), dw.seq_lens[:C],
                        int(np.max(np.diff(w.cu_q_lens))), w.scale)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags() & pa.PA_DEVERR_BLOCK_ID
    ref, _ = _oracle_prefill(w)
    r2 = slice(int(w.cu_q_lens[2]), int(w.cu_q_lens[3]))
    assert_close(out[r2], ref[r2], "clean chunk beside chunks with bad block ids")
    assert bool(torch.isfinite(out).all()), "bad block ids must read as zeros, not garbage"


def test_prefill_flags_chunk_rows_past_the_query_tensor(pa, cuda_device):
    # the second chunk's rows end past total_q_tokens: it is skipped (no row
    # beyond the output tensor is written) and the first chunk is still exact
    w = W.prefill_batch([(0, 20), (10, 20)], Hq=8, Hkv=2, D=128, seed=10)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    # chunk 1 (30 tokens in its sequence) claims rows 20 .. 49 from position 0:
    # consistent with its sequence, but T = 40 rows exist
    cu_bad = w.cu_q_lens.copy()
    cu_bad[C] = T + 10
    start_bad = w.q_start_pos.copy()
    start_bad[1] = 0
    Hq, D = w.num_q_heads, w.head_dim
    buf = torch.full((T + 64, Hq, D), 7.0, dtype=torch.bfloat16, device=cuda_device)
    pa.pa_device_error_flags(reset=True)
    pa.pa_prefill_chunk(buf[:T], dw.q[:T], dw.k_cache, dw.v_cache, dw.block_tables[:C],
                        torch.from_numpy(cu_bad).to(cuda_device),
                        torch.from_numpy(start_bad).to(cuda_device), dw.seq_lens[:C], 30,
                        w.scale)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags() & pa.PA_DEVERR_CHUNK
    assert bool((buf[T:] == 7.0).all()), "rows past the tensor were written"
    assert bool((buf[20:T] == 7.0).all()), "the skipped chunk wrote rows"
    ref, _ = _oracle_prefill(w)
    assert_close(buf[:20], ref[:20], "good chunk beside one past the tensor")


def test_prefill_rejects_unsupported_shapes(pa, cuda_device):
    w = W.prefill_batch([(0, 20)], Hq=6, Hkv=2, D=128, seed=10)  # group 3 does not tile 128 rows
    dw = DeviceWorkload(w, cuda_device)
    with pytest.raises(pa.PAError) as e:
        _prefill(pa, dw)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def _hybrid_call(pa, dw, ws, chunk_sms=0, with_lse=True):
    w = dw.w
    dev = dw.q.device
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    out_c = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    out_d = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse_c = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    lse_d = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=dev) if with_lse else None
    pa.pa_hybrid_attention(out_c, dw.q[:T], dw.block_tables[:C],
                           torch.from_numpy(w.cu_q_lens).to(dev),
                           torch.from_numpy(w.q_start_pos).to(dev), dw.seq_lens[:C],
                           int(np.max(np.diff(w.cu_q_lens))), out_d, dw.dq, dw.dtables, dw.dlens,
                           dw.k_cache, dw.v_cache, w.scale, ws, chunk_sms=chunk_sms,
                           chunk_lse=lse_c, decode_lse=lse_d)
    return out_c, out_d, lse_c, lse_d


def _hybrid_ws(pa, w, dev):
    return pa.alloc_workspace(pa.pa_hybrid_workspace_size(
        w.num_decode_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq), dev)


@pytest.mark.parametrize("chunk_sms", [0, 1, 8, 32, 64, 151, 1000])
def test_sarathi_hybrid_co_scheduled_matches_oracle(pa, cuda_device, chunk_sms):
    """pa_hybrid_attention, one launch: the decode on its first CTAs, the
    chunk's tile pairs on the rest; both match the oracle, and the chunk is
    bit for bit the output of pa_prefill_chunk (the same CTA-pair tiles)."""
    w, ref_c, ref_c_lse, ref_d = _hybrid()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    ws = _hybrid_ws(pa, w, cuda_device)
    out_c, out_d, lse_c, lse_d = _hybrid_call(pa, dw, ws, chunk_sms)
    alone, alone_lse = _prefill(pa, dw)
    torch.cuda.synchronize()
    assert_close(out_c, ref_c, f"co-scheduled chunk, chunk_sms {chunk_sms}")
    assert_close(lse_c.cpu().numpy(), ref_c_lse, "co-scheduled chunk lse")
    assert_close(out_d, ref_d, f"co-scheduled decode, chunk_sms {chunk_sms}")
    assert torch.isfinite(lse_d).all()
    assert torch.equal(out_c.view(torch.int16), alone.view(torch.int16))
    assert torch.equal(lse_c, alone_lse)
    assert pa.pa_device_error_flags() == 0


def test_sarathi_hybrid_co_scheduled_repeats_and_leaves_workspace_zeroed(pa, cuda_device):
    """Ten calls in a row on one workspace (the decode's tickets reset
    themselves, the reserved head stays zero); every call gives the same
    bits."""
    w, _, _, ref_d = _hybrid()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    ws = _hybrid_ws(pa, w, cuda_device)
    outs = [_hybrid_call(pa, dw, ws, 32, with_lse=False)[:2] for _ in range(10)]
    torch.cuda.synchronize()
    for c, d in outs[1:]:
        assert torch.equal(c.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(d.view(torch.int16), outs[0][1].view(torch.int16))
    assert_close(outs[-1][1], ref_d, "repeated co-scheduled decode")
    assert int(ws[:256].count_nonzero()) == 0
    assert pa.pa_device_error_flags() == 0


def test_hybrid_without_chunks_or_decodes(pa, cuda_device):
    """With no decode the call is the chunk alone; with no chunk, the decode
    alone; both still match the oracle."""
    w, ref_c, _, ref_d = _hybrid()
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    dev = cuda_device
    ws = _hybrid_ws(pa, w, dev)
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    # no decodes
    out_c = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    none_d = torch.empty((0, Hq, D), dtype=torch.bfloat16, device=dev)
    pa.pa_hybrid_attention(out_c, dw.q[:T], dw.block_tables[:C],
                           torch.from_numpy(w.cu_q_lens).to(dev),
                           torch.from_numpy(w.q_start_pos).to(dev), dw.seq_lens[:C],
                           int(np.max(np.diff(w.cu_q_lens))), none_d, none_d,
                           dw.dtables[:0], dw.dlens[:0], dw.k_cache, dw.v_cache, w.scale, ws)
    # no chunks
    out_d = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=dev)
    none_c = torch.empty((0, Hq, D), dtype=torch.bfloat16, device=dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.pa_hybrid_attention(none_c, none_c, dw.block_tables[:1], zero, zero[:0], zero[:0], 0,
                           out_d, dw.dq, dw.dtables, dw.dlens, dw.k_cache, dw.v_cache, w.scale, ws)
    torch.cuda.synchronize()
    assert_close(out_c, ref_c, "hybrid call, chunk only")
    assert_close(out_d, ref_d, "hybrid call, decode only")
    assert pa.pa_device_error_flags() == 0


def test_hybrid_rejects_bad_arguments_before_launching(pa, cuda_device):
    w, _, _, _ = _hybrid()
    dw = DeviceWorkload(w, cuda_device)
    ws = _hybrid_ws(pa, w, cuda_device)
    small = ws[:256]
    with pytest.raises(pa.PAError) as e:
        _hybrid_call(pa, dw, small)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    with pytest.raises(pa.PAError) as e:
        _hybrid_call(pa, dw, ws, chunk_sms=-1)
    assert e.value.status == pa.PA_ERR_INVALID
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags() == 0


HYBRID_SHAPES = [
    # (chunk_tokens, chunk_start, num_decode, dec_lo, dec_hi, Hq, Hkv, seed)
    (96, 200, 20, 1, 300, 16, 8, 1),     # group 2, decodes from one token up
    (130, 0, 50, 16, 700, 32, 4, 2),     # group 8, chunk from position 0, a ragged tile
    (1, 5000, 300, 100, 2000, 8, 8, 3),  # group 1, a one-token chunk beside many decodes
    (256, 64, 7, 2000, 9000, 32, 8, 4),  # group 4, few long decodes: pieces split across CTAs
]


@pytest.mark.parametrize("ct,cs,nd,lo,hi,Hq,Hkv,seed", HYBRID_SHAPES)
def test_hybrid_one_launch_shapes_match_oracle(pa, cuda_device, ct, cs, nd, lo, hi, Hq, Hkv,
                                               seed):
    """The one-launch hybrid kernel (decode CTAs and prefill CTA pairs in one
    grid) on other shapes than the Sarathi batch, NaN in every unused slot:
    both results match the oracle, at the default chunk share and at a
    narrow one."""
    w = W.sarathi_hybrid(seed=900 + seed, poison=True, chunk_tokens=ct, chunk_start=cs,
                         num_decode=nd, dec_lo=lo, dec_hi=hi, Hq=Hq, Hkv=Hkv, D=128)
    kc, vc = oracle_scattered(w)
    ref_c, ref_c_lse = oracle.prefill(w.chunk_q, kc, vc, w.block_tables[:1], w.cu_q_lens,
                                      w.q_start_pos, w.seq_lens[:1], w.scale)
    ref_d, ref_d_lse = oracle.decode(w.decode_q, kc, vc, w.decode_block_tables,
                                     w.decode_seq_lens, w.scale)
    dw = DeviceWorkload(w, cuda_device)
    dw.scatter(pa)
    ws = _hybrid_ws(pa, w, cuda_device)
    for chunk_sms in (0, 8):
        out_c, out_d, lse_c, lse_d = _hybrid_call(pa, dw, ws, chunk_sms)
        torch.cuda.synchronize()
        what = f"hybrid G={Hq // Hkv} chunk {ct}@{cs} decodes {nd}, chunk_sms {chunk_sms}"
        assert_close(out_c, ref_c, what + " chunk")
        assert_close(lse_c.cpu().numpy(), ref_c_lse, what + " chunk lse")
        assert_close(out_d, ref_d, what + " decodes")
        assert_close(lse_d.cpu().numpy(), ref_d_lse, what + " decodes lse")
    assert int(ws[:256].count_nonzero()) == 0
    assert pa.pa_device_error_flags() == 0

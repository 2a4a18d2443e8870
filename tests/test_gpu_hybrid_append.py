"""pa_hybrid_attention_append: a Sarathi hybrid step with its slot scatter in
the same launch.

The step's new rows go into their slots ("03 - Engines Papers", section 2
PagedAttention: the step's K/V are written into the blocks, then attention
gathers them) while the chunk and the decodes attend ("03 - Engines Papers",
section 3 Sarathi / Sarathi-Serve).  Checked bit for bit against
pa_reshape_and_cache followed by pa_hybrid_attention (both pools, both
outputs, both lse arrays), and elementwise against the fp64 oracle.  The
pools' copies of every new slot hold NaN beforehand, so the launch must
attend the rows it was given, not what the pool held there."""
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


def _poisoned_pools(w):
    """The pools with NaN in every slot the step writes."""
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    for slot in w.slot_mapping:
        if slot >= 0:
            b, o = divmod(int(slot), 16)
            kc[b, o] = W.BF16_NAN
            vc[b, o] = W.BF16_NAN
    return kc, vc


def _outputs(w, dev):
    T = int(w.cu_q_lens[w.num_chunks])
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    nan = float("nan")
    return (torch.full((T, Hq, D), nan, dtype=torch.bfloat16, device=dev),
            torch.full((S, Hq, D), nan, dtype=torch.bfloat16, device=dev),
            torch.full((T, Hq), nan, dtype=torch.float32, device=dev),
            torch.full((S, Hq), nan, dtype=torch.float32, device=dev))


def _ws(pa, w, dev):
    return pa.alloc_workspace(pa.pa_hybrid_workspace_size(
        w.num_decode_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.max_blocks_per_seq), dev)


def _fused(pa, w, dev, chunk_sms=0, ws=None, key=None, value=None):
    """The fused step on fresh device pools whose new slots hold NaN."""
    kc0, vc0 = _poisoned_pools(w)
    kc, vc = bits_to_dev(kc0, dev), bits_to_dev(vc0, dev)
    q = bits_to_dev(w.q, dev)
    key = bits_to_dev(w.key, dev) if key is None else key
    value = bits_to_dev(w.value, dev) if value is None else value
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    s0 = w.decode_seq0
    out_c, out_d, lse_c, lse_d = _outputs(w, dev)
    ws = _ws(pa, w, dev) if ws is None else ws
    pa.pa_hybrid_attention_append(
        out_c, q[:T], key[:T], value[:T], bt[:C], torch.from_numpy(w.cu_q_lens).to(dev),
        torch.from_numpy(w.q_start_pos).to(dev), sl[:C], int(np.max(np.diff(w.cu_q_lens))),
        out_d, q[T:T + w.num_decode_seqs], key[T:], value[T:], bt[s0:], sl[s0:], kc, vc,
        w.scale, ws, chunk_sms=chunk_sms, chunk_lse=lse_c, decode_lse=lse_d)
    return out_c, out_d, lse_c, lse_d, kc, vc, ws


def _two_launches(pa, w, dev, chunk_sms=0):
    """pa_reshape_and_cache, then pa_hybrid_attention."""
    dw = DeviceWorkload(w, dev)
    dw.scatter(pa)
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    out_c, out_d, lse_c, lse_d = _outputs(w, dev)
    pa.pa_hybrid_attention(out_c, dw.q[:T], dw.block_tables[:C],
                           torch.from_numpy(w.cu_q_lens).to(dev),
                           torch.from_numpy(w.q_start_pos).to(dev), dw.seq_lens[:C],
                           int(np.max(np.diff(w.cu_q_lens))), out_d, dw.dq, dw.dtables, dw.dlens,
                           dw.k_cache, dw.v_cache, w.scale, _ws(pa, w, dev), chunk_sms=chunk_sms,
                           chunk_lse=lse_c, decode_lse=lse_d)
    return out_c, out_d, lse_c, lse_d, dw.k_cache, dw.v_cache


SHAPES = [
    # (chunk_tokens, chunk_start, num_decode, dec_lo, dec_hi, Hq, Hkv, seed); every
    # chunk starts a block
    (512, 1536, 128, 256, 4096, 32, 8, 0),  # the Sarathi batch
    (96, 208, 20, 1, 300, 16, 8, 1),        # group 2, decodes from one token up
    (130, 0, 50, 16, 700, 32, 4, 2),        # group 8, chunk from position 0, a ragged tile
    (1, 4992, 300, 100, 2000, 8, 8, 3),     # group 1, a one-token chunk beside many decodes
    (250, 64, 7, 2000, 9000, 32, 8, 4),     # group 4, few long decodes, a ragged last block
    (64, 32, 5, 10, 400, 8, 1, 5),          # one kv head, group 8
    (48, 16, 6, 10, 300, 4, 2, 6),          # two kv heads, group 2
]


@pytest.mark.parametrize("ct,cs,nd,lo,hi,Hq,Hkv,seed", SHAPES)
def test_fused_step_equals_scatter_then_hybrid(pa, cuda_device, ct, cs, nd, lo, hi, Hq, Hkv,
                                               seed):
    w = W.sarathi_hybrid(seed=950 + seed, poison=True, chunk_tokens=ct, chunk_start=cs,
                         num_decode=nd, dec_lo=lo, dec_hi=hi, Hq=Hq, Hkv=Hkv, D=128)
    kc_ref, vc_ref = oracle_scattered(w)
    ref_c, ref_c_lse = oracle.prefill(w.chunk_q, kc_ref, vc_ref, w.block_tables[:1],
                                      w.cu_q_lens, w.q_start_pos, w.seq_lens[:1], w.scale)
    ref_d, ref_d_lse = oracle.decode(w.decode_q, kc_ref, vc_ref, w.decode_block_tables,
                                     w.decode_seq_lens, w.scale)
    for chunk_sms in (0, 8):
        fc, fd, flc, fld, fk, fv, ws = _fused(pa, w, cuda_device, chunk_sms)
        tc, td, tlc, tld, tk, tv = _two_launches(pa, w, cuda_device, chunk_sms)
        torch.cuda.synchronize()
        what = f"fused hybrid G={Hq // Hkv} chunk {ct}@{cs} decodes {nd}, chunk_sms {chunk_sms}"
        # the pools, every byte (poison outside the written slots included)
        assert np.array_equal(dev_to_bits(fk), kc_ref), what + ": K pool"
        assert np.array_equal(dev_to_bits(fv), vc_ref), what + ": V pool"
        assert np.array_equal(dev_to_bits(fk), dev_to_bits(tk))
        # the two launches' results, bit for bit
        assert np.array_equal(dev_to_bits(fc), dev_to_bits(tc)), what + ": chunk bits"
        assert np.array_equal(dev_to_bits(fd), dev_to_bits(td)), what + ": decode bits"
        assert torch.equal(flc, tlc) and torch.equal(fld, tld), what + ": lse bits"
        # and the oracle
        assert_close(fc, ref_c, what + " chunk")
        assert_close(flc.cpu().numpy(), ref_c_lse, what + " chunk lse")
        assert_close(fd, ref_d, what + " decodes")
        assert_close(fld.cpu().numpy(), ref_d_lse, what + " decodes lse")
        assert int(ws[:256].count_nonzero()) == 0
    assert pa.pa_device_error_flags() == 0


def test_fused_step_repeats_bit_for_bit(pa, cuda_device):
    """Ten fused steps in a row on one workspace give the same bits."""
    w = W.sarathi_hybrid()
    dev = cuda_device
    ws = _ws(pa, w, dev)
    outs = [_fused(pa, w, dev, 32, ws=ws)[:2] for _ in range(10)]
    torch.cuda.synchronize()
    for c, d in outs[1:]:
        assert torch.equal(c.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(d.view(torch.int16), outs[0][1].view(torch.int16))
    assert int(ws[:256].count_nonzero()) == 0
    assert pa.pa_device_error_flags() == 0


def test_fused_step_without_decodes_or_chunk(pa, cuda_device):
    """No decodes: the launch is the chunk alone (its new rows written too);
    no chunk: the call is pa_decode_append."""
    w = W.sarathi_hybrid(seed=961, poison=True, chunk_tokens=200, chunk_start=96, num_decode=9,
                         dec_lo=20, dec_hi=900, Hq=16, Hkv=4, D=128)
    dev = cuda_device
    kc_ref, vc_ref = oracle_scattered(w)
    ref_c, _ = oracle.prefill(w.chunk_q, kc_ref, vc_ref, w.block_tables[:1], w.cu_q_lens,
                              w.q_start_pos, w.seq_lens[:1], w.scale)
    ref_d, _ = oracle.decode(w.decode_q, kc_ref, vc_ref, w.decode_block_tables,
                             w.decode_seq_lens, w.scale)
    kc0, vc0 = _poisoned_pools(w)
    q, key, value = (bits_to_dev(a, dev) for a in (w.q, w.key, w.value))
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    T, S, Hq, D = 200, 9, 16, 128
    cu = torch.from_numpy(w.cu_q_lens).to(dev)
    qs = torch.from_numpy(w.q_start_pos).to(dev)
    # the chunk alone (no workspace needed)
    kc, vc = bits_to_dev(kc0, dev), bits_to_dev(vc0, dev)
    out_c = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    none = torch.empty((0, Hq, D), dtype=torch.bfloat16, device=dev)
    none_kv = key[:0]
    pa.pa_hybrid_attention_append(out_c, q[:T], key[:T], value[:T], bt[:1], cu, qs, sl[:1], T,
                                  none, none, none_kv, none_kv, bt[1:1], sl[1:1], kc, vc,
                                  w.scale, None)
    torch.cuda.synchronize()
    assert_close(out_c, ref_c, "fused call, chunk only")
    rows = [int(s) for s in w.slot_mapping[:T]]
    kb = dev_to_bits(kc).reshape(-1, *kc_ref.shape[2:])
    assert np.array_equal(kb[rows], kc_ref.reshape(-1, *kc_ref.shape[2:])[rows])
    # the decodes alone
    kc, vc = bits_to_dev(kc0, dev), bits_to_dev(vc0, dev)
    out_d = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=dev)
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.pa_hybrid_attention_append(none, none, none_kv, none_kv, bt[:1], zero, zero[:0],
                                  zero[:0], 0, out_d, q[T:], key[T:], value[T:], bt[1:], sl[1:],
                                  kc, vc, w.scale, _ws(pa, w, dev))
    torch.cuda.synchronize()
    assert_close(out_d, ref_d, "fused call, decodes only")
    rows = [int(s) for s in w.slot_mapping[T:]]
    kb = dev_to_bits(kc).reshape(-1, *kc_ref.shape[2:])
    assert np.array_equal(kb[rows], kc_ref.reshape(-1, *kc_ref.shape[2:])[rows])
    assert pa.pa_device_error_flags() == 0


def test_fused_step_flags_a_chunk_that_does_not_start_a_block(pa, cuda_device):
    """A chunk starting inside a block cannot read its own keys from its new
    rows: it is skipped and flagged, and the decodes are still exact."""
    w = W.sarathi_hybrid(seed=962, chunk_tokens=64, chunk_start=100, num_decode=12, dec_lo=30,
                         dec_hi=600, Hq=16, Hkv=4, D=128)
    kc_ref, vc_ref = oracle_scattered(w)
    ref_d, _ = oracle.decode(w.decode_q, kc_ref, vc_ref, w.decode_block_tables,
                             w.decode_seq_lens, w.scale)
    _, fd, _, _, _, _, _ = _fused(pa, w, cuda_device)
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags(reset=True) == pa.PA_DEVERR_CHUNK
    assert_close(fd, ref_d, "decodes beside a flagged chunk")
    assert pa.pa_device_error_flags() == 0


def test_fused_step_rejects_bad_arguments_before_launching(pa, cuda_device):
    w = W.sarathi_hybrid(seed=963, chunk_tokens=32, chunk_start=16, num_decode=4, dec_lo=20,
                         dec_hi=80, Hq=8, Hkv=2, D=128)
    dev = cuda_device
    key = bits_to_dev(w.key, dev)
    wide = torch.zeros((key.shape[0], 2 * 128 + 4), dtype=torch.bfloat16, device=dev)
    odd = wide.as_strided(key.shape, (2 * 128 + 4, 128, 1))  # stride not a multiple of 8
    with pytest.raises(pa.PAError) as e:
        _fused(pa, w, dev, key=odd, value=odd)
    assert e.value.status == pa.PA_ERR_INVALID
    with pytest.raises(pa.PAError) as e:
        _fused(pa, w, dev, ws=_ws(pa, w, dev)[:256])
    assert e.value.status == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert pa.pa_device_error_flags() == 0


def test_fused_step_several_chunks_without_decodes(pa, cuda_device):
    """Three chunks (one of them ragged, all starting a block), no decodes:
    the launch writes every chunk's new rows and attends each chunk's own keys
    from them; bit for bit pa_reshape_and_cache + pa_prefill_chunk, and the
    oracle elementwise."""
    w = W.prefill_batch([(0, 40), (32, 72), (160, 130)], Hq=16, Hkv=4, D=128, seed=964,
                        poison=True)
    dev = cuda_device
    kc_ref, vc_ref = oracle_scattered(w)
    C = w.num_chunks
    T = int(w.cu_q_lens[C])
    ref, ref_lse = oracle.prefill(w.q[:T], kc_ref, vc_ref, w.block_tables[:C], w.cu_q_lens,
                                  w.q_start_pos, w.seq_lens[:C], w.scale)
    kc0, vc0 = _poisoned_pools(w)
    kc, vc = bits_to_dev(kc0, dev), bits_to_dev(vc0, dev)
    q, key, value = (bits_to_dev(a, dev) for a in (w.q, w.key, w.value))
    bt = torch.from_numpy(w.block_tables).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    cu = torch.from_numpy(w.cu_q_lens).to(dev)
    qs = torch.from_numpy(w.q_start_pos).to(dev)
    max_q = int(np.max(np.diff(w.cu_q_lens)))
    Hq, D = w.num_q_heads, w.head_dim
    out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=dev)
    none = torch.empty((0, Hq, D), dtype=torch.bfloat16, device=dev)
    pa.pa_hybrid_attention_append(out, q[:T], key[:T], value[:T], bt[:C], cu, qs, sl[:C], max_q,
                                  none, none, key[:0], value[:0], bt[:0], sl[:0], kc, vc, w.scale,
                                  None, chunk_lse=lse)
    # the two-launch form on the same inputs
    dw = DeviceWorkload(w, dev)
    dw.scatter(pa)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    pa.pa_prefill_chunk(out2, dw.q[:T], dw.k_cache, dw.v_cache, dw.block_tables[:C], cu, qs,
                        dw.seq_lens[:C], max_q, w.scale, out_lse=lse2)
    torch.cuda.synchronize()
    assert np.array_equal(dev_to_bits(kc), kc_ref) and np.array_equal(dev_to_bits(vc), vc_ref)
    assert np.array_equal(dev_to_bits(out), dev_to_bits(out2))
    assert torch.equal(lse, lse2)
    assert_close(out, ref, "fused chunks")
    assert_close(lse.cpu().numpy(), ref_lse, "fused chunks lse")
    assert pa.pa_device_error_flags() == 0


def test_fused_step_strided_rows(pa, cuda_device):
    """New K / V rows with a token stride above Hkv * D (rows of a fused QKV
    buffer): the same bits as with contiguous rows."""
    w = W.sarathi_hybrid(seed=965, poison=True, chunk_tokens=96, chunk_start=48, num_decode=10,
                         dec_lo=30, dec_hi=700, Hq=16, Hkv=4, D=128)
    dev = cuda_device
    rows, Hkv, D = w.key.shape
    pad = 3 * 128  # the rest of a fused row
    wide_k = torch.zeros((rows, Hkv * D + pad), dtype=torch.bfloat16, device=dev)
    wide_v = torch.zeros_like(wide_k)
    wide_k[:, :Hkv * D] = bits_to_dev(w.key, dev).view(rows, Hkv * D)
    wide_v[:, :Hkv * D] = bits_to_dev(w.value, dev).view(rows, Hkv * D)
    key = wide_k.as_strided((rows, Hkv, D), (Hkv * D + pad, D, 1))
    value = wide_v.as_strided((rows, Hkv, D), (Hkv * D + pad, D, 1))
    sc, sd, slc, sld, sk, sv, _ = _fused(pa, w, dev, key=key, value=value)
    fc, fd, flc, fld, fk, fv, _ = _fused(pa, w, dev)
    torch.cuda.synchronize()
    for x, y in ((sc, fc), (sd, fd), (sk, fk), (sv, fv)):
        assert np.array_equal(dev_to_bits(x), dev_to_bits(y))
    assert torch.equal(slc, flc) and torch.equal(sld, fld)
    kc_ref, _ = oracle_scattered(w)
    assert np.array_equal(dev_to_bits(sk), kc_ref)
    assert pa.pa_device_error_flags() == 0

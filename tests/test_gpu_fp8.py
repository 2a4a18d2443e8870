"""FP8 (E4M3) KV cache on the GPU, through the C ABI, against the oracle.

* The quantizing scatter is bit-exact against the oracle's quantizer over
  whole pools (untouched bytes included), per-head and per-tensor scales.
* The E4M3 decode matches the oracle's decode over the dequantized cache
  (fp64), within the same tolerance as the bf16 path, in all three split
  modes, on the Llama-3-8B-shaped layer, the copy-on-write mix (group 8, with
  pa_copy_blocks_fp8), the long-context batch at full size, edge shapes, NaN
  codes in unused slots, and queries far from unit scale.
The initial pools are the workloads' bf16 pools quantized by the oracle (the
scales calibrated as max |x| / 448 per head); NaN poison becomes NaN codes.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_218_gb300 import workload as W
from tests.gpu_common import assert_close, bits_to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa(cuda_device):
    from paged_kv_cache_218_gb300 import binding
    return binding


def calibrate(pool_bits, new_bits, per_tensor):
    x = np.concatenate([W.bf16_bits_to_f32(pool_bits).reshape(-1, pool_bits.shape[2],
                                                              pool_bits.shape[3]),
                        W.bf16_bits_to_f32(new_bits)], axis=0)
    amax = np.nanmax(np.abs(x), axis=(0, 2))
    if per_tensor:
        amax = np.full_like(amax, amax.max())
    return np.maximum(amax / 448.0, 1e-8).astype(np.float32)


class Fp8Case:
    """A workload with E4M3 pools on host (oracle) and device."""

    def __init__(self, w, dev, per_tensor=False, q_mult=1.0):
        self.w = w
        nb, bs, Hkv, D = w.k_cache.shape
        self.ks = calibrate(w.k_cache, w.key, per_tensor)
        self.vs = calibrate(w.v_cache, w.value, per_tensor)
        all_slots = np.arange(nb * bs, dtype=np.int64)
        z = np.zeros((nb, bs, Hkv, D), np.uint8)
        self.kc0, self.vc0 = oracle.reshape_and_cache_fp8(
            w.k_cache.reshape(nb * bs, Hkv, D), w.v_cache.reshape(nb * bs, Hkv, D), z, z,
            all_slots, self.ks, self.vs)
        q = w.q
        if q_mult != 1.0:
            q = W.f32_to_bf16_bits((W.bf16_bits_to_f32(q) * q_mult).astype(np.float32))
        self.q = q
        self.dev = dev
        self.dk = torch.from_numpy(self.kc0).to(dev)
        self.dv = torch.from_numpy(self.vc0).to(dev)
        self.dks = torch.from_numpy(self.ks).to(dev)
        self.dvs = torch.from_numpy(self.vs).to(dev)
        self.dq = bits_to_dev(q, dev)
        self.bt = torch.from_numpy(w.block_tables).to(dev)
        self.lens = torch.from_numpy(w.seq_lens).to(dev)

    def step_on_gpu(self, pa):
        w = self.w
        if w.cow_pairs.shape[0]:
            pa.pa_copy_blocks_fp8(self.dk, self.dv, torch.from_numpy(w.cow_pairs).to(self.dev))
        pa.pa_reshape_and_cache_fp8(bits_to_dev(w.key, self.dev), bits_to_dev(w.value, self.dev),
                                    self.dk, self.dv, torch.from_numpy(w.slot_mapping).to(self.dev),
                                    self.dks, self.dvs)

    def step_on_oracle(self):
        w = self.w
        kc, vc = oracle.copy_blocks_fp8(self.kc0, self.vc0, w.cow_pairs)
        return oracle.reshape_and_cache_fp8(w.key, w.value, kc, vc, w.slot_mapping, self.ks,
                                            self.vs)

    def decode(self, pa, partition, with_lse=True):
        w = self.w
        S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
        out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=self.dev)
        lse = torch.full((S, Hq), float("nan"), dtype=torch.float32, device=self.dev) \
            if with_lse else None
        ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                            w.max_blocks_per_seq, 16, partition),
                                self.dev)
        pa.pa_decode_fp8(out, self.dq[w.q_decode_row0:w.q_decode_row0 + S], self.dk, self.dv,
                         self.dks, self.dvs, self.bt[w.decode_seq0:], self.lens[w.decode_seq0:],
                         w.scale, partition_tokens=partition, out_lse=lse, workspace=ws)
        torch.cuda.synchronize()
        return out, lse


def run_case(pa, c, partition):
    kc, vc = c.step_on_oracle()
    c.step_on_gpu(pa)
    torch.cuda.synchronize()
    assert np.array_equal(c.dk.cpu().numpy(), kc), "K pool differs from the oracle's quantizer"
    assert np.array_equal(c.dv.cpu().numpy(), vc), "V pool differs from the oracle's quantizer"
    w = c.w
    S = w.num_decode_seqs
    ref, ref_lse = oracle.decode_fp8(c.q[w.q_decode_row0:w.q_decode_row0 + S], kc, vc, c.ks,
                                     c.vs, w.decode_block_tables, w.decode_seq_lens, w.scale)
    out, lse = c.decode(pa, partition)
    assert_close(out, ref, f"{w.name} fp8 decode, partition {partition}")
    assert_close(lse.cpu().numpy(), ref_lse, f"{w.name} fp8 lse, partition {partition}")
    assert pa.pa_device_error_flags() == 0


@pytest.mark.parametrize("partition", [0, 512, -1])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_fp8_llama3_layer(pa, cuda_device, partition, per_tensor):
    run_case(pa, Fp8Case(W.llama3_8b_layer(), cuda_device, per_tensor), partition)


@pytest.mark.parametrize("partition", [0, 512])
def test_fp8_cow_mix_group8(pa, cuda_device, partition):
    run_case(pa, Fp8Case(W.cow_mix(poison=True), cuda_device), partition)


@pytest.mark.parametrize("partition", [0, 512])
def test_fp8_long_context_full_size(pa, cuda_device, partition):
    run_case(pa, Fp8Case(W.long_context_split(), cuda_device), partition)


EDGE = [  # S, lo, hi, Hq, Hkv, seed
    (5, 1, 40, 8, 8, 1), (7, 1, 17, 8, 1, 2), (9, 15, 33, 6, 2, 3), (3, 16, 16, 16, 2, 4),
    (11, 1, 300, 24, 3, 5), (4, 100, 900, 40, 5, 6), (6, 1, 64, 7, 1, 7), (200, 1, 60, 32, 4, 8),
]


@pytest.mark.parametrize("S,lo,hi,Hq,Hkv,seed", EDGE)
@pytest.mark.parametrize("partition", [0, 32, -1])
def test_fp8_edge_shapes_with_nan_poison(pa, cuda_device, S, lo, hi, Hq, Hkv, seed, partition):
    w = W.decode_batch(S, lo, hi, Hq, Hkv, 128, seed, poison=True)
    run_case(pa, Fp8Case(w, cuda_device), partition)


@pytest.mark.parametrize("q_mult", [2000.0, 1e-3, 3e4])
def test_fp8_queries_far_from_unit_scale(pa, cuda_device, q_mult):
    w = W.decode_batch(12, 1, 500, 32, 8, 128, 31, poison=True)
    run_case(pa, Fp8Case(w, cuda_device, q_mult=q_mult), 0)


@pytest.mark.parametrize("partition", [0, 256, -1])
def test_fp8_scores_climbing_along_the_sequence(pa, cuda_device, partition):
    """Queries all 1 and every key at position p equal to 0.75 (p // 128)
    before quantization: scores climb by about 12 log2 units per 128 keys,
    so the running maximum moves at almost every block (two blocks per step
    on this path) and split pieces carry log-sum-exps far apart."""
    w = W.decode_batch(6, 100, 3000, 32, 8, 128, seed=960)
    w.q[:] = W.f32_to_bf16_bits(np.float32(1.0))
    for s_ in range(w.num_decode_seqs):
        n = int(w.seq_lens[s_])
        for pos in range(n - 1):
            w.k_cache[w.block_tables[s_, pos // 16], pos % 16] = \
                W.f32_to_bf16_bits(np.float32(0.75 * (pos // 128)))
        w.key[s_] = W.f32_to_bf16_bits(np.float32(0.75 * ((n - 1) // 128)))
    run_case(pa, Fp8Case(w, cuda_device), partition)


def test_fp8_rejects_head_dim_64(pa, cuda_device):
    w = W.tiny()
    c_k = torch.zeros(w.k_cache.shape, dtype=torch.uint8, device=cuda_device)
    sc = torch.ones(w.num_kv_heads, dtype=torch.float32, device=cuda_device)
    out = torch.empty((w.num_decode_seqs, w.num_q_heads, w.head_dim), dtype=torch.bfloat16,
                      device=cuda_device)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_fp8(out, bits_to_dev(w.decode_q, cuda_device), c_k, c_k, sc, sc,
                         torch.from_numpy(w.block_tables).to(cuda_device),
                         torch.from_numpy(w.seq_lens).to(cuda_device), w.scale,
                         partition_tokens=-1)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED

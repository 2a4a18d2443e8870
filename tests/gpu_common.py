"""Helpers shared by the GPU parity tests: move a seeded workload to the
device, run this step's copy-on-write + slot scatter through the C ABI, and
compare bf16 outputs with the fp64 oracle elementwise."""
import numpy as np
import torch

from paged_kv_cache_218_gb300.workload import bf16_bits_to_f32

ATOL = 1e-2
RTOL = 1e-2


def bits_to_dev(a, device):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def dev_to_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def dev_to_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


class DeviceWorkload:
    def __init__(self, w, device):
        self.w = w
        self.k_cache = bits_to_dev(w.k_cache, device)
        self.v_cache = bits_to_dev(w.v_cache, device)
        self.q = bits_to_dev(w.q, device)
        self.key = bits_to_dev(w.key, device)
        self.value = bits_to_dev(w.value, device)
        self.block_tables = torch.from_numpy(w.block_tables).to(device)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(device)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).to(device)
        self.cow_pairs = torch.from_numpy(w.cow_pairs).to(device)

    def scatter(self, pa):
        if self.cow_pairs.shape[0]:
            pa.pa_copy_blocks(self.k_cache, self.v_cache, self.cow_pairs)
        pa.pa_reshape_and_cache(self.key, self.value, self.k_cache, self.v_cache,
                                self.slot_mapping)

    # decode part of the batch
    @property
    def dq(self):
        w = self.w
        return self.q[w.q_decode_row0:w.q_decode_row0 + w.num_decode_seqs]

    @property
    def dtables(self):
        return self.block_tables[self.w.decode_seq0:]

    @property
    def dlens(self):
        return self.seq_lens[self.w.decode_seq0:]


def oracle_scattered(w):
    import oracle
    kc, vc = oracle.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs)
    return oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping)


def assert_close(got_bf16, ref_f64, what="", atol=ATOL, rtol=RTOL):
    got = dev_to_f64(got_bf16) if isinstance(got_bf16, torch.Tensor) else np.asarray(got_bf16)
    ref = np.asarray(ref_f64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside |d| <= {atol} + {rtol}|ref|;"
            f" max err {float(np.nanmax(err))}; first {idx.tolist()} got "
            f"{[float(got[tuple(i)]) for i in idx]} ref {[float(ref[tuple(i)]) for i in idx]}")
    return float(err.max()) if err.size else 0.0

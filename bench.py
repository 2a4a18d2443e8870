"""Benchmark: paged decode KV-read GB/s (and decode tokens/s) on GB300.

Default workload: one Llama-3-8B-shaped decode layer -- 64 sequences with
lengths uniform[128, 2048], 32 q / 8 kv heads, head_dim 128, 16-token blocks
drawn at random from a pool 1.25x the need, bf16 N(0, 1) data (seeded,
synthetic).  One step = the slot scatter of the 64 new tokens followed by
balanced paged decode over every sequence (the whole decode hot path), on
one of 8 independent copies of the KV pool in rotation so that the working
set (~2.7 GB) is far above the 129 MB L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--config llama3_8b_decode_layer|long_context_split_kv|
                              cow_prefix_mix|sarathi_hybrid]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload on its own GPU (the decode path needs no exchange);
value = all ranks' KV bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV-read GB/s & % of GB300 HBM peak; decode tokens/s at batch"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0

CONFIG_TEXT = {
    "llama3_8b_decode_layer": "Llama-3-8B-shaped decode layer: 64 seqs, seq_lens U[128,2048], "
                              "32 q / 8 kv heads, head_dim 128, block 16, bf16 N(0,1)",
    "long_context_split_kv": "long-context decode: 8 seqs, seq_lens U[32768,131072], 32 q / 8 kv "
                             "heads, head_dim 128, block 16, bf16 N(0,1)",
    "cow_prefix_mix": "continuous-batching mix: 256 seqs, lognormal(median 512, sigma 1) lengths "
                      "in [1,8192], 64 q / 8 kv heads, head_dim 128, groups of 4 alias a "
                      "256-token prefix with copy-on-write",
    "sarathi_hybrid": "Sarathi hybrid batch: prefill chunk of 512 queries at positions "
                      "1536-2047 + 128 decodes with seq_lens U[256,4096], 32 q / 8 kv heads, "
                      "head_dim 128, token budget 640",
    "shared_prompt_batch": "shared system prompt: 128 seqs in 16 groups of 8, each group aliasing "
                           "one 2048-token prompt, private suffixes lognormal(median 256, sigma 1), "
                           "32 q / 8 kv heads, head_dim 128",
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def source_hash(files):
    """Hash of the kernel sources' code: comments and runs of white space are
    dropped first, so that only a change of code invalidates a profile."""
    import re
    h = hashlib.sha256()
    for f in files:
        text = open(os.path.join(ROOT, "paged_kv_cache_218_gb300", "csrc", f)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(re.sub(r"\s+", " ", text).strip().encode())
    return h.hexdigest()[:16]


def profile_traffic(kernel_files, summary: str, key: str = "traffic_bytes_per_launch"):
    """A figure recorded by an ncu capture in profiles/ (by default the per-launch
    DRAM bytes), valid only while the kernel sources still hash to the value
    the summary was taken at; None otherwise."""
    try:
        fields = {}
        for line in open(os.path.join(ROOT, "profiles", summary)):
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
        if fields.get("source_sha256_16") != source_hash(kernel_files):
            return None
        return float(fields[key])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxs) if maxs else None,
                "samples": len(sms), "reasons": sorted(reasons)}


def reduce_over_ranks(elapsed_ms, units, device=None):
    """Slowest rank's elapsed time and the units (bytes, tokens) of all ranks;
    the identity when torch.distributed is not initialised or has one rank."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(elapsed_ms), float(units)
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    tdist.all_reduce(u, op=tdist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ----------------------------------------------------------------------------- workload

def make_workload(name):
    from paged_kv_cache_218_gb300 import workload as W
    return {"llama3_8b_decode_layer": W.llama3_8b_layer, "long_context_split_kv": W.long_context_split,
            "cow_prefix_mix": W.cow_mix, "sarathi_hybrid": W.sarathi_hybrid,
            "shared_prompt_batch": W.shared_prompt_batch}[name]()


class Replica:
    """One device-resident copy of the step's state (KV pools, tables, inputs)."""

    def __init__(self, w, dev, src=None):
        import numpy as np
        import torch

        def bits(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

        if src is None:
            self.k_cache = bits(w.k_cache)
            self.v_cache = bits(w.v_cache)
        else:
            self.k_cache = src.k_cache.clone()
            self.v_cache = src.v_cache.clone()
        self.q = bits(w.q)
        self.key = bits(w.key)
        self.value = bits(w.value)
        self.block_tables = torch.from_numpy(w.block_tables).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).to(dev)
        S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
        self.out = torch.empty((S, Hq, D), dtype=torch.bfloat16, device=dev)
        self.cow_pairs = torch.from_numpy(w.cow_pairs).to(dev) if len(w.cow_pairs) else None
        C = w.num_chunks
        if C:
            T = int(w.cu_q_lens[C])
            self.out_chunk = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
            self.cu = torch.from_numpy(w.cu_q_lens).to(dev)
            self.qs = torch.from_numpy(w.q_start_pos).to(dev)


def decode_args(w, r):
    s0, q0, S = w.decode_seq0, w.q_decode_row0, w.num_decode_seqs
    return (r.out, r.q[q0:q0 + S], r.k_cache, r.v_cache, r.block_tables[s0:], r.seq_lens[s0:])


def kv_bytes_decode(w):
    from paged_kv_cache_218_gb300 import workload as W
    return W.logical_kv_bytes(w.decode_seq_lens, w.num_kv_heads, w.head_dim)


def decode_algorithmic_bytes(w, append=False):
    """Minimal bytes one decode launch must move: every K/V token once, the
    queries, the outputs, the used block-table entries and the lengths; with
    the step's new token fused in (pa_decode_append), that token also written
    to its slot (its read, from the step's key / value rows instead of the
    pool, is already in the K/V tokens)."""
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    nb = sum((int(n) + 15) // 16 for n in w.decode_seq_lens)
    new = S * 2 * w.num_kv_heads * D * 2 if append else 0
    return kv_bytes_decode(w) + 2 * S * Hq * D * 2 + nb * 4 + S * 4 + new


def chunk_flops(w):
    """Causal (q, k) pairs of the prefill chunk x heads x 4 x head_dim
    (QK^T and PV, 2 flops per multiply-add)."""
    pairs = 0
    for c in range(w.num_chunks):
        n = int(w.cu_q_lens[c + 1] - w.cu_q_lens[c])
        p0 = int(w.q_start_pos[c])
        pairs += n * p0 + n * (n + 1) // 2
    return 4.0 * pairs * w.num_q_heads * w.head_dim


# ----------------------------------------------------------------------------- arms

def run_gpu(args, rank, world, local_rank):
    import torch

    from paged_kv_cache_218_gb300 import binding as pa

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = make_workload(args.config)
    R = args.replicas
    reps = [Replica(w, dev)]
    for _ in range(R - 1):
        reps.append(Replica(w, dev, src=reps[0]))
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    P = args.partition_tokens
    ws = [pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                         w.max_blocks_per_seq, 16, P), dev)
          for _ in range(R)]
    hybrid = w.num_chunks > 0
    max_q = int(max(w.cu_q_lens[1:] - w.cu_q_lens[:-1])) if hybrid else 0
    T = int(w.cu_q_lens[w.num_chunks]) if hybrid else 0
    main = torch.cuda.current_stream()
    s_chunk = torch.cuda.Stream(device=dev) if hybrid else None
    hws = [pa.alloc_workspace(pa.pa_hybrid_workspace_size(S, Hq, w.num_kv_heads, D,
                                                          w.max_blocks_per_seq), dev)
           for _ in range(R)] if hybrid else None
    cow = len(w.cow_pairs) > 0
    # a decode-only step fuses the slot scatter into the decode (pa_decode_append),
    # a hybrid step into its one launch (pa_hybrid_attention_append); eager
    # hybrid steps run scatter, chunk and decode as three launches
    use_graphs_cfg = not args.no_graphs
    launches_per_step = (1 if (use_graphs_cfg or not hybrid) else 3) + (1 if P > 0 else 0) \
        + (1 if cow else 0)

    def append(i):
        r = reps[i % R]
        out, q, kc, vc, bt, sl = decode_args(w, r)
        pa.pa_decode_append(out, q, r.key, r.value, kc, vc, bt, sl, w.scale, partition_tokens=P,
                            workspace=ws[i % R])

    def step(i, ev=None, cev=None):
        r = reps[i % R]
        cur = torch.cuda.current_stream()
        if cow:  # private copies of shared blocks about to be written (copy on write)
            pa.pa_copy_blocks(r.k_cache, r.v_cache, r.cow_pairs)
        if not hybrid:  # the new tokens' slot scatter fused into the decode
            if ev is not None:
                ev[0].record(cur)
            append(i)
            if ev is not None:
                ev[1].record(cur)
            return
        if hybrid and ev is None:
            # the hybrid batch in one call and one launch: the step's slot
            # scatter, and the chunk's tile pairs beside the decode on the SMs
            # it leaves free
            s0, q0, S_ = w.decode_seq0, w.q_decode_row0, w.num_decode_seqs
            pa.pa_hybrid_attention_append(
                r.out_chunk, r.q[:T], r.key[:T], r.value[:T], r.block_tables[:w.num_chunks],
                r.cu, r.qs, r.seq_lens[:w.num_chunks], max_q, r.out, r.q[q0:q0 + S_],
                r.key[T:T + S_], r.value[T:T + S_], r.block_tables[s0:], r.seq_lens[s0:],
                r.k_cache, r.v_cache, w.scale, hws[i % R])
            return
        pa.pa_reshape_and_cache(r.key, r.value, r.k_cache, r.v_cache, r.slot_mapping)
        if hybrid:  # timed kernel by kernel (no graphs): chunk and decode on two streams
            s_chunk.wait_stream(cur)
            if cev is not None:
                cev[0].record(s_chunk)
            pa.pa_prefill_chunk(r.out_chunk, r.q[:T], r.k_cache, r.v_cache,
                                r.block_tables[:w.num_chunks], r.cu, r.qs,
                                r.seq_lens[:w.num_chunks], max_q, w.scale, stream=s_chunk)
            if cev is not None:
                cev[1].record(s_chunk)
        if ev is not None:
            ev[0].record(cur)
        pa.pa_decode(*decode_args(w, r), w.scale, partition_tokens=P, workspace=ws[i % R])
        if ev is not None:
            ev[1].record(cur)
        if hybrid:
            cur.wait_stream(s_chunk)

    def chunk_only(i):
        r = reps[i % R]
        pa.pa_prefill_chunk(r.out_chunk, r.q[:T], r.k_cache, r.v_cache,
                            r.block_tables[:w.num_chunks], r.cu, r.qs,
                            r.seq_lens[:w.num_chunks], max_q, w.scale)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if pa.pa_device_error_flags() != 0:
        raise RuntimeError("device error flags set during warm-up")

    # Graph replay: one CUDA graph per round of R steps (every replica's
    # scatter, then its decode; the hybrid step's call co-schedules the prefill
    # chunk beside the decode), each kernel a programmatic dependent of the one before,
    # so consecutive kernels overlap launch and prologue with the previous
    # one's drain.  Single-step graphs cover a remainder of K mod R steps.
    use_graphs = not args.no_graphs
    if use_graphs:
        g_round, g_dec_round, g_chunk_round = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(),
                                               torch.cuda.CUDAGraph() if hybrid else None)
        with torch.cuda.graph(g_round):
            for r in range(R):
                step(r)
        with torch.cuda.graph(g_dec_round):  # the step's attention kernel alone
            for r in range(R):
                if hybrid:
                    pa.pa_decode(*decode_args(w, reps[r]), w.scale, partition_tokens=P,
                                 workspace=ws[r])
                else:
                    append(r)
        if hybrid:
            with torch.cuda.graph(g_chunk_round):
                for r in range(R):
                    chunk_only(r)
        g_step = []
        for r in range(args.steps % R):
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1):
                step(r)
            g_step.append(g1)
        for i in range(max(1, args.warmup // R)):
            g_round.replay()
        torch.cuda.synchronize()

    dist = world > 1
    if dist:
        import torch.distributed as tdist
    K = args.steps
    if use_graphs:
        evs = []
        cevs = [None] * K
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        cevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K)] if hybrid else [None] * K
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.6)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        tdist.barrier()
    torch.cuda.synchronize()
    t_start.record(main)
    if use_graphs:
        for _ in range(K // R):
            g_round.replay()
        for g1 in g_step:
            g1.replay()
    else:
        for i in range(K):
            step(i, evs[i], cevs[i])
    t_end.record(main)
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    clocks = sampler.stop()
    elapsed_ms, kv_all = reduce_over_ranks(t_start.elapsed_time(t_end), kv_bytes_decode(w) * K, dev)

    def back_to_back(g, n_launch):
        # CUDA events on the launching stream around n rounds of R launches
        n = max(1, n_launch // R)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(main)
        for _ in range(n):
            g.replay()
        b.record(main)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (n * R)

    if use_graphs:
        K2 = min(K, args.kernel_steps)
        dec_ms = back_to_back(g_dec_round, K2)
        chunk_ms = back_to_back(g_chunk_round, K2) if hybrid else None
    else:
        dec_ms = sum(a.elapsed_time(b) for a, b in evs) / K
        chunk_ms = sum(a.elapsed_time(b) for a, b in cevs) / K if hybrid else None
    flags = pa.pa_device_error_flags()
    if flags:
        raise RuntimeError(f"device error flags {flags} after the timed region")

    e2e = run_e2e(args, w, reps, ws, dev, pa, dist, s_chunk, max_q, T, hws)
    fp8 = measure_fp8_decode(args, w, reps, ws, dev, pa) if (use_graphs and w.head_dim == 128) \
        else None
    casc = measure_cascade(args, w, reps, dev, pa, CASCADE_GROUP[args.config]) \
        if (use_graphs and args.config in CASCADE_GROUP) else None
    prefill = measure_prefill_chunk(args, dev, pa) if use_graphs else None
    return dict(w=w, elapsed_ms=elapsed_ms, kv_all=kv_all, dec_ms=dec_ms, chunk_ms=chunk_ms,
                clocks=clocks, e2e=e2e, launches=launches_per_step * K, graphs=use_graphs,
                fp8=fp8, cascade=casc, prefill=prefill)


def measure_fp8_decode(args, w, reps, ws, dev, pa):
    """The same decode over E4M3 copies of each replica's pools (per-kv-head
    scales max |x| / 448, quantized by pa_reshape_and_cache_fp8 at set-up),
    timed like the bf16 kernel: back-to-back launches from graphs of R."""
    import torch
    R = len(reps)
    nb, bs, Hkv, D = reps[0].k_cache.shape
    P = args.partition_tokens
    pools = []
    for r in reps:
        kf = torch.empty((nb, bs, Hkv, D), dtype=torch.uint8, device=dev)
        vf = torch.empty_like(kf)
        ks = (r.k_cache.float().abs().amax(dim=(0, 1, 3)) / 448.0).clamp_min(1e-8).contiguous()
        vs = (r.v_cache.float().abs().amax(dim=(0, 1, 3)) / 448.0).clamp_min(1e-8).contiguous()
        slots = torch.arange(nb * bs, dtype=torch.int64, device=dev)
        pa.pa_reshape_and_cache_fp8(r.k_cache.view(nb * bs, Hkv, D), r.v_cache.view(nb * bs, Hkv, D),
                                    kf, vf, slots, ks, vs)
        pools.append((kf, vf, ks, vs))
    torch.cuda.synchronize()

    def dec(i):
        r = reps[i]
        out, q, _, _, bt, sl = decode_args(w, r)
        kf, vf, ks, vs = pools[i]
        pa.pa_decode_fp8(out, q, kf, vf, ks, vs, bt, sl, w.scale, partition_tokens=P,
                         workspace=ws[i])

    for i in range(max(3, args.warmup // 4)):
        dec(i % R)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(R):
            dec(i)
    g.replay()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, args.kernel_steps) // R)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (n * R)
    if pa.pa_device_error_flags() != 0:
        raise RuntimeError("device error flags set by the E4M3 decode")
    S, Hq = w.num_decode_seqs, w.num_q_heads
    kv = kv_bytes_decode(w) // 2
    alg = kv + 2 * S * Hq * D * 2 + sum((int(x) + 15) // 16 for x in w.decode_seq_lens) * 4 + S * 4
    del pools
    return {"launch_ms": ms, "bytes_per_launch": alg, "kernel": "decode_kernel<128, E4M3>",
            "kv_bytes_per_token": 2 * Hkv * D, "tokens_per_s": S / (ms * 1e-3),
            "achieved_gbs": alg / (ms * 1e-3) / 1e9,
            "scales": "per kv head, max |x| / 448"}


PREFILL_REPLICAS = 16  # chunk replicas in rotation: ~290 MB, more than L2


def measure_prefill_chunk(args, dev, pa):
    """The Sarathi batch's prefill chunk alone (512 queries at positions
    1536-2047 attending causally over 2048 paged keys; Llama-3-8B heads) on
    the tensor cores: PREFILL_REPLICAS independent copies of the chunk's
    state rotate, so no launch finds its K/V or queries in L2, timed as
    back-to-back launches from CUDA graphs of one launch per copy."""
    import torch

    from paged_kv_cache_218_gb300 import workload as W
    w = W.sarathi_hybrid(num_decode=0)
    reps = [Replica(w, dev)]
    for _ in range(PREFILL_REPLICAS - 1):
        reps.append(Replica(w, dev, src=reps[0]))
    T = int(w.cu_q_lens[w.num_chunks])
    max_q = int(max(w.cu_q_lens[1:] - w.cu_q_lens[:-1]))
    for r in reps:
        pa.pa_reshape_and_cache(r.key, r.value, r.k_cache, r.v_cache, r.slot_mapping)

    def chunk(r):
        pa.pa_prefill_chunk(r.out_chunk, r.q[:T], r.k_cache, r.v_cache,
                            r.block_tables[:w.num_chunks], r.cu, r.qs,
                            r.seq_lens[:w.num_chunks], max_q, w.scale)

    for _ in range(3):
        for r in reps:
            chunk(r)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in reps:
            chunk(r)
    g.replay()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, args.kernel_steps) // PREFILL_REPLICAS)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    if pa.pa_device_error_flags() != 0:
        raise RuntimeError("device error flags set by the prefill chunk")
    ms = a.elapsed_time(b) / (n * PREFILL_REPLICAS)
    del reps
    return {"launch_ms": ms, "gflop": chunk_flops(w) / 1e9, "kernel": "prefill_kernel<2>",
            "workload": "prefill chunk of 512 queries at positions 1536-2047 over its 2048 "
                        "paged keys, 32 q / 8 kv heads, head_dim 128 (the Sarathi batch's chunk)",
            "l2": f"{PREFILL_REPLICAS} copies of the chunk's K/V, queries and output in rotation "
                  "(~290 MB) > 129 MB L2",
            "timing": f"back-to-back launches from CUDA graphs of {PREFILL_REPLICAS}; "
                      "time / launches"}


# batches whose consecutive sequences share prefix blocks, and their group size
CASCADE_GROUP = {"cow_prefix_mix": 4, "shared_prompt_batch": 8}
E2E_PASSES = 4  # passes over the replicas per end-to-end graph round


def measure_cascade(args, w, reps, dev, pa, group):
    """Cascade decode of a batch with shared prefixes (each group's shared
    prefix attended once for its members, then each suffix): two launches per
    call, timed like the plain decode over back-to-back calls from graphs of R."""
    import torch

    from paged_kv_cache_218_gb300 import workload as W
    R = len(reps)
    P = args.partition_tokens
    go, pt, sb = W.cascade_groups(w, group)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    meta = [torch.from_numpy(x).to(dev) for x in (go, pt, sb)]
    wss = [pa.alloc_workspace(pa.pa_cascade_workspace_size(S, Hq, w.num_kv_heads, D,
                                                           w.max_blocks_per_seq, 16, P), dev)
           for _ in range(R)]

    def call(i):
        out, q, kc, vc, bt, sl = decode_args(w, reps[i])
        pa.pa_cascade_decode(out, q, kc, vc, bt, sl, meta[0], group, meta[1], meta[2], w.scale,
                             partition_tokens=P, workspace=wss[i])

    for i in range(max(3, args.warmup // 4)):
        call(i % R)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(R):
            call(i)
    g.replay()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, args.kernel_steps) // R)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(n):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (n * R)
    if pa.pa_device_error_flags() != 0:
        raise RuntimeError("device error flags set by the cascade decode")
    logical = kv_bytes_decode(w)
    unique = W.unique_kv_bytes(w.decode_block_tables, w.decode_seq_lens, w.num_kv_heads, D)
    return {"launch_ms": ms, "launches_per_call": 2, "groups": int(len(go) - 1),
            "group_size": group, "shared_prefix_blocks": int(pt.shape[1]),
            "logical_kv_bytes": logical, "unique_kv_bytes": unique,
            "unique_gbs": unique / (ms * 1e-3) / 1e9, "logical_gbs": logical / (ms * 1e-3) / 1e9,
            "tokens_per_s": S / (ms * 1e-3)}


def run_e2e(args, w, reps, ws, dev, pa, dist, s_chunk, max_q, T, hws):
    """Same metric through the public API with host buffers, run the way a
    serving loop runs it.  Every step uploads its inputs (queries, new K/V,
    slots, copy-on-write pairs, block tables, lengths; the chunk's metadata in
    the hybrid batch) from one pinned host buffer in one copy, runs the step's
    kernels on views of the uploaded buffer, and reads its outputs back into
    pinned host memory.  Three streams pipeline the steps: uploads run ahead of
    the kernels, read-backs follow them.  A replica's buffers are reused only
    after the step that last used them has finished its kernels (for the
    upload) and its read-back (for the outputs).  With graphs (the default) one
    CUDA graph holds a round of E2E_PASSES passes over the R replicas, and
    rounds replay back to back (a round's first upload and last read-back do
    not overlap the next round, so longer rounds spread that cost); without,
    the steps are issued one by one.  In a graph the upload buffers and the
    outputs alternate between two sets by pass, so a pass's uploads run during
    the pass before it, and the kernel stream joins them (and the read-backs
    of the output set it overwrites) once per pass: a cross-stream wait in
    front of a kernel ends its
    programmatic overlap with the kernel before it (measured 55.0 us per step
    with one join per step on the Llama-3-8B layer, against 49.3 us for the
    kernels alone)."""
    import torch

    R = len(reps)
    K = max(args.warmup + 1, min(args.steps, args.e2e_steps))
    RS = R * E2E_PASSES  # steps per graph round
    if not args.no_graphs:
        K = (K + RS - 1) // RS * RS
    hybrid = w.num_chunks > 0
    s0, q0, S, C = w.decode_seq0, w.q_decode_row0, w.num_decode_seqs, w.num_chunks
    P = args.partition_tokens
    names = ["q", "key", "value", "slot_mapping", "block_tables", "seq_lens"]
    names += ["cow_pairs"] if reps[0].cow_pairs is not None else []
    names += ["cu", "qs"] if hybrid else []
    layout, total = {}, 0
    for n in names:
        t = getattr(reps[0], n)
        layout[n] = (total, t.dtype, tuple(t.shape), t.numel() * t.element_size())
        total += (layout[n][3] + 255) // 256 * 256
    host = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for n, (o, _, _, nb) in layout.items():
        host[o:o + nb].copy_(getattr(reps[0], n).cpu().contiguous().view(-1).view(torch.uint8))
    # two upload buffers per replica: passes alternate between the sets
    arenas = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2 * R)]
    views = [{n: ar[o:o + nb].view(dt).view(shape) for n, (o, dt, shape, nb) in layout.items()}
             for ar in arenas]
    # two output sets per replica, alternating by pass like the upload buffers
    results = [[r.out] + ([r.out_chunk] if hybrid else []) for r in reps]
    results += [[torch.empty_like(x) for x in res] for res in results]
    host_out = [[torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in res]
                for res in results[:R]]
    d2h = sum(x.numel() * x.element_size() for x in results[0])

    comp = torch.cuda.current_stream()
    s_up, s_dn = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_up = [torch.cuda.Event() for _ in range(2 * R)]
    ev_k = [torch.cuda.Event() for _ in range(2 * R)]  # by upload buffer
    ev_dn = [torch.cuda.Event() for _ in range(2 * R)]  # by output set
    used = [False] * (2 * R)

    def kernels(j, a=None):  # on the current stream; replica j, buffer set a // R
        r, v = reps[j], views[j if a is None else a]
        out = results[j if a is None else a][0]
        out_chunk = results[j if a is None else a][1] if hybrid else None
        comp = torch.cuda.current_stream()
        if "cow_pairs" in v:
            pa.pa_copy_blocks(r.k_cache, r.v_cache, v["cow_pairs"])
        if not hybrid:  # slot scatter fused into the decode
            pa.pa_decode_append(out, v["q"][q0:q0 + S], v["key"], v["value"], r.k_cache,
                                r.v_cache, v["block_tables"][s0:], v["seq_lens"][s0:], w.scale,
                                partition_tokens=P, workspace=ws[j])
            return
        if hybrid and not args.no_graphs:  # slot scatter fused into the hybrid launch
            pa.pa_hybrid_attention_append(
                out_chunk, v["q"][:T], v["key"][:T], v["value"][:T], v["block_tables"][:C],
                v["cu"], v["qs"], v["seq_lens"][:C], max_q, out, v["q"][q0:q0 + S],
                v["key"][T:T + S], v["value"][T:T + S], v["block_tables"][s0:],
                v["seq_lens"][s0:], r.k_cache, r.v_cache, w.scale, hws[j])
            return
        pa.pa_reshape_and_cache(v["key"], v["value"], r.k_cache, r.v_cache, v["slot_mapping"])
        if hybrid:
            s_chunk.wait_stream(comp)
            pa.pa_prefill_chunk(out_chunk, v["q"][:T], r.k_cache, r.v_cache,
                                v["block_tables"][:C], v["cu"], v["qs"], v["seq_lens"][:C],
                                max_q, w.scale, stream=s_chunk)
        pa.pa_decode(out, v["q"][q0:q0 + S], r.k_cache, r.v_cache, v["block_tables"][s0:],
                     v["seq_lens"][s0:], w.scale, partition_tokens=P, workspace=ws[j])
        if hybrid:
            comp.wait_stream(s_chunk)

    def one(i):
        j = i % R
        if used[j]:
            s_up.wait_event(ev_k[j])
        with torch.cuda.stream(s_up):
            arenas[j].copy_(host, non_blocking=True)
        ev_up[j].record(s_up)
        comp.wait_event(ev_up[j])
        if used[j]:
            comp.wait_event(ev_dn[j])
        kernels(j)
        ev_k[j].record(comp)
        s_dn.wait_event(ev_k[j])
        with torch.cuda.stream(s_dn):
            for dst, src in zip(host_out[j], results[j]):
                dst.copy_(src, non_blocking=True)
        ev_dn[j].record(s_dn)
        used[j] = True

    def uploads(p):  # a pass's inputs into upload set p % 2 (captured into the round)
        for j in range(R):
            a = (p % 2) * R + j
            if p >= 2:  # the set's last reader: pass p - 2's kernels
                s_up.wait_event(ev_k[a])
            with torch.cuda.stream(s_up):
                arenas[a].copy_(host, non_blocking=True)
            ev_up[a].record(s_up)

    def round_body():  # E2E_PASSES x R pipelined steps, captured into one graph
        # Pass 0's inputs were uploaded by the round before (or the prologue
        # below): the graph of a round completes before the next one starts.
        # The round uploads passes 1 .. E2E_PASSES - 1 and the next round's
        # pass 0, each one pass ahead of its kernels.
        cap = torch.cuda.current_stream()
        s_up.wait_stream(cap)
        s_dn.wait_stream(cap)
        for p in range(E2E_PASSES):
            uploads(p + 1)  # runs while pass p's kernels do
            # one join per pass: this pass's uploads, and the read-backs of
            # the output set this pass overwrites (pass p - 2's)
            for j in range(R):
                a = (p % 2) * R + j
                if p >= 1:
                    cap.wait_event(ev_up[a])
                if p >= 2:
                    cap.wait_event(ev_dn[a])
            for j in range(R):
                a = (p % 2) * R + j
                kernels(j, a)
                ev_k[a].record(cap)
                s_dn.wait_event(ev_k[a])
                with torch.cuda.stream(s_dn):
                    for dst, src in zip(host_out[j], results[a]):
                        dst.copy_(src, non_blocking=True)
                ev_dn[a].record(s_dn)
        cap.wait_stream(s_up)
        cap.wait_stream(s_dn)

    g = None
    if not args.no_graphs:
        assert E2E_PASSES % 2 == 0  # a round ends on the upload set it starts on
        for i in range(args.warmup):
            one(i)
        for j in range(R):  # the prologue: the first round's pass 0 inputs
            arenas[j].copy_(host, non_blocking=True)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            round_body()
        for _ in range(max(1, args.warmup // RS)):
            g.replay()
    else:
        for i in range(args.warmup):
            one(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        import torch.distributed as tdist
        tdist.barrier()
    torch.cuda.synchronize()
    a.record(comp)
    if g is not None:
        for _ in range(K // RS):
            g.replay()
    else:
        s_up.wait_stream(comp)
        for i in range(K):
            one(args.warmup + i)
        comp.wait_stream(s_dn)
    b.record(comp)
    torch.cuda.synchronize()
    if pa.pa_device_error_flags() != 0:
        raise RuntimeError("device error flags set in the end-to-end run")
    ms, kv_all = reduce_over_ranks(a.elapsed_time(b), kv_bytes_decode(w) * K, dev)
    return dict(ms=ms, steps=K, h2d=total, d2h=d2h, kv_all=kv_all,
                pipeline=(f"one CUDA graph per round of {RS} steps ({E2E_PASSES} passes over "
                          f"{R} replicas); " if g is not None else "")
                + "upload (one copy from pinned host memory), kernels and read-back on three "
                  "streams, uploads running a pass ahead of the kernels (two sets of upload and "
                  "output buffers per replica) and read-backs following them; the kernel stream "
                  "joins the copies once per pass")


def run_oracle(w, min_seconds):
    """The fp64 CPU oracle as it stands, on the host cores: decode attention
    over the whole batch (its KV already holding the new tokens), repeated
    until at least `min_seconds` of CPU time; returns (seconds per pass,
    passes, threads, kv bytes per pass)."""
    import oracle
    kc, vc = oracle.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs)
    kc, vc = oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping)
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(w.decode_q, kc, vc, w.decode_block_tables, w.decode_seq_lens, w.scale)
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or passes >= 1000:
            break
    return el / passes, passes, oracle.num_threads(), kv_bytes_decode(w)


def cpu_baseline_obj(w, min_seconds):
    """The oracle on every host core (OpenMP over sequence and kv head), then
    a bounded single-threaded sample of the same work (at most a few seconds,
    at least one pass)."""
    import oracle
    sec, passes, cores, kvb = run_oracle(w, min_seconds)
    n_all = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        sec1, passes1, _, _ = run_oracle(w, min(3.0, min_seconds / 4))
    finally:
        oracle.set_num_threads(n_all)
    return {"value": kvb / sec / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle decode over the whole batch ({w.num_decode_seqs} seqs, "
                      f"{kvb / 1e6:.1f} MB of bf16 KV), repeated {passes}x in {sec * passes:.1f} s; "
                      f"slot scatter excluded", "tokens_per_s": w.num_decode_seqs / sec,
            "single_thread": {"value": kvb / sec1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"the same pass repeated {passes1}x on one thread"}}


def block_manager_timing(steps=64, seqs=256, group=4, system_tokens=256):
    """Host block manager at serving scale, the C++ manager (through its C ABI)
    and the plain-Python oracle manager on the same script: admit a
    continuous-batching mix (``seqs`` requests; groups of ``group`` share a
    ``system_tokens``-token system prompt through the prefix cache; suffix
    lengths lognormal, median 512, clipped to [1, 8192]), fork one member per
    group, then decode steps of one appended token per sequence, each ended
    with its copy pairs and the batch's block tables."""
    import numpy as np

    from oracle.block_manager import BlockManagerOracle
    from paged_kv_cache_218_gb300.block_manager import BlockManager
    rng = np.random.default_rng(4004)
    systems = [rng.integers(0, 32000, system_tokens).tolist() for _ in range(seqs // group)]
    prompts = [systems[i // group] + rng.integers(
        0, 32000, int(np.clip(np.rint(np.exp(np.log(512.0) + rng.standard_normal())), 1, 8192))
    ).tolist() for i in range(seqs)]
    toks = rng.integers(0, 32000, (steps, seqs + seqs // group)).tolist()
    nb = sum(-(-(len(p) + steps) // 16) for p in prompts) + 2 * seqs
    max_blocks = max(-(-(len(p) + steps) // 16) for p in prompts)

    def run(m, oracle_side):
        t0 = time.perf_counter()
        for i, p in enumerate(prompts):
            m.add_sequence(i, p)
        for g in range(seqs // group):
            m.fork(g * group, seqs + g)
        m.end_step()
        t1 = time.perf_counter()
        ids = list(range(seqs + seqs // group))
        for st in range(steps):
            if oracle_side:
                for i in ids:
                    m.append_token(i, toks[st][i])
            else:
                m.append_tokens(ids, toks[st])
            m.end_step()
            m.build_tables(ids, max_blocks)
        t2 = time.perf_counter()
        return (t1 - t0) / seqs * 1e6, (t2 - t1) / steps * 1e6

    m = BlockManager(nb, 16, True)
    admit_us, step_us = run(m, False)
    cached = m.num_cached_blocks()
    m.close()
    o_admit_us, o_step_us = run(BlockManagerOracle(nb, 16, True), True)
    return {"unit": "us", "admit_us_per_seq": admit_us, "decode_step_us": step_us,
            "batch": seqs + seqs // group, "cached_blocks": cached,
            "oracle_admit_us_per_seq": o_admit_us, "oracle_decode_step_us": o_step_us,
            "workload": f"{seqs} requests, groups of {group} sharing a {system_tokens}-token "
                        "system prompt, lognormal(median 512) suffixes, one fork per group; "
                        f"{steps} decode steps of one token per sequence + copy pairs + tables"}


def reference_arm(args):
    """K timed steps of the oracle, each a bounded sample of the workload: a
    rotating subset of the sequences sized so that warm-up + K steps take
    about --cpu-seconds in total."""
    import numpy as np

    import oracle
    from paged_kv_cache_218_gb300 import workload as W
    w = make_workload(args.config)
    kc, vc = oracle.copy_blocks(w.k_cache, w.v_cache, w.cow_pairs)
    kc, vc = oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slot_mapping)
    q, bt, sl = w.decode_q, w.decode_block_tables, w.decode_seq_lens
    S = w.num_decode_seqs
    t0 = time.perf_counter()
    oracle.decode(q, kc, vc, bt, sl, w.scale)
    full = time.perf_counter() - t0
    per_step = args.cpu_seconds / (args.steps + args.warmup)
    n = int(max(1, min(S, round(S * per_step / full))))

    def step(i):
        idx = (np.arange(n) + i * n) % S
        oracle.decode(q[idx], kc, vc, bt[idx], sl[idx], w.scale)
        return W.logical_kv_bytes(sl[idx], w.num_kv_heads, w.head_dim)

    for i in range(args.warmup):
        step(i)
    kvb = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        kvb += step(args.warmup + i)
    el = time.perf_counter() - t0
    value = kvb / el / 1e9
    cores = oracle.num_threads()
    sample = (f"each step: fp64 oracle decode of {n} of the {S} sequences (rotating), "
              f"KV already holding the new tokens; slot scatter excluded")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": CONFIG_TEXT[args.config], "name": args.config},
            "tokens_per_s": n * args.steps / el,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def profile_case(args):
    """Three launches of one kernel on a small case, for an ncu capture (ncu
    is run on this command; see profiles/): the decode (bf16 or E4M3) on the
    Llama-3-8B-shaped layer, or the Sarathi prefill chunk."""
    import numpy as np
    import torch

    from paged_kv_cache_218_gb300 import binding as pa
    from paged_kv_cache_218_gb300 import workload as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = {"prefill": W.sarathi_hybrid, "cascade": W.cow_mix}.get(args.profile_case,
                                                                 W.llama3_8b_layer)()
    r = Replica(w, dev)
    pa.pa_reshape_and_cache(r.key, r.value, r.k_cache, r.v_cache, r.slot_mapping)
    S, Hq, D = w.num_decode_seqs, w.num_q_heads, w.head_dim
    if args.profile_case == "prefill":
        T = int(w.cu_q_lens[w.num_chunks])
        max_q = int(max(w.cu_q_lens[1:] - w.cu_q_lens[:-1]))
        for _ in range(3):
            pa.pa_prefill_chunk(r.out_chunk, r.q[:T], r.k_cache, r.v_cache,
                                r.block_tables[:w.num_chunks], r.cu, r.qs,
                                r.seq_lens[:w.num_chunks], max_q, w.scale)
    elif args.profile_case == "cascade":
        go, pt, sb = W.cascade_groups(w, 4)
        meta = [torch.from_numpy(x).to(dev) for x in (go, pt, sb)]
        ws = pa.alloc_workspace(pa.pa_cascade_workspace_size(S, Hq, w.num_kv_heads, D,
                                                             w.max_blocks_per_seq, 16, 0), dev)
        out, q, kc, vc, bt, sl = decode_args(w, r)
        for _ in range(3):
            pa.pa_cascade_decode(out, q, kc, vc, bt, sl, meta[0], 4, meta[1], meta[2], w.scale,
                                 partition_tokens=0, workspace=ws)
    else:
        ws = pa.alloc_workspace(pa.pa_decode_workspace_size(S, Hq, w.num_kv_heads, D,
                                                            w.max_blocks_per_seq, 16, 0), dev)
        args_d = decode_args(w, r)
        if args.profile_case == "decode":
            for _ in range(3):
                pa.pa_decode(*args_d, w.scale, partition_tokens=0, workspace=ws)
        elif args.profile_case == "append":
            out, q, kc, vc, bt, sl = args_d
            for _ in range(3):
                pa.pa_decode_append(out, q, r.key, r.value, kc, vc, bt, sl, w.scale,
                                    partition_tokens=0, workspace=ws)
        else:
            nb, bs, Hkv, _ = r.k_cache.shape
            kf = torch.empty((nb, bs, Hkv, D), dtype=torch.uint8, device=dev)
            vf = torch.empty_like(kf)
            ks = (r.k_cache.float().abs().amax(dim=(0, 1, 3)) / 448.0).contiguous()
            vs = (r.v_cache.float().abs().amax(dim=(0, 1, 3)) / 448.0).contiguous()
            pa.pa_reshape_and_cache_fp8(r.k_cache.view(nb * bs, Hkv, D),
                                        r.v_cache.view(nb * bs, Hkv, D), kf, vf,
                                        torch.arange(nb * bs, dtype=torch.int64, device=dev),
                                        ks, vs)
            out, q, _, _, bt, sl = args_d
            for _ in range(3):
                pa.pa_decode_fp8(out, q, kf, vf, ks, vs, bt, sl, w.scale, partition_tokens=0,
                                 workspace=ws)
    torch.cuda.synchronize()
    if pa.pa_device_error_flags() != 0:
        raise RuntimeError("device error flags set")
    print("ok")


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="llama3_8b_decode_layer", choices=sorted(CONFIG_TEXT))
    ap.add_argument("--partition-tokens", type=int, default=None,
                    help="decode split mode (0 balanced, >0 fixed partitions, <0 single pass)")
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--kernel-steps", type=int, default=2000,
                    help="decode-only launches timed for the roofline's kernel duration")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch every kernel from Python instead of replaying CUDA graphs")
    ap.add_argument("--profile-case", default=None,
                    choices=["decode", "append", "decode_fp8", "prefill", "cascade"],
                    help="run three launches of one kernel on a small case (for ncu) and exit")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.partition_tokens is None:
        args.partition_tokens = 0

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    hbm, bf16, peak_src = load_peaks()

    if args.impl == "reference":
        # the reference arm is the fp64 oracle on the host cores; rank 0 only
        if rank != 0:
            return
        print(json.dumps(reference_arm(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    w = res["w"]
    K = args.steps
    kvb = kv_bytes_decode(w)
    step_ms = res["elapsed_ms"] / K
    value = res["kv_all"] / (res["elapsed_ms"] * 1e-3) / 1e9
    fused = w.num_chunks == 0  # the step's decode carries the slot scatter (pa_decode_append)
    alg = decode_algorithmic_bytes(w, append=fused)
    achieved = alg / (res["dec_ms"] * 1e-3) / 1e9
    traffic = profile_traffic(["pa_decode.cu", "pa_decode_body.cuh", "pa_ptx.cuh",
                               "pa_internal.h"],
                              "decode_append_kernel_llama3_8b_decode_layer.md") \
        if args.config == "llama3_8b_decode_layer" else None
    e = res["e2e"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": CONFIG_TEXT[args.config], "name": args.config,
                   "partition_tokens": args.partition_tokens,
                   "accumulate": "fp32",
                   "l2": f"{args.replicas} independent KV pools in rotation "
                         f"({args.replicas * 2 * w.k_cache.nbytes / 1e9:.2f} GB) >> 129 MB L2",
                   "parallelism": f"replicas x{world}",
                   "launch": (f"CUDA graph per round of {args.replicas} steps ("
                              + ("copy-on-write block copies, " if len(w.cow_pairs) else "")
                              + ("pa_hybrid_attention_append: one launch with the slot scatter "
                                 "fused in, the decode on its first CTAs, the chunk's CTA pairs on "
                                 "the SMs it leaves free; "
                                 if w.num_chunks else
                                 "pa_decode_append: the slot scatter fused into the decode; ")
                              + "programmatic dependent launches)") if res["graphs"]
                             else "eager launches from Python"},
        "tokens_per_s": w.num_decode_seqs * world * K / (res["elapsed_ms"] * 1e-3),
        "pct_of_nominal_8tbps": 100.0 * value / world / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": "decode_kernel<128> with the slot scatter (pa_decode_append)"
                               if fused else "decode_kernel<128>",
                     "peak_source": f"{peak_src} (hbm_gbs)",
                     "bytes_per_launch": alg, "launch_ms": res["dec_ms"],
                     "launch_timing": ("CUDA events on the launching stream around back-to-back "
                                       f"launches of that kernel alone (graphs of {args.replicas}, "
                                       "one per KV pool, each launch a programmatic dependent of "
                                       "the one before); time / launches") if res["graphs"]
                                      else "CUDA events around each decode launch in the timed region"},
        "e2e": {"value": e["kv_all"] / (e["ms"] * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                "steps": e["steps"], "ms_per_step": e["ms"] / e["steps"],
                "pipeline": e["pipeline"]},
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
    }
    if res.get("cascade") is not None:
        c = res["cascade"]
        plain_ms = res["dec_ms"]
        line["cascade"] = dict(c, peak=hbm, frac_unique=c["unique_gbs"] / hbm,
                               plain_decode_ms=plain_ms,
                               plain_unique_gbs=c["unique_kv_bytes"] / (plain_ms * 1e-3) / 1e9,
                               speedup_vs_plain=plain_ms / c["launch_ms"])
    if res.get("fp8") is not None:
        f = res["fp8"]
        line["fp8_kv"] = dict(f, peak=hbm, frac=f["achieved_gbs"] / hbm,
                              peak_source=f"{peak_src} (hbm_gbs)",
                              tokens_per_s_vs_bf16=f["tokens_per_s"] /
                              (w.num_decode_seqs / (res["dec_ms"] * 1e-3)))
    if res.get("prefill") is not None:
        pf = res["prefill"]
        tf = pf["gflop"] / pf["launch_ms"]  # GFLOP / ms = TFLOP/s
        line["prefill_chunk"] = dict(pf, bound="tensor", tflops=tf, peak=bf16,
                                     frac_of_bf16_peak=tf / bf16,
                                     peak_source=f"{peak_src} (bf16_tflops, burst: timed alone)",
                                     tensor_pipe_ncu=profile_traffic(
                                         ["pa_prefill.cu", "pa_prefill_body.cuh",
                                          "pa_ptx.cuh", "pa_internal.h"],
                                         "prefill_kernel_sarathi_chunk.md", "tensor_pipe_active_pct"))
    if res["chunk_ms"] is not None:
        if res["graphs"]:
            line["hybrid_step"] = {
                "step_ms": step_ms, "decode_alone_ms": res["dec_ms"],
                "chunk_alone_ms": res["chunk_ms"],
                "chunk_hidden_frac": max(0.0, min(1.0, (res["dec_ms"] + res["chunk_ms"] - step_ms)
                                                  / res["chunk_ms"])),
                "how": "pa_hybrid_attention_append: one launch whose first CTAs run the decode "
                       "(each writing its sequences' new tokens) and whose other CTAs run the "
                       "chunk's query tiles as tensor-core CTA pairs on the SMs the decode leaves "
                       "free (each writing its tile's new rows); step = that call"}
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline_obj(w, args.cpu_seconds)
        line["host_block_manager"] = block_manager_timing()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()

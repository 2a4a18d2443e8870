"""fp64 CPU oracle for paged attention (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links
or calls it, and it shares no code with the CUDA library: the arithmetic lives
in ``pa_oracle.c`` (plain C loops in fp64), this module only marshals numpy
arrays into it.

Every function takes bf16 data as ``numpy.uint16`` bit patterns, exactly as
the seeded generators in ``paged_kv_cache_218_gb300.workload`` produce them.
Citations for each computed quantity are in the header of ``pa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into liboracle.so with gcc and OpenMP."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_int64
            D = ctypes.c_double
            sigs = {
                "oracle_reshape_and_cache": [P, P, L, L, P, P, P, I, I, I, I, L],
                "oracle_copy_blocks": [P, P, P, I, I, I, I, L],
                "oracle_decode": [P, P, P, P, I, P, I, I, I, I, I, L, D, P, P],
                "oracle_decode_pairs": [P, P, P, P, I, P, I, I, I, I, L, D, P, I, P, P],
                "oracle_attend_range": [P, P, P, P, I, I, I, L, L, I, I, I, I, L, D, P, P],
                "oracle_merge": [P, P, P, I, I, I, I, P, P],
                "oracle_prefill": [P, P, P, P, I, P, P, P, I, I, I, I, I, L, D, P, P],
                "oracle_reshape_and_cache_fp8": [P, P, L, L, P, P, P, P, P, I, I, I, I, L],
                "oracle_decode_fp8": [P, P, P, P, P, P, I, P, I, I, I, I, I, L, D, P, P],
                "oracle_e4m3_encode": [ctypes.c_float],
                "oracle_num_threads": [],
                "oracle_set_num_threads": [I],
            }
            for name, args in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int if name != "oracle_set_num_threads" else None
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle: invalid metadata in {what}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, block_size=16):
    """Scatter new tokens' K/V ([T, Hkv, D] uint16) into copies of the pools.

    Returns the updated (k_cache, v_cache) copies; the inputs are untouched.
    """
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    slots = _c(slot_mapping, np.int64)
    T, Hkv, D = key.shape
    nb = kc.shape[0]
    rc = _load().oracle_reshape_and_cache(
        _ptr(key), _ptr(value), Hkv * D, Hkv * D, _ptr(kc), _ptr(vc), _ptr(slots),
        T, Hkv, D, block_size, nb)
    _check(rc, "reshape_and_cache")
    return kc, vc


def copy_blocks(k_cache, v_cache, pairs):
    """Copy whole physical blocks src -> dst (pairs [n, 2] int64) in copies."""
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    pairs = _c(np.asarray(pairs, dtype=np.int64).reshape(-1, 2), np.int64)
    nb, bs, Hkv, D = kc.shape
    rc = _load().oracle_copy_blocks(_ptr(kc), _ptr(vc), _ptr(pairs), pairs.shape[0],
                                    Hkv, D, bs, nb)
    _check(rc, "copy_blocks")
    return kc, vc


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale):
    """Decode attention: q [S, Hq, D] -> (out [S, Hq, D] fp64, lse [S, Hq])."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    out = np.zeros((S, Hq, D), dtype=np.float64)
    lse = np.zeros((S, Hq), dtype=np.float64)
    rc = _load().oracle_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1],
                               _ptr(sl), S, Hq, Hkv, D, bs, nb, float(scale), _ptr(out),
                               _ptr(lse))
    _check(rc, "decode")
    return out, lse


def decode_pairs(q, k_cache, v_cache, block_tables, seq_lens, scale, pairs):
    """Decode attention for listed (seq, q head) pairs only -> (out [n, D], lse [n])."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    pairs = _c(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), np.int32)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    n = pairs.shape[0]
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_decode_pairs(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                     bt.shape[1], _ptr(sl), Hq, Hkv, D, bs, nb,
                                     float(scale), _ptr(pairs), n, _ptr(out), _ptr(lse))
    _check(rc, "decode_pairs")
    return out, lse


def attend_range(q, k_cache, v_cache, block_tables, s, h, a, b, scale):
    """Partial attention of (seq s, q head h) over key positions [a, b)."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    out = np.zeros((D,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    rc = _load().oracle_attend_range(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                     bt.shape[1], int(s), int(h), int(a), int(b), Hq, Hkv,
                                     D, bs, nb, float(scale), _ptr(out), _ptr(lse))
    _check(rc, "attend_range")
    return out, float(lse[0])


def merge(part_o, part_lse, num_parts):
    """LSE merge: part_o [S, Hq, P, D], part_lse [S, Hq, P], num_parts [S]."""
    part_o = _c(np.asarray(part_o, dtype=np.float64), np.float64)
    part_lse = _c(np.asarray(part_lse, dtype=np.float64), np.float64)
    num_parts = _c(np.asarray(num_parts, dtype=np.int32), np.int32)
    S, Hq, P, D = part_o.shape
    out = np.zeros((S, Hq, D), dtype=np.float64)
    lse = np.zeros((S, Hq), dtype=np.float64)
    rc = _load().oracle_merge(_ptr(part_o), _ptr(part_lse), _ptr(num_parts), S, Hq, D, P,
                              _ptr(out), _ptr(lse))
    _check(rc, "merge")
    return out, lse


def prefill(q, k_cache, v_cache, block_tables, cu_q_lens, q_start_pos, seq_lens, scale):
    """Causal prefill chunks: q [Tq, Hq, D] -> (out [Tq, Hq, D], lse [Tq, Hq])."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint16)
    v_cache = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_q_lens, np.int32)
    qs = _c(q_start_pos, np.int32)
    sl = _c(seq_lens, np.int32)
    Tq, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    C = qs.shape[0]
    out = np.zeros((Tq, Hq, D), dtype=np.float64)
    lse = np.zeros((Tq, Hq), dtype=np.float64)
    rc = _load().oracle_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), bt.shape[1],
                                _ptr(cu), _ptr(qs), _ptr(sl), C, Hq, Hkv, D, bs, nb,
                                float(scale), _ptr(out), _ptr(lse))
    _check(rc, "prefill")
    return out, lse


# ----------------------------------------------------------------- FP8 (E4M3) KV cache

def e4m3_value(code: int) -> float:
    """The value of one E4M3 byte (NaN for 0x7F / 0xFF)."""
    return float(_load().oracle_e4m3_value(int(code) & 0xFF))


def e4m3_encode(v: float) -> int:
    """The E4M3 code nearest to the fp32 value v (ties to even, saturating)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(v))))


def reshape_and_cache_fp8(key, value, k_cache, v_cache, slot_mapping, k_scales, v_scales,
                          block_size=16):
    """Quantizing scatter of bf16 key/value [T, Hkv, D] into copies of uint8
    E4M3 pools: code = E4M3(x / scale[h]), the division in IEEE fp32."""
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    kc = np.array(k_cache, dtype=np.uint8, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint8, copy=True, order="C")
    slots = _c(slot_mapping, np.int64)
    ks = _c(np.asarray(k_scales, dtype=np.float32), np.float32)
    vs = _c(np.asarray(v_scales, dtype=np.float32), np.float32)
    T, Hkv, D = key.shape
    rc = _load().oracle_reshape_and_cache_fp8(
        _ptr(key), _ptr(value), Hkv * D, Hkv * D, _ptr(kc), _ptr(vc), _ptr(slots), _ptr(ks),
        _ptr(vs), T, Hkv, D, block_size, kc.shape[0])
    _check(rc, "reshape_and_cache_fp8")
    return kc, vc


def copy_blocks_fp8(k_cache, v_cache, pairs):
    """Whole-block copies src -> dst of uint8 pools (copies returned)."""
    kc = np.array(k_cache, dtype=np.uint8, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint8, copy=True, order="C")
    for src, dst in np.asarray(pairs, dtype=np.int64).reshape(-1, 2):
        kc[dst] = kc[src]
        vc[dst] = vc[src]
    return kc, vc


def decode_fp8(q, k_cache, v_cache, k_scales, v_scales, block_tables, seq_lens, scale):
    """Decode over E4M3 pools, dequantized exactly in fp64:
    q [S, Hq, D] -> (out [S, Hq, D], lse [S, Hq])."""
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint8)
    v_cache = _c(v_cache, np.uint8)
    ks = _c(np.asarray(k_scales, dtype=np.float32), np.float32)
    vs = _c(np.asarray(v_scales, dtype=np.float32), np.float32)
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    out = np.zeros((S, Hq, D), dtype=np.float64)
    lse = np.zeros((S, Hq), dtype=np.float64)
    rc = _load().oracle_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs),
                                   _ptr(bt), bt.shape[1], _ptr(sl), S, Hq, Hkv, D, bs, nb,
                                   float(scale), _ptr(out), _ptr(lse))
    _check(rc, "decode_fp8")
    return out, lse


# ----------------------------------------------------------------- cascade

def cascade_decode(q, k_cache, v_cache, block_tables, seq_lens, group_offsets, prefix_tables,
                   shared_blocks, scale):
    """Cascade decode in the steps of the pages' two-level attention
    ("03 - Engines Papers", section 12): per sequence, attention over its
    group's shared prefix (tokens [0, min(len, 16 * shared)) through the
    group's prefix table), attention over its private suffix (tokens
    [16 * shared, len) through its own table), and their log-sum-exp merge.
    Returns (out [S, Hq, D], lse [S, Hq])."""
    bt = np.asarray(block_tables, dtype=np.int32)
    sl = np.asarray(seq_lens, dtype=np.int32)
    go = np.asarray(group_offsets, dtype=np.int64)
    pt = np.asarray(prefix_tables, dtype=np.int32).reshape(len(go) - 1, -1)
    sb = np.asarray(shared_blocks, dtype=np.int64)
    S, mb = bt.shape
    pre_bt = np.full((S, max(pt.shape[1], 1)), -1, dtype=np.int32)
    pre_len = np.zeros(S, dtype=np.int32)
    suf_bt = np.full((S, mb), -1, dtype=np.int32)
    suf_len = np.zeros(S, dtype=np.int32)
    for g in range(len(go) - 1):
        for s in range(go[g], go[g + 1]):
            k = int(min(sb[s], -(-int(sl[s]) // 16)))
            pre_bt[s, :pt.shape[1]] = pt[g]
            pre_len[s] = min(int(sl[s]), 16 * int(sb[s]))
            rest = bt[s, k:]
            suf_bt[s, :len(rest)] = rest
            suf_len[s] = int(sl[s]) - 16 * k if int(sl[s]) > 16 * k else 0
    o_pre, l_pre = decode(q, k_cache, v_cache, pre_bt, pre_len, scale)
    o_suf, l_suf = decode(q, k_cache, v_cache, suf_bt, suf_len, scale)
    part_o = np.stack([o_pre, o_suf], axis=2)
    part_lse = np.stack([l_pre, l_suf], axis=2)
    return merge(part_o, part_lse, np.full(S, 2, dtype=np.int32))

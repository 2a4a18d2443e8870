"""The C-ABI library on a machine without a GPU: it loads, exports every
symbol include/pa.h declares, and its host-side logic (status strings,
workspace sizing, metadata validation, argument checks that return before
any launch) behaves as documented.  No call here reaches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

from paged_kv_cache_218_gb300 import workload as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")
LIB = os.path.join(ROOT, "paged_kv_cache_218_gb300", "libpa.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from paged_kv_cache_218_gb300 import build
        build.build()
    return ctypes.CDLL(LIB)


def declared_functions():
    """Every function declared in include/*.h."""
    import glob
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_prefill_chunk", "pa_merge_partials",
              "pa_decode_workspace_size", "pa_copy_blocks", "pa_validate_metadata",
              "pa_bm_create", "pa_bm_add_sequence", "pa_bm_append_token", "pa_bm_end_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in pa.h but not exported"


def test_status_strings(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(-1) == b"PA_ERR_INVALID"
    assert lib.pa_status_string(-4) == b"PA_ERR_WORKSPACE"
    assert lib.pa_status_string(123) == b"PA_ERR_UNKNOWN"
    assert lib.pa_version() >> 16 == 1


def _ws(lib, *args):
    f = lib.pa_decode_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 7
    return f(*args)


def test_workspace_sizes(lib):
    # single pass needs none
    assert _ws(lib, 64, 32, 8, 128, 128, 16, -1) == 0
    # fixed partitions: [S, Hq, P_max, D] fp32 + [S, Hq, P_max] fp32, each 256-aligned
    S, Hq, D, mb, P = 64, 32, 128, 128, 512
    pmax = (mb * 16 + P - 1) // P
    rows = S * Hq * pmax
    expect = -(-rows * D * 4 // 256) * 256 + -(-rows * 4 // 256) * 256
    assert _ws(lib, S, Hq, 8, D, mb, 16, P) == expect
    # balanced: independent of the batch, positive
    b1 = _ws(lib, 64, 32, 8, 128, 128, 16, 0)
    b2 = _ws(lib, 4096, 32, 8, 128, 128, 16, 0)
    assert b1 > 0 and b1 == b2
    # invalid or unsupported shapes report 0
    assert _ws(lib, 64, 32, 8, 96, 128, 16, 0) == 0
    assert _ws(lib, 64, 30, 8, 128, 128, 16, 0) == 0
    assert _ws(lib, 64, 32, 8, 128, 128, 32, 0) == 0
    assert _ws(lib, 64, 32, 8, 128, 128, 16, 24) == 0


def test_hybrid_and_cascade_workspace_sizes(lib):
    f = lib.pa_hybrid_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 6
    dec = _ws(lib, 128, 32, 8, 128, 256, 16, 0)
    # the balanced decode's workspace after 256 bytes for the chunk's finish counter
    assert f(128, 32, 8, 128, 256, 16) == 256 + dec
    assert f(128, 32, 8, 96, 256, 16) == 0
    g = lib.pa_cascade_workspace_size
    g.restype = ctypes.c_size_t
    g.argtypes = [ctypes.c_int] * 7
    S, Hq, Hkv = 256, 64, 8
    o = -(-S * Hq * 128 * 4 // 256) * 256
    l = -(-S * Hq * 4 // 256) * 256
    t = -(-S * Hkv * 4 // 256) * 256
    # prefix result and the partials of up to three more prefix parts, tickets, then the decode's
    assert g(S, Hq, Hkv, 128, 512, 16, 0) == 4 * (o + l) + t + _ws(lib, S, Hq, Hkv, 128, 512, 16, 0)
    assert g(S, Hq, Hkv, 64, 512, 16, 0) == 0


def test_hybrid_checks_arguments_before_launching(lib):
    f = lib.pa_hybrid_attention
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, I, P, P, P, I, I, I, P, P, P, P, I, P, I, P, P, P, I, I, I, I,
                  ctypes.c_int64, ctypes.c_float, I, P, ctypes.c_size_t, P]
    f.restype = I

    def call(**kw):
        a = dict(oc=P(256), qc=P(256), cbt=P(256), cmb=4, cu=P(256), qs=P(256), csl=P(256),
                 C=1, T=32, mq=32, clse=None, od=P(256), qd=P(256), dbt=P(256), dmb=4,
                 dsl=P(256), S=2, dlse=None, k=P(256), v=P(256), Hq=8, Hkv=2, D=128, bs=16,
                 nb=10, scale=0.1, cs=0, ws=P(256), wsb=1 << 30, st=None)
        a.update(kw)
        return f(*a.values())

    assert call(D=64) == -2              # the chunk's tensor-core path needs head_dim 128
    assert call(Hq=6, Hkv=2) == -2       # group 3 does not tile 128 rows
    assert call(scale=0.0) == -1
    assert call(cs=-1) == -1             # chunk_sms must be >= 0
    assert call(S=-1) == -1
    assert call(ws=None) == -4           # workspace missing
    assert call(wsb=100) == -4           # workspace too small
    assert call(ws=P(272)) == -4         # workspace misaligned
    assert call(oc=None) == -1


def test_hybrid_append_checks_arguments_before_launching(lib):
    f = lib.pa_hybrid_attention_append
    P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [P, P, P, P, P, I, P, P, P, I, I, I, P, P, P, P, P, P, I, P, I, P, L, L,
                  P, P, I, I, I, I, L, ctypes.c_float, I, P, ctypes.c_size_t, P]
    f.restype = I

    def call(**kw):
        a = dict(oc=P(256), qc=P(256), kc=P(256), vc=P(256), cbt=P(256), cmb=4, cu=P(256),
                 qs=P(256), csl=P(256), C=1, T=32, mq=32, clse=None, od=P(256), qd=P(256),
                 kd=P(256), vd=P(256), dbt=P(256), dmb=4, dsl=P(256), S=2, dlse=None,
                 kst=256, vst=256, k=P(256), v=P(256), Hq=8, Hkv=2, D=128, bs=16, nb=10,
                 scale=0.1, cs=0, ws=P(256), wsb=1 << 30, st=None)
        a.update(kw)
        return f(*a.values())

    assert call(D=64) == -2              # the chunk's tensor-core path needs head_dim 128
    assert call(scale=0.0) == -1
    assert call(cs=-1) == -1
    assert call(S=-1) == -1
    assert call(kst=255) == -1           # a token stride below Hkv * D
    assert call(vst=260) == -1           # not a multiple of 8 elements
    assert call(kc=None) == -1           # the chunk's new rows are missing
    assert call(vc=P(264)) == -1         # misaligned
    assert call(kd=None) == -1           # the decodes' new rows are missing
    assert call(oc=None) == -1


def _decode_args(**kw):
    P = ctypes.c_void_p
    a = dict(out=P(16), q=P(16), k=P(16), v=P(16), bt=P(16), mb=4, sl=P(16), S=2, Hq=8, Hkv=2,
             D=128, bs=16, nb=10, scale=0.1, part=-1, lse=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return a


def _decode(lib, **kw):
    a = _decode_args(**kw)
    f = lib.pa_decode
    P, I, L, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    f.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, L, F, I, P, P, S, P]
    f.restype = I
    return f(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["sl"], a["S"], a["Hq"],
             a["Hkv"], a["D"], a["bs"], a["nb"], a["scale"], a["part"], a["lse"], a["ws"],
             a["wsb"], a["stream"])


def test_decode_argument_checks_return_before_launch(lib):
    assert _decode(lib, D=96) == -2           # head_dim not 64/128
    assert _decode(lib, bs=32) == -2          # block_size not 16
    assert _decode(lib, Hq=6, Hkv=4) == -1    # Hq not a multiple of Hkv
    assert _decode(lib, Hq=32, Hkv=2) == -2   # group 16 > 8
    assert _decode(lib, scale=0.0) == -1
    assert _decode(lib, scale=float("nan")) == -1
    assert _decode(lib, out=None) == -1
    assert _decode(lib, S=0, out=None) == 0   # empty batch: nothing to do
    assert _decode(lib, mb=0) == -1
    assert _decode(lib, part=24) == -1        # partition not a multiple of 16
    assert _decode(lib, q=ctypes.c_void_p(18)) == -1  # misaligned


def test_other_calls_check_arguments(lib):
    P = ctypes.c_void_p
    lib.pa_reshape_and_cache.argtypes = [P, P, ctypes.c_int64, ctypes.c_int64, P, P, P,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int64, P]
    assert lib.pa_reshape_and_cache(None, None, 256, 256, None, None, None, 0, 2, 128, 16, 10,
                                    None) == 0
    assert lib.pa_reshape_and_cache(P(16), P(16), 256, 256, P(16), P(16), P(16), 3, 2, 128, 32,
                                    10, None) == -2
    assert lib.pa_reshape_and_cache(P(16), P(16), 100, 256, P(16), P(16), P(16), 3, 2, 128, 16,
                                    10, None) == -1
    lib.pa_merge_partials.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, P]
    assert lib.pa_merge_partials(P(16), None, P(16), P(16), P(16), 2, 4, 96, 3, None) == -2
    assert lib.pa_merge_partials(None, None, P(16), P(16), P(16), 2, 4, 128, 3, None) == -1
    f = lib.pa_prefill_chunk
    I = ctypes.c_int
    f.argtypes = [P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, ctypes.c_int64, ctypes.c_float,
                  P, P]
    assert f(P(16), P(16), P(16), P(16), P(16), 4, P(16), P(16), P(16), 1, 32, 32, 8, 2, 64, 16,
             10, 0.1, None, None) == -2   # head_dim 64 not served by the tensor-core path
    assert f(P(16), P(16), P(16), P(16), P(16), 4, P(16), P(16), P(16), 1, 32, 32, 6, 2, 128, 16,
             10, 0.1, None, None) == -2   # group 3 does not tile 128 rows
    assert f(None, P(16), P(16), P(16), P(16), 4, P(16), P(16), P(16), 1, 32, 32, 8, 2, 128, 16,
             10, 0.1, None, None) == -1


def _validate(lib, bt, sl, slots=None, ref=None, nb=16, bs=16):
    f = lib.pa_validate_metadata
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int64,
                  ctypes.c_int]
    bt = np.ascontiguousarray(bt, dtype=np.int32)
    sl = np.ascontiguousarray(sl, dtype=np.int32)
    sm = None if slots is None else np.ascontiguousarray(slots, dtype=np.int64)
    rc = None if ref is None else np.ascontiguousarray(ref, dtype=np.int32)
    p = lambda a: None if a is None else a.ctypes.data_as(P)
    return f(p(bt), bt.shape[1], p(sl), sl.shape[0], p(sm), 0 if sm is None else sm.shape[0],
             p(rc), nb, bs)


def test_validate_metadata(lib):
    w = W.tiny()
    assert _validate(lib, w.block_tables, w.seq_lens, w.slot_mapping, w.refcount) == 0
    bt = w.block_tables.copy()
    bt[3, 2] = 16
    assert _validate(lib, bt, w.seq_lens) == -1               # block id outside the pool
    lens = w.seq_lens.copy()
    lens[0] = 49
    assert _validate(lib, w.block_tables, lens) == -1         # longer than the table
    slots = w.slot_mapping.copy()
    slots[1] = slots[0]
    assert _validate(lib, w.block_tables, w.seq_lens, slots) == -1   # duplicate slot
    slots = w.slot_mapping.copy()
    slots[1] = -1
    assert _validate(lib, w.block_tables, w.seq_lens, slots) == 0    # padding is fine
    ref = w.refcount.copy()
    ref[int(w.slot_mapping[2]) // 16] = 2
    assert _validate(lib, w.block_tables, w.seq_lens, w.slot_mapping, ref) == -1  # write into shared


def test_validate_metadata_on_copy_on_write_mix(lib):
    w = W.cow_mix()
    assert _validate(lib, w.block_tables, w.seq_lens, w.slot_mapping, w.refcount,
                     nb=w.num_blocks) == 0
    # undo one copy: the write would land in a block shared by the group
    src, dst = w.cow_pairs[0]
    bt = w.block_tables.copy()
    bt[bt == dst] = src
    s = int(np.argwhere(w.block_tables == dst)[0][0])
    n = int(w.seq_lens[s])
    slots = w.slot_mapping.copy()
    slots[s] = int(src) * 16 + (n - 1) % 16
    ref = w.refcount.copy()
    ref[src] += 1
    assert _validate(lib, bt, w.seq_lens, slots, ref, nb=w.num_blocks) == -1

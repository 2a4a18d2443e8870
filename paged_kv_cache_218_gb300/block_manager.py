"""ctypes binding of the host block manager (include/pa_block_manager.h).

Argument marshalling only: every call goes to the C++ manager in libpa.so.
Host-only; needs neither torch nor a GPU.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libpa.so not found at {_LIB_PATH}; build it first with "
                      "`python -m paged_kv_cache_218_gb300.build`")
_lib = ctypes.CDLL(_LIB_PATH)

PA_OK = 0
PA_ERR_INVALID = -1
PA_ERR_NO_BLOCKS = -6
PA_ERR_BM_STEP = -7

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_SIGS = {
    "pa_bm_create": ([_L, _I, _I], _P),
    "pa_bm_destroy": ([_P], None),
    "pa_bm_add_sequence": ([_P, _L, _P, _I, _P, ctypes.POINTER(_I)], _I),
    "pa_bm_append_token": ([_P, _L, ctypes.c_int32, ctypes.POINTER(_L)], _I),
    "pa_bm_append_tokens": ([_P, _P, _P, _I, _P, ctypes.POINTER(_I)], _I),
    "pa_bm_fork": ([_P, _L, _L], _I),
    "pa_bm_free_sequence": ([_P, _L], _I),
    "pa_bm_num_step_copies": ([_P], _L),
    "pa_bm_end_step": ([_P, _P, _I], _I),
    "pa_bm_build_tables": ([_P, _P, _I, _P, _I, _P], _I),
    "pa_bm_num_free_blocks": ([_P], _L),
    "pa_bm_num_parked_blocks": ([_P], _L),
    "pa_bm_num_cached_blocks": ([_P], _L),
    "pa_bm_num_evictable_blocks": ([_P], _L),
    "pa_bm_refcount": ([_P, _L], _I),
    "pa_bm_seq_len": ([_P, _L], _L),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class BlockManagerError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed with status {status}")
        self.status = status


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class BlockManager:
    """Refcounted block pool, block tables, copy on write, fork and prefix
    cache; every method is one C call.  Methods raise BlockManagerError on a
    non-zero status (``.status`` holds it)."""

    def __init__(self, num_blocks: int, block_size: int = 16, prefix_caching: bool = True):
        self._h = _lib.pa_bm_create(int(num_blocks), int(block_size), int(bool(prefix_caching)))
        if not self._h:
            raise ValueError("pa_bm_create rejected its arguments")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self) -> None:
        if self._h:
            _lib.pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    @staticmethod
    def _check(fn: str, rc: int) -> None:
        if rc != PA_OK:
            raise BlockManagerError(fn, rc)

    def add_sequence(self, seq_id: int, tokens) -> tuple[np.ndarray, int]:
        """Admit a prompt; returns (slots int64 [n], -1 for reused tokens; num_cached)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        slots = np.empty(t.shape[0], dtype=np.int64)
        cached = ctypes.c_int(0)
        self._check("pa_bm_add_sequence", _lib.pa_bm_add_sequence(
            self._h, int(seq_id), _ptr(t), int(t.shape[0]), _ptr(slots), ctypes.byref(cached)))
        return slots, int(cached.value)

    def append_token(self, seq_id: int, token: int) -> int:
        slot = ctypes.c_int64(0)
        self._check("pa_bm_append_token",
                    _lib.pa_bm_append_token(self._h, int(seq_id), int(token), ctypes.byref(slot)))
        return int(slot.value)

    def append_tokens(self, seq_ids, tokens) -> np.ndarray:
        """One token per listed sequence, in order; returns the slots (int64).
        On a failure the appends before it stay done and the error's
        ``.done`` tells how many."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        if ids.shape != t.shape:
            raise ValueError("seq_ids and tokens differ in length")
        slots = np.empty(ids.shape[0], dtype=np.int64)
        st = ctypes.c_int(0)
        done = _lib.pa_bm_append_tokens(self._h, _ptr(ids), _ptr(t), int(ids.shape[0]),
                                        _ptr(slots), ctypes.byref(st))
        if st.value != PA_OK:
            err = BlockManagerError("pa_bm_append_tokens", st.value)
            err.done = int(done)
            raise err
        return slots

    def fork(self, parent_id: int, child_id: int) -> None:
        self._check("pa_bm_fork", _lib.pa_bm_fork(self._h, int(parent_id), int(child_id)))

    def free_sequence(self, seq_id: int) -> None:
        self._check("pa_bm_free_sequence", _lib.pa_bm_free_sequence(self._h, int(seq_id)))

    def end_step(self) -> np.ndarray:
        """End the step; returns its copy pairs as int64 [n, 2] (src, dst)."""
        n = int(_lib.pa_bm_num_step_copies(self._h))
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        rc = _lib.pa_bm_end_step(self._h, _ptr(pairs), n)
        if rc < 0:
            raise BlockManagerError("pa_bm_end_step", rc)
        return pairs[:rc]

    def build_tables(self, seq_ids, max_blocks: int) -> tuple[np.ndarray, np.ndarray]:
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tables = np.empty((ids.shape[0], max_blocks), dtype=np.int32)
        lens = np.empty(ids.shape[0], dtype=np.int32)
        self._check("pa_bm_build_tables", _lib.pa_bm_build_tables(
            self._h, _ptr(ids), int(ids.shape[0]), _ptr(tables), int(max_blocks), _ptr(lens)))
        return tables, lens

    def num_free_blocks(self) -> int:
        return int(_lib.pa_bm_num_free_blocks(self._h))

    def num_parked_blocks(self) -> int:
        return int(_lib.pa_bm_num_parked_blocks(self._h))

    def num_cached_blocks(self) -> int:
        return int(_lib.pa_bm_num_cached_blocks(self._h))

    def num_evictable_blocks(self) -> int:
        return int(_lib.pa_bm_num_evictable_blocks(self._h))

    def refcount(self, block: int) -> int:
        return int(_lib.pa_bm_refcount(self._h, int(block)))

    def seq_len(self, seq_id: int) -> int:
        return int(_lib.pa_bm_seq_len(self._h, int(seq_id)))

"""Python binding of the host block manager and serving loop in
``include/pa_blocks.h`` (argument marshalling only; the logic runs in the
library's C++)."""
from __future__ import annotations

import ctypes

import numpy as np

from . import pa as _pa

PA_BM_FULL = 1
EV_ADMIT, EV_PREEMPT, EV_FINISH = 0, 1, 2
_EV_NAMES = {EV_ADMIT: "admit", EV_PREEMPT: "preempt", EV_FINISH: "finish"}
_bound = False


def _lib():
    global _bound
    lib = _pa.load()
    if not _bound:
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        sigs = {
            "pa_bm_create": (P, [i32, i32, P, i32]),
            "pa_bm_destroy": (None, [P]),
            "pa_bm_num_free": (i32, [P]),
            "pa_bm_can_allocate": (i32, [P, i64]),
            "pa_bm_add_sequence": (ctypes.c_int, [P, i64, P, i64, i64, P]),
            "pa_bm_fork": (ctypes.c_int, [P, i64, i64]),
            "pa_bm_append": (ctypes.c_int, [P, i64, i32, P, P, P]),
            "pa_bm_free": (ctypes.c_int, [P, i64]),
            "pa_bm_table": (i32, [P, i64, P, i32]),
            "pa_bm_seq_len": (i64, [P, i64]),
            "pa_bm_refcount": (i32, [P, i32]),
            "pa_bm_batch": (ctypes.c_int, [P, P, i32, P, i32, i32, P]),
            "pa_bm_common_prefix": (i32, [P, P, i32]),
            "pa_loop_create": (P, [P]),
            "pa_loop_destroy": (None, [P]),
            "pa_loop_submit": (ctypes.c_int, [P, i64, i64, i64]),
            "pa_loop_step": (ctypes.c_int, [P, P, i32, P, P, i32, P, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _bound = True
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class BlockManager:
    """A pool of ``num_blocks`` blocks; ``free_order``'s last entry is handed
    out first."""

    def __init__(self, num_blocks: int, block_size: int = 16, free_order=None,
                 prefix_caching: bool = False):
        self._l = _lib()
        fo = None
        if free_order is not None:
            fo = np.ascontiguousarray(free_order, dtype=np.int32)
            if fo.shape != (num_blocks,):
                raise ValueError("free_order must list every block")
        self._h = self._l.pa_bm_create(int(num_blocks), int(block_size),
                                       _ptr(fo) if fo is not None else None,
                                       int(bool(prefix_caching)))
        if not self._h:
            raise ValueError("bad block manager arguments")
        self.block_size = block_size
        self.num_blocks = num_blocks

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._l.pa_bm_destroy(h)
            self._h = None

    @staticmethod
    def _check(fn, rc):
        if rc < 0:
            raise _pa.PAError(fn, rc)
        return rc

    def num_free(self) -> int:
        return int(self._l.pa_bm_num_free(self._h))

    def can_allocate(self, n_tokens: int) -> bool:
        return bool(self._l.pa_bm_can_allocate(self._h, int(n_tokens)))

    def add_sequence(self, seq_id, tokens, extra=0):
        """Number of tokens found cached, or None if the pool is too small."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        nc = ctypes.c_int64(0)
        rc = self._check("pa_bm_add_sequence", self._l.pa_bm_add_sequence(
            self._h, int(seq_id), _ptr(t) if t.size else None, t.size, int(extra),
            ctypes.byref(nc)))
        return None if rc == PA_BM_FULL else int(nc.value)

    def fork(self, parent, child):
        self._check("pa_bm_fork", self._l.pa_bm_fork(self._h, int(parent), int(child)))

    def append(self, seq_id, token):
        """(slot, (src, dst) or None), or None if no block is free."""
        slot, cs, cd = ctypes.c_int64(0), ctypes.c_int32(0), ctypes.c_int32(0)
        rc = self._check("pa_bm_append", self._l.pa_bm_append(
            self._h, int(seq_id), int(token), ctypes.byref(slot), ctypes.byref(cs),
            ctypes.byref(cd)))
        if rc == PA_BM_FULL:
            return None
        return int(slot.value), (None if cs.value < 0 else (int(cs.value), int(cd.value)))

    def free_sequence(self, seq_id):
        self._check("pa_bm_free", self._l.pa_bm_free(self._h, int(seq_id)))

    def table(self, seq_id):
        n = self._l.pa_bm_table(self._h, int(seq_id), None, 0)
        if n < 0:
            raise KeyError(seq_id)
        out = np.zeros(max(n, 1), dtype=np.int32)
        self._l.pa_bm_table(self._h, int(seq_id), _ptr(out), n)
        return out[:n].tolist()

    def seq_len(self, seq_id) -> int:
        n = int(self._l.pa_bm_seq_len(self._h, int(seq_id)))
        if n < 0:
            raise KeyError(seq_id)
        return n

    def refcount(self, block) -> int:
        return int(self._l.pa_bm_refcount(self._h, int(block)))

    def batch(self, seq_ids, width, pad=2**31 - 1):
        """(tables int32 [n, width] padded with ``pad``, seq_lens int32 [n])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tables = np.zeros((ids.size, width), dtype=np.int32)
        lens = np.zeros(ids.size, dtype=np.int32)
        self._check("pa_bm_batch", self._l.pa_bm_batch(
            self._h, _ptr(ids), ids.size, _ptr(tables), int(width), int(pad), _ptr(lens)))
        return tables, lens

    def common_prefix(self, seq_ids) -> int:
        """Leading blocks all of ``seq_ids`` share, each full in every one of
        them (the prefix block list of a cascade decode is the first of their
        tables cut to this length)."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = int(self._l.pa_bm_common_prefix(self._h, _ptr(ids), ids.size))
        if n < 0:
            raise KeyError("unknown sequence id")
        return n


class ServingLoop:
    """The serving loop of ``include/pa_blocks.h`` over ``bm`` (kept alive by
    this object)."""

    def __init__(self, bm: BlockManager):
        self._l = _lib()
        self.bm = bm
        self._h = self._l.pa_loop_create(bm._h)
        if not self._h:
            raise ValueError("could not create the loop")
        self.n_requests = 0

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._l.pa_loop_destroy(h)
            self._h = None

    def submit(self, rid, tokens, max_new):
        rc = self._l.pa_loop_submit(self._h, int(rid), int(tokens), int(max_new))
        if rc < 0:
            raise _pa.PAError("pa_loop_submit", rc)
        self.n_requests += 1

    def step(self):
        """One iteration: (more, step, events [(step, what, id, tokens, free)],
        written [(id, slot)])."""
        n = max(self.n_requests, 1)
        ev = np.zeros((3 * n + 8, 5), dtype=np.int64)
        wr = np.zeros((n, 2), dtype=np.int64)
        ne, nw, st = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int64(0)
        rc = self._l.pa_loop_step(self._h, _ptr(ev), ev.shape[0], ctypes.byref(ne), _ptr(wr),
                                  wr.shape[0], ctypes.byref(nw), ctypes.byref(st))
        if rc < 0:
            raise _pa.PAError("pa_loop_step", rc)
        events = [(int(e[0]), _EV_NAMES[int(e[1])], int(e[2]), int(e[3]), int(e[4]))
                  for e in ev[:ne.value]]
        written = [(int(w[0]), int(w[1])) for w in wr[:nw.value]]
        return rc == 1, int(st.value), events, written

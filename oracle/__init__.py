"""CPU oracle for OasisKV's per-layer look-ahead sparse decode step.

TEST INFRASTRUCTURE ONLY.  The oracle is a plain, sequential C++ restatement
of the method (``oasis_oracle.cpp``, fp64 sums, one rounding) plus this thin
ctypes wrapper.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import it.  It shares no code with
the CUDA library and never reads a value produced by it: its inputs come from
the seeded workload generators and its own earlier results.

Arrays are numpy: bf16 data as ``uint16`` bit patterns, ids/stamps as
``int32``, scores and attention outputs as ``float32``.  Layouts follow
``oasis_oracle.h``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oasis_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboasis_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``liboasis_oracle.so`` (g++, no CUDA)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < max(
                os.path.getmtime(_SRC),
                os.path.getmtime(os.path.join(_HERE, "oasis_oracle.h")))):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-o", tmp, _SRC
        ])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        sig = {
            "orc_summary_build": [P, P, I, I, I, I, I, P],
            "orc_attention_rh": [P, P, P, P, P, I, I, I, I, I, I, I, I, D, I, I, P],
            "orc_score_rh": [P, P, P, I, I, I, I, I, I, I, I, I, P],
            "orc_topk_rh": [P, I, I, P],
            "orc_admit_evict_rh": [P, P, P, I, I, I, P, P, P, P],
            "orc_step_rh": [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, D,
                            I, I, P, P, P, P, P, P, P],
            "orc_demand_rh": [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P, P, P, P, P, P],
            "orc_stall_step_rh": [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, D,
                                  I, I, P, P, P, P, P, P, P, P, P, P, P, P, P],
            "orc_append_token": [P, P, P, P, P, I, I, I, I, I, I],
            "orc_remote_fetch_rh": [P, I, P, P, I, I, P, P, P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray, dtype) -> ctypes.c_void_p:
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("array must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def _ok(rc: int, name: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {name} rejected its arguments")


def num_blocks(ctx: int, B: int) -> int:
    return 0 if ctx <= 0 else (ctx + B - 1) // B


def summary_build(host_kv: np.ndarray, ctx_len: np.ndarray) -> np.ndarray:
    """Per-block min/max key summaries, ``[R][Hkv][NBmax][2][d]`` uint16."""
    R, Hkv, NBmax, _, B, d = host_kv.shape
    summ = np.zeros((R, Hkv, NBmax, 2, d), dtype=np.uint16)
    _ok(_load().orc_summary_build(_p(host_kv, np.uint16), _p(ctx_len, np.int32),
                                  R, Hkv, NBmax, B, d, _p(summ, np.uint16)),
        "summary_build")
    return summ


def drafts(qd: np.ndarray) -> int:
    """Number of draft queries D in ``qd``: ``[R][Hq][d]`` is one draft,
    ``[D][R][Hq][d]`` is D of them."""
    if qd.ndim == 3:
        return 1
    if qd.ndim == 4 and qd.shape[0] >= 1:
        return qd.shape[0]
    raise ValueError("draft queries must be [R][Hq][d] or [D][R][Hq][d]")


def attention_rh(host_kv, ctx_len, res, q, qd, r, h, scale=None):
    """Attention outputs ``[1 + D][G][d]`` float32 of one (r, h): the normal
    query, then each draft query."""
    R, Hkv, NBmax, _, B, d = host_kv.shape
    Hq = q.shape[1]
    K = res.shape[-1]
    D = drafts(qd)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty((1 + D, Hq // Hkv, d), dtype=np.float32)
    _ok(_load().orc_attention_rh(
        _p(host_kv, np.uint16), _p(ctx_len, np.int32), _p(res, np.int32),
        _p(q, np.uint16), _p(qd, np.uint16), D, R, Hq, Hkv, NBmax, B, d, K,
        float(scale), r, h, _p(out, np.float32)), "attention_rh")
    return out


def score_rh(summ, ctx_len, qd, r, h, B):
    """Summary scores ``[NBmax]`` float32 of one (r, h) (-inf past the context)."""
    R, Hkv, NBmax, _, d = summ.shape
    D = drafts(qd)
    Hq = qd.shape[-2]
    s = np.empty(NBmax, dtype=np.float32)
    _ok(_load().orc_score_rh(_p(summ, np.uint16), _p(ctx_len, np.int32),
                             _p(qd, np.uint16), D, R, Hq, Hkv, NBmax, d, B, r, h,
                             _p(s, np.float32)), "score_rh")
    return s


def topk_rh(scores: np.ndarray, nb: int, K: int) -> np.ndarray:
    """Block ids in rank order (score desc, id asc), ``[K]`` int32, -1 padded."""
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    out = np.empty(K, dtype=np.int32)
    _ok(_load().orc_topk_rh(_p(scores, np.float32), nb, K, _p(out, np.int32)),
        "topk_rh")
    return out


def admit_evict_rh(res_row, stamp_row, topk, C, step):
    """Capped LRS eviction of one (r, h); updates ``res_row``/``stamp_row`` in
    place and returns ``(admit_ids, admit_slots, evict_ids, n_admit)``."""
    K = res_row.shape[0]
    a = np.empty(max(C, 1), dtype=np.int32)
    s = np.empty(max(C, 1), dtype=np.int32)
    e = np.empty(max(C, 1), dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    _ok(_load().orc_admit_evict_rh(_p(res_row, np.int32), _p(stamp_row, np.int32),
                                   _p(topk, np.int32), K, C, step, _p(a, np.int32),
                                   _p(s, np.int32), _p(e, np.int32),
                                   _p(n, np.int32)), "admit_evict_rh")
    return a[:C], s[:C], e[:C], int(n[0])


def demand_rh(summ, ctx_len, res, stamp, q, r, h, K, step, B):
    """Miss-stall demand fetch of one (r, h): rank with the normal query
    ``q`` ([R][Hq][d]), then admit every missing block of its top-K (no cap).
    ``res``/``stamp`` are the whole ``[R][Hkv][K]`` tables, updated in place
    for (r, h).  Returns a dict with scores [NBmax], topk [K], admit_ids,
    admit_slots, evict_ids [K] (-1 padded) and n_admit."""
    R, Hkv, NBmax, _, d = summ.shape
    Hq = q.shape[1]
    out = dict(scores=np.empty(NBmax, dtype=np.float32), topk=np.empty(K, dtype=np.int32),
               admit_ids=np.empty(K, dtype=np.int32), admit_slots=np.empty(K, dtype=np.int32),
               evict_ids=np.empty(K, dtype=np.int32))
    n = np.zeros(1, dtype=np.int32)
    _ok(_load().orc_demand_rh(
        _p(summ, np.uint16), _p(ctx_len, np.int32), _p(res, np.int32), _p(stamp, np.int32),
        _p(q, np.uint16), R, Hq, Hkv, NBmax, B, d, K, step, r, h,
        _p(out["scores"], np.float32), _p(out["topk"], np.int32),
        _p(out["admit_ids"], np.int32), _p(out["admit_slots"], np.int32),
        _p(out["evict_ids"], np.int32), _p(n, np.int32)), "demand_rh")
    out["n_admit"] = int(n[0])
    return out


def append_token(host_kv, summ, ctx_len, k_new, v_new, r):
    """Write one token (``[Hkv][d]`` keys and values) at position ctx_len[r]
    and fold its key into the tail summary; ctx_len is not changed."""
    R, Hkv, NBmax, _, B, d = host_kv.shape
    _ok(_load().orc_append_token(_p(host_kv, np.uint16), _p(summ, np.uint16),
                                 _p(ctx_len, np.int32), _p(k_new, np.uint16),
                                 _p(v_new, np.uint16), R, Hkv, NBmax, B, d, r),
        "append_token")


def remote_fetch_rh(ids, local_map_row, count, capacity):
    """Remote-tier slot assignment of one (r, h).  ``local_map_row`` ([NBmax]
    int32) is updated in place; ``count`` is a 1-element int32 array updated
    in place.  Returns ``(miss_ids, miss_slots, full)``."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n = ids.shape[0]
    mi = np.full(max(n, 1), -1, dtype=np.int32)
    ms = np.full(max(n, 1), -1, dtype=np.int32)
    nm = np.zeros(1, dtype=np.int32)
    rc = _load().orc_remote_fetch_rh(_p(ids, np.int32), n, _p(local_map_row, np.int32),
                                     _p(count, np.int32), capacity, local_map_row.shape[0],
                                     _p(mi, np.int32), _p(ms, np.int32), _p(nm, np.int32))
    if rc < 0:
        raise ValueError("oracle remote_fetch_rh rejected its arguments")
    k = int(nm[0])
    return mi[:k].copy(), ms[:k].copy(), bool(rc)


class LayerOracle:
    """Oracle state of one layer restricted to a set of (r, h) pairs.

    The pairs are independent in every stage of the step, so a sample of them
    can be followed at full problem size.  ``res``/``stamp`` hold the whole
    ``[R][Hkv][K]`` tables but only the tracked pairs are advanced.
    """

    def __init__(self, host_kv, summ, ctx_len, res0, K, C, pairs, scale=None,
                 remote_capacity=None):
        self.host_kv, self.summ, self.ctx_len = host_kv, summ, ctx_len
        self.R, self.Hkv, self.NBmax, _, self.B, self.d = host_kv.shape
        self.K, self.C = K, C
        self.res = np.array(res0, dtype=np.int32, copy=True)
        self.stamp = np.full_like(self.res, -1)
        self.pairs = [tuple(int(x) for x in p) for p in pairs]
        self.scale = 1.0 / np.sqrt(self.d) if scale is None else scale
        self._scores = np.empty(self.NBmax, dtype=np.float32)
        # Remote tier: the decode side's slot map and slot count per pair.
        # At load the initial resident set is fetched (in slot order), then
        # the block each context ends in when it ends inside a block (decoding
        # appends there).  initial_misses is that last assignment.
        self.remote_capacity = remote_capacity
        self.resident_misses, self.initial_misses = {}, {}
        if remote_capacity is not None:
            self.local_map = np.full((self.R, self.Hkv, self.NBmax), -1, dtype=np.int32)
            self.local_count = np.zeros((self.R, self.Hkv), dtype=np.int32)
            for (r, h) in self.pairs:
                self.resident_misses[(r, h)] = self._fetch(r, h, self.res[r, h])
                c = int(self.ctx_len[r])
                tail = [c // self.B] if c > 0 and c % self.B else []
                self.initial_misses[(r, h)] = self._fetch(r, h, np.array(tail, dtype=np.int32))

    def append_local(self, r):
        """Remote tier: a token appended to request r at position ctx_len[r]
        goes to its block's local slot; a block it opens takes the next slot.
        Returns True if some head found no slot left."""
        full = False
        c = int(self.ctx_len[r])
        for (rr, h) in self.pairs:
            if rr == r:
                full |= self._fetch(r, h, np.array([c // self.B], dtype=np.int32))["full"]
        return full

    def _fetch(self, r, h, ids):
        cnt = self.local_count[r, h:h + 1].copy()
        row = self.local_map[r, h]
        mi, ms, full = remote_fetch_rh(ids, row, cnt, self.remote_capacity)
        self.local_count[r, h] = cnt[0]
        return dict(miss_ids=mi, miss_slots=ms, n_miss=len(mi), full=full)

    def _step_outputs(self, Hq, D):
        C1 = max(self.C, 1)
        return dict(attn=np.empty((1 + D, Hq // self.Hkv, self.d), dtype=np.float32),
                    scores=np.empty(self.NBmax, dtype=np.float32),
                    topk=np.empty(self.K, dtype=np.int32),
                    admit_ids=np.empty(C1, dtype=np.int32),
                    admit_slots=np.empty(C1, dtype=np.int32),
                    evict_ids=np.empty(C1, dtype=np.int32))

    def _finish(self, v, n, r, h):
        for k in ("admit_ids", "admit_slots", "evict_ids"):
            v[k] = v[k][:self.C]
        v["n_admit"] = int(n[0])
        if self.remote_capacity is not None:
            v.update(self._fetch(r, h, v["admit_ids"][:v["n_admit"]]))
        return v

    def step(self, q, qd, t):
        """Run one layer-step (``orc_step_rh``: attention on the table as it
        stands, then scan, top-K and capped admission) for every tracked
        pair, on the oracle's own state only.  ``qd`` holds one draft
        ``[R][Hq][d]`` or D of them ``[D][R][Hq][d]``.  Returns a dict keyed
        by (r, h) with attn [1+D][G][d], scores, topk, admit_ids,
        admit_slots, evict_ids, n_admit (and, with a remote tier, the slot
        assignment's miss lists)."""
        L = _load()
        Hq = q.shape[1]
        D = drafts(qd)
        out = {}
        for (r, h) in self.pairs:
            v = self._step_outputs(Hq, D)
            n = np.zeros(1, dtype=np.int32)
            _ok(L.orc_step_rh(
                _p(self.host_kv, np.uint16), _p(self.summ, np.uint16),
                _p(self.ctx_len, np.int32), _p(self.res, np.int32), _p(self.stamp, np.int32),
                _p(q, np.uint16), _p(qd, np.uint16), D, self.R, Hq, self.Hkv, self.NBmax,
                self.B, self.d, self.K, self.C, t, float(self.scale), r, h,
                _p(v["attn"], np.float32), _p(v["scores"], np.float32),
                _p(v["topk"], np.int32), _p(v["admit_ids"], np.int32),
                _p(v["admit_slots"], np.int32), _p(v["evict_ids"], np.int32),
                _p(n, np.int32)), "step_rh")
            out[(r, h)] = self._finish(v, n, r, h)
        return out

    def stall_step(self, q, qd, t):
        """Run one miss-stall layer-step (``orc_stall_step_rh``: the demand
        fetch of the normal query's whole top-K, then ``step`` on the
        resulting table) for every tracked pair.  Returns the dict of
        ``step`` with, per pair, the demand lists under dm_scores, dm_topk,
        dm_admit_ids, dm_admit_slots, dm_evict_ids ([K] each) and
        dm_n_admit.  Not available with a remote tier."""
        if self.remote_capacity is not None:
            raise ValueError("the miss-stall step has no remote tier")
        L = _load()
        Hq = q.shape[1]
        D = drafts(qd)
        out = {}
        for (r, h) in self.pairs:
            v = self._step_outputs(Hq, D)
            dm = dict(dm_scores=np.empty(self.NBmax, dtype=np.float32),
                      dm_topk=np.empty(self.K, dtype=np.int32),
                      dm_admit_ids=np.empty(self.K, dtype=np.int32),
                      dm_admit_slots=np.empty(self.K, dtype=np.int32),
                      dm_evict_ids=np.empty(self.K, dtype=np.int32))
            dn = np.zeros(1, dtype=np.int32)
            n = np.zeros(1, dtype=np.int32)
            _ok(L.orc_stall_step_rh(
                _p(self.host_kv, np.uint16), _p(self.summ, np.uint16),
                _p(self.ctx_len, np.int32), _p(self.res, np.int32), _p(self.stamp, np.int32),
                _p(q, np.uint16), _p(qd, np.uint16), D, self.R, Hq, self.Hkv, self.NBmax,
                self.B, self.d, self.K, self.C, t, float(self.scale), r, h,
                _p(dm["dm_scores"], np.float32), _p(dm["dm_topk"], np.int32),
                _p(dm["dm_admit_ids"], np.int32), _p(dm["dm_admit_slots"], np.int32),
                _p(dm["dm_evict_ids"], np.int32), _p(dn, np.int32),
                _p(v["attn"], np.float32), _p(v["scores"], np.float32),
                _p(v["topk"], np.int32), _p(v["admit_ids"], np.int32),
                _p(v["admit_slots"], np.int32), _p(v["evict_ids"], np.int32),
                _p(n, np.int32)), "stall_step_rh")
            dm["dm_n_admit"] = int(dn[0])
            v.update(dm)
            out[(r, h)] = self._finish(v, n, r, h)
        return out

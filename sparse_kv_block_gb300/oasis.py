"""ctypes binding of the C ABI in ``include/oasis.h`` (``liboasis.so``).

Every function here marshals arguments and calls the library; all device
work runs in the library's CUDA kernels.  PyTorch is used only to allocate
device / pinned memory and to name streams.  If the library is missing the
import fails loudly: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint32, c_void_p
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboasis.so")

OASIS_OK, OASIS_EINVAL, OASIS_ENOMEM, OASIS_ECUDA = 0, -1, -2, -3
OASIS_ETIMEOUT, OASIS_ESTATE, OASIS_EDEVICE = -4, -5, -6
STATUS_NAMES = {0: "OK", -1: "EINVAL", -2: "ENOMEM", -3: "ECUDA", -4: "ETIMEOUT",
                -5: "ESTATE", -6: "EDEVICE"}


class oasis_config(ctypes.Structure):
    _fields_ = [("num_layers", c_int32), ("num_requests", c_int32), ("max_blocks", c_int32),
                ("num_q_heads", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("block_size", c_int32), ("topk", c_int32), ("fetch_ratio", c_float),
                ("softmax_scale", c_float), ("out_fp32", c_int32), ("device", c_int32),
                ("side_groups", c_int32), ("schedule", c_int32), ("num_drafts", c_int32)]


SCHEDULE_SCAN_FIRST, SCHEDULE_CONCURRENT, SCHEDULE_THREE_STREAMS, SCHEDULE_AUTO = 0, 1, 2, 3
SCHEDULE_EARLY_SCAN = 4


class oasis_sizes(ctypes.Structure):
    _fields_ = [("kv_pool_bytes", c_size_t), ("summaries_bytes", c_size_t),
                ("host_kv_bytes", c_size_t), ("res_ids_bytes", c_size_t),
                ("stamps_bytes", c_size_t), ("phys_bytes", c_size_t),
                ("ctx_len_bytes", c_size_t), ("workspace_bytes", c_size_t),
                ("fetch_cap", c_int32), ("units_per_head", c_int32)]


class oasis_buffers(ctypes.Structure):
    _fields_ = [("kv_pool", POINTER(c_void_p)), ("summaries", POINTER(c_void_p)),
                ("host_kv", POINTER(c_void_p)), ("res_ids", POINTER(c_void_p)),
                ("stamps", POINTER(c_void_p)), ("phys", POINTER(c_void_p)),
                ("ctx_len", c_void_p), ("workspace", c_void_p)]


class oasis_remote_config(ctypes.Structure):
    _fields_ = [("capacity", c_int32), ("gbps", c_float), ("threads", c_int32)]


class oasis_remote_sizes(ctypes.Structure):
    _fields_ = [("local_tier_bytes", c_size_t), ("local_map_bytes", c_size_t),
                ("miss_lists_bytes", c_size_t)]


DEVERR_NOT_LOCAL = 0x8


class OasisError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


# Declared exports: name -> (restype, argtypes).  Tests check this list against
# include/oasis.h.
_P = c_void_p
EXPORTS = {
    "oasis_config_error": (c_char_p, [POINTER(oasis_config)]),
    "oasis_query_sizes": (c_int, [POINTER(oasis_config), POINTER(oasis_sizes)]),
    "oasis_init": (c_int, [POINTER(oasis_config), POINTER(oasis_buffers), POINTER(c_void_p)]),
    "oasis_destroy": (c_int, [_P]),
    "oasis_last_error": (c_char_p, [_P]),
    "oasis_sync": (c_int, [_P, POINTER(c_uint32)]),
    "oasis_build_summaries": (c_int, [_P, c_int, c_int, _P]),
    "oasis_load_resident": (c_int, [_P, c_int, c_int, _P]),
    "oasis_resume_resident": (c_int, [_P, c_int, c_int, _P]),
    "oasis_lookahead_attn": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P]),
    "oasis_dense_attn": (c_int, [_P, _P, c_int, _P, _P, _P, _P, _P]),
    "oasis_score_topk": (c_int, [_P, c_int, c_int, _P, _P, _P, _P]),
    "oasis_admit_evict": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P, _P]),
    "oasis_score_admit_noalloc": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P, _P]),
    "oasis_prefetch": (c_int, [_P, c_int, c_int, _P, _P, _P, _P]),
    "oasis_step": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P]),
    "oasis_wait": (c_int, [_P, c_int, c_double]),
    "oasis_join": (c_int, [_P, c_int, _P]),
    "oasis_step_host": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P]),
    "oasis_step_host_async": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P]),
    "oasis_wait_outputs": (c_int, [_P, c_int, c_int, c_double]),
    "oasis_step_lists": (c_int, [_P, c_int, c_int, POINTER(c_void_p), POINTER(c_void_p),
                                 POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p),
                                 POINTER(c_void_p)]),
    "oasis_append_token": (c_int, [_P, c_int, c_int, _P, _P, _P]),
    "oasis_refresh_blocks": (c_int, [_P, c_int, c_int, _P, _P, c_int, _P]),
    "oasis_advance_context": (c_int, [_P, c_int, c_int, _P]),
    "oasis_remote_query_sizes": (c_int, [POINTER(oasis_config), POINTER(oasis_remote_config),
                                         POINTER(oasis_remote_sizes)]),
    "oasis_remote_attach": (c_int, [_P, c_int, POINTER(oasis_remote_config), _P, _P, _P]),
    "oasis_remote_stats": (c_int, [_P, c_int, POINTER(c_int64), POINTER(c_int64),
                                   POINTER(c_double), POINTER(c_int64)]),
    "oasis_demand_topk": (c_int, [_P, c_int, c_int, _P, _P, _P, _P]),
    "oasis_admit_demand": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P, _P]),
    "oasis_fetch_demand": (c_int, [_P, c_int, c_int, _P, _P, _P, _P]),
    "oasis_step_stall": (c_int, [_P, c_int, c_int, _P, _P, _P, _P, _P]),
    "oasis_stall_lists": (c_int, [_P, c_int, c_int, POINTER(c_void_p), POINTER(c_void_p),
                                  POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p),
                                  POINTER(c_void_p)]),
    "oasis_set_wait_limit": (c_int, [_P, ctypes.c_longlong]),
    "oasis_profile_enable": (c_int, [_P, c_int]),
    "oasis_profile_read_n": (c_int, [_P, c_int, POINTER(c_double), POINTER(c_int64),
                                     POINTER(c_double)]),
    "oasis_profile_read": (c_int, [_P, POINTER(c_double), POINTER(c_int64), POINTER(c_double)]),
}

PROFILE_KINDS = ["attention", "score_topk", "admit_evict", "prefetch", "demand_score",
                 "demand_gather", "topk_select"]

_lib = None


def lib():
    """Load liboasis.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        import torch.cuda  # noqa: F401  (loads the CUDA runtime the library links)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s) -> Optional[int]:
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_config(R, NBmax, Hq, Hkv, K, fetch_ratio, layers=1, softmax_scale=0.0,
                out_fp32=False, device=0, d=128, B=16, side_groups=0,
                schedule=SCHEDULE_AUTO, num_drafts=1) -> oasis_config:
    """``num_drafts`` D: draft queries per step; q_draft / out_draft then hold
    D planes ``[D][R][Hq][d]`` (a ``[R][Hq][d]`` tensor is the one-draft case).
    ``schedule``: one of SCHEDULE_*; with SCHEDULE_EARLY_SCAN the device-buffer
    oasis_step reads q_draft when it is called, so it must be complete then."""
    return oasis_config(layers, R, NBmax, Hq, Hkv, d, B, K, fetch_ratio, softmax_scale,
                        1 if out_fp32 else 0, device, side_groups, schedule, num_drafts)


def oasis_config_error(cfg: oasis_config) -> Optional[str]:
    m = lib().oasis_config_error(ctypes.byref(cfg))
    return None if m is None else m.decode()


def oasis_query_sizes(cfg: oasis_config) -> oasis_sizes:
    out = oasis_sizes()
    rc = lib().oasis_query_sizes(ctypes.byref(cfg), ctypes.byref(out))
    if rc != OASIS_OK:
        raise OasisError(rc, oasis_config_error(cfg) or "query_sizes failed")
    return out


def oasis_remote_query_sizes(cfg: oasis_config, rcfg: oasis_remote_config) -> oasis_remote_sizes:
    out = oasis_remote_sizes()
    rc = lib().oasis_remote_query_sizes(ctypes.byref(cfg), ctypes.byref(rcfg), ctypes.byref(out))
    if rc != OASIS_OK:
        raise OasisError(rc, "remote_query_sizes: bad config or remote config")
    return out


class Oasis:
    """A library context plus the caller-owned buffers it was given.

    Buffers are allocated with torch (device memory and pinned host memory
    for the KV store unless ``host_kv`` tensors are passed in) and kept alive
    here.  Methods map one-to-one onto the C ABI calls.
    """

    def __init__(self, cfg: oasis_config, host_kv: Optional[Sequence[torch.Tensor]] = None):
        self.cfg = cfg
        self.sizes = oasis_query_sizes(cfg)
        L, R, Hkv = cfg.num_layers, cfg.num_requests, cfg.num_kv_heads
        K, U, NB = cfg.topk, self.sizes.units_per_head, cfg.max_blocks
        self.C, self.U = self.sizes.fetch_cap, U
        dev = torch.device("cuda", cfg.device)
        self.device = dev
        if host_kv is None:
            host_kv = [torch.zeros((R, Hkv, NB, 2, 16, 128), dtype=torch.bfloat16,
                                   pin_memory=True) for _ in range(L)]
        if len(host_kv) != L:
            raise ValueError("need one host store per layer")
        for t in host_kv:
            if t.numel() * t.element_size() != self.sizes.host_kv_bytes or not t.is_pinned():
                raise ValueError("host_kv must be pinned and of host_kv_bytes")
        self.host_kv = list(host_kv)
        self.kv_pool = [torch.zeros((R, Hkv, U, 2, 16, 128), dtype=torch.bfloat16, device=dev)
                        for _ in range(L)]
        self.summaries = [torch.zeros((R, Hkv, NB, 2, 128), dtype=torch.bfloat16, device=dev)
                          for _ in range(L)]
        self.res_ids = [torch.full((2, R, Hkv, K), -1, dtype=torch.int32, device=dev)
                        for _ in range(L)]
        self.stamps = [torch.full((R, Hkv, K), -1, dtype=torch.int32, device=dev)
                       for _ in range(L)]
        self.phys = [torch.zeros((2, R, Hkv, U), dtype=torch.int32, device=dev) for _ in range(L)]
        self.ctx_len = torch.zeros((2, R), dtype=torch.int32, device=dev)
        self.workspace = torch.zeros(self.sizes.workspace_bytes, dtype=torch.uint8, device=dev)

        def arr(ts):
            a = (c_void_p * L)(*[t.data_ptr() for t in ts])
            return a
        self._arrs = [arr(self.kv_pool), arr(self.summaries), arr(self.host_kv),
                      arr(self.res_ids), arr(self.stamps), arr(self.phys)]
        bufs = oasis_buffers(*[ctypes.cast(a, POINTER(c_void_p)) for a in self._arrs],
                             self.ctx_len.data_ptr(), self.workspace.data_ptr())
        handle = c_void_p()
        torch.cuda.synchronize(dev)
        rc = lib().oasis_init(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(handle))
        if rc != OASIS_OK:
            raise OasisError(rc, oasis_config_error(cfg) or "oasis_init failed "
                             "(buffers not pinned/mapped, or CUDA error)")
        self.ctx = handle.value

    # ------------------------------------------------------------------ util
    def _check(self, rc: int) -> None:
        if rc != OASIS_OK:
            raise OasisError(rc, lib().oasis_last_error(self.ctx).decode())

    def close(self) -> None:
        if getattr(self, "ctx", None):
            lib().oasis_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ C ABI calls
    def oasis_sync(self) -> int:
        bits = c_uint32(0)
        rc = lib().oasis_sync(self.ctx, ctypes.byref(bits))
        if rc not in (OASIS_OK, OASIS_EDEVICE):
            self._check(rc)
        if rc == OASIS_EDEVICE:
            raise OasisError(rc, f"device error bits 0x{bits.value:x}")
        return bits.value

    def oasis_build_summaries(self, layer: int, table: int = 0, stream=None) -> None:
        self._check(lib().oasis_build_summaries(self.ctx, layer, table, _stream(stream)))

    def oasis_load_resident(self, layer: int, first_step: int = 0, stream=None) -> None:
        self._check(lib().oasis_load_resident(self.ctx, layer, first_step, _stream(stream)))

    def oasis_resume_resident(self, layer: int, first_step: int, stream=None) -> None:
        self._check(lib().oasis_resume_resident(self.ctx, layer, first_step, _stream(stream)))

    def _sized(self, q=None, qd=None, out=None, outd=None) -> None:
        """Refuse torch tensors smaller than the call reads or writes (the
        library takes plain pointers and cannot check their extent)."""
        c = self.cfg
        D = c.num_drafts if c.num_drafts > 0 else 1
        qb = c.num_requests * c.num_q_heads * c.head_dim * 2
        ob = qb * (2 if c.out_fp32 else 1)
        for name, x, need in (("q", q, qb), ("q_draft", qd, D * qb), ("out", out, ob),
                              ("out_draft", outd, D * ob)):
            if isinstance(x, torch.Tensor) and x.numel() * x.element_size() < need:
                raise ValueError(f"{name} holds {x.numel() * x.element_size()} bytes, "
                                 f"the call needs {need}")

    def oasis_lookahead_attn(self, layer, step, q, qd, out, outd, stream=None) -> None:
        self._sized(q, qd, out, outd)
        self._check(lib().oasis_lookahead_attn(self.ctx, layer, step, _ptr(q), _ptr(qd),
                                               _ptr(out), _ptr(outd), _stream(stream)))

    def oasis_dense_attn(self, kv_dense, table, q, qd, out, outd, stream=None) -> None:
        self._sized(q, qd, out, outd)
        self._check(lib().oasis_dense_attn(self.ctx, _ptr(kv_dense), table, _ptr(q), _ptr(qd),
                                           _ptr(out), _ptr(outd), _stream(stream)))

    def oasis_score_topk(self, layer, step, qd, topk_ids, topk_scores=None, stream=None) -> None:
        self._sized(qd=qd)
        self._check(lib().oasis_score_topk(self.ctx, layer, step, _ptr(qd), _ptr(topk_ids),
                                           _ptr(topk_scores), _stream(stream)))

    def oasis_admit_evict(self, layer, step, topk_ids, admit_ids, admit_slots, evict_ids,
                          n_admit, stream=None) -> None:
        self._check(lib().oasis_admit_evict(self.ctx, layer, step, _ptr(topk_ids),
                                            _ptr(admit_ids), _ptr(admit_slots),
                                            _ptr(evict_ids), _ptr(n_admit), _stream(stream)))

    def oasis_score_admit_noalloc(self, layer, step, qd, admit_ids, admit_slots, evict_ids,
                                  n_admit, stream=None) -> None:
        self._sized(qd=qd)
        self._check(lib().oasis_score_admit_noalloc(self.ctx, layer, step, _ptr(qd),
                                                    _ptr(admit_ids), _ptr(admit_slots),
                                                    _ptr(evict_ids), _ptr(n_admit),
                                                    _stream(stream)))

    def oasis_prefetch(self, layer, step, admit_ids, admit_slots, n_admit, stream=None) -> None:
        self._check(lib().oasis_prefetch(self.ctx, layer, step, _ptr(admit_ids),
                                         _ptr(admit_slots), _ptr(n_admit), _stream(stream)))

    def oasis_step(self, layer, step, q, qd, out, outd, stream=None) -> None:
        self._sized(q, qd, out, outd)
        self._check(lib().oasis_step(self.ctx, layer, step, _ptr(q), _ptr(qd), _ptr(out),
                                     _ptr(outd), _stream(stream)))

    def oasis_demand_topk(self, layer, step, q, topk_ids, topk_scores=None, stream=None) -> None:
        self._sized(q=q)
        self._check(lib().oasis_demand_topk(self.ctx, layer, step, _ptr(q), _ptr(topk_ids),
                                            _ptr(topk_scores), _stream(stream)))

    def oasis_admit_demand(self, layer, step, topk_ids, admit_ids, admit_slots, evict_ids,
                           n_admit, stream=None) -> None:
        """Lists [R][Hkv][K] int32 and n_admit [R][Hkv] int32 (device)."""
        self._check(lib().oasis_admit_demand(self.ctx, layer, step, _ptr(topk_ids),
                                             _ptr(admit_ids), _ptr(admit_slots),
                                             _ptr(evict_ids), _ptr(n_admit), _stream(stream)))

    def oasis_fetch_demand(self, layer, step, admit_ids, admit_slots, n_admit,
                           stream=None) -> None:
        self._check(lib().oasis_fetch_demand(self.ctx, layer, step, _ptr(admit_ids),
                                             _ptr(admit_slots), _ptr(n_admit), _stream(stream)))

    def oasis_step_stall(self, layer, step, q, qd, out, outd, stream=None) -> None:
        self._sized(q, qd, out, outd)
        self._check(lib().oasis_step_stall(self.ctx, layer, step, _ptr(q), _ptr(qd), _ptr(out),
                                           _ptr(outd), _stream(stream)))

    def oasis_stall_lists(self, layer: int, step: int) -> dict:
        ps = [c_void_p() for _ in range(6)]
        self._check(lib().oasis_stall_lists(self.ctx, layer, step,
                                            *[ctypes.byref(p) for p in ps]))
        return dict(zip(["topk_ids", "topk_scores", "admit_ids", "admit_slots", "evict_ids",
                         "n_admit"], [p.value for p in ps]))

    def oasis_wait(self, layer: int, timeout_ms: float) -> bool:
        """True when the layer's side work is done, False on timeout."""
        rc = lib().oasis_wait(self.ctx, layer, float(timeout_ms))
        if rc == OASIS_ETIMEOUT:
            return False
        self._check(rc)
        return True

    def oasis_join(self, layer, stream=None) -> None:
        self._check(lib().oasis_join(self.ctx, layer, _stream(stream)))

    def oasis_step_host(self, layer, step, q_host, qd_host, out_host, outd_host,
                        stream=None) -> None:
        self._sized(q_host, qd_host, out_host, outd_host)
        self._check(lib().oasis_step_host(self.ctx, layer, step, _ptr(q_host), _ptr(qd_host),
                                          _ptr(out_host), _ptr(outd_host), _stream(stream)))

    def oasis_step_host_async(self, layer, step, q_host, qd_host, out_host, outd_host,
                              stream=None) -> None:
        self._sized(q_host, qd_host, out_host, outd_host)
        self._check(lib().oasis_step_host_async(self.ctx, layer, step, _ptr(q_host),
                                                _ptr(qd_host), _ptr(out_host), _ptr(outd_host),
                                                _stream(stream)))

    def oasis_wait_outputs(self, layer: int, step: int, timeout_ms: float) -> bool:
        """True when the outputs of host-buffer step `step` are in host
        memory, False on timeout."""
        rc = lib().oasis_wait_outputs(self.ctx, layer, step, float(timeout_ms))
        if rc == OASIS_ETIMEOUT:
            return False
        self._check(rc)
        return True

    def oasis_step_lists(self, layer: int, step: int) -> dict:
        ps = [c_void_p() for _ in range(6)]
        self._check(lib().oasis_step_lists(self.ctx, layer, step,
                                           *[ctypes.byref(p) for p in ps]))
        return dict(zip(["topk_ids", "topk_scores", "admit_ids", "admit_slots", "evict_ids",
                         "n_admit"], [p.value for p in ps]))

    def oasis_append_token(self, layer, step, k_new, v_new, stream=None) -> None:
        self._check(lib().oasis_append_token(self.ctx, layer, step, _ptr(k_new), _ptr(v_new),
                                             _stream(stream)))

    def oasis_refresh_blocks(self, layer, step, ids, n_ids, stream=None) -> None:
        """ids: int32 [R][Hkv][max_ids] (device), n_ids: int32 [R][Hkv] (device)."""
        self._check(lib().oasis_refresh_blocks(self.ctx, layer, step, _ptr(ids), _ptr(n_ids),
                                               int(ids.shape[-1]), _stream(stream)))

    def oasis_advance_context(self, step, grow=1, stream=None) -> None:
        self._check(lib().oasis_advance_context(self.ctx, step, grow, _stream(stream)))

    def oasis_remote_attach(self, layer: int, capacity: int, gbps: float = 0.0,
                            threads: int = 0) -> dict:
        """Allocate the remote tier's buffers (pinned local tier and miss
        lists, device local map), attach them to `layer` and return them as
        tensors: local_tier [R][Hkv][capacity][2][16][128] bf16, local_map
        [R][Hkv][NBmax] int32, local_count [R][Hkv] int32 (a view into the
        same buffer), miss_lists (flat int32)."""
        rcfg = oasis_remote_config(capacity, gbps, threads)
        sz = oasis_remote_query_sizes(self.cfg, rcfg)
        R, Hkv, NB = self.cfg.num_requests, self.cfg.num_kv_heads, self.cfg.max_blocks
        local = torch.zeros((R, Hkv, capacity, 2, 16, 128), dtype=torch.bfloat16,
                            pin_memory=True)
        assert local.numel() * 2 == sz.local_tier_bytes
        mp = torch.empty(sz.local_map_bytes // 4, dtype=torch.int32, device=self.device)
        lists = torch.zeros(sz.miss_lists_bytes // 4, dtype=torch.int32, pin_memory=True)
        self._check(lib().oasis_remote_attach(self.ctx, layer, ctypes.byref(rcfg),
                                              local.data_ptr(), mp.data_ptr(),
                                              lists.data_ptr()))
        pairs = R * Hkv
        M = max(self.cfg.topk, self.C)
        t = dict(local_tier=local, local_map=mp[:pairs * NB].view(R, Hkv, NB),
                 local_count=mp[pairs * NB:pairs * NB + pairs].view(R, Hkv),
                 local_base=mp[pairs * NB + pairs:].view(R, Hkv), miss_lists=lists,
                 n_miss=lists[:pairs].view(R, Hkv),
                 miss_ids=lists[pairs:pairs + pairs * M].view(R, Hkv, M),
                 miss_slots=lists[pairs + pairs * M:pairs + 2 * pairs * M].view(R, Hkv, M))
        if not hasattr(self, "remote"):
            self.remote = {}
        self.remote[layer] = t
        return t

    def oasis_remote_stats(self, layer: int) -> dict:
        u, n, b = c_int64(0), c_int64(0), c_int64(0)
        sec = c_double(0.0)
        self._check(lib().oasis_remote_stats(self.ctx, layer, ctypes.byref(u), ctypes.byref(n),
                                             ctypes.byref(sec), ctypes.byref(b)))
        return dict(units=u.value, transfers=n.value, seconds=sec.value, bad_entries=b.value)

    def oasis_set_wait_limit(self, cycles: int) -> None:
        """Barrier-wait limit of the following launches in clock cycles
        (<= 0: the default, about a second)."""
        self._check(lib().oasis_set_wait_limit(self.ctx, int(cycles)))

    def oasis_profile_enable(self, enable: bool = True) -> None:
        self._check(lib().oasis_profile_enable(self.ctx, 1 if enable else 0))

    def oasis_profile_read(self, nkinds: int = 4) -> tuple:
        """(summed ms, launch counts, summed start offsets in ms) per kernel
        kind, for the first `nkinds` of PROFILE_KINDS."""
        ms = (c_double * nkinds)()
        cnt = (c_int64 * nkinds)()
        off = (c_double * nkinds)()
        self._check(lib().oasis_profile_read_n(self.ctx, nkinds, ms, cnt, off))
        return list(ms), list(cnt), list(off)

    # ------------------------------------------------------- tensor views
    def step_lists(self, layer: int, step: int) -> dict:
        """The workspace lists of oasis_step(layer, step) as torch tensors
        (views, no copy; valid until step + 2 is issued)."""
        return self._list_views(self.oasis_step_lists(layer, step), max(self.C, 1))

    def stall_lists(self, layer: int, step: int) -> dict:
        """The demand lists of oasis_step_stall(layer, step) as torch tensors
        (views, no copy; admission lists [R][Hkv][K])."""
        return self._list_views(self.oasis_stall_lists(layer, step), self.cfg.topk)

    def _list_views(self, p: dict, width: int) -> dict:
        R, Hkv, K = self.cfg.num_requests, self.cfg.num_kv_heads, self.cfg.topk
        out = {}
        for name, shape, dt in [("topk_ids", (R, Hkv, K), torch.int32),
                                ("topk_scores", (R, Hkv, K), torch.float32),
                                ("admit_ids", (R, Hkv, width), torch.int32),
                                ("admit_slots", (R, Hkv, width), torch.int32),
                                ("evict_ids", (R, Hkv, width), torch.int32),
                                ("n_admit", (R, Hkv), torch.int32)]:
            n = 1
            for s in shape:
                n *= s
            off = p[name] - self.workspace.data_ptr()
            es = torch.tensor([], dtype=dt).element_size()
            out[name] = self.workspace[off:off + n * es].view(dt).view(shape)
        return out

    def set_context(self, lens) -> None:
        """Set both ctx_len tables (plain host-to-device copy)."""
        t = torch.as_tensor(lens, dtype=torch.int32)
        self.ctx_len.copy_(t.view(1, -1).expand(2, -1))

    def set_resident(self, layer: int, res, first_step: int = 0) -> None:
        """Write the caller's resident table for `first_step` (host-to-device copy)."""
        self.res_ids[layer][first_step & 1].copy_(torch.as_tensor(res, dtype=torch.int32))

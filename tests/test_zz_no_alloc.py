"""oasis_score_admit_noalloc (top-K list in the library's fixed device
scratch) against the existing oasis_score_topk + oasis_admit_evict (top-K
list in a caller buffer), on two consecutive steps of identical contexts:
admission lists and tables equal bit for bit.  Also: an oversize
configuration is refused with a message, before any device work.

Collected last on purpose (file name), so it runs both alone and after the
rest of the suite has used the device."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from sparse_kv_block_gb300 import oasis as ob
from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("shape_name,R,ratio", [("tiny", 5, 0.25), ("qwen3_8b_16k", 8, 0.05)])
def test_noalloc_matches_stage_calls_on_two_steps(dev, shape_name, R, ratio):
    sh = dataclasses.replace(workload.SHAPES[shape_name], R=R)
    A = H.make_layer(sh, seed=31, steps=2, fetch_ratio=ratio)
    B = H.make_layer(sh, seed=31, steps=2, fetch_ratio=ratio)
    sh = A.shape
    K, C, Hk = sh.K, max(sh.C, 1), sh.Hkv

    def lists():
        aid = torch.full((sh.R, Hk, C), -7, dtype=torch.int32, device=dev)
        return aid, torch.full_like(aid, -7), torch.full_like(aid, -7), \
            torch.full((sh.R, Hk), -7, dtype=torch.int32, device=dev)

    for t in range(2):
        qd = A.qd[t].to(dev)
        topk = torch.empty((sh.R, Hk, K), dtype=torch.int32, device=dev)
        la, lb = lists(), lists()
        A.eng.oasis_score_topk(0, t, qd, topk)
        A.eng.oasis_admit_evict(0, t, topk, *la)
        B.eng.oasis_score_admit_noalloc(0, t, qd, *lb)
        A.eng.oasis_sync()
        B.eng.oasis_sync()
        for x, y in zip(la, lb):
            assert torch.equal(x, y), t
        nxt = (t + 1) & 1
        assert torch.equal(A.eng.res_ids[0][nxt], B.eng.res_ids[0][nxt])
        assert torch.equal(A.eng.phys[0][nxt], B.eng.phys[0][nxt])
        assert torch.equal(A.eng.stamps[0], B.eng.stamps[0])
        # both sides gather their admissions, so step t + 1 starts equal
        A.eng.oasis_prefetch(0, t, la[0], la[1], la[3])
        B.eng.oasis_prefetch(0, t, lb[0], lb[1], lb[3])
        A.eng.oasis_sync()
        B.eng.oasis_sync()
    assert torch.equal(A.eng.kv_pool[0], B.eng.kv_pool[0])
    A.eng.close()
    B.eng.close()


def test_noalloc_refuses_oversize_config(dev):
    # 1025 (request, KV head) pairs x K = 256 > 262144 scratch entries.  The
    # context gets small real buffers: the call must refuse before touching
    # any of them (only oasis_init's clear of the error word runs).
    cfg = ob.make_config(R=1025, NBmax=256, Hq=4, Hkv=1, K=256, fetch_ratio=0.0)
    small = [torch.zeros(1 << 16, dtype=torch.uint8, device=dev) for _ in range(5)]
    host = torch.zeros(1 << 16, dtype=torch.uint8, pin_memory=True)
    ctx_len = torch.zeros(2 * 1025, dtype=torch.int32, device=dev)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    arr = lambda t: ctypes.cast((ctypes.c_void_p * 1)(t.data_ptr()), ctypes.POINTER(ctypes.c_void_p))
    bufs = ob.oasis_buffers(arr(small[0]), arr(small[1]), arr(host), arr(small[2]),
                            arr(small[3]), arr(small[4]), ctx_len.data_ptr(), ws.data_ptr())
    h = ctypes.c_void_p()
    assert ob.lib().oasis_init(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(h)) == 0
    out = torch.zeros(4, dtype=torch.int32, device=dev)
    rc = ob.lib().oasis_score_admit_noalloc(h.value, 0, 0, out.data_ptr(), out.data_ptr(),
                                            out.data_ptr(), out.data_ptr(), out.data_ptr(),
                                            None)
    msg = ob.lib().oasis_last_error(h.value).decode()
    ob.lib().oasis_destroy(h.value)
    assert rc == ob.OASIS_EINVAL
    assert "262144" in msg and "262400" in msg

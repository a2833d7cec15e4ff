"""Failure detection without a GPU fault: a host-side bounded wait that runs
out (the side work is held up by a slow emulated network transfer on the
remote tier's host worker thread, not by a GPU spin) and then succeeds; argument and state errors
reported as status codes with messages."""
import dataclasses
import time

import pytest
import torch

from sparse_kv_block_gb300 import oasis as ob
from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu
TINY = workload.SHAPES["tiny"]


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def test_bounded_wait_times_out_then_completes(dev):
    # 0.001 GB/s: the step's first transfer of up to 2 x 2 x 4 units (64 KiB)
    # takes the remote tier's worker thread ~65 ms; the gather waits for it.
    L = H.make_layer(TINY, seed=61, steps=2, fetch_ratio=0.25, remote_capacity=TINY.NBmax,
                     remote_gbps=0.001)
    eng = L.eng
    out = torch.empty((TINY.R, TINY.Hq, 128), dtype=torch.bfloat16, device=dev)
    outd = torch.empty_like(out)
    t0 = time.perf_counter()
    eng.oasis_step(0, 0, L.q[0].to(dev), L.qd[0].to(dev), out, outd)
    assert time.perf_counter() - t0 < 0.05                   # issuing does not wait for it
    assert eng.oasis_wait(0, 1.0) is False                   # still transferring
    assert "not done" in ob.lib().oasis_last_error(eng.ctx).decode()
    assert eng.oasis_wait(0, 30000.0) is True                # then it finishes
    eng.oasis_sync()
    eng.close()


def test_wait_without_side_work_and_bad_arguments(dev):
    L = H.make_layer(TINY, seed=62, steps=1)
    eng = L.eng
    assert eng.oasis_wait(0, 0.0) is True                    # nothing outstanding
    with pytest.raises(ob.OasisError) as e:
        eng.oasis_wait(5, 1.0)                               # layer out of range
    assert e.value.status == ob.OASIS_EINVAL
    with pytest.raises(ob.OasisError) as e:
        eng.oasis_lookahead_attn(0, 0, None, None, None, None)
    assert e.value.status == ob.OASIS_EINVAL
    eng.close()


def test_step_before_load_is_refused(dev):
    cfg = ob.make_config(TINY.R, TINY.NBmax, TINY.Hq, TINY.Hkv, TINY.K, TINY.fetch_ratio)
    eng = ob.Oasis(cfg)
    q = torch.zeros((TINY.R, TINY.Hq, 128), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ob.OasisError) as e:
        eng.oasis_step(0, 0, q, q, q, q)
    assert e.value.status == ob.OASIS_ESTATE
    eng.close()


def test_init_refuses_a_host_store_that_is_not_page_locked(dev):
    # The library itself (not only the binding) refuses a pageable host store
    # with OASIS_EINVAL and no context; the same buffers with a pinned store
    # give a working context.
    import ctypes
    sh = TINY
    cfg = ob.make_config(sh.R, sh.NBmax, sh.Hq, sh.Hkv, sh.K, sh.fetch_ratio)
    sz = ob.oasis_query_sizes(cfg)
    U = sz.units_per_head
    pool = torch.zeros((sh.R, sh.Hkv, U, 2, 16, 128), dtype=torch.bfloat16, device=dev)
    summ = torch.zeros((sh.R, sh.Hkv, sh.NBmax, 2, 128), dtype=torch.bfloat16, device=dev)
    res = torch.full((2, sh.R, sh.Hkv, sh.K), -1, dtype=torch.int32, device=dev)
    stamps = torch.full((sh.R, sh.Hkv, sh.K), -1, dtype=torch.int32, device=dev)
    phys = torch.zeros((2, sh.R, sh.Hkv, U), dtype=torch.int32, device=dev)
    ctx_len = torch.zeros((2, sh.R), dtype=torch.int32, device=dev)
    ws = torch.zeros(sz.workspace_bytes, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    def init_with(host):
        arrs = [(ctypes.c_void_p * 1)(t.data_ptr()) for t in (pool, summ, host, res, stamps, phys)]
        bufs = ob.oasis_buffers(*[ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)) for a in arrs],
                                ctx_len.data_ptr(), ws.data_ptr())
        h = ctypes.c_void_p()
        rc = ob.lib().oasis_init(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(h))
        return rc, h.value

    pageable = torch.zeros((sh.R, sh.Hkv, sh.NBmax, 2, 16, 128), dtype=torch.bfloat16)
    assert not pageable.is_pinned()
    rc, h = init_with(pageable)
    assert rc == ob.OASIS_EINVAL and h is None
    pinned = pageable.pin_memory()
    rc, h = init_with(pinned)
    assert rc == ob.OASIS_OK and h is not None
    assert ob.lib().oasis_destroy(h) == ob.OASIS_OK

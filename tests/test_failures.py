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

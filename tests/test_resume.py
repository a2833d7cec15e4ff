"""Checkpoint and resume: a layer's state between steps is its caller-owned
buffers (resident table, stamps, context lengths).  Saving them after step
t - 1 and resuming a fresh context with oasis_resume_resident at step t
continues bit for bit like the original context."""
import dataclasses

import numpy as np
import pytest
import torch

from sparse_kv_block_gb300 import workload
from sparse_kv_block_gb300.oasis import Oasis, make_config
from tests import _harness as H

pytestmark = pytest.mark.gpu
TINY = workload.SHAPES["tiny"]


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def test_resume_matches_continuing(dev):
    sh = dataclasses.replace(TINY, R=4)
    A = H.make_layer(sh, seed=71, steps=6, fetch_ratio=0.25, out_fp32=True)
    eng = A.eng
    outs = lambda: (torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev),
                    torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev))
    for t in range(3):
        o, od = outs()
        eng.oasis_step(0, t, A.q[t].to(dev), A.qd[t].to(dev), o, od)
    eng.oasis_join(0)
    eng.oasis_sync()
    t = 3
    saved_res = eng.res_ids[0][t & 1].clone()
    saved_stamps = eng.stamps[0].clone()
    saved_ctx = eng.ctx_len[t & 1].clone()

    cfg = make_config(sh.R, sh.NBmax, sh.Hq, sh.Hkv, sh.K, sh.fetch_ratio, out_fp32=True)
    B = Oasis(cfg, host_kv=[A.host])
    B.ctx_len[t & 1].copy_(saved_ctx)
    B.ctx_len[(t + 1) & 1].copy_(saved_ctx)
    B.res_ids[0][t & 1].copy_(saved_res)
    B.stamps[0].copy_(saved_stamps)
    B.oasis_build_summaries(0, t & 1)
    B.oasis_resume_resident(0, t)
    B.oasis_sync()
    assert torch.equal(B.stamps[0], saved_stamps)
    for t in range(3, 6):
        oa, oda = outs()
        ob_, odb = outs()
        eng.oasis_step(0, t, A.q[t].to(dev), A.qd[t].to(dev), oa, oda)
        B.oasis_step(0, t, A.q[t].to(dev), A.qd[t].to(dev), ob_, odb)
        eng.oasis_join(0)
        B.oasis_join(0)
        eng.oasis_sync()
        B.oasis_sync()
        assert torch.equal(oa, ob_) and torch.equal(oda, odb), t
        nxt = (t + 1) & 1
        assert torch.equal(eng.res_ids[0][nxt], B.res_ids[0][nxt]), t
        assert torch.equal(eng.stamps[0], B.stamps[0]), t
    eng.close()
    B.close()

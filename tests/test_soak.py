"""Soak: thousands of fused steps issued back to back (double-buffered
tables and lists, side streams reused every step) keep every invariant: no
device error bits, a full set of distinct resident ids in range, each
table's units a permutation, and every resident pool unit byte-equal to its
host block.  (Parity with the oracle is covered by the lockstep tests; here
no oracle is fed anything the GPU produced.)"""
import dataclasses

import numpy as np
import pytest
import torch

from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu
TINY = workload.SHAPES["tiny"]


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def test_three_thousand_steps(dev):
    sh = dataclasses.replace(TINY, R=4, ctx=2048)
    nq = 16
    L = H.make_layer(sh, seed=81, steps=nq, fetch_ratio=0.25, out_fp32=True, schedule=3)
    eng = L.eng
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    step = 0
    for chunk in range(6):
        for _ in range(499):
            eng.oasis_step(0, step, qg[step % nq], qdg[step % nq], out, outd)
            step += 1
        t = step
        eng.oasis_step(0, t, qg[t % nq], qdg[t % nq], out, outd)
        step += 1
        eng.oasis_join(0)
        assert eng.oasis_sync() == 0
        # tables after step t (the next step's) and the pool
        nxt = (t + 1) & 1
        resn = eng.res_ids[0][nxt].cpu().numpy()
        for r in range(sh.R):
            for h in range(sh.Hkv):
                ids = resn[r, h][resn[r, h] >= 0]
                assert len(set(ids.tolist())) == len(ids) == sh.K
                assert ids.min() >= 0 and ids.max() < sh.NBmax
        H.check_pool(L, nxt)
    eng.close()

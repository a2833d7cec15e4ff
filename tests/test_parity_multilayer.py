"""GPU parity of a multi-layer decode loop: several layers, each with its own
host store, summaries and resident state, stepped in layer order on one main
stream while every layer's side work (scan, top-K, admission, gather) runs on
the context's shared side streams and overlaps the next layers."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_kv_block_gb300 import workload
from sparse_kv_block_gb300.oasis import Oasis, make_config
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("schedule", [0, 1, 2, 3, 4])
def test_three_layers_interleaved(dev, schedule):
    sh = dataclasses.replace(workload.SHAPES["tiny"], R=3, ctx=900, layers=3)
    nl, steps = 3, 5
    lens = workload.ctx_lens(sh)
    hosts, qs, qds, res0s = [], [], [], []
    for l in range(nl):
        h = torch.empty((sh.R, sh.Hkv, sh.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                        pin_memory=True)
        workload.host_kv(sh, 21, l, lens, out=h)
        q, qd = workload.queries(sh, 21, l, steps)
        hosts.append(h)
        qs.append(q)
        qds.append(qd)
        res0s.append(workload.initial_resident(sh, 21, l, lens))
    cfg = make_config(sh.R, sh.NBmax, sh.Hq, sh.Hkv, sh.K, sh.fetch_ratio, layers=nl,
                      out_fp32=True, side_groups=2, schedule=schedule)
    eng = Oasis(cfg, host_kv=hosts)
    eng.set_context(lens)
    orcs = []
    for l in range(nl):
        eng.set_resident(l, res0s[l], 0)
        eng.oasis_build_summaries(l, 0)
        eng.oasis_load_resident(l, 0)
        hb = workload.bf16_bits(hosts[l])
        orcs.append(oracle.LayerOracle(hb, oracle.summary_build(hb, lens), lens, res0s[l],
                                       sh.K, sh.C, [(r, h) for r in range(sh.R)
                                                    for h in range(sh.Hkv)]))
    eng.oasis_sync()
    outs = [torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev) for _ in range(nl)]
    outds = [torch.empty_like(o) for o in outs]
    qg = [q.to(dev) for q in qs]
    qdg = [q.to(dev) for q in qds]
    torch.cuda.synchronize()  # the early-scan schedule reads q_draft when the call is made
    for t in range(steps):
        for l in range(nl):      # no host sync between layers
            eng.oasis_step(l, t, qg[l][t], qdg[l][t], outs[l], outds[l])
        for l in range(nl):
            eng.oasis_join(l)
        eng.oasis_sync()
        for l in range(nl):
            ref = orcs[l].step(workload.bf16_bits(qs[l][t]), workload.bf16_bits(qds[l][t]), t)
            H.check_attention([outs[l].cpu().numpy(), outds[l].cpu().numpy()], ref, sh.G)
            lists = {k: v.cpu().numpy() for k, v in eng.step_lists(l, t).items()}
            for (r, h), v in ref.items():
                assert np.array_equal(lists["topk_ids"][r, h], v["topk"])
                assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
            assert (eng.res_ids[l][(t + 1) & 1].cpu().numpy() == orcs[l].res).all()
            pool = workload.bf16_bits(eng.kv_pool[l].cpu())
            res = eng.res_ids[l][(t + 1) & 1].cpu().numpy()
            phys = eng.phys[l][(t + 1) & 1].cpu().numpy()
            hb = workload.bf16_bits(hosts[l])
            for r in range(sh.R):
                for h in range(sh.Hkv):
                    for s in range(sh.K):
                        if res[r, h, s] >= 0:
                            np.testing.assert_array_equal(pool[r, h, phys[r, h, s]],
                                                          hb[r, h, res[r, h, s]])
    eng.close()

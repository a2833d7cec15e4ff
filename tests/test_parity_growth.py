"""GPU parity for growing contexts (one decoded token appended per request per
step, crossing block boundaries): the append writes the host store, folds the
key into the tail summary and patches the resident copy; ctx_len advances.
The oracle works on its own copy of the host store, so the bytes the GPU
writes into pinned memory are checked, not shared."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("ctx0,steps", [(1000, 40), (250, 30)])
def test_append_and_advance_match_oracle(dev, ctx0, steps):
    sh = dataclasses.replace(workload.SHAPES["tiny"], ctx=ctx0, grow_steps=steps)
    L = H.make_layer(sh, seed=11, steps=steps, out_fp32=True)
    eng = L.eng
    hb_orc = L.hb.copy()                       # the oracle's own host store
    summ_orc = L.summ.copy()
    lens = L.lens.copy()
    orc = oracle.LayerOracle(hb_orc, summ_orc, lens, L.res0, sh.K, sh.C, L.orc.pairs)
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    for t in range(steps):
        eng.oasis_step(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        k_new, v_new = workload.new_tokens(sh, 11, 0, t)
        eng.oasis_append_token(0, t, k_new.to(dev), v_new.to(dev))
        eng.oasis_advance_context(t, 1)
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        kb, vb = workload.bf16_bits(k_new), workload.bf16_bits(v_new)
        for r in range(sh.R):
            oracle.append_token(hb_orc, summ_orc, lens, kb[r], vb[r], r)
        lens += 1
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
        for (r, h), v in ref.items():
            assert np.array_equal(lists["topk_ids"][r, h], v["topk"])
            assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
        nxt = (t + 1) & 1
        assert (eng.ctx_len[nxt].cpu().numpy() == lens).all()
        assert (eng.res_ids[0][nxt].cpu().numpy() == orc.res).all()
        # host store written by the GPU == the oracle's copy (all blocks)
        np.testing.assert_array_equal(L.hb, hb_orc)
        gs = workload.bf16_bits(eng.summaries[0].cpu())
        for r in range(sh.R):
            nb = -(-int(lens[r]) // 16)
            np.testing.assert_array_equal(H.bits_to_float(gs[r, :, :nb]),
                                          H.bits_to_float(summ_orc[r, :, :nb]))
        # resident copies include the appended token
        res = eng.res_ids[0][nxt].cpu().numpy()
        phys = eng.phys[0][nxt].cpu().numpy()
        pool = workload.bf16_bits(eng.kv_pool[0].cpu())
        for r in range(sh.R):
            for h in range(sh.Hkv):
                for s in range(sh.K):
                    if res[r, h, s] >= 0:
                        np.testing.assert_array_equal(pool[r, h, phys[r, h, s]],
                                                      hb_orc[r, h, res[r, h, s]])
    eng.close()


@pytest.mark.parametrize("schedule", [0, 4])
def test_growth_steps_back_to_back(dev, schedule):
    # Steps, appends and context advances issued with no host wait at all.
    # Under the early-scan schedule the scan of step t + 1 runs on its own
    # stream and must still see the token appended after step t (the tail
    # summary) and the advanced context length.
    steps = 24
    sh = dataclasses.replace(workload.SHAPES["tiny"], R=3, ctx=990, grow_steps=steps)
    L = H.make_layer(sh, seed=12, lens=[990, 1000, 31], steps=steps, out_fp32=True,
                     schedule=schedule)
    eng = L.eng
    hb_orc = L.hb.copy()
    summ_orc = L.summ.copy()
    lens = L.lens.copy()
    orc = oracle.LayerOracle(hb_orc, summ_orc, lens, L.res0, sh.K, sh.C, L.orc.pairs)
    outs = [torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
            for _ in range(2 * steps)]
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    toks = [workload.new_tokens(sh, 12, 0, t) for t in range(steps)]
    toks_d = [(k.to(dev), v.to(dev)) for k, v in toks]
    torch.cuda.synchronize()  # the early-scan schedule reads q_draft when the call is made
    for t in range(steps):
        eng.oasis_step(0, t, qg[t], qdg[t], outs[2 * t], outs[2 * t + 1])
        eng.oasis_append_token(0, t, *toks_d[t])
        eng.oasis_advance_context(t, 1)
    eng.oasis_join(0)
    eng.oasis_sync()
    for t in range(steps):
        ref = orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        kb, vb = workload.bf16_bits(toks[t][0]), workload.bf16_bits(toks[t][1])
        for r in range(sh.R):
            oracle.append_token(hb_orc, summ_orc, lens, kb[r], vb[r], r)
        lens += 1
        H.check_attention([outs[2 * t].cpu().numpy(), outs[2 * t + 1].cpu().numpy()], ref, sh.G)
        if t >= steps - 2:   # the lists of the last two steps are still in place
            lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
            for (r, h), v in ref.items():
                assert np.array_equal(lists["topk_ids"][r, h], v["topk"])
    nxt = steps & 1
    assert (eng.ctx_len[nxt].cpu().numpy() == lens).all()
    assert (eng.res_ids[0][nxt].cpu().numpy() == orc.res).all()
    assert (eng.stamps[0].cpu().numpy() == orc.stamp).all()
    np.testing.assert_array_equal(L.hb, hb_orc)
    gs = workload.bf16_bits(eng.summaries[0].cpu())
    for r in range(sh.R):
        nb = -(-int(lens[r]) // 16)
        np.testing.assert_array_equal(H.bits_to_float(gs[r, :, :nb]),
                                      H.bits_to_float(summ_orc[r, :, :nb]))
    eng.close()

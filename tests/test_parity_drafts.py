"""GPU parity with several draft queries per step (D = 2 or 3): every draft's
attention over the one resident set, and the summary scan with the drafts'
bounds summed, through the C ABI against the oracle, on the tiny workload and
its edge cases, on the fused and host-buffer steps, on the dense anchor, and
on sampled pairs of the full 128 x 16K Qwen3-8B-shaped layer."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu

TINY = workload.SHAPES["tiny"]


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def check_lists(eng, t, ref, C):
    lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
    for (r, h), v in ref.items():
        # a different list inside the tie window would end the lockstep run
        assert np.array_equal(lists["topk_ids"][r, h], v["topk"]), "tie window hit"
        assert lists["n_admit"][r, h] == v["n_admit"]
        assert (lists["admit_ids"][r, h, :C] == v["admit_ids"]).all()
        assert (lists["admit_slots"][r, h, :C] == v["admit_slots"]).all()
        assert (lists["evict_ids"][r, h, :C] == v["evict_ids"]).all()


@pytest.mark.parametrize("D,out_fp32", [(2, True), (3, True), (3, False)])
def test_staged_steps(dev, D, out_fp32):
    L = H.make_layer(TINY, seed=20, steps=5, out_fp32=out_fp32, num_drafts=D)
    assert tuple(L.qd.shape[1:3]) == (D, TINY.R)
    for t in range(5):
        H.run_staged_step(L, t, dev)
    L.eng.close()


@pytest.mark.parametrize("D,Hq,lens", [(2, 4, [700, 33, 0, 1024, 16]),
                                       (3, 2, [1024, 1, 500, 999, 64]),
                                       (3, 8, [0, 0, 17, 1024, 513])])
def test_small_groups_ragged_contexts(dev, D, Hq, lens):
    # G = 2, G = 1 and G = 4 with 2 or 3 drafts: 6 to 16 query columns per
    # KV head; empty, one-token and ragged contexts.
    sh = dataclasses.replace(TINY, R=5, Hq=Hq, Hkv=2)
    L = H.make_layer(sh, seed=21, lens=lens, steps=3, out_fp32=True, num_drafts=D)
    H.check_summaries(L)
    for t in range(3):
        H.run_staged_step(L, t, dev)
    L.eng.close()


@pytest.mark.parametrize("schedule,groups", [(0, 0), (1, 3), (2, 3), (3, 0), (4, 2)])
def test_fused_steps_back_to_back(dev, schedule, groups):
    # oasis_step with three drafts, six steps issued with no host wait between
    # them; the draft planes are staged per step by the library (on the scan
    # stream under the early-scan schedule).
    D = 3
    sh = dataclasses.replace(TINY, R=5)
    L = H.make_layer(sh, seed=22, steps=6, out_fp32=True, side_groups=groups,
                     schedule=schedule, num_drafts=D)
    eng = L.eng
    outs = [torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev) for _ in range(6)]
    outds = [torch.empty((D, sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
             for _ in range(6)]
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    torch.cuda.synchronize()  # the early-scan schedule reads q_draft when the call is made
    for t in range(6):
        eng.oasis_step(0, t, qg[t], qdg[t], outs[t], outds[t])
    eng.oasis_join(0)
    eng.oasis_sync()
    for t in range(6):
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([outs[t].cpu().numpy(), outds[t].cpu().numpy()], ref, sh.G)
        if t >= 4:   # the lists of the last two steps are still in place
            check_lists(eng, t, ref, sh.C)
    assert (eng.res_ids[0][6 & 1].cpu().numpy() == L.orc.res).all()
    assert (eng.stamps[0].cpu().numpy() == L.orc.stamp).all()
    H.check_pool(L, 6 & 1)
    eng.close()


def test_host_buffer_steps(dev):
    D = 2
    sh = dataclasses.replace(TINY, R=5)
    L = H.make_layer(sh, seed=23, steps=4, out_fp32=False, num_drafts=D)
    eng = L.eng
    bufs = []
    for t in range(4):
        q = torch.empty((sh.R, sh.Hq, 128), dtype=torch.bfloat16, pin_memory=True)
        qd = torch.empty((D, sh.R, sh.Hq, 128), dtype=torch.bfloat16, pin_memory=True)
        o = torch.empty_like(q).pin_memory()
        od = torch.empty_like(qd).pin_memory()
        q.copy_(L.q[t])
        qd.copy_(L.qd[t])
        bufs.append((q, qd, o, od))
        eng.oasis_step_host(0, t, q, qd, o, od)
    torch.cuda.synchronize()
    eng.oasis_join(0)
    eng.oasis_sync()
    for t in range(4):
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([bufs[t][2].float().numpy(), bufs[t][3].float().numpy()], ref, sh.G)
    assert (eng.res_ids[0][4 & 1].cpu().numpy() == L.orc.res).all()
    eng.close()


def test_binding_refuses_a_one_plane_draft_tensor(dev):
    # With D = 2 a [R][Hq][d] draft tensor is half the bytes the call reads.
    L = H.make_layer(TINY, seed=24, steps=1, num_drafts=2)
    q = L.q[0].to(dev)
    out = torch.empty((TINY.R, TINY.Hq, 128), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError, match="q_draft"):
        L.eng.oasis_step(0, 0, q, q, out, torch.empty((2,) + tuple(out.shape), dtype=out.dtype,
                                                      device=dev))
    with pytest.raises(ValueError, match="out_draft"):
        L.eng.oasis_lookahead_attn(0, 0, q, L.qd[0].to(dev), out, out)
    L.eng.close()


def test_dense_anchor_with_drafts(dev):
    D = 3
    L = H.make_layer(TINY, seed=25, lens=[1000, 37], steps=1, out_fp32=True, num_drafts=D)
    sh, eng = L.shape, L.eng
    kv_dense = L.host.to(dev)
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty((D, sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    eng.oasis_dense_attn(kv_dense, 0, L.q[0].to(dev), L.qd[0].to(dev), out, outd)
    eng.oasis_sync()
    every = np.broadcast_to(np.arange(sh.NBmax, dtype=np.int32), (sh.R, sh.Hkv, sh.NBmax)).copy()
    qb, qdb = workload.bf16_bits(L.q[0]), workload.bf16_bits(L.qd[0])
    ref = {(r, h): {"attn": oracle.attention_rh(L.hb, L.lens, every, qb, qdb, r, h)}
           for r in range(sh.R) for h in range(sh.Hkv)}
    H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
    eng.close()


def test_full_size_layer_three_drafts_sampled(dev):
    # 128 requests x 16K tokens, three drafts: staged lockstep steps, then
    # fused steps on the sampled pairs (a pair leaves the check if its list
    # differs inside the tie window).
    sh = workload.SHAPES["qwen3_8b_16k"]
    sample = [(0, 0), (9, 3), (64, 7), (127, 5)]
    D = 3
    L = H.make_layer(sh, seed=26, steps=5, gen_device="cuda", pairs=sample, num_drafts=D)
    for t in range(2):
        H.run_staged_step(L, t, dev, check_pool_every=False)
        H.check_pool(L, (t + 1) & 1, sample)
    eng = L.eng
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.bfloat16, device=dev)
    outd = torch.empty((D, sh.R, sh.Hq, 128), dtype=torch.bfloat16, device=dev)
    live = list(sample)
    for t in range(2, 5):
        eng.oasis_step(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        L.orc.pairs = live
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([out.float().cpu().numpy(), outd.float().cpu().numpy()], ref, sh.G)
        lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
        res_n = eng.res_ids[0][(t + 1) & 1].cpu().numpy()
        keep = []
        for (r, h), v in ref.items():
            assert H.topk_agrees(lists["topk_ids"][r, h], v["topk"], v["scores"], sh.K)
            if not np.array_equal(lists["topk_ids"][r, h], v["topk"]):
                continue
            assert lists["n_admit"][r, h] == v["n_admit"]
            assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
            assert (res_n[r, h] == L.orc.res[r, h]).all()
            keep.append((r, h))
        live = keep
        assert len(live) >= len(sample) - 1
        H.check_pool(L, (t + 1) & 1, live)
    eng.close()


def test_drafts_with_remote_tier(dev):
    # Three drafts with the emulated remote tier: the admitted blocks that the
    # drafts' summed bounds select are fetched into the local tier first.
    D = 3
    sh = dataclasses.replace(TINY, R=4)
    L = H.make_layer(sh, seed=27, steps=5, fetch_ratio=0.25, out_fp32=True, side_groups=2,
                     remote_capacity=48, num_drafts=D)
    eng = L.eng
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty((D, sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    for t in range(5):
        eng.oasis_step(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        check_lists(eng, t, ref, sh.C)
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        H.check_remote(L, ref)
        H.check_pool(L, (t + 1) & 1)
    eng.close()


@pytest.mark.parametrize("schedule", [0, 4])
def test_drafts_with_growing_contexts(dev, schedule):
    # Two drafts while every request grows by one token per step (appends and
    # context advances issued back to back with the steps, no host wait).
    D, steps = 2, 20
    sh = dataclasses.replace(TINY, R=3, ctx=990, grow_steps=steps)
    L = H.make_layer(sh, seed=28, lens=[990, 1000, 47], steps=steps, out_fp32=True,
                     schedule=schedule, num_drafts=D)
    eng = L.eng
    hb_orc, summ_orc, lens = L.hb.copy(), L.summ.copy(), L.lens.copy()
    orc = oracle.LayerOracle(hb_orc, summ_orc, lens, L.res0, sh.K, sh.C, L.orc.pairs)
    outs = [torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev) for _ in range(steps)]
    outds = [torch.empty((D, sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
             for _ in range(steps)]
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    toks = [workload.new_tokens(sh, 28, 0, t) for t in range(steps)]
    toks_d = [(k.to(dev), v.to(dev)) for k, v in toks]
    torch.cuda.synchronize()  # the early-scan schedule reads q_draft when the call is made
    for t in range(steps):
        eng.oasis_step(0, t, qg[t], qdg[t], outs[t], outds[t])
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
        H.check_attention([outs[t].cpu().numpy(), outds[t].cpu().numpy()], ref, sh.G)
    assert (eng.res_ids[0][steps & 1].cpu().numpy() == orc.res).all()
    assert (eng.stamps[0].cpu().numpy() == orc.stamp).all()
    np.testing.assert_array_equal(L.hb, hb_orc)
    eng.close()

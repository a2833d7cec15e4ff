"""GPU parity on the tiny workload (2 requests x 1024 tokens, 8 q / 2 KV heads,
K = 16, cap 0.25) and its edge cases, through the C ABI, against the oracle."""
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
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("out_fp32", [True, False])
def test_staged_eight_steps(dev, out_fp32):
    L = H.make_layer(TINY, seed=0, steps=8, out_fp32=out_fp32)
    H.check_summaries(L)
    H.check_pool(L, 0)
    for t in range(8):
        H.run_staged_step(L, t, dev)
    L.eng.close()


def test_dense_when_k_covers_every_block(dev):
    # K = NB = 64: sparse attention equals dense attention over the context.
    L = H.make_layer(TINY, seed=1, steps=2, K=64, fetch_ratio=0.25, out_fp32=True)
    for t in range(2):
        ref = H.run_staged_step(L, t, dev)
        for v in ref.values():
            assert v["n_admit"] == 0
    L.eng.close()


@pytest.mark.parametrize("lens", [[1000, 37], [16, 1024], [0, 5], [1024, 1], [0, 0]])
def test_ragged_contexts(dev, lens):
    L = H.make_layer(TINY, seed=2, lens=lens, steps=3, out_fp32=True)
    H.check_summaries(L)
    for t in range(3):
        H.run_staged_step(L, t, dev)
    L.eng.close()


@pytest.mark.parametrize("ratio", [0.0, 1.0, 0.0625])
def test_fetch_cap_extremes(dev, ratio):
    L = H.make_layer(TINY, seed=3, steps=3, fetch_ratio=ratio, out_fp32=True)
    for t in range(3):
        ref = H.run_staged_step(L, t, dev)
        if ratio == 1.0:   # fetch-all: the resident set becomes the top-K set
            for (r, h), v in ref.items():
                assert set(L.orc.res[r, h].tolist()) == set(v["topk"].tolist())
    L.eng.close()


def test_small_groups_and_many_requests(dev):
    sh = dataclasses.replace(TINY, R=5, Hq=4, Hkv=2, ctx=700)   # G = 2, ragged tail
    L = H.make_layer(sh, seed=4, steps=3, out_fp32=True)
    for t in range(3):
        H.run_staged_step(L, t, dev)
    L.eng.close()


@pytest.mark.parametrize("groups,R,schedule", [(0, 2, 0), (3, 5, 0), (10, 5, 0), (3, 5, 1),
                                               (3, 5, 2), (0, 2, 2), (0, 5, 3), (0, 2, 4),
                                               (3, 5, 4)])
def test_fused_step_matches_oracle(dev, groups, R, schedule):
    # oasis_step: fused scan + top-K + admission per request group on one side
    # stream, gathers per group on another; uneven and one-pair groups too;
    # both schedules.
    sh = dataclasses.replace(TINY, R=R)
    L = H.make_layer(sh, seed=5, steps=6, out_fp32=True, side_groups=groups, schedule=schedule)
    eng = L.eng
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    for t in range(6):
        qg, qdg = L.q[t].to(dev), L.qd[t].to(dev)
        torch.cuda.synchronize()  # the early-scan schedule reads q_draft when the call is made
        eng.oasis_step(0, t, qg, qdg, out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
        for (r, h), v in ref.items():
            # a different list inside the tie window would end the lockstep run
            assert np.array_equal(lists["topk_ids"][r, h], v["topk"]), "tie window hit"
            assert lists["n_admit"][r, h] == v["n_admit"]
            assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
            assert (lists["admit_slots"][r, h, :sh.C] == v["admit_slots"]).all()
            assert (lists["evict_ids"][r, h, :sh.C] == v["evict_ids"]).all()
        assert (eng.res_ids[0][(t + 1) & 1].cpu().numpy() == L.orc.res).all()
        assert (eng.stamps[0].cpu().numpy() == L.orc.stamp).all()
        H.check_pool(L, (t + 1) & 1)
    eng.close()


@pytest.mark.parametrize("lens", [None, [0]])
def test_single_pair_fused_steps(dev, lens):
    # One request with one KV head (G = 4): one-CTA grids everywhere; also
    # with an empty context (nothing to rank, admit or attend: zero outputs).
    sh = dataclasses.replace(TINY, R=1, Hq=4, Hkv=1)
    L = H.make_layer(sh, seed=8, steps=4, lens=lens, out_fp32=True)
    eng = L.eng
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    for t in range(4):
        eng.oasis_step(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        if lens == [0]:
            assert not out.any() and not outd.any()
        lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
        v = ref[(0, 0)]
        assert np.array_equal(lists["topk_ids"][0, 0], v["topk"])
        assert lists["n_admit"][0, 0] == v["n_admit"]
        assert (eng.res_ids[0][(t + 1) & 1].cpu().numpy() == L.orc.res).all()
        assert (eng.stamps[0].cpu().numpy() == L.orc.stamp).all()
        H.check_pool(L, (t + 1) & 1)
    eng.close()


def test_host_buffer_step_matches_device_step(dev):
    L = H.make_layer(TINY, seed=6, steps=3, out_fp32=False)
    sh, eng = L.shape, L.eng
    qh = torch.empty((sh.R, sh.Hq, 128), dtype=torch.bfloat16, pin_memory=True)
    qdh = torch.empty_like(qh).pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    odh = torch.empty_like(qh).pin_memory()
    for t in range(3):
        qh.copy_(L.q[t])
        qdh.copy_(L.qd[t])
        eng.oasis_step_host(0, t, qh, qdh, oh, odh)
        torch.cuda.synchronize()
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([oh.float().numpy(), odh.float().numpy()], ref, sh.G)
        assert (eng.res_ids[0][(t + 1) & 1].cpu().numpy() == L.orc.res).all()
    eng.close()


def test_host_buffer_step_pageable_outputs(dev):
    # Outputs in pageable host memory cannot be written through a device
    # mapping: the step falls back to the workspace and a copy back.
    L = H.make_layer(TINY, seed=10, steps=2, out_fp32=True)
    sh, eng = L.shape, L.eng
    for t in range(2):
        qh = L.q[t].clone().pin_memory()
        qdh = L.qd[t].clone().pin_memory()
        oh = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32)      # pageable
        odh = torch.empty_like(oh)
        assert not oh.is_pinned()
        eng.oasis_step_host(0, t, qh, qdh, oh, odh)
        torch.cuda.synchronize()
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([oh.numpy(), odh.numpy()], ref, sh.G)
    eng.close()


@pytest.mark.parametrize("schedule", [0, 1, 3, 4])
def test_host_buffer_steps_back_to_back(dev, schedule):
    # oasis_step_host issued for consecutive steps with no host wait between
    # them: step t + 1's input copies may overlap step t's side work; every
    # schedule but the pages' three streams (the automatic one is scan-first).
    sh = dataclasses.replace(TINY, R=5)
    L = H.make_layer(sh, seed=9, steps=6, fetch_ratio=0.25, out_fp32=False, schedule=schedule)
    eng = L.eng

    def pinned():
        return torch.empty((sh.R, sh.Hq, 128), dtype=torch.bfloat16, pin_memory=True)
    bufs = [[pinned() for _ in range(4)] for _ in range(6)]
    for t in range(6):
        bufs[t][0].copy_(L.q[t])
        bufs[t][1].copy_(L.qd[t])
        eng.oasis_step_host(0, t, *bufs[t])
    torch.cuda.synchronize()
    eng.oasis_join(0)
    eng.oasis_sync()
    for t in range(6):
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([bufs[t][2].float().numpy(), bufs[t][3].float().numpy()], ref, sh.G)
    assert (eng.res_ids[0][6 & 1].cpu().numpy() == L.orc.res).all()
    H.check_pool(L, 6 & 1)
    eng.close()


@pytest.mark.parametrize("schedule,mixed", [(3, False), (0, False), (1, False), (3, True)])
def test_host_buffer_async_outputs(dev, schedule, mixed):
    # oasis_step_host_async: the outputs of step t come back on the library's
    # output stream; the host waits for them with oasis_wait_outputs, two
    # steps later, in a two-deep ring of output buffers.  `mixed` alternates
    # with the stream-ordered oasis_step_host (slot reuse across both).
    sh = dataclasses.replace(TINY, R=5)
    L = H.make_layer(sh, seed=15, steps=8, fetch_ratio=0.25, out_fp32=False, schedule=schedule)
    eng = L.eng

    def pinned():
        return torch.empty((sh.R, sh.Hq, 128), dtype=torch.bfloat16, pin_memory=True)
    qh, qdh = [pinned() for _ in range(8)], [pinned() for _ in range(8)]
    for t in range(8):
        qh[t].copy_(L.q[t])
        qdh[t].copy_(L.qd[t])
    oh, odh = [pinned(), pinned()], [pinned(), pinned()]
    got = {}
    for t in range(8):
        b = t & 1
        if t >= 2:
            assert eng.oasis_wait_outputs(0, t - 2, 30000.0)
            got[t - 2] = (oh[b].float().numpy().copy(), odh[b].float().numpy().copy())
        if mixed and t % 2:
            eng.oasis_step_host(0, t, qh[t], qdh[t], oh[b], odh[b])
        else:
            eng.oasis_step_host_async(0, t, qh[t], qdh[t], oh[b], odh[b])
    for t in (6, 7):
        assert eng.oasis_wait_outputs(0, t, 30000.0)
        got[t] = (oh[t & 1].float().numpy().copy(), odh[t & 1].float().numpy().copy())
    with pytest.raises(Exception) as ei:       # step 5's slot now holds step 7
        eng.oasis_wait_outputs(0, 5, 1.0)
    assert "no outputs of step 5" in str(ei.value)
    eng.oasis_join(0)
    eng.oasis_sync()
    for t in range(8):
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([got[t][0], got[t][1]], ref, sh.G)
    assert (eng.res_ids[0][8 & 1].cpu().numpy() == L.orc.res).all()
    H.check_pool(L, 8 & 1)
    eng.close()


def test_device_error_word_on_bad_block_id(dev):
    # An id past the context is reported through oasis_sync, not a fault:
    # the kernels skip it and set a bit in the device error word.
    L = H.make_layer(TINY, seed=7, steps=1)
    bad = L.res0.copy()
    bad[0, 0, 0] = 63
    L.eng.set_context([1000, 1024])     # block 63 starts at token 1008 >= 1000
    L.eng.set_resident(0, bad, 0)
    out = torch.empty((TINY.R, TINY.Hq, 128), dtype=torch.bfloat16, device=dev)
    L.eng.oasis_lookahead_attn(0, 0, L.q[0].to(dev), L.qd[0].to(dev), out, torch.empty_like(out))
    with pytest.raises(Exception) as ei:
        L.eng.oasis_sync()
    assert "0x1" in str(ei.value)
    assert L.eng.oasis_sync() == 0      # bits were cleared
    L.eng.close()


@pytest.mark.parametrize("ratio,groups,schedule", [(1.0, 3, 0), (0.25, 0, 1), (1.0, 1, 1),
                                                    (1.0, 3, 2), (0.25, 0, 4), (1.0, 3, 4)])
def test_back_to_back_steps_without_host_sync(dev, ratio, groups, schedule):
    # Steps issued back to back: step t+1's scan and admission may run while
    # step t's gathers are still copying, so the step lists must be per step.
    sh = dataclasses.replace(TINY, R=5)
    L = H.make_layer(sh, seed=8, steps=8, fetch_ratio=ratio, out_fp32=True,
                     side_groups=groups, schedule=schedule)
    eng, sh = L.eng, L.shape
    outs = [torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev) for _ in range(16)]
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    torch.cuda.synchronize()  # the early-scan schedule reads q_draft when the call is made
    for t in range(8):
        eng.oasis_step(0, t, qg[t], qdg[t], outs[2 * t], outs[2 * t + 1])
    eng.oasis_join(0)
    eng.oasis_sync()
    for t in range(8):
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([outs[2 * t].cpu().numpy(), outs[2 * t + 1].cpu().numpy()], ref, sh.G)
        if t >= 6:   # the lists of the last two steps are still in place
            lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
            for (r, h), v in ref.items():
                assert np.array_equal(lists["topk_ids"][r, h], v["topk"])
                assert lists["n_admit"][r, h] == v["n_admit"]
                assert (lists["admit_slots"][r, h, :sh.C] == v["admit_slots"]).all()
    assert (eng.res_ids[0][8 & 1].cpu().numpy() == L.orc.res).all()
    assert (eng.stamps[0].cpu().numpy() == L.orc.stamp).all()
    H.check_pool(L, 8 & 1)
    eng.close()

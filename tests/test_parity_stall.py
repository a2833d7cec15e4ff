"""GPU parity of the miss-stall step (the other outcome of a look-ahead miss,
"Pith review of OasisKV", section "What would settle it": fetch on demand
and stall instead of dropping context) through the C ABI against the
oracle's stall step: the demand ranking with the normal query, its uncapped
in-place admission and gather, the attention over the updated table, then
the look-ahead part of the step.

Stage by stage (oasis_demand_topk, oasis_admit_demand, oasis_fetch_demand,
then the look-ahead stages) with the oracle's lists driving both admissions,
and fused (oasis_step_stall), on the tiny workload, its edge cases, mixed
with look-ahead steps, and on sampled pairs of the full 128 x 16K layer."""
import dataclasses

import numpy as np
import pytest
import torch

from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu

TINY = workload.SHAPES["tiny"]
QWEN = workload.SHAPES["qwen3_8b_16k"]
# 64 pairs spread over every KV head, the first, middle and last requests
# (so over the first and last waves of the one-CTA-per-pair grids).
QWEN_SAMPLE = sorted({(r, (r * 5 + k) % 8) for r in list(range(0, 128, 4)) for k in (0, 3)})


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def bits(x):
    return workload.bf16_bits(x)


@pytest.mark.parametrize("out_fp32", [True, False])
def test_staged_stall_steps(dev, out_fp32):
    L = H.make_layer(TINY, seed=10, steps=6, out_fp32=out_fp32)
    for t in range(6):
        H.run_staged_stall_step(L, t, dev)
    L.eng.close()


@pytest.mark.parametrize("lens,ratio", [([1000, 37], 0.25), ([0, 5], 0.25), ([16, 1024], 0.0),
                                        ([1024, 1], 1.0)])
def test_staged_stall_edge_cases(dev, lens, ratio):
    # ragged tails, an empty request, fewer blocks than K, no look-ahead
    # fetch at all, fetch-all look-ahead
    L = H.make_layer(TINY, seed=11, lens=lens, fetch_ratio=ratio, steps=3, out_fp32=True)
    for t in range(3):
        H.run_staged_stall_step(L, t, dev)
    L.eng.close()


@pytest.mark.parametrize("groups,R,num_drafts", [(0, 2, 1), (3, 5, 1), (0, 2, 2)])
def test_fused_stall_steps_match_oracle(dev, groups, R, num_drafts):
    sh = dataclasses.replace(TINY, R=R)
    L = H.make_layer(sh, seed=12, steps=5, out_fp32=True, side_groups=groups,
                     num_drafts=num_drafts)
    eng = L.eng
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty(tuple(L.qd[0].shape), dtype=torch.float32, device=dev)
    for t in range(5):
        eng.oasis_step_stall(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = L.orc.stall_step(bits(L.q[t]), bits(L.qd[t]), t)
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        H.check_stall_step(L, t, ref, exact=True)
        H.check_pool(L, t & 1)          # the demand fetch filled the table attended
        H.check_pool(L, (t + 1) & 1)    # the look-ahead gathers filled the next one
    eng.close()


def test_stall_and_lookahead_steps_mix(dev):
    # drop, stall, stall, drop, stall on one layer, back to back with no host
    # synchronisation, against the oracle's step / stall step in that order
    L = H.make_layer(TINY, seed=13, steps=5, out_fp32=True)
    eng = L.eng
    kinds = ["drop", "stall", "stall", "drop", "stall"]
    outs = [torch.empty((TINY.R, TINY.Hq, 128), dtype=torch.float32, device=dev)
            for _ in range(2 * len(kinds))]
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    for t, k in enumerate(kinds):
        fn = eng.oasis_step_stall if k == "stall" else eng.oasis_step
        fn(0, t, qg[t], qdg[t], outs[2 * t], outs[2 * t + 1])
    eng.oasis_join(0)
    eng.oasis_sync()
    for t, k in enumerate(kinds):
        if k == "stall":
            ref = L.orc.stall_step(bits(L.q[t]), bits(L.qd[t]), t)
        else:
            ref = L.orc.step(bits(L.q[t]), bits(L.qd[t]), t)
        H.check_attention([outs[2 * t].cpu().numpy(), outs[2 * t + 1].cpu().numpy()], ref, TINY.G)
    assert (eng.res_ids[0][len(kinds) & 1].cpu().numpy() == L.orc.res).all()
    assert (eng.stamps[0].cpu().numpy() == L.orc.stamp).all()
    H.check_pool(L, len(kinds) & 1)
    eng.close()


def test_stall_attends_over_the_query_topk(dev):
    # With at least K blocks, the stall step's attention reads exactly the
    # normal query's top-K (the oracle's stall step is pinned to that): the
    # demand lists leave no block of the GPU's own top-K missing.
    L = H.make_layer(TINY, seed=14, steps=3, out_fp32=True)
    eng = L.eng
    out = torch.empty((TINY.R, TINY.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    for t in range(3):
        before = eng.res_ids[0][t & 1].cpu().numpy().copy()
        eng.oasis_step_stall(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        dm = {k: v.cpu().numpy() for k, v in eng.stall_lists(0, t).items()}
        cur = eng.res_ids[0][t & 1].cpu().numpy()
        for r in range(TINY.R):
            for h in range(TINY.Hkv):
                T = set(dm["topk_ids"][r, h].tolist())
                assert set(cur[r, h].tolist()) == T
                n = dm["n_admit"][r, h]
                assert n == len(T - set(before[r, h].tolist()))
                assert (dm["admit_ids"][r, h, n:] == -1).all()
    eng.close()


@pytest.fixture(scope="module")
def qwen_layer(dev):
    L = H.make_layer(QWEN, seed=20, steps=6, gen_device="cuda", pairs=QWEN_SAMPLE)
    yield L
    L.eng.close()


def test_qwen3_layer_staged_stall_steps(dev, qwen_layer):
    # The initial resident set is a random subset: the first demand fetch
    # brings nearly the whole top-K of every pair; later ones only misses.
    L = qwen_layer
    fetched = []
    for t in range(2):
        dm, ref = H.run_staged_stall_step(L, t, dev, check_pool_every=False)
        H.check_pool(L, t & 1, QWEN_SAMPLE)
        H.check_pool(L, (t + 1) & 1, QWEN_SAMPLE)
        fetched.append(np.mean([v["n_admit"] for v in dm.values()]))
    # from a random start the first demand fetch brings most of the top-K;
    # the second only what the previous step's top-K and look-ahead missed
    assert fetched[1] < fetched[0]


def test_qwen3_layer_fused_stall_steps(dev, qwen_layer):
    L = qwen_layer
    eng = L.eng
    out = torch.empty((QWEN.R, QWEN.Hq, 128), dtype=torch.bfloat16, device=dev)
    outd = torch.empty_like(out)
    live = list(QWEN_SAMPLE)
    for t in range(2, 5):
        eng.oasis_step_stall(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        L.orc.pairs = live
        ref = L.orc.stall_step(bits(L.q[t]), bits(L.qd[t]), t)
        H.check_attention([out.float().cpu().numpy(), outd.float().cpu().numpy()], ref, QWEN.G)
        live = H.check_stall_step(L, t, ref, exact=False)
        assert len(live) >= len(QWEN_SAMPLE) - 3
        H.check_pool(L, t & 1, live)
        H.check_pool(L, (t + 1) & 1, live)
    # properties on every pair: distinct resident ids, the pool a permutation
    res = eng.res_ids[0][1]
    srt, _ = torch.sort(res, dim=-1)
    assert (srt[..., 1:] != srt[..., :-1]).all()
    phys = eng.phys[0][1]
    ps, _ = torch.sort(phys, dim=-1)
    assert torch.equal(ps, torch.arange(eng.U, device=dev, dtype=torch.int32).expand_as(ps))

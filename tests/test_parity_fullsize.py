"""GPU parity at the full sizes of the other benchmark workloads, in their
launch configurations, on sampled (request, KV head) pairs that the oracle
follows one by one:
* one layer of the 36-layer workload (90 requests x 16K tokens: 720 pairs,
  for which the launcher picks the 4-warp scan), staged and fused steps,
  then blocks rewritten in the store and refreshed;
* the growing Llama-shaped layer (64 requests from 32K tokens, 2064 blocks)
  with one token appended per request and step;
* the fetch caps 0.01 and 1.0 on the 128 x 16K layer."""
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
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def fused_steps(L, dev, steps, sample, K):
    """oasis_step on the sampled pairs; a pair whose top-K differs inside the
    tie window leaves the check (the two sides then diverge legitimately)."""
    eng, sh = L.eng, L.shape
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32 if eng.cfg.out_fp32
                      else torch.bfloat16, device=dev)
    outd = torch.empty_like(out)
    live = list(sample)
    for t in steps:
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
            assert H.topk_agrees(lists["topk_ids"][r, h], v["topk"], v["scores"], K)
            if not np.array_equal(lists["topk_ids"][r, h], v["topk"]):
                continue
            assert lists["n_admit"][r, h] == v["n_admit"]
            assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
            assert (res_n[r, h] == L.orc.res[r, h]).all()
            keep.append((r, h))
        live = keep
        assert len(live) >= len(sample) - 2
        H.check_pool(L, (t + 1) & 1, live)
    return live


def test_36_layer_workload_layer(dev):
    sh = workload.SHAPES["qwen3_8b_36l"]
    sample = [(0, 0), (13, 5), (44, 2), (61, 3), (89, 7)]
    L = H.make_layer(sh, seed=91, steps=4, gen_device="cuda", pairs=sample)
    H.check_summaries(L, sample)
    # the scan + top-K of all 720 pairs (the 4-warp variant) against the oracle
    topk = torch.empty((sh.R, sh.Hkv, sh.K), dtype=torch.int32, device=dev)
    scores = torch.empty((sh.R, sh.Hkv, sh.K), dtype=torch.float32, device=dev)
    L.eng.oasis_score_topk(0, 0, L.qd[0].to(dev), topk, scores)
    L.eng.oasis_sync()
    ref_s, ref_t = H.oracle_scan_all_pairs(L, workload.bf16_bits(L.qd[0]))
    differ = H.check_scan_all_pairs(L, topk.cpu().numpy(), scores.cpu().numpy(), ref_s, ref_t)
    assert len(differ) <= 8, differ
    for t in range(2):
        H.run_staged_step(L, t, dev, check_pool_every=False)
        H.check_pool(L, (t + 1) & 1, sample)
    live = fused_steps(L, dev, range(2, 4), sample, sh.K)
    # rewrite a few blocks of the sampled pairs (resident and not), refresh
    rng = np.random.default_rng(5)
    gen = torch.Generator().manual_seed(5)
    res = L.eng.res_ids[0][4 & 1].cpu().numpy()
    ids = np.full((sh.R, sh.Hkv, 4), -1, dtype=np.int32)
    nid = np.zeros((sh.R, sh.Hkv), dtype=np.int32)
    for (r, h) in live:
        blocks = [int(res[r, h, 0]), int(res[r, h, 1])] + \
            [int(x) for x in rng.choice(sh.NBmax, size=2, replace=False)]
        blocks = list(dict.fromkeys(blocks))
        ids[r, h, :len(blocks)] = blocks
        nid[r, h] = len(blocks)
        for b in blocks:
            L.host[r, h, b] = torch.randn((2, 16, 128), generator=gen).to(torch.bfloat16)
    L.eng.oasis_refresh_blocks(0, 4, torch.from_numpy(ids).to(dev), torch.from_numpy(nid).to(dev))
    L.eng.oasis_sync()
    gs = workload.bf16_bits(L.eng.summaries[0].cpu())
    for (r, h) in live:
        one = np.ascontiguousarray(L.hb[r:r + 1])
        want = oracle.summary_build(one, np.ascontiguousarray(L.lens[r:r + 1]))
        np.testing.assert_array_equal(H.bits_to_float(gs[r, h]), H.bits_to_float(want[0, h]))
    H.check_pool(L, 4 & 1, live)
    L.eng.close()


def test_growing_llama_shaped_layer(dev):
    sh = workload.SHAPES["llama31_8b_32k"]
    steps = 3
    sample = [(0, 0), (17, 6), (42, 3), (63, 7)]
    L = H.make_layer(sh, seed=92, steps=steps, gen_device="cuda", pairs=sample, out_fp32=True)
    eng = L.eng
    lens = L.lens                       # the oracle's context lengths (shared array)
    live = list(sample)
    for t in range(steps):
        k_new, v_new = workload.new_tokens(sh, 92, 0, t)
        live = fused_steps(L, dev, [t], live, sh.K)
        eng.oasis_append_token(0, t, k_new.to(dev), v_new.to(dev))
        eng.oasis_advance_context(t, 1)
        eng.oasis_sync()
        kb, vb = workload.bf16_bits(k_new), workload.bf16_bits(v_new)
        for (r, h) in live:               # the GPU wrote the token into the store
            p = int(lens[r])
            np.testing.assert_array_equal(L.hb[r, h, p // 16, 0, p % 16], kb[r, h])
            np.testing.assert_array_equal(L.hb[r, h, p // 16, 1, p % 16], vb[r, h])
        for r in sorted({r for (r, _) in sample}):
            oracle.append_token(L.hb, L.summ, lens, kb[r], vb[r], r)
        lens += 1
        assert (eng.ctx_len[(t + 1) & 1].cpu().numpy() == lens).all()
        gs = workload.bf16_bits(eng.summaries[0].cpu())
        for (r, h) in live:
            b = (int(lens[r]) - 1) // 16
            np.testing.assert_array_equal(H.bits_to_float(gs[r, h, b]),
                                          H.bits_to_float(L.summ[r, h, b]))
    eng.close()


@pytest.mark.parametrize("ratio", [0.01, 1.0])
def test_fetch_cap_extremes_full_layer(dev, ratio):
    sh = workload.SHAPES["qwen3_8b_16k"]
    sample = [(0, 0), (50, 4), (127, 7)]
    L = H.make_layer(sh, seed=93, steps=2, fetch_ratio=ratio, gen_device="cuda", pairs=sample)
    for t in range(2):
        ref = H.run_staged_step(L, t, dev, check_pool_every=False)
        H.check_pool(L, (t + 1) & 1, sample)
        for v in ref.values():
            assert v["n_admit"] <= L.shape.C
    L.eng.close()


def test_remote_tier_full_layer(dev):
    # The remote tier on the 128 x 16K layer (local tier of NBmax slots): the
    # sampled pairs' slot assignment, slot map, local copies and pool follow
    # the oracle through staged and fused steps.
    sh = workload.SHAPES["qwen3_8b_16k"]
    sample = [(3, 1), (64, 5), (126, 2)]
    L = H.make_layer(sh, seed=94, steps=4, gen_device="cuda", pairs=sample,
                     remote_capacity=sh.NBmax)
    H.check_remote(L, L.orc.initial_misses)
    for t in range(2):
        ref = H.run_staged_step(L, t, dev, check_pool_every=False)
        H.check_remote(L, ref)
        H.check_pool(L, (t + 1) & 1, sample)
    live = fused_steps(L, dev, range(2, 4), sample, sh.K)
    assert L.eng.oasis_remote_stats(0)["bad_entries"] == 0
    L.eng.close()


def test_two_layers_of_the_36_layer_workload(dev):
    # Two full-size layers (90 x 16K each, own stores) stepped in layer order
    # on one stream without host synchronisation, as the multi-layer
    # benchmark does: each layer's side work overlaps the next layer.
    from sparse_kv_block_gb300.oasis import Oasis, make_config
    sh = workload.SHAPES["qwen3_8b_36l"]
    nl, steps = 2, 3
    sample = [(2, 0), (45, 6), (88, 3)]
    lens = workload.ctx_lens(sh)
    hosts, qs, qds, res0s, orcs = [], [], [], [], []
    for l in range(nl):
        h = torch.empty((sh.R, sh.Hkv, sh.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                        pin_memory=True)
        workload.host_kv(sh, 95, l, lens, device="cuda", out=h)
        q, qd = workload.queries(sh, 95, l, steps, device="cuda")
        hosts.append(h)
        qs.append(q.cpu())
        qds.append(qd.cpu())
        res0s.append(workload.initial_resident(sh, 95, l, lens))
    eng = Oasis(make_config(sh.R, sh.NBmax, sh.Hq, sh.Hkv, sh.K, sh.fetch_ratio, layers=nl,
                            out_fp32=True), host_kv=hosts)
    eng.set_context(lens)
    for l in range(nl):
        eng.set_resident(l, res0s[l], 0)
        eng.oasis_build_summaries(l, 0)
        eng.oasis_load_resident(l, 0)
        hb = workload.bf16_bits(hosts[l])
        orcs.append(oracle.LayerOracle(hb, oracle.summary_build(hb, lens), lens, res0s[l],
                                       sh.K, sh.C, sample))
    eng.oasis_sync()
    outs = [torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev) for _ in range(nl)]
    outds = [torch.empty_like(o) for o in outs]
    live = [list(sample) for _ in range(nl)]
    for t in range(steps):
        for l in range(nl):
            eng.oasis_step(l, t, qs[l][t].to(dev), qds[l][t].to(dev), outs[l], outds[l])
        for l in range(nl):
            eng.oasis_join(l)
        eng.oasis_sync()
        for l in range(nl):
            orcs[l].pairs = live[l]
            ref = orcs[l].step(workload.bf16_bits(qs[l][t]), workload.bf16_bits(qds[l][t]), t)
            H.check_attention([outs[l].cpu().numpy(), outds[l].cpu().numpy()], ref, sh.G)
            lists = {k: v.cpu().numpy() for k, v in eng.step_lists(l, t).items()}
            res_n = eng.res_ids[l][(t + 1) & 1].cpu().numpy()
            keep = []
            for (r, h), v in ref.items():
                assert H.topk_agrees(lists["topk_ids"][r, h], v["topk"], v["scores"], sh.K)
                if np.array_equal(lists["topk_ids"][r, h], v["topk"]):
                    assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
                    assert (res_n[r, h] == orcs[l].res[r, h]).all()
                    keep.append((r, h))
            live[l] = keep
            assert len(keep) >= len(sample) - 1
    eng.close()

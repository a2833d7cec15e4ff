"""Remote tier (emulated prefill-decode disaggregation with remote partial
fetch) on the GPU against the oracle: slot assignment lists, slot map and
counts bit-exact, local tier and pool byte-exact, attention within the usual
tolerance; tier overflow reported through the device error word; the
throttle honoured."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from sparse_kv_block_gb300 import workload
from sparse_kv_block_gb300.oasis import DEVERR_NOT_LOCAL, OASIS_ESTATE, OasisError
from tests import _harness as H

pytestmark = pytest.mark.gpu
TINY = workload.SHAPES["tiny"]


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def test_remote_staged_steps_match_oracle(dev):
    sh = dataclasses.replace(TINY, R=3)
    L = H.make_layer(sh, seed=11, steps=6, fetch_ratio=0.25, remote_capacity=sh.NBmax)
    H.check_remote(L, L.orc.initial_misses)
    for t in range(6):
        ref = H.run_staged_step(L, t, dev)
        H.check_remote(L, ref)
    st = L.eng.oasis_remote_stats(0)
    assert st["units"] == int(L.orc.local_count.sum()) and st["bad_entries"] == 0
    L.eng.close()


@pytest.mark.parametrize("groups,schedule", [(0, 0), (3, 0), (2, 2), (2, 4)])
def test_remote_fused_steps_match_oracle(dev, groups, schedule):
    sh = dataclasses.replace(TINY, R=4)
    L = H.make_layer(sh, seed=12, steps=6, fetch_ratio=0.25, out_fp32=True, side_groups=groups,
                     schedule=schedule, remote_capacity=48)
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
        lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
        for (r, h), v in ref.items():
            assert np.array_equal(lists["topk_ids"][r, h], v["topk"]), "tie window hit"
            assert not v["full"]
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        H.check_remote(L, ref)
        H.check_pool(L, (t + 1) & 1)
    eng.close()


def test_remote_back_to_back_steps(dev):
    # The worker thread's transfer between the slot assignment and the
    # gather of every step, steps issued without host synchronisation.
    sh = dataclasses.replace(TINY, R=5)
    L = H.make_layer(sh, seed=13, steps=8, fetch_ratio=0.25, out_fp32=True,
                     remote_capacity=sh.NBmax)
    eng = L.eng
    outs = [torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev) for _ in range(16)]
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    for t in range(8):
        eng.oasis_step(0, t, qg[t], qdg[t], outs[2 * t], outs[2 * t + 1])
    eng.oasis_join(0)
    eng.oasis_sync()
    for t in range(8):
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([outs[2 * t].cpu().numpy(), outs[2 * t + 1].cpu().numpy()], ref, sh.G)
    H.check_remote(L, ref)
    H.check_pool(L, 8 & 1)
    eng.close()


def test_remote_tier_overflow_is_reported(dev):
    # capacity K + 1: the first admissions overflow the tier.  The oracle runs
    # its own steps (its top-K drives both sides' admission); the GPU reports
    # OASIS_DEVERR_NOT_LOCAL exactly when the oracle's assignment overflows,
    # and the slot map, counts and lists stay equal to the oracle's.
    sh = dataclasses.replace(TINY, R=2)
    cap = sh.K + 1
    L = H.make_layer(sh, seed=14, steps=4, fetch_ratio=0.25, remote_capacity=cap)
    eng = L.eng
    R, Hk, K, C = sh.R, sh.Hkv, sh.K, sh.C
    saw_full = False
    for t in range(4):
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        feed = np.full((R, Hk, K), -1, dtype=np.int32)
        for (r, h), v in ref.items():
            feed[r, h] = v["topk"]
        aid = torch.empty((R, Hk, C), dtype=torch.int32, device=dev)
        asl, evi = torch.empty_like(aid), torch.empty_like(aid)
        nad = torch.empty((R, Hk), dtype=torch.int32, device=dev)
        eng.oasis_admit_evict(0, t, torch.from_numpy(feed).to(dev), aid, asl, evi, nad)
        eng.oasis_prefetch(0, t, aid, asl, nad)
        full = False
        try:
            eng.oasis_sync()
        except OasisError as e:
            assert f"0x{DEVERR_NOT_LOCAL:x}" in str(e)
            full = True
        want_full = any(v["full"] for v in ref.values())
        assert full == want_full, t
        saw_full |= full
        H.check_remote(L, ref)
    assert saw_full
    eng.close()


def test_remote_throttle_and_refresh_refused(dev):
    sh = dataclasses.replace(TINY, R=2)
    gbps = 0.25
    L = H.make_layer(sh, seed=15, steps=3, fetch_ratio=0.25, remote_capacity=sh.NBmax,
                     remote_gbps=gbps)
    for t in range(3):
        H.run_staged_step(L, t, dev)
    st = L.eng.oasis_remote_stats(0)
    assert st["transfers"] == 5   # the load (resident set, then tail blocks), one per step
    assert st["units"] == int(L.orc.local_count.sum())
    assert st["seconds"] >= st["units"] * 8192 / (gbps * 1e9) * 0.999
    ids = torch.zeros((sh.R, sh.Hkv, 1), dtype=torch.int32, device=dev)
    n = torch.zeros((sh.R, sh.Hkv), dtype=torch.int32, device=dev)
    with pytest.raises(OasisError) as e:
        L.eng.oasis_refresh_blocks(0, 3, ids, n)
    assert e.value.status == OASIS_ESTATE
    L.eng.close()


@pytest.mark.parametrize("lens0", [[1000, 37], [992, 16]])
def test_remote_with_growing_contexts(dev, lens0):
    # Decoding with a remote tier: the load also brings each context's
    # partial tail block to the local tier; appended tokens go to local slots
    # (a block a token opens takes the next slot); the remote store is never
    # written.  The oracle keeps its own copy of the store with the appends.
    steps = 30
    sh = dataclasses.replace(TINY, ctx=max(lens0), grow_steps=steps)
    lens = np.array(lens0, dtype=np.int32)
    L = H.make_layer(sh, seed=16, steps=steps, lens=lens, fetch_ratio=0.25, out_fp32=True,
                     remote_capacity=sh.NBmax)
    eng = L.eng
    remote_before = L.hb.copy()
    hb_orc, summ_orc, lens_o = L.hb.copy(), L.summ.copy(), L.lens.copy()
    orc = oracle.LayerOracle(hb_orc, summ_orc, lens_o, L.res0, sh.K, sh.C, L.orc.pairs,
                             remote_capacity=sh.NBmax)
    T = L.remote
    assert (T["local_map"].cpu().numpy() == orc.local_map).all()
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    for t in range(steps):
        eng.oasis_step(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        k_new, v_new = workload.new_tokens(sh, 16, 0, t)
        eng.oasis_append_token(0, t, k_new.to(dev), v_new.to(dev))
        eng.oasis_advance_context(t, 1)
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        kb, vb = workload.bf16_bits(k_new), workload.bf16_bits(v_new)
        for r in range(sh.R):
            assert not orc.append_local(r)
            oracle.append_token(hb_orc, summ_orc, lens_o, kb[r], vb[r], r)
        lens_o += 1
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        lmap = T["local_map"].cpu().numpy()
        assert (lmap == orc.local_map).all(), t
        assert (T["local_count"].cpu().numpy() == orc.local_count).all(), t
        local = workload.bf16_bits(T["local_tier"])
        for (r, h) in orc.pairs:
            for b in np.nonzero(lmap[r, h] >= 0)[0]:
                np.testing.assert_array_equal(local[r, h, lmap[r, h, b]], hb_orc[r, h, b])
        nxt = (t + 1) & 1
        res = eng.res_ids[0][nxt].cpu().numpy()
        phys = eng.phys[0][nxt].cpu().numpy()
        pool = workload.bf16_bits(eng.kv_pool[0].cpu())
        for (r, h) in orc.pairs:
            for s_ in range(sh.K):
                if res[r, h, s_] >= 0:
                    np.testing.assert_array_equal(pool[r, h, phys[r, h, s_]], hb_orc[r, h, res[r, h, s_]])
    np.testing.assert_array_equal(L.hb, remote_before)      # the remote store is untouched
    eng.close()

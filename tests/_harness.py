"""Shared GPU-test harness: one layer of a workload on both the CUDA path (via
the C ABI) and the CPU oracle, on the same seeded bytes.

Parity protocol (tolerances of the build target):
* summaries: equal values (bf16 min/max are exact);
* top-K ids: equal, except ids whose oracle fp32 score lies within 1e-5
  relative of the K-th score (the tie window); afterwards the oracle's list
  drives both sides' eviction so the resident state stays in lockstep;
* admit/evict lists, resident table, stamps: bit-exact given that list;
* pool: byte-exact against the host store for every resident slot;
* attention: max-abs <= 1e-2 and mean-abs <= 1e-3 against the fp32 oracle.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from sparse_kv_block_gb300 import workload
from sparse_kv_block_gb300.oasis import Oasis, make_config

ATT_MAX_ABS = 1e-2
ATT_MEAN_ABS = 1e-3
TIE_REL = 1e-5


@dataclasses.dataclass
class Layer:
    shape: workload.Shape
    lens: np.ndarray
    host: torch.Tensor
    q: torch.Tensor
    qd: torch.Tensor
    res0: np.ndarray
    eng: Oasis
    orc: oracle.LayerOracle
    hb: np.ndarray
    summ: np.ndarray
    remote: dict = None
    D: int = 1  # draft queries per step; qd is [steps][D][R][Hq][d] when D > 1


def make_layer(shape, seed=0, lens=None, steps=4, K=None, fetch_ratio=None, out_fp32=False,
               gen_device="cpu", pairs=None, res0=None, side_groups=0,
               schedule=0, remote_capacity=None, remote_gbps=0.0, num_drafts=1,
               mutate_host=None) -> Layer:
    if K is not None or fetch_ratio is not None:
        shape = dataclasses.replace(shape, K=K if K is not None else shape.K,
                                    fetch_ratio=shape.fetch_ratio if fetch_ratio is None else fetch_ratio)
    lens = workload.ctx_lens(shape) if lens is None else np.asarray(lens, dtype=np.int32)
    host = torch.empty((shape.R, shape.Hkv, shape.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                       pin_memory=True)
    workload.host_kv(shape, seed, 0, lens, device=gen_device, out=host)
    if mutate_host is not None:   # a test's own structure on top of the draw
        mutate_host(host)
    if num_drafts == 1:
        q, qd = workload.queries(shape, seed, 0, steps, device=gen_device)
    else:
        q, qd = workload.draft_queries(shape, seed, 0, steps, num_drafts, device=gen_device)
    q, qd = q.cpu(), qd.cpu()
    if res0 is None:
        res0 = workload.initial_resident(shape, seed, 0, lens)
    cfg = make_config(shape.R, shape.NBmax, shape.Hq, shape.Hkv, shape.K, shape.fetch_ratio,
                      out_fp32=out_fp32, side_groups=side_groups, schedule=schedule,
                      num_drafts=num_drafts)
    eng = Oasis(cfg, host_kv=[host])
    eng.set_context(lens)
    eng.set_resident(0, res0, 0)
    eng.oasis_build_summaries(0, 0)
    remote = None
    if remote_capacity is not None:
        remote = eng.oasis_remote_attach(0, remote_capacity, remote_gbps)
    eng.oasis_load_resident(0, 0)
    eng.oasis_sync()
    hb = workload.bf16_bits(host)
    summ = oracle.summary_build(hb, lens)
    if pairs is None:
        pairs = [(r, h) for r in range(shape.R) for h in range(shape.Hkv)]
    orc = oracle.LayerOracle(hb, summ, lens, res0, shape.K, shape.C, pairs,
                             remote_capacity=remote_capacity)
    return Layer(shape, lens, host, q, qd, res0, eng, orc, hb, summ, remote, num_drafts)


def check_remote(L: Layer, misses: dict):
    """Remote tier against the oracle: the last slot assignment's lists per
    pair (bit-exact), the slot map and counts, and every held block's local
    copy against the host store, byte for byte."""
    T = L.remote
    n_miss = T["n_miss"].numpy()
    mi, ms = T["miss_ids"].numpy(), T["miss_slots"].numpy()
    for (r, h), v in misses.items():
        n = v["n_miss"]
        assert n_miss[r, h] == n, (r, h)
        assert (mi[r, h, :n] == v["miss_ids"]).all(), (r, h)
        assert (ms[r, h, :n] == v["miss_slots"]).all(), (r, h)
    lmap = T["local_map"].cpu().numpy()
    cnt = T["local_count"].cpu().numpy()
    base = T["local_base"].cpu().numpy()
    for (r, h) in misses:
        assert base[r, h] == cnt[r, h] - n_miss[r, h], (r, h)
    local = workload.bf16_bits(T["local_tier"])
    for (r, h) in misses:
        assert (lmap[r, h] == L.orc.local_map[r, h]).all(), (r, h)
        assert cnt[r, h] == L.orc.local_count[r, h], (r, h)
        for b in np.nonzero(lmap[r, h] >= 0)[0]:
            np.testing.assert_array_equal(local[r, h, lmap[r, h, b]], L.hb[r, h, b])


def bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def check_summaries(L: Layer, pairs=None):
    gs = workload.bf16_bits(L.eng.summaries[0].cpu())
    B = 16
    for (r, h) in (pairs or L.orc.pairs):
        nb = -(-int(L.lens[r]) // B)
        np.testing.assert_array_equal(bits_to_float(gs[r, h, :nb]), bits_to_float(L.summ[r, h, :nb]))


def topk_agrees(gpu_ids, ref_ids, ref_scores, K):
    """Ids equal except inside the tie window around the K-th oracle score."""
    if np.array_equal(gpu_ids, ref_ids):
        return True
    valid = ref_ids[ref_ids >= 0]
    if len(valid) < K:
        return False
    kth = ref_scores[valid[-1]]
    window = TIE_REL * max(abs(kth), 1e-30)
    g = set(gpu_ids.tolist()) - {-1}
    o = set(valid.tolist())
    for b in g ^ o:
        if abs(ref_scores[b] - kth) > window:
            return False
    return True


def check_attention(out_gpu: list, ref: dict, G: int):
    """out_gpu = [out, out_draft]; out_draft is [R][Hq][d] for one draft or
    [D][R][Hq][d] for D of them (compared plane by plane)."""
    planes = [out_gpu[0]]
    for x in out_gpu[1:]:
        planes += list(x) if x.ndim == 4 else [x]
    errs = []
    for (r, h), v in ref.items():
        assert len(planes) == v["attn"].shape[0]
        for which in range(len(planes)):
            d = np.abs(planes[which][r, h * G:(h + 1) * G].astype(np.float64) - v["attn"][which])
            errs.append(d)
    e = np.concatenate([x.ravel() for x in errs])
    assert e.max() <= ATT_MAX_ABS, f"attention max-abs {e.max():.3e}"
    assert e.mean() <= ATT_MEAN_ABS, f"attention mean-abs {e.mean():.3e}"
    return float(e.max()), float(e.mean())


def check_pool(L: Layer, table: int, pairs=None):
    """Every occupied slot's pool unit equals the host store's block, byte for byte."""
    res = L.eng.res_ids[0][table].cpu().numpy()
    phys = L.eng.phys[0][table].cpu().numpy()
    pool = workload.bf16_bits(L.eng.kv_pool[0].cpu())
    for (r, h) in (pairs or L.orc.pairs):
        for s in range(L.shape.K):
            b = res[r, h, s]
            if b < 0:
                continue
            u = phys[r, h, s]
            assert 0 <= u < L.eng.U
            np.testing.assert_array_equal(pool[r, h, u], L.hb[r, h, b])
        # the table's units are distinct
        assert len(set(phys[r, h].tolist())) == L.eng.U


def run_staged_step(L: Layer, t: int, dev, check_pool_every=True):
    """One layer-step through the separate C-ABI stages, compared stage by stage."""
    sh, eng = L.shape, L.eng
    qg, qdg = L.q[t].to(dev), L.qd[t].to(dev)
    odt = torch.float32 if eng.cfg.out_fp32 else torch.bfloat16
    out = torch.empty((sh.R, sh.Hq, 128), dtype=odt, device=dev)
    outd = torch.empty(tuple(L.qd[t].shape), dtype=odt, device=dev)
    R, H, K, C = sh.R, sh.Hkv, sh.K, max(sh.C, 1)
    topk = torch.empty((R, H, K), dtype=torch.int32, device=dev)
    scores = torch.empty((R, H, K), dtype=torch.float32, device=dev)
    eng.oasis_lookahead_attn(0, t, qg, qdg, out, outd)
    eng.oasis_score_topk(0, t, qdg, topk, scores)
    eng.oasis_sync()
    gpu_topk = topk.cpu().numpy()

    qb, qdb = workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t])
    # Oracle step; its own top-K drives its eviction.
    ref = L.orc.step(qb, qdb, t)
    for (r, h), v in ref.items():
        assert topk_agrees(gpu_topk[r, h], v["topk"], v["scores"], K), (t, r, h)
        nv = (v["topk"] >= 0).sum()
        got = scores.cpu().numpy()[r, h, :nv]
        np.testing.assert_allclose(got, v["scores"][v["topk"][:nv]], rtol=2e-6, atol=1e-4)
    check_attention([out.float().cpu().numpy(), outd.float().cpu().numpy()], ref, sh.G)

    # Lockstep: the oracle's top-K drives the GPU eviction too.
    feed = gpu_topk.copy()
    for (r, h), v in ref.items():
        feed[r, h] = v["topk"]
    feed_d = torch.from_numpy(feed).to(dev)
    aid = torch.empty((R, H, C), dtype=torch.int32, device=dev)
    asl = torch.empty_like(aid)
    evi = torch.empty_like(aid)
    nad = torch.empty((R, H), dtype=torch.int32, device=dev)
    eng.oasis_admit_evict(0, t, feed_d, aid, asl, evi, nad)
    eng.oasis_prefetch(0, t, aid, asl, nad)
    eng.oasis_sync()
    aid, asl, evi, nad = (x.cpu().numpy() for x in (aid, asl, evi, nad))
    nxt = (t + 1) & 1
    res_n = eng.res_ids[0][nxt].cpu().numpy()
    st = eng.stamps[0].cpu().numpy()
    for (r, h), v in ref.items():
        n = v["n_admit"]
        assert nad[r, h] == n
        assert (aid[r, h, :sh.C] == v["admit_ids"]).all()
        assert (asl[r, h, :sh.C] == v["admit_slots"]).all()
        assert (evi[r, h, :sh.C] == v["evict_ids"]).all()
        assert (res_n[r, h] == L.orc.res[r, h]).all()
        assert (st[r, h] == L.orc.stamp[r, h]).all()
    if check_pool_every:
        check_pool(L, nxt)
    return ref


def run_staged_stall_step(L: Layer, t: int, dev, check_pool_every=True):
    """One miss-stall layer-step through the separate C-ABI stages: the
    demand ranking with the normal query, the uncapped in-place demand
    admission fed the oracle's list (lockstep) and the demand gather,
    compared with the oracle's demand fetch (oracle.demand_rh, whose pairing
    with LayerOracle.step is pinned equal to the oracle's stall step); then
    the look-ahead stages of run_staged_step on the updated table."""
    sh, eng = L.shape, L.eng
    R, H, K = sh.R, sh.Hkv, sh.K
    qg = L.q[t].to(dev)
    dtk = torch.empty((R, H, K), dtype=torch.int32, device=dev)
    dsc = torch.empty((R, H, K), dtype=torch.float32, device=dev)
    eng.oasis_demand_topk(0, t, qg, dtk, dsc)
    eng.oasis_sync()
    gpu_dtk, gpu_dsc = dtk.cpu().numpy(), dsc.cpu().numpy()
    qb = workload.bf16_bits(L.q[t])
    dm = {(r, h): oracle.demand_rh(L.summ, L.lens, L.orc.res, L.orc.stamp, qb, r, h, K, t, 16)
          for (r, h) in L.orc.pairs}
    feed = gpu_dtk.copy()
    for (r, h), v in dm.items():
        assert topk_agrees(gpu_dtk[r, h], v["topk"], v["scores"], K), (t, r, h)
        nv = (v["topk"] >= 0).sum()
        np.testing.assert_allclose(gpu_dsc[r, h, :nv], v["scores"][v["topk"][:nv]],
                                   rtol=2e-6, atol=1e-4)
        feed[r, h] = v["topk"]
    aid = torch.empty((R, H, K), dtype=torch.int32, device=dev)
    asl, evi = torch.empty_like(aid), torch.empty_like(aid)
    nad = torch.empty((R, H), dtype=torch.int32, device=dev)
    eng.oasis_admit_demand(0, t, torch.from_numpy(feed).to(dev), aid, asl, evi, nad)
    eng.oasis_fetch_demand(0, t, aid, asl, nad)
    eng.oasis_sync()
    aid, asl, evi, nad = (x.cpu().numpy() for x in (aid, asl, evi, nad))
    cur = t & 1
    res_c = eng.res_ids[0][cur].cpu().numpy()
    st = eng.stamps[0].cpu().numpy()
    for (r, h), v in dm.items():
        n = v["n_admit"]
        assert nad[r, h] == n, (t, r, h)
        assert (aid[r, h] == v["admit_ids"]).all()
        assert (asl[r, h] == v["admit_slots"]).all()
        assert (evi[r, h] == v["evict_ids"]).all()
        assert (res_c[r, h] == L.orc.res[r, h]).all()
        assert (st[r, h] == L.orc.stamp[r, h]).all()
    if check_pool_every:
        check_pool(L, cur)
    ref = run_staged_step(L, t, dev, check_pool_every)
    return dm, ref


def check_stall_step(L: Layer, t: int, ref: dict, pairs=None, exact=True):
    """Lists of oasis_step_stall(t) and the tables after it against the
    oracle's stall step.  exact: every pair's two top-K lists must equal the
    oracle's; otherwise a pair whose list differs inside the tie window is
    dropped from the returned set of pairs still in lockstep."""
    sh, eng = L.shape, L.eng
    dm = {k: v.cpu().numpy() for k, v in eng.stall_lists(0, t).items()}
    la = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
    res_n = eng.res_ids[0][(t + 1) & 1].cpu().numpy()
    st = eng.stamps[0].cpu().numpy()
    keep = []
    for (r, h), v in ref.items():
        if pairs is not None and (r, h) not in pairs:
            continue
        assert topk_agrees(dm["topk_ids"][r, h], v["dm_topk"], v["dm_scores"], sh.K)
        assert topk_agrees(la["topk_ids"][r, h], v["topk"], v["scores"], sh.K)
        same = (np.array_equal(dm["topk_ids"][r, h], v["dm_topk"]) and
                np.array_equal(la["topk_ids"][r, h], v["topk"]))
        if not same:
            assert not exact, f"tie window hit at step {t}, pair {(r, h)}"
            continue
        assert dm["n_admit"][r, h] == v["dm_n_admit"]
        assert (dm["admit_ids"][r, h] == v["dm_admit_ids"]).all()
        assert (dm["admit_slots"][r, h] == v["dm_admit_slots"]).all()
        assert (dm["evict_ids"][r, h] == v["dm_evict_ids"]).all()
        assert la["n_admit"][r, h] == v["n_admit"]
        assert (la["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
        assert (la["admit_slots"][r, h, :sh.C] == v["admit_slots"]).all()
        assert (la["evict_ids"][r, h, :sh.C] == v["evict_ids"]).all()
        assert (res_n[r, h] == L.orc.res[r, h]).all()
        assert (st[r, h] == L.orc.stamp[r, h]).all()
        keep.append((r, h))
    return keep


def oracle_scan_all_pairs(L: Layer, qd_bits: np.ndarray, threads: int = 0):
    """The oracle's summary scores and top-K of every (request, KV head) pair
    of the layer for draft queries qd_bits, on a pool of host threads (the
    oracle's C functions release the interpreter lock).  Returns
    (scores [R][Hkv][NBmax] float32, topk [R][Hkv][K] int32)."""
    import concurrent.futures
    import os
    sh = L.shape
    scores = np.empty((sh.R, sh.Hkv, sh.NBmax), dtype=np.float32)
    topk = np.empty((sh.R, sh.Hkv, sh.K), dtype=np.int32)

    def one(p):
        r, h = divmod(p, sh.Hkv)
        s = oracle.score_rh(L.summ, L.lens, qd_bits, r, h, 16)
        scores[r, h] = s
        topk[r, h] = oracle.topk_rh(s, oracle.num_blocks(int(L.lens[r]), 16), sh.K)

    n = threads or min(32, os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(one, range(sh.R * sh.Hkv)))
    return scores, topk


def check_scan_all_pairs(L: Layer, gpu_topk: np.ndarray, gpu_scores: np.ndarray,
                         ref_scores: np.ndarray, ref_topk: np.ndarray):
    """Every pair's GPU top-K against the oracle's (tie-window rule) and its
    scores in rank order (rtol 2e-6); returns the pairs whose lists differ
    inside the tie window."""
    sh = L.shape
    differ = []
    for r in range(sh.R):
        for h in range(sh.Hkv):
            assert topk_agrees(gpu_topk[r, h], ref_topk[r, h], ref_scores[r, h], sh.K), (r, h)
            if not np.array_equal(gpu_topk[r, h], ref_topk[r, h]):
                differ.append((r, h))
            nv = int((ref_topk[r, h] >= 0).sum())
            np.testing.assert_allclose(gpu_scores[r, h, :nv],
                                       ref_scores[r, h][ref_topk[r, h, :nv]],
                                       rtol=2e-6, atol=1e-4)
    return differ

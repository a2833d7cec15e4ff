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
               schedule=0, remote_capacity=None, remote_gbps=0.0, num_drafts=1) -> Layer:
    if K is not None or fetch_ratio is not None:
        shape = dataclasses.replace(shape, K=K if K is not None else shape.K,
                                    fetch_ratio=shape.fetch_ratio if fetch_ratio is None else fetch_ratio)
    lens = workload.ctx_lens(shape) if lens is None else np.asarray(lens, dtype=np.int32)
    host = torch.empty((shape.R, shape.Hkv, shape.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                       pin_memory=True)
    workload.host_kv(shape, seed, 0, lens, device=gen_device, out=host)
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

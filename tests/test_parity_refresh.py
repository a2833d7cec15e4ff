"""oasis_refresh_blocks on the GPU against the oracle: after blocks of the
pinned host store are rewritten between steps, their summaries equal the
oracle's summaries of the new store, resident copies equal the host store
byte for byte, and the following steps stay in parity."""
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
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def test_refresh_rewritten_blocks(dev):
    sh = dataclasses.replace(TINY, R=3)
    lens = np.array([1024, 1000, 37], dtype=np.int32)   # ragged, with tail blocks
    L = H.make_layer(sh, seed=21, steps=5, lens=lens, fetch_ratio=0.25)
    eng = L.eng
    rng = np.random.default_rng(3)
    gen = torch.Generator().manual_seed(3)
    for t in range(4):
        H.run_staged_step(L, t, dev)
        nxt = t + 1
        # Rewrite a few blocks per pair: some resident, some not, some tails.
        res = eng.res_ids[0][nxt & 1].cpu().numpy()
        max_ids = 6
        ids = np.full((sh.R, sh.Hkv, max_ids), -1, dtype=np.int32)
        nid = np.zeros((sh.R, sh.Hkv), dtype=np.int32)
        for r in range(sh.R):
            nb = -(-int(lens[r]) // 16)
            for h in range(sh.Hkv):
                cand = [int(b) for b in res[r, h] if b >= 0][:2] + [nb - 1]
                cand += [int(x) for x in rng.choice(nb, size=min(2, nb), replace=False)]
                cand = list(dict.fromkeys(cand))[:max_ids - 1]
                ids[r, h, :len(cand)] = cand
                ids[r, h, len(cand)] = -1         # a skipped entry inside n_ids
                nid[r, h] = len(cand) + 1
                for b in cand:
                    valid = min(16, int(lens[r]) - b * 16)
                    # unit variance, like every input the tolerances are set for
                    new = torch.randn((2, valid, 128), generator=gen)
                    L.host[r, h, b, :, :valid] = new.to(torch.bfloat16)
        eng.oasis_refresh_blocks(0, nxt, torch.from_numpy(ids).to(dev),
                                 torch.from_numpy(nid).to(dev))
        eng.oasis_sync()
        # the oracle sees the same pinned bytes; its summaries are rebuilt
        L.summ[...] = oracle.summary_build(L.hb, L.lens)
        L.orc.summ = L.summ
        H.check_summaries(L)
        H.check_pool(L, nxt & 1)
    H.run_staged_step(L, 4, dev)
    eng.close()


@pytest.mark.parametrize("schedule", [0, 4])
def test_refresh_between_fused_steps(dev, schedule):
    # Blocks rewritten between fused steps, the refresh issued with no host
    # wait before the next oasis_step: under the early-scan schedule that
    # step's scan runs on its own stream and must still read the refreshed
    # summaries (a rewritten block's bound changes, and so does the ranking).
    sh = dataclasses.replace(TINY, R=3)
    lens = np.array([1024, 1000, 37], dtype=np.int32)
    L = H.make_layer(sh, seed=22, steps=5, lens=lens, fetch_ratio=0.25, out_fp32=True,
                     schedule=schedule)
    eng = L.eng
    rng = np.random.default_rng(4)
    gen = torch.Generator().manual_seed(4)
    qg, qdg = L.q.to(dev), L.qd.to(dev)
    torch.cuda.synchronize()  # the early-scan schedule reads q_draft when the call is made
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    for t in range(5):
        eng.oasis_step(0, t, qg[t], qdg[t], out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
        for (r, h), v in ref.items():
            assert np.array_equal(lists["topk_ids"][r, h], v["topk"]), (t, r, h)
            assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
        assert (eng.res_ids[0][(t + 1) & 1].cpu().numpy() == L.orc.res).all()
        H.check_pool(L, (t + 1) & 1)
        if t == 4:
            break
        # Rewrite the keys of several blocks per pair to a strong shift along
        # the queries' mean (they move up the ranking), then refresh.
        nxt = t + 1
        ids = np.full((sh.R, sh.Hkv, 6), -1, dtype=np.int32)
        nid = np.zeros((sh.R, sh.Hkv), dtype=np.int32)
        for r in range(sh.R):
            nb = -(-int(lens[r]) // 16)
            for h in range(sh.Hkv):
                cand = [int(x) for x in rng.choice(nb, size=min(5, nb), replace=False)]
                ids[r, h, :len(cand)] = cand
                nid[r, h] = len(cand)
                for b in cand:
                    valid = min(16, int(lens[r]) - b * 16)
                    new = torch.randn((2, valid, 128), generator=gen)
                    new[0] += 2.0 * L.q[t + 1, r, h * sh.G].float() / L.q[t + 1, r, h * sh.G].float().norm()
                    L.host[r, h, b, :, :valid] = new.to(torch.bfloat16)
        eng.oasis_refresh_blocks(0, nxt, torch.from_numpy(ids).to(dev),
                                 torch.from_numpy(nid).to(dev))
        L.summ[...] = oracle.summary_build(L.hb, L.lens)
        L.orc.summ = L.summ
    eng.close()

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

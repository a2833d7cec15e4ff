"""GPU parity across the shape limits the kernels are specialised for: K in
every top-K register width (K <= 32, 64, 128, 256, including K that is not a
multiple of 32), every query-group size G = 1..4, and the largest NBmax the
fused admission accepts (131072 blocks = 2M tokens for one request)."""
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
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("K,ratio", [(40, 0.25), (100, 0.1), (200, 0.05), (256, 0.25)])
def test_topk_widths(dev, K, ratio):
    sh = dataclasses.replace(TINY, R=2, ctx=8192)          # 512 blocks
    lens = np.array([8192, 5000], dtype=np.int32)          # ragged, 313-block tail request
    L = H.make_layer(sh, seed=41, steps=3, K=K, fetch_ratio=ratio, lens=lens, out_fp32=True)
    for t in range(3):
        H.run_staged_step(L, t, dev)
    L.eng.close()


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (6, 2), (8, 2), (12, 3)])
def test_group_sizes(dev, Hq, Hkv):
    sh = dataclasses.replace(TINY, R=3, Hq=Hq, Hkv=Hkv, ctx=1500)
    L = H.make_layer(sh, seed=42, steps=3, out_fp32=True)
    for t in range(3):
        H.run_staged_step(L, t, dev)
    L.eng.close()


def test_largest_nbmax(dev):
    # One request of 131072 blocks (2M tokens, a 1 GiB host store), K = 256.
    sh = dataclasses.replace(TINY, R=1, Hq=4, Hkv=1, ctx=131072 * 16, K=256)
    L = H.make_layer(sh, seed=43, steps=3, fetch_ratio=0.25, out_fp32=True, gen_device=dev)
    H.check_summaries(L)
    for t in range(2):
        H.run_staged_step(L, t, dev)
    # and the fused scan + top-K + admission of oasis_step at this size
    eng, t = L.eng, 2
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    eng.oasis_step(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
    eng.oasis_join(0)
    eng.oasis_sync()
    ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
    H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
    lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
    for (r, h), v in ref.items():
        assert H.topk_agrees(lists["topk_ids"][r, h], v["topk"], v["scores"], sh.K)
        if np.array_equal(lists["topk_ids"][r, h], v["topk"]):
            assert lists["n_admit"][r, h] == v["n_admit"]
            assert (eng.res_ids[0][(t + 1) & 1].cpu().numpy()[r, h] == L.orc.res[r, h]).all()
    H.check_pool(L, (t + 1) & 1)   # the GPU's own resident table, against the store
    eng.close()

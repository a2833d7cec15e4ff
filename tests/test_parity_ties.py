"""GPU parity when block scores tie exactly: blocks whose keys are copies of
one another have bit-identical summaries, so both the oracle and the GPU
give them the same score, and the head-wise top-K must order them by lower
block id (the reading of the top-K's tie-break) and cut a tied group at K
exactly like the oracle.  Lists, tables and stamps bit-exact, stage by stage
and fused, through the look-ahead step and the miss-stall step."""
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


def all_equal_keys(host):
    host[:, :, :, 0] = host[:, :, :1, 0]          # every block's keys = block 0's


def eight_patterns(host):
    # block b carries key pattern b % 8 (8 groups of 8 blocks): 8 distinct
    # scores per head, each shared by 8 blocks, so K = 12 cuts the second
    # group after its 4 lowest ids
    nb = host.shape[2]
    for b in range(8, nb):
        host[:, :, b, 0] = host[:, :, b % 8, 0]


@pytest.mark.parametrize("mutate,K,lens", [(all_equal_keys, 16, None),
                                           (eight_patterns, 12, None),
                                           (eight_patterns, 12, [1000, 600])])
def test_ties_staged(dev, mutate, K, lens):
    L = H.make_layer(TINY, seed=40, steps=3, K=K, out_fp32=True, lens=lens, mutate_host=mutate)
    for t in range(3):
        ref = H.run_staged_step(L, t, dev)
        for v in ref.values():
            tk = v["topk"]
            s = v["scores"][tk]
            # the oracle itself: equal scores in increasing id
            for i in range(len(tk) - 1):
                assert s[i] > s[i + 1] or (s[i] == s[i + 1] and tk[i] < tk[i + 1])
    L.eng.close()


@pytest.mark.parametrize("mutate,K", [(all_equal_keys, 16), (eight_patterns, 12)])
def test_ties_fused_and_stall(dev, mutate, K):
    L = H.make_layer(TINY, seed=41, steps=4, K=K, out_fp32=True, mutate_host=mutate)
    eng, sh = L.eng, L.shape
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    for t in range(4):
        stall = t % 2 == 1
        fn = eng.oasis_step_stall if stall else eng.oasis_step
        fn(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        eng.oasis_sync()
        qb, qdb = workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t])
        if stall:
            ref = L.orc.stall_step(qb, qdb, t)
            H.check_stall_step(L, t, ref, exact=True)
        else:
            ref = L.orc.step(qb, qdb, t)
            lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
            for (r, h), v in ref.items():
                assert np.array_equal(lists["topk_ids"][r, h], v["topk"])
                assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
            assert (eng.res_ids[0][(t + 1) & 1].cpu().numpy() == L.orc.res).all()
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        H.check_pool(L, (t + 1) & 1)
    eng.close()

"""GPU parity of the dense anchor (oasis_dense_attn): full-context decode
attention over a dense HBM copy of the KV store, against the oracle's
attention with every block of the context resident."""
import numpy as np
import pytest
import torch

import oracle
from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def dense_check(L, dev, pairs, out_dtype):
    sh, eng = L.shape, L.eng
    kv_dense = L.host.to(dev)
    out = torch.empty((sh.R, sh.Hq, 128), dtype=out_dtype, device=dev)
    outd = torch.empty_like(out)
    eng.oasis_dense_attn(kv_dense, 0, L.q[0].to(dev), L.qd[0].to(dev), out, outd)
    eng.oasis_sync()
    every = np.broadcast_to(np.arange(sh.NBmax, dtype=np.int32),
                            (sh.R, sh.Hkv, sh.NBmax)).copy()
    qb, qdb = workload.bf16_bits(L.q[0]), workload.bf16_bits(L.qd[0])
    ref = {(r, h): {"attn": oracle.attention_rh(L.hb, L.lens, every, qb, qdb, r, h)}
           for (r, h) in pairs}
    return H.check_attention([out.float().cpu().numpy(), outd.float().cpu().numpy()], ref, sh.G)


@pytest.mark.parametrize("lens", [[1024, 1024], [1000, 37], [0, 17]])
def test_dense_tiny(dev, lens):
    L = H.make_layer(workload.SHAPES["tiny"], seed=9, lens=lens, steps=1, out_fp32=True)
    dense_check(L, dev, [(r, h) for r in range(2) for h in range(2)], torch.float32)
    L.eng.close()


def test_dense_full_size_sampled(dev):
    sh = workload.SHAPES["qwen3_8b_16k"]
    sample = [(0, 0), (17, 5), (64, 3), (127, 7)]
    L = H.make_layer(sh, seed=4, steps=1, gen_device="cuda", pairs=sample)
    dense_check(L, dev, sample, torch.bfloat16)
    L.eng.close()

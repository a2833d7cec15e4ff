"""The kernel variants that the launchers pick only for some grid sizes or
on request, each checked against the oracle in a child process whose
environment selects it: the 4- and 8-consumer-warp scans (picked by grid
size), the 3-warp attention (a tuning override), the one-kernel scan +
ranking on short contexts (picked for contexts over 1024 blocks) and the
split scan + ranking on long contexts, where the ranking stages the scores
in shared memory (2064 blocks) or re-reads them from global memory (9000
blocks)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import dataclasses, sys
import torch
sys.path.insert(0, {root!r})
from sparse_kv_block_gb300 import workload
from tests import _harness as H
dev = torch.device("cuda", 0)
sh = dataclasses.replace(workload.SHAPES["tiny"], R=5, ctx=2000)
L = H.make_layer(sh, seed=51, steps=3, fetch_ratio=0.25, out_fp32=True)
for t in range(3):
    H.run_staged_step(L, t, dev)
out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
outd = torch.empty_like(out)
L2 = H.make_layer(sh, seed=52, steps=3, fetch_ratio=0.25, out_fp32=True)
for t in range(3):
    L2.eng.oasis_step(0, t, L2.q[t].to(dev), L2.qd[t].to(dev), out, outd)
    L2.eng.oasis_join(0)
    L2.eng.oasis_sync()
    import numpy as np
    from sparse_kv_block_gb300 import workload as w
    ref = L2.orc.step(w.bf16_bits(L2.q[t]), w.bf16_bits(L2.qd[t]), t)
    H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
    assert (L2.eng.res_ids[0][(t + 1) & 1].cpu().numpy() == L2.orc.res).all()
    H.check_pool(L2, (t + 1) & 1)
print("variant ok")
'''


CHILD_LONG = r'''
import dataclasses, sys
import torch
sys.path.insert(0, {root!r})
from sparse_kv_block_gb300 import workload
from tests import _harness as H
dev = torch.device("cuda", 0)
for ctx in (2064 * 16, 9000 * 16 - 5):
    sh = dataclasses.replace(workload.SHAPES["tiny"], R=2, Hq=4, Hkv=1, ctx=ctx, K=128)
    L = H.make_layer(sh, seed=53, steps=2, fetch_ratio=0.05, out_fp32=True)
    for t in range(2):
        H.run_staged_step(L, t, dev)
    L.eng.close()
print("variant ok")
'''


@pytest.mark.parametrize("env,child", [({"OASIS_SCAN_WARPS": "4"}, CHILD),
                                       ({"OASIS_SCAN_WARPS": "8"}, CHILD),
                                       ({"OASIS_ATTN_WARPS": "3"}, CHILD),
                                       ({"OASIS_SCAN": "fused"}, CHILD),
                                       ({"OASIS_SCAN": "split"}, CHILD_LONG)],
                         ids=["scan-4-warps", "scan-8-warps", "attention-3-warps",
                              "one-kernel-scan", "split-scan-long-contexts"])
def test_variant_matches_oracle(env, child):
    import __graft_entry__
    __graft_entry__.build()
    e = dict(os.environ)
    e.update(env)
    p = subprocess.run([sys.executable, "-c", child.format(root=ROOT)], cwd=ROOT, env=e,
                       capture_output=True, text=True, timeout=900)
    assert p.returncode == 0 and "variant ok" in p.stdout, p.stdout[-2000:] + p.stderr[-4000:]

"""The kernels' bounded barrier waits, made to run out on purpose.

Every wait of the attention and scan kernels on a stage of their shared
memory rings is bounded; a wait that runs out sets the device error word's
timeout bit and the kernel ends early, after waiting (with the default limit)
for the copies it has already issued.  Here the limit is set to a few clock
cycles, so that the first wait runs out before its copy lands: no fault, no
hang, nothing is left in flight.  The tests check that oasis_sync reports
the timeout, that the context stays usable, and that steps issued with the
default limit afterwards (for the fused step: after resuming from the
caller's saved state) match the oracle again."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from sparse_kv_block_gb300 import oasis as ob
from sparse_kv_block_gb300 import workload
from tests import _harness as H

pytestmark = pytest.mark.gpu

TINY = workload.SHAPES["tiny"]
SHORT = 4   # clock cycles: the first wait of every warp runs out


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda", 0)


def sync_bits(eng):
    bits = ctypes.c_uint32(0)
    rc = ob.lib().oasis_sync(eng.ctx, ctypes.byref(bits))
    return rc, bits.value


def test_stage_calls_time_out_then_recover(dev):
    # 512 blocks per request: the scan streams 16 chunks through its 2-stage
    # ring, so its producer must wait for consumed stages (with two chunks
    # both copies are issued at once and land before any wait).
    sh = dataclasses.replace(TINY, ctx=512 * 16)
    L = H.make_layer(sh, seed=50, steps=3, out_fp32=True)
    eng, sh = L.eng, L.shape
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    topk = torch.empty((sh.R, sh.Hkv, sh.K), dtype=torch.int32, device=dev)
    eng.oasis_set_wait_limit(SHORT)
    eng.oasis_lookahead_attn(0, 0, L.q[0].to(dev), L.qd[0].to(dev), out, outd)
    rc, bits = sync_bits(eng)
    assert rc == ob.OASIS_EDEVICE and bits & 0x2, (rc, bits)
    eng.oasis_score_topk(0, 0, L.qd[0].to(dev), topk)
    rc, bits = sync_bits(eng)
    assert rc == ob.OASIS_EDEVICE and bits & 0x2, (rc, bits)
    assert sync_bits(eng) == (ob.OASIS_OK, 0)      # the bits were cleared
    # default limit again: the stage calls above wrote no table, so the
    # staged steps continue from the loaded state in parity
    eng.oasis_set_wait_limit(0)
    for t in range(2):
        H.run_staged_step(L, t, dev)
    eng.close()


def test_fused_step_times_out_then_resumes(dev):
    L = H.make_layer(TINY, seed=51, steps=3, out_fp32=True)
    eng, sh = L.eng, L.shape
    out = torch.empty((sh.R, sh.Hq, 128), dtype=torch.float32, device=dev)
    outd = torch.empty_like(out)
    saved_res = eng.res_ids[0][0].clone()
    saved_stamps = eng.stamps[0].clone()
    eng.oasis_set_wait_limit(SHORT)
    eng.oasis_step(0, 0, L.q[0].to(dev), L.qd[0].to(dev), out, outd)
    eng.oasis_join(0)
    rc, bits = sync_bits(eng)
    assert rc == ob.OASIS_EDEVICE and bits & 0x2, (rc, bits)
    # The step's results are undefined, but its admission still left a
    # well-formed table: distinct ids per (request, KV head), the units a
    # permutation.
    res = eng.res_ids[0][1]
    srt, _ = torch.sort(res, dim=-1)
    valid = srt >= 0
    assert not ((srt[..., 1:] == srt[..., :-1]) & valid[..., 1:]).any()
    ps, _ = torch.sort(eng.phys[0][1], dim=-1)
    assert torch.equal(ps, torch.arange(eng.U, device=dev, dtype=torch.int32).expand_as(ps))
    # The caller resumes from the state it saved before the step.
    eng.oasis_set_wait_limit(0)
    eng.res_ids[0][0].copy_(saved_res)
    eng.stamps[0].copy_(saved_stamps)
    eng.oasis_resume_resident(0, 0)
    eng.oasis_sync()
    for t in range(3):
        eng.oasis_step(0, t, L.q[t].to(dev), L.qd[t].to(dev), out, outd)
        eng.oasis_join(0)
        assert sync_bits(eng) == (ob.OASIS_OK, 0)
        ref = L.orc.step(workload.bf16_bits(L.q[t]), workload.bf16_bits(L.qd[t]), t)
        H.check_attention([out.cpu().numpy(), outd.cpu().numpy()], ref, sh.G)
        lists = {k: v.cpu().numpy() for k, v in eng.step_lists(0, t).items()}
        for (r, h), v in ref.items():
            assert np.array_equal(lists["topk_ids"][r, h], v["topk"])
            assert (lists["admit_ids"][r, h, :sh.C] == v["admit_ids"]).all()
        assert (eng.res_ids[0][(t + 1) & 1].cpu().numpy() == L.orc.res).all()
        assert (eng.stamps[0].cpu().numpy() == L.orc.stamp).all()
        H.check_pool(L, (t + 1) & 1)
    eng.close()

"""CPU-side checks of the C ABI: the library loads, exports every symbol that
include/oasis.h declares, and its pure host calls (configuration checks and
buffer sizes) behave without a GPU."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from sparse_kv_block_gb300 import oasis as ob

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "oasis.h")).read()
    return sorted(set(re.findall(r"OASIS_API\s+[\w\s\*]+?\b(oasis_\w+)\s*\(", src)))


def test_header_declarations_are_exported_and_bound():
    names = declared_symbols()
    assert len(names) >= 20
    L = ctypes.CDLL(ob.LIB_PATH)
    for n in names:
        assert hasattr(L, n), f"{n} declared but not exported"
    assert sorted(ob.EXPORTS) == names


def test_query_sizes_qwen3_8b_layer():
    cfg = ob.make_config(R=128, NBmax=1024, Hq=32, Hkv=8, K=128, fetch_ratio=0.05)
    s = ob.oasis_query_sizes(cfg)
    assert s.fetch_cap == 6 and s.units_per_head == 134
    assert s.kv_pool_bytes == 128 * 8 * 134 * 8192
    assert s.summaries_bytes == 128 * 8 * 1024 * 512          # 512 MiB
    assert s.host_kv_bytes == 8 << 30                          # 8 GiB
    assert s.summaries_bytes * 16 == s.host_kv_bytes           # summaries = 1/16 of KV
    assert s.res_ids_bytes == 2 * 128 * 8 * 128 * 4
    assert s.ctx_len_bytes == 2 * 128 * 4
    assert s.workspace_bytes % 256 == 0


def test_workspace_grows_with_draft_planes():
    # q_draft / out_draft staging holds D planes; nothing else changes.
    base = ob.make_config(R=128, NBmax=1024, Hq=32, Hkv=8, K=128, fetch_ratio=0.05)
    plane = 128 * 32 * 128 * 2
    w = [ob.oasis_query_sizes(ob.make_config(R=128, NBmax=1024, Hq=32, Hkv=8, K=128,
                                             fetch_ratio=0.05, num_drafts=D)).workspace_bytes
         for D in (1, 2, 3)]
    assert ob.oasis_query_sizes(base).workspace_bytes == w[0]
    # qd_stage x2, qd_ring x2 and outd_stage x2 (a bf16 plane each) per extra draft
    assert w[1] - w[0] == 6 * plane and w[2] - w[1] == 6 * plane
    zero = ob.make_config(R=128, NBmax=1024, Hq=32, Hkv=8, K=128, fetch_ratio=0.05,
                          num_drafts=0)
    assert ob.oasis_query_sizes(zero).workspace_bytes == w[0]


@pytest.mark.parametrize("ratio,K,cap", [(0.05, 128, 6), (0.01, 128, 1), (0.25, 128, 32),
                                         (1.0, 128, 128), (0.25, 16, 4), (0.0, 16, 0)])
def test_fetch_cap_is_floor(ratio, K, cap):
    cfg = ob.make_config(R=2, NBmax=256, Hq=8, Hkv=2, K=K, fetch_ratio=ratio)
    assert ob.oasis_query_sizes(cfg).fetch_cap == cap


@pytest.mark.parametrize("field,value,msg", [
    ("head_dim", 64, "head_dim"), ("block_size", 32, "block_size"),
    ("topk", 0, "topk"), ("topk", 300, "topk"), ("num_q_heads", 40, "per KV head"),
    ("num_q_heads", 31, "multiple"), ("fetch_ratio", 1.5, "fetch_ratio"),
    ("max_blocks", 8, "topk must be <= max_blocks"), ("num_requests", 0, "num_requests"),
    ("num_drafts", 4, "num_drafts"), ("num_drafts", -1, "num_drafts"),
    ("schedule", 5, "schedule"), ("schedule", -1, "schedule"),
])
def test_config_errors(field, value, msg):
    cfg = ob.make_config(R=2, NBmax=64, Hq=8, Hkv=2, K=16, fetch_ratio=0.25)
    assert ob.oasis_config_error(cfg) is None
    setattr(cfg, field, value)
    err = ob.oasis_config_error(cfg)
    assert err is not None and msg in err
    with pytest.raises(ob.OasisError):
        ob.oasis_query_sizes(cfg)


def test_init_rejects_null_buffers_without_touching_the_gpu():
    cfg = ob.make_config(R=2, NBmax=64, Hq=8, Hkv=2, K=16, fetch_ratio=0.25)
    bufs = ob.oasis_buffers()
    h = ctypes.c_void_p()
    assert ob.lib().oasis_init(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(h)) == ob.OASIS_EINVAL
    assert h.value is None
    assert ob.lib().oasis_init(ctypes.byref(cfg), None, ctypes.byref(h)) == ob.OASIS_EINVAL
    # calls on a null context are rejected, not crashed
    assert ob.lib().oasis_step(None, 0, 0, None, None, None, None, None) == ob.OASIS_EINVAL
    assert ob.lib().oasis_last_error(None) == b"null context"
    assert ob.lib().oasis_destroy(None) == ob.OASIS_OK

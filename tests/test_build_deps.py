"""The in-tree build recompiles an object when any header its source reaches
through ``#include "..."`` changes (no GPU needed)."""
import os

from sparse_kv_block_gb300 import build as b


def test_every_kernel_source_depends_on_the_headers_it_includes():
    d = {s: {os.path.basename(x) for x in b.deps(os.path.join(b.CSRC, s))} for s in b.SOURCES}
    assert {"admit.cuh", "sortnet.cuh", "common.cuh", "kernels.h"} <= d["score_topk.cu"]
    assert {"admit.cuh", "sortnet.cuh", "common.cuh", "kernels.h"} <= d["admit_gather.cu"]
    assert "oasis.h" in d["api.cu"]
    # every header under csrc/ is reached by some source
    headers = {f for f in os.listdir(b.CSRC) if f.endswith((".cuh", ".h"))}
    assert headers <= set().union(*d.values())


def test_a_touched_nested_header_makes_the_object_stale(tmp_path):
    (tmp_path / "inner.cuh").write_text("#pragma once\n")
    (tmp_path / "outer.cuh").write_text('#pragma once\n#include "inner.cuh"\n')
    src = tmp_path / "k.cu"
    src.write_text('#include "outer.cuh"\n#include <cuda.h>\n')
    obj = tmp_path / "k.o"
    obj.write_text("")
    got = {os.path.basename(x) for x in b.deps(str(src))}
    assert got == {"k.cu", "outer.cuh", "inner.cuh"}
    t = os.path.getmtime(obj)
    for f in (src, tmp_path / "outer.cuh", tmp_path / "inner.cuh"):
        os.utime(f, (t - 10, t - 10))
    assert not b._stale(str(obj), b.deps(str(src)))
    os.utime(tmp_path / "inner.cuh", (t + 10, t + 10))
    assert b._stale(str(obj), b.deps(str(src)))

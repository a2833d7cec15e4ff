"""The C ABI from a plain C program (no Python, no torch): compile
sparse_kv_block_gb300/examples/c_client.c against include/oasis.h, link
liboasis.so, run it.  Host-only calls, so no GPU is needed."""
import ctypes
import os
import shutil
import subprocess

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_sizes_and_refusal(tmp_path):
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    __graft_entry__.build()
    pkg = os.path.join(ROOT, "sparse_kv_block_gb300")
    exe = str(tmp_path / "c_client")
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           os.path.join(pkg, "examples", "c_client.c"), "-L", pkg, "-loasis",
                           f"-Wl,-rpath,{pkg}", "-o", exe])
    p = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stdout + p.stderr
    lines = p.stdout.splitlines()
    assert lines[0] == "fetch_cap 6 units_per_head 134"
    assert f"kv_pool_bytes {128 * 8 * 134 * 8192} summaries_bytes {512 << 20} " \
           f"host_kv_bytes {8 << 30}" == lines[1]
    assert lines[-1].startswith("refused: head_dim")


def test_binding_structs_match_the_header(tmp_path):
    """Every field of the ctypes mirrors in the binding sits at the offset the
    C compiler gives it in include/oasis.h, and the sizes agree."""
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    from sparse_kv_block_gb300 import oasis as ob
    structs = [ob.oasis_config, ob.oasis_sizes, ob.oasis_buffers, ob.oasis_remote_config,
               ob.oasis_remote_sizes]
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "oasis.h"',
             'int main(void) {']
    for st in structs:
        n = st.__name__
        lines.append(f'  printf("{n} %zu\\n", sizeof({n}));')
        for f, _ in st._fields_:
            lines.append(f'  printf("{n}.{f} %zu\\n", offsetof({n}, {f}));')
    lines += ['  return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = str(tmp_path / "layout")
    subprocess.check_call([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-o", exe])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60, check=True).stdout
    got = dict(line.rsplit(" ", 1) for line in out.splitlines())
    for st in structs:
        n = st.__name__
        assert int(got[n]) == ctypes.sizeof(st), n
        for f, _ in st._fields_:
            assert int(got[f"{n}.{f}"]) == getattr(st, f).offset, f"{n}.{f}"

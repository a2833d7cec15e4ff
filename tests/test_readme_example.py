"""The Python usage example in README.md runs as written."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    import __graft_entry__
    __graft_entry__.build()
    text = open(os.path.join(ROOT, "README.md")).read()
    m = re.search(r"## Using the step from Python\s+```python\n(.*?)```", text, re.S)
    assert m, "example block not found"
    scope = {}
    exec(compile(m.group(1), "README.md", "exec"), scope)
    assert scope["out"].abs().sum().item() > 0
    n = scope["lists"]["n_admit"]
    assert int(n.min()) >= 0 and int(n.max()) <= scope["shape"].K
    scope["eng"].close()

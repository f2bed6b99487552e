"""The README's usage example runs as written on the GPU."""

import os
import re

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def setup_module(module):
    import __graft_entry__
    __graft_entry__.build()


def test_readme_example_runs():
    with open(os.path.join(ROOT, "README.md")) as fh:
        text = fh.read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example in README.md"
    scope = {}
    exec(compile(blocks[0], "README.md example", "exec"), scope)
    d, nxt = scope["d"], scope["nxt"]
    assert int(d.t["status"].item()) == 0 and int(d.t["wstatus"].item()) == 0
    assert int(nxt["status"].item()) == 0

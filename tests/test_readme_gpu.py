"""The usage example of the README runs as written (shapes and finite
results; parity itself is covered by the other GPU tests)."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example(gpu):
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example in the README"
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)  # noqa: S102 (the README's own example)
    torch.cuda.synchronize()
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    for name, shape in (("o", (4, 512, 32, 128)), ("dq", (4, 512, 32, 128)), ("o1", (4, 1, 32, 128)),
                        ("lse", (4, 32, 512)), ("lse1", (4, 32, 1))):
        t = scope[name]
        assert tuple(t.shape) == shape
        assert torch.isfinite(t.float()).all()

"""The usage example in README.md runs as written on the GPU."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_readme_python_example_runs():
    import torch
    from residual_sp_rs_gb300 import build
    build.build()
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README.md has no python example"
    ns = {}
    exec(compile(blocks[0], "README.md", "exec"), ns)
    torch.cuda.synchronize()
    T, S, B, H = ns["T"], ns["S"], ns["B"], ns["H"]
    assert ns["f"]["h"].shape == (S * B, H) and ns["f"]["mask"].dtype == torch.uint8
    assert ns["g"]["d_sum"].shape == (S * B, H) and ns["g"]["dgamma"].shape == (H,)
    assert ns["y_hp"].shape == (T, S * B, H // T)
    assert torch.isfinite(ns["g"]["dgamma"]).all()

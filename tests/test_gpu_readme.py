"""The README's usage examples run as written on the GPU (in order, in one
namespace) and give finite results."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_examples_run(cuda_ok):
    blocks = re.findall(r"```python\n(.*?)```", open(README, encoding="utf-8").read(), flags=re.S)
    assert len(blocks) >= 3
    ns = {}
    for code in blocks:
        exec(compile(code, README, "exec"), ns)
    torch.cuda.synchronize()
    for name in ("out", "lse", "out_h", "lse_h", "out_v", "lse_v", "out_s", "lse_s"):
        assert name in ns, name
        assert torch.isfinite(ns[name].float()).all(), name
    import hybrid_sliding_window_02_b300 as swa
    assert swa.device_error() == 0

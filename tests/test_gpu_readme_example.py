"""The README's example runs as written: its code block is executed, and both GEMM results are
compared with the product of the decoded codes (torch's float8 decoding of the same bytes, times the
scales the casts returned), within the GEMM tolerance."""
import os
import re

import pytest
import torch

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example() -> str:
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert len(blocks) == 1, "the README has one python example"
    return blocks[0]


def test_readme_example_runs_and_multiplies():
    require_gpu()
    src = _example()
    mx_at = src.index("# MXFP8")
    env: dict = {}
    exec(compile(src[:mx_at], "README.md", "exec"), env)  # per-tensor part
    torch.cuda.synchronize()

    def check(y, a, b):
        ref = a.float() @ b.float().t()
        tol = 1e-3 * (a.float().abs() @ b.float().abs().t()) + ref.abs() * 2.0 ** -8
        assert torch.all((y.float() - ref).abs() <= tol)

    qx, qw, sx, sw, y = env["qx"], env["qw"], env["sx"], env["sw"], env["y"]
    dec = lambda c: c.view(torch.float8_e4m3fn).float()
    check(y, dec(qx) * sx, dec(qw) * sw)

    exec(compile(src[mx_at:], "README.md", "exec"), env)  # MXFP8 part, same namespace
    torch.cuda.synchronize()
    qx, qw, sfx, sfw, y = env["qx"], env["qw"], env["sfx"], env["sfw"], env["y"]
    e8m0 = lambda s: torch.exp2(s.float() - 127.0).repeat_interleave(32, dim=1)
    check(y, dec(qx) * e8m0(sfx), dec(qw) * e8m0(sfw))

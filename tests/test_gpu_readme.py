"""The README's Python example runs as written and matches the oracle (needs a GB300)."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_matches_the_oracle():
    import torch

    from tests._util import check_bf16, run_oracle
    from tp_reduce_moe_gb300 import build
    build.build()
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "README has no python example"
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    torch.cuda.synchronize()
    out, residual_out = scope["out"], scope["residual_out"]
    assert out.shape == residual_out.shape == (scope["T"], scope["H"])
    # the example's own inputs, copied back, through the CPU oracle
    inp = dict(E=[e.cpu() for e in scope["E"]], S=[s.cpu() for s in scope["S"]],
               perm=scope["perm"].cpu(), w=scope["w"].cpu(), residual=scope["residual"].cpu(),
               gamma=scope["gamma"].cpu(), weight_bias=0.0, eps=1e-6)
    ref = run_oracle(inp)
    check_bf16(out, ref["out"], "README example out")
    check_bf16(residual_out, ref["h"], "README example residual_out")

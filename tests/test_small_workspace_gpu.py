"""The smallest workspaces rra_init accepts (1 MiB) and a small one (8 MiB),
each in a process of its own (rra_init sizes the workspace once per
device): every schedule and form, at sizes from one tile to many, either
runs and matches the oracle bit for bit or returns RRA_ERR_WORKSPACE before
any launch; no call ever leaves a device error behind."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

_CHILD = r"""
import os, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import collective_all_reduce_rank_gb300 as rra
import oracle
from collective_all_reduce_rank_gb300 import inputs

torch.cuda.set_device(0)
rra.rra_init(0, int(sys.argv[2]))
ALGO = {"ring": rra.RRA_ALGO_RING, "oneshot": rra.RRA_ALGO_ONE_SHOT, "twoshot": rra.RRA_ALGO_TWO_SHOT,
        "tree": rra.RRA_ALGO_TREE}
FORMS = {"ring": ("RRA_RING_PROTO", ("", "ll", "staged", "simple")), "tree": ("RRA_TREE_PROTO", ("", "ll", "staged"))}
seen = {"ok": 0, "workspace": 0}
for dtype, code in (("float32", rra.RRA_FLOAT32), ("bfloat16", rra.RRA_BFLOAT16)):
    for n in (2, 8):
        for S in (1 << 10, 1 << 20, 16 << 20):
            count = S // (4 if dtype == "float32" else 2) + 3
            xs = inputs.make_ranks(n, count, dtype, "normal", seed=S + n)
            if dtype == "bfloat16":
                ins = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in xs]
            else:
                ins = [torch.from_numpy(x).cuda() for x in xs]
            for name, algo in ALGO.items():
                var, forms = FORMS.get(name, (None, ("",)))
                want = None
                for form in forms:
                    if var:
                        os.environ.pop(var, None)
                        if form:
                            os.environ[var] = form
                    outs = [torch.empty_like(t) for t in ins]
                    st = rra.rra_allreduce(ins, outs, count, code, rra.RRA_SUM, algo, check=False)
                    if st == rra.RRA_ERR_WORKSPACE:
                        seen["workspace"] += 1
                        continue
                    assert st == rra.RRA_SUCCESS, (name, form, n, S, st)
                    dst, info = rra.rra_query_status()
                    assert dst == rra.RRA_SUCCESS, (name, form, n, S, info)
                    if want is None:
                        want, _, _ = oracle.allreduce(name, xs, dtype)
                    for r in (0, n - 1):
                        got = outs[r].view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bfloat16" \
                            else outs[r].cpu().numpy()
                        assert got.tobytes() == want[r].tobytes(), (name, form, n, S, r)
                    seen["ok"] += 1
                if var:
                    os.environ.pop(var, None)
print("small workspace ok", seen)
"""


@pytest.mark.parametrize("workspace", [1 << 20, 8 << 20])
def test_small_workspace_runs_or_refuses(workspace):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    p = subprocess.run([sys.executable, "-c", _CHILD, root, str(workspace)], capture_output=True, text=True,
                       timeout=900)
    assert p.returncode == 0 and "small workspace ok" in p.stdout, p.stdout[-3000:] + p.stderr[-3000:]
    # the smallest workspace refuses some forms (the staged ring's and
    # tree's slots for 16 MiB per rank do not fit 384 KiB)
    if workspace == 1 << 20:
        assert "'workspace': 0}" not in p.stdout, p.stdout

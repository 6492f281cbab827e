"""The sampled-window check of the sweep's parity test, pinned on the CPU:
on a problem small enough for the oracle in full, the windowed problems
(n chunks of m elements for the ring, one-shot and two-shot; two parts for
the tree) reproduce the full result at those positions bit for bit."""
import numpy as np

import oracle
from collective_all_reduce_rank_gb300 import inputs
from test_sweep_parity_gpu import AR, _parts, _windows


def test_window_reduction_reproduces_full_oracle():
    n, dtype = 5, "float32"
    xs = inputs.make_ranks(n, 4 * 5000 + 3, dtype, "normal", seed=3)
    count = xs[0].size
    for name in AR:
        full, _, _ = oracle.allreduce(name, xs, dtype)
        bounds = _parts(count, 2 if name == "tree" else n, dtype)
        for win in _windows(bounds, 64):
            sub = [np.concatenate([x[o:o + 64] for o in win]) for x in xs]
            want, _, _ = oracle.allreduce(name, sub, dtype)
            idx = np.concatenate([np.arange(o, o + 64) for o in win])
            assert want[0].tobytes() == full[0][idx].tobytes(), (name, win)

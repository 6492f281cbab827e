"""Host <-> device helpers for the GPU tests (numpy <-> torch CUDA tensors)."""
import numpy as np
import torch

import collective_all_reduce_rank_gb300 as rra

TORCH = {"int32": torch.int32, "float32": torch.float32, "bfloat16": torch.bfloat16}
CODE = {"int32": rra.RRA_INT32, "float32": rra.RRA_FLOAT32, "bfloat16": rra.RRA_BFLOAT16}


def to_dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bfloat16":
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "bfloat16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def empty(n: int, count: int, dtype: str, fill=None):
    """n output buffers, poisoned so unwritten elements show."""
    outs = []
    for _ in range(n):
        t = torch.empty(count, dtype=TORCH[dtype], device="cuda")
        if dtype == "int32":
            t.fill_(-0x5A5A5A5A if fill is None else fill)
        else:
            t.view(torch.int16 if dtype == "bfloat16" else torch.int32).fill_(-1 if fill is None else fill)
        outs.append(t)
    return outs


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what=""):
    if got.tobytes() != want.tobytes():
        g = got.view(np.uint16 if got.dtype == np.uint16 else np.uint32)
        w = want.view(np.uint16 if want.dtype == np.uint16 else np.uint32)
        bad = np.nonzero(g != w)[0]
        raise AssertionError("%s: %d of %d elements differ, first at %d: got %r want %r"
                             % (what, bad.size, g.size, bad[0], got[bad[0]], want[bad[0]]))


def bf16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rel_ok(got: np.ndarray, want: np.ndarray, rel=1e-2, abs_=1e-3):
    """The bfloat16 bar: |g - r| <= rel |r| + abs for every element."""
    g = bf16_bits_to_f64(got)
    r = bf16_bits_to_f64(want)
    return bool(np.all(np.abs(g - r) <= rel * np.abs(r) + abs_))

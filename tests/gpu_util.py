"""Device-side helpers for the GPU tests: move a workload's arrays to the GPU and
back (bit patterns only, no arithmetic)."""
from __future__ import annotations

import numpy as np
import torch

import adapter_sgmv_bgmv_gb300 as L


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


def from_dev(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def upload_table(ctx, case):
    a_pool = to_dev(case["a_pool"])
    b_pool = a_pool if case["b_pool"] is case["a_pool"] else to_dev(case["b_pool"])
    return L.AdapterTable(ctx, a_pool, b_pool, case["rank"], case["scale"], case["a_pages"],
                          case["b_pages"])


def sample_rows(case, k=64, seed=0):
    """Rows to check against the oracle: the first and last row of every segment
    run plus a seeded random sample, released rows included."""
    ids = np.asarray(case["ids"])
    n = ids.shape[0]
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    edges = np.flatnonzero(np.diff(ids) != 0)
    pick.update(edges.tolist())
    pick.update((edges + 1).tolist())
    pick.update([0, n - 1])
    return np.array(sorted(p for p in pick if 0 <= p < n), np.int64)

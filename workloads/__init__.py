"""Seeded synthetic inputs for the multi-LoRA delta.

This module only draws random numbers and lays them out (bf16 bit patterns in
uint16 arrays, page tables, adapter ids).  It holds none of the method's
arithmetic and imports neither the library nor the oracle; both the tests and the
benchmark feed the same arrays to each side.

Shapes and distributions follow the workloads the pages describe:

* ``tiny_decode``       -- 16 single-token requests, d=256, 4 rank-8 adapters.
* ``llama7b_decode_het`` / ``llama7b_decode_hom`` -- Llama-7B projection (4096x4096),
  64 single-token requests, rank 16; 64 distinct adapters vs all rows on one
  (Punica's heterogeneous vs homogeneous batch of 64, "BEE-30060", Background).
* ``slora_prefill``     -- 8 prefill requests with log-normal lengths, ranks from
  {8,16,32,64}, 1000 registered adapters of which only the 8 referenced ones are
  resident in a unified pool of 4096-wide pages in shuffled order (S-LoRA page,
  Unified Paging).
* ``valora_prefill``    -- Qwen-VL-7B MLP up-projection 4096->11008, 16 requests of
  1024 visual + 32 text tokens, 4 rank-64 adapters with Zipf(1.2) popularity
  (VaLoRA blog, section 5.2 models; long visual-token inputs, section 5.3.1).
* ``valora_merge``      -- the same adapters and a 4096x11008 base weight for the
  merge / unmerge mode switch (VaLoRA blog, section 4.4.1).
* ``lorazor_decode``    -- 70B projection (8192x8192), 256 single-token requests,
  512 resident rank-16 adapters (Zipf(1.0)) in 8192-wide shuffled pages; at step t
  the first 128+t entries of a fixed random permutation of the rows are released
  (adapter id -1) (LoRazor page: permanent early release, active-row kernels).

Values: x ~ N(0,1), A ~ N(0, 1/d_in), B ~ N(0, 1/r), W ~ N(0, 1/d_in), scale
s = alpha/r with alpha = 16; everything drawn in fp32 and rounded to bf16.
"""
from __future__ import annotations

import math

import numpy as np
import torch

ALPHA = 16.0
CONFIG_NAMES = ("tiny_decode", "llama7b_decode_het", "llama7b_decode_hom",
                "slora_prefill", "valora_prefill", "valora_merge", "lorazor_decode")


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 values -> bf16 bit patterns (uint16), via torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, std):
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def _zipf_probs(n: int, a: float) -> np.ndarray:
    p = np.arange(1, n + 1, dtype=np.float64) ** (-a)
    return p / p.sum()


def _contiguous_table(rng, n_adapters, ranks, d_in, d_out, max_rank):
    """A and B of every adapter in two dense row blocks (no paging): the page of
    A's column j of adapter k is row offset[k]+j of a [sum r, d_in] array."""
    ranks = np.asarray(ranks, np.int32)
    offs = np.concatenate([[0], np.cumsum(ranks)]).astype(np.int64)
    total = int(offs[-1])
    a_pool = np.empty((total, d_in), np.uint16)
    b_pool = np.empty((total, d_out), np.uint16)
    a_pages = np.full((n_adapters, max_rank), -1, np.int32)
    b_pages = np.full((n_adapters, max_rank), -1, np.int32)
    for k in range(n_adapters):
        r = int(ranks[k])
        a_pool[offs[k]:offs[k] + r] = _normal(rng, (r, d_in), 1.0 / math.sqrt(d_in))
        b_pool[offs[k]:offs[k] + r] = _normal(rng, (r, d_out), 1.0 / math.sqrt(r))
        a_pages[k, :r] = np.arange(offs[k], offs[k] + r)
        b_pages[k, :r] = np.arange(offs[k], offs[k] + r)
    return a_pool, b_pool, a_pages, b_pages


def _paged_table(rng, n_adapters, ranks, resident, page_width, d_in, d_out, max_rank):
    """Unified pool of page_width-wide pages holding A columns and B rows of the
    resident adapters only, in shuffled page order; others get page id -1."""
    ranks = np.asarray(ranks, np.int32)
    resident = [int(k) for k in resident]
    n_pages = int(sum(2 * int(ranks[k]) for k in resident))
    order = rng.permutation(n_pages).astype(np.int32)
    pool = np.zeros((n_pages, page_width), np.uint16)
    a_pages = np.full((n_adapters, max_rank), -1, np.int32)
    b_pages = np.full((n_adapters, max_rank), -1, np.int32)
    nxt = 0
    for k in resident:
        r = int(ranks[k])
        pa = order[nxt:nxt + r]
        pb = order[nxt + r:nxt + 2 * r]
        nxt += 2 * r
        pool[pa, :d_in] = _normal(rng, (r, d_in), 1.0 / math.sqrt(d_in))
        pool[pb, :d_out] = _normal(rng, (r, d_out), 1.0 / math.sqrt(r))
        a_pages[k, :r] = pa
        b_pages[k, :r] = pb
    return pool, pool, a_pages, b_pages


def _finish(case, rng, y_mode):
    n, d_out = case["n"], case["d_out"]
    if y_mode == "zero":
        case["y"] = np.zeros((n, d_out), np.uint16)
    elif y_mode == "randn":
        case["y"] = _normal(rng, (n, d_out), 1.0)
    else:
        raise ValueError(y_mode)
    return case


def make_W(d_in: int, d_out: int, seed: int = 0) -> np.ndarray:
    """Base weight W [d_in, d_out] ~ N(0, 1/d_in), bf16 bits."""
    rng = np.random.default_rng(10_000 + seed)
    return _normal(rng, (d_in, d_out), 1.0 / math.sqrt(d_in))


def make(name: str, seed: int = 0, y_mode: str = "randn", step: int = 0) -> dict:
    """Build one workload.  Returned keys: n, d_in, d_out, x [n,d_in], y [n,d_out],
    a_pool, b_pool (page arrays), rank, scale, a_pages, b_pages [n_adapters,max_rank],
    ids [n] (int32, -1 = released), plus config-specific extras."""
    rng = np.random.default_rng(seed)
    if name == "tiny_decode":
        d, n, na, r = 256, 16, 4, 8
        ranks = np.full(na, r, np.int32)
        a_pool, b_pool, ap, bp = _contiguous_table(rng, na, ranks, d, d, r)
        ids = rng.integers(0, na, n).astype(np.int32)
        case = dict(n=n, d_in=d, d_out=d, ids=ids, paged=False)
    elif name in ("llama7b_decode_het", "llama7b_decode_hom"):
        d, n, na, r = 4096, 64, 64, 16
        ranks = np.full(na, r, np.int32)
        a_pool, b_pool, ap, bp = _contiguous_table(rng, na, ranks, d, d, r)
        if name.endswith("het"):
            ids = rng.permutation(na).astype(np.int32)
        else:
            ids = np.zeros(n, np.int32)
        case = dict(n=n, d_in=d, d_out=d, ids=ids, paged=False)
    elif name == "slora_prefill":
        d, n_req, na, mr = 4096, 8, 1000, 64
        z = rng.standard_normal(n_req)
        lens = np.clip(np.round(np.exp(math.log(512.0) + 0.6 * z)), 16, 2048).astype(np.int64)
        ranks = rng.choice(np.array([8, 16, 32, 64], np.int32), size=na)
        chosen = rng.choice(na, size=n_req, replace=False)
        a_pool, b_pool, ap, bp = _paged_table(rng, na, ranks, chosen, d, d, d, mr)
        ids = np.concatenate([np.full(l, k, np.int32) for l, k in zip(lens, chosen)])
        case = dict(n=int(lens.sum()), d_in=d, d_out=d, ids=ids, paged=True,
                    request_lens=lens, request_adapter=chosen.astype(np.int32))
    elif name in ("valora_prefill", "valora_merge"):
        d_in, d_out, na, r = 4096, 11008, 4, 64
        n_req, per_req = 16, 1024 + 32
        ranks = np.full(na, r, np.int32)
        a_pool, b_pool, ap, bp = _contiguous_table(rng, na, ranks, d_in, d_out, r)
        req_ad = rng.choice(na, size=n_req, p=_zipf_probs(na, 1.2)).astype(np.int32)
        ids = np.repeat(req_ad, per_req).astype(np.int32)
        n = n_req * per_req if name == "valora_prefill" else 0
        case = dict(n=n, d_in=d_in, d_out=d_out, ids=ids[:n], paged=False,
                    request_adapter=req_ad)
        if name == "valora_merge":
            case["merge_adapter"] = 0
    elif name == "lorazor_decode":
        d, n, na, r = 8192, 256, 512, 16
        ranks = np.full(na, r, np.int32)
        a_pool, b_pool, ap, bp = _paged_table(rng, na, ranks, range(na), d, d, d, r)
        base = rng.choice(na, size=n, p=_zipf_probs(na, 1.0)).astype(np.int32)
        pi = rng.permutation(n)
        case = dict(n=n, d_in=d, d_out=d, paged=True, base_ids=base,
                    release_order=pi.astype(np.int32))
        case["ids"] = lorazor_ids(case, step)
    else:
        raise KeyError(name)
    case.update(name=name, seed=seed, a_pool=a_pool, b_pool=b_pool, rank=ranks,
                scale=(ALPHA / ranks.astype(np.float32)).astype(np.float32),
                a_pages=ap, b_pages=bp)
    if case["n"] > 0:
        case["x"] = _normal(rng, (case["n"], case["d_in"]), 1.0)
    else:
        case["x"] = np.zeros((0, case["d_in"]), np.uint16)
    _finish(case, rng, y_mode)
    if name == "valora_merge":
        case["W"] = make_W(case["d_in"], case["d_out"], seed)
    return case


def lorazor_ids(case: dict, step: int) -> np.ndarray:
    """Adapter ids at decode step t: rows release_order[:128+t] are released (-1)."""
    ids = case["base_ids"].copy()
    n = ids.shape[0]
    k = min(n, n // 2 + int(step))
    ids[case["release_order"][:k]] = -1
    return ids


def small(seed: int, n: int, d_in: int, d_out: int, n_adapters: int, ranks,
          paged: bool = False, release_frac: float = 0.0, y_mode: str = "randn",
          page_width: int | None = None, ids=None) -> dict:
    """A free-form small case for sweeps (ragged sizes, mixed ranks, releases)."""
    rng = np.random.default_rng(seed)
    ranks = np.asarray(ranks, np.int32)
    mr = int(ranks.max()) if ranks.size else 8
    if paged:
        pw = page_width or max(d_in, d_out)
        a_pool, b_pool, ap, bp = _paged_table(rng, n_adapters, ranks, range(n_adapters),
                                              pw, d_in, d_out, mr)
    else:
        a_pool, b_pool, ap, bp = _contiguous_table(rng, n_adapters, ranks, d_in, d_out, mr)
    if ids is None:
        ids = rng.integers(0, n_adapters, n).astype(np.int32)
        if release_frac > 0:
            ids[rng.random(n) < release_frac] = -1
    case = dict(name="small", seed=seed, n=n, d_in=d_in, d_out=d_out,
                ids=np.asarray(ids, np.int32), paged=paged, a_pool=a_pool,
                b_pool=b_pool, rank=ranks,
                scale=(ALPHA / np.maximum(ranks, 1).astype(np.float32)).astype(np.float32),
                a_pages=ap, b_pages=bp)
    case["x"] = _normal(rng, (n, d_in), 1.0)
    return _finish(case, rng, y_mode)

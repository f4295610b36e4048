"""A seeded sweep of small random cases through the C ABI, each against the oracle.

Every case draws its own shape (d_in, d_out any multiples of 8 up to 2048, 1 to
400 rows), adapter count and ranks (8 to 64), storage (contiguous or a paged pool
of a wider page), released fraction, id layout (uniform, or request-like runs so
that some reach the tensor-core tiles) and y_in (N(0,1) or zero), then runs with
drawn options (early page copies and early input, B copied over A or not, the
tile path on or off, a fixed minimum run).  Checked: lora_fused under the bar with
released rows bit-exact, and on every third case lora_shrink (the same cells
written, within fp32 rounding of the oracle) and lora_expand of the oracle's v.
Drawn cases also go through lora_base_fused, lora_merge / lora_unmerge on both
merge kernels, and lora_fused_device_ids in both modes."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_parity
from tests.conftest import MAX_ABS_RMS, REL_FROB

pytestmark = pytest.mark.gpu

L = pytest.importorskip("adapter_sgmv_bgmv_gb300")
from tests.gpu_util import from_dev, to_dev, upload_table  # noqa: E402

N_CASES = 160


@pytest.fixture(scope="module")
def ctx():
    c = L.Context(0, max_rows=1024, max_rank=64)
    yield c
    c.close()


def draw(seed):
    rng = np.random.default_rng(7000 + seed)
    n = int(rng.integers(1, 401))
    d_in, d_out = (8 * int(v) for v in rng.integers(1, 257, 2))
    na = int(rng.integers(1, 9))
    ranks = [8 * int(v) for v in rng.integers(1, 9, na)]
    paged = bool(rng.random() < 0.5)
    pw = max(d_in, d_out) + 8 * int(rng.integers(0, 4)) if paged else None
    release = float(rng.choice([0.0, 0.3, 0.7]))
    if rng.random() < 0.5:
        # request-like runs: each run one adapter, some long enough for a tile
        lens, tot = [], 0
        while tot < n:
            m = int(min(n - tot, rng.choice([1, 3, 17, 64, 130, 260])))
            lens.append(m)
            tot += m
        ids = np.repeat(rng.integers(0, na, len(lens)), lens).astype(np.int32)
        ids[rng.random(n) < release * 0.2] = -1
    else:
        ids = None
    case = workloads.small(seed=7000 + seed, n=n, d_in=d_in, d_out=d_out, n_adapters=na,
                           ranks=ranks, paged=paged, release_frac=release if ids is None else 0.0,
                           y_mode=str(rng.choice(["randn", "zero"])), page_width=pw, ids=ids)
    opts = {L.OPT_EARLY_PAGES: int(rng.integers(0, 2)),
            L.OPT_EARLY_INPUT: int(rng.integers(0, 2)),
            L.OPT_ROWS_B_OVER_A: int(rng.integers(-1, 2)),
            L.OPT_TILE_PATH: int(rng.random() < 0.8),
            L.OPT_TILE_MIN_RUN: int(rng.choice([0, 0, 32, 128]))}
    return case, opts


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case_matches_oracle(ctx, seed):
    c, opts = draw(seed)
    for k, v in opts.items():
        ctx.set_option(k, v)
    try:
        table = upload_table(ctx, c)
        t = oracle.Table.from_case(c)
        x = to_dev(c["x"])
        y = to_dev(c["y"])
        L.lora_fused(ctx, table, c["ids"], x, y)
        ctx.sync_status()
        got = from_dev(y)
        what = (f"seed {seed}: n={c['n']} d_in={c['d_in']} d_out={c['d_out']} "
                f"ranks={list(c['rank'])} paged={c['paged']} opts={opts} "
                f"path={ctx.last_path()[0]}")
        ref = oracle.fused(t, c["ids"], c["x"], c["y"], nthreads=4)
        assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, what)
        rel = c["ids"] < 0
        np.testing.assert_array_equal(got[rel], c["y"][rel], err_msg=what)
        if seed % 3 == 0:
            v_ref = oracle.shrink(t, c["ids"], c["x"])
            v = torch.full(v_ref.shape, float("nan"), device="cuda")
            L.lora_shrink(ctx, table, c["ids"], x, v)
            ctx.sync_status()
            vg = v.cpu().numpy()
            np.testing.assert_array_equal(np.isnan(vg), np.isnan(v_ref), err_msg=what)
            m = ~np.isnan(v_ref)
            if m.any():
                # fp32 accumulation of d_in products against the oracle's double sum
                scale = np.sqrt(np.mean(v_ref[m] ** 2)) + 1e-30
                assert np.abs(vg[m] - v_ref[m]).max() <= 1e-4 * scale * 64, what
            v0 = np.where(np.isnan(v_ref), 0, v_ref).astype(np.float32)
            y2 = to_dev(c["y"])
            L.lora_expand(ctx, table, c["ids"], torch.from_numpy(v0).cuda(), y2)
            ctx.sync_status()
            assert_parity(from_dev(y2), oracle.expand(t, c["ids"], v0, c["y"]), REL_FROB,
                          MAX_ABS_RMS, what + " expand")
    finally:
        ctx.set_option(L.OPT_EARLY_PAGES, 0)
        ctx.set_option(L.OPT_EARLY_INPUT, 0)
        ctx.set_option(L.OPT_ROWS_B_OVER_A, 0)
        ctx.set_option(L.OPT_TILE_PATH, 1)
        ctx.set_option(L.OPT_TILE_MIN_RUN, 0)


N_OTHER = 40


@pytest.mark.parametrize("seed", range(N_OTHER))
def test_random_base_projection_matches_oracle(ctx, seed):
    """lora_base_fused on a drawn case: y = bf16(x W + s (x A) B), x W alone for
    released rows, every element against the oracle."""
    c, _ = draw(10_000 + seed)
    table = upload_table(ctx, c)
    W = workloads.make_W(c["d_in"], c["d_out"], seed=seed)
    y = torch.empty((c["n"], c["d_out"]), dtype=torch.bfloat16, device="cuda")
    L.lora_base_fused(ctx, table, c["ids"], to_dev(c["x"]), to_dev(W), y)
    ctx.sync_status()
    ref = oracle.base_fused(oracle.Table.from_case(c), c["ids"], c["x"], W, nthreads=4)
    assert_parity(from_dev(y), ref, REL_FROB, MAX_ABS_RMS,
                  f"seed {seed}: n={c['n']} d_in={c['d_in']} d_out={c['d_out']}")


@pytest.mark.parametrize("seed", range(N_OTHER))
def test_random_merge_and_unmerge_match_oracle(ctx, seed):
    """lora_merge then lora_unmerge of a drawn adapter on a drawn W, on the kernel the
    library picks and on the CUDA-core one, every element against the oracle."""
    c, _ = draw(20_000 + seed)
    table = upload_table(ctx, c)
    t = oracle.Table.from_case(c)
    k = seed % len(c["rank"])
    W = workloads.make_W(c["d_in"], c["d_out"], seed=seed)
    for path in (0, 1):
        ctx.set_option(L.OPT_MERGE_KERNEL, path)
        try:
            Wd = to_dev(W)
            L.lora_merge(ctx, table, k, Wd)
            ctx.sync_status()
            merged = from_dev(Wd)
            ref = oracle.merge(t, k, W, +1)
            assert_parity(merged, ref, REL_FROB, MAX_ABS_RMS, f"seed {seed} merge path {path}")
            L.lora_unmerge(ctx, table, k, Wd)
            ctx.sync_status()
            assert_parity(from_dev(Wd), oracle.merge(t, k, merged, -1), REL_FROB, MAX_ABS_RMS,
                          f"seed {seed} unmerge path {path}")
        finally:
            ctx.set_option(L.OPT_MERGE_KERNEL, 0)


@pytest.mark.parametrize("seed", range(N_OTHER))
def test_random_device_ids_match_host_planned(ctx, seed):
    """lora_fused_device_ids on a drawn case, in both modes, against the oracle."""
    c, opts = draw(30_000 + seed)
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    ids_dev = torch.from_numpy(np.ascontiguousarray(c["ids"], np.int32)).cuda()
    try:
        for mode in (0, 1):
            ctx.set_option(L.OPT_DEVICE_PLAN, mode)
            ctx.set_option(L.OPT_EARLY_INPUT, opts[L.OPT_EARLY_INPUT])
            y = to_dev(c["y"])
            L.lora_fused_device_ids(ctx, table, ids_dev, x, y)
            ctx.sync_status()
            ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=4)
            assert_parity(from_dev(y), ref, REL_FROB, MAX_ABS_RMS, f"seed {seed} mode {mode}")
            rel = c["ids"] < 0
            np.testing.assert_array_equal(from_dev(y)[rel], c["y"][rel])
    finally:
        ctx.set_option(L.OPT_DEVICE_PLAN, 0)
        ctx.set_option(L.OPT_EARLY_INPUT, 0)

"""lora_fused_noalloc: the fused delta for callers that must not allocate device or
pinned memory while it runs (an allocator hook, a fixed memory budget): its
scratch is fixed arrays inside the library, committed when the context is created.
It must give the results of lora_fused and of the oracle, call after call, and
leave the GPU's free memory unchanged from its very first call on.  Collected last
on purpose: a failure here comes after every other test has run."""
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


def _case(seed):
    # long same-adapter runs (tensor-core tiles) and scattered rows (row-gather)
    ids = np.concatenate([np.full(300, 0), np.array([1, 2, 1, 3, -1, 2, 3, 1]),
                          np.full(200, 2), np.full(40, 3)]).astype(np.int32)
    return workloads.small(seed=seed, n=ids.size, d_in=512, d_out=768, n_adapters=4,
                           ranks=[16, 32, 8, 64], paged=True, ids=ids)


def test_noalloc_matches_fused_and_oracle_on_two_calls_and_allocates_nothing():
    ctx = L.Context(0, max_rows=4096, max_rank=64)
    cases = [_case(71), _case(72)]
    tables = [upload_table(ctx, c) for c in cases]
    xs = [to_dev(c["x"]) for c in cases]
    y_ref = [to_dev(c["y"]) for c in cases]
    y_got = [to_dev(c["y"]) for c in cases]
    for c, t, x, y in zip(cases, tables, xs, y_ref):      # the existing entry point
        L.lora_fused(ctx, t, c["ids"], x, y)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]            # before the first no-alloc call
    for c, t, x, y in zip(cases, tables, xs, y_got):      # two calls in a row
        L.lora_fused_noalloc(ctx, t, c["ids"], x, y)
        assert ctx.last_path()[0] == 3                    # tiles and row-gather both ran
    ctx.sync_status()
    assert torch.cuda.mem_get_info()[0] == free_before
    for k in range(2):
        got = from_dev(y_got[k])
        assert_parity(got, from_dev(y_ref[k]), REL_FROB, MAX_ABS_RMS, f"call {k} vs lora_fused")
        ref = oracle.fused(oracle.Table.from_case(cases[k]), cases[k]["ids"], cases[k]["x"],
                           cases[k]["y"], nthreads=8)
        assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, f"call {k} vs oracle")
        rel = cases[k]["ids"] < 0
        np.testing.assert_array_equal(got[rel], cases[k]["y"][rel])
    ctx.close()


def _refused(ctx, c):
    t = upload_table(ctx, c)
    y = to_dev(c["y"])
    with pytest.raises(L.LoraError) as e:
        L.lora_fused_noalloc(ctx, t, c["ids"], to_dev(c["x"]), y)
    assert e.value.name == "LORA_E_CAPACITY"
    assert ctx.last_path() == (0, 0)                      # nothing launched
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(y), c["y"])    # nothing written


def test_noalloc_rejects_more_tiles_than_its_partial_v_slots():
    ctx = L.Context(0, max_rows=1 << 15, max_rank=64)
    # 65 tiles of 128 rows: one more than the 64 partial-V slots
    _refused(ctx, workloads.small(seed=73, n=65 * 128, d_in=64, d_out=64, n_adapters=1,
                                  ranks=[8], ids=np.zeros(65 * 128, np.int32)))
    ctx.close()


def test_noalloc_rejects_dense_rows_beyond_its_fixed_array():
    ctx = L.Context(0, max_rows=1 << 15, max_rank=64)
    # nine rank-64 adapters in shuffled pages, 128 rows each: their dense rows take
    # 9 x 64 x (4096 + 4096) x 2 B = 9 MB, past the 8 MB array
    ids = np.repeat(np.arange(9, dtype=np.int32), 128)
    _refused(ctx, workloads.small(seed=74, n=ids.size, d_in=4096, d_out=4096, n_adapters=9,
                                  ranks=[64] * 9, paged=True, ids=ids))
    ctx.close()


def test_noalloc_rejects_more_scattered_rows_than_its_parameter_plan():
    ctx = L.Context(0, max_rows=1 << 15, max_rank=64)
    # 600 rows alternating between two adapters: no run reaches a tile, so all 600
    # go to the row-gather kernel, past the 512 rows its in-parameter plan holds
    ids = np.tile(np.array([0, 1], np.int32), 300)
    _refused(ctx, workloads.small(seed=75, n=ids.size, d_in=64, d_out=64, n_adapters=2,
                                  ranks=[8, 8], ids=ids))
    ctx.close()


@pytest.mark.parametrize("seed", range(24))
def test_noalloc_on_drawn_cases_matches_the_oracle(seed):
    """lora_fused_noalloc on drawn cases within its limits (the sweep's shapes,
    storage, releases, id layouts and options): the oracle's result, released rows
    bit-exact."""
    from tests.test_gpu_sweep import draw
    c, opts = draw(40_000 + seed)
    ctx = L.Context(0, max_rows=1024, max_rank=64)
    try:
        for k, v in opts.items():
            if k != L.OPT_TILE_MIN_RUN:
                ctx.set_option(k, v)
        table = upload_table(ctx, c)
        y = to_dev(c["y"])
        try:
            L.lora_fused_noalloc(ctx, table, c["ids"], to_dev(c["x"]), y)
        except L.LoraError as e:
            # past a fixed limit: refused before any launch, y untouched
            assert e.name == "LORA_E_CAPACITY"
            np.testing.assert_array_equal(from_dev(y), c["y"])
            return
        ctx.sync_status()
        got = from_dev(y)
        ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=4)
        assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, f"seed {seed}")
        rel = c["ids"] < 0
        np.testing.assert_array_equal(got[rel], c["y"][rel])
    finally:
        ctx.close()

"""The offline shape -> configuration search through the C ABI: it finds a
configuration, stores it under the runtime's key, and results stay correct with it."""
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


def test_tune_rows_then_results_still_match(tmp_path):
    ctx = L.Context(0, max_rows=4096, max_rank=64)
    c = workloads.make("tiny_decode", seed=4)
    table = upload_table(ctx, c)
    scratch_y = to_dev(c["y"])
    us = L.lora_tune_shape(ctx, table, L.KIND_ROWS_FUSED, c["ids"], to_dev(c["x"]), scratch_y,
                           iters=5)
    assert us > 0 and ctx.tiles_count() == 1
    path = tmp_path / "tiles.tbl"
    ctx.tiles_save(str(path))
    fresh = L.Context(0, max_rows=4096, max_rank=64)
    fresh.tiles_load(str(path))
    t2 = upload_table(fresh, c)
    y = to_dev(c["y"])
    L.lora_fused(fresh, t2, c["ids"], to_dev(c["x"]), y)
    fresh.sync_status()
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"])
    assert_parity(from_dev(y), ref, REL_FROB, MAX_ABS_RMS, "tuned rows")
    fresh.close()
    ctx.close()


def test_tune_merge_and_tiles():
    ctx = L.Context(0, max_rows=4096, max_rank=64)
    c = workloads.small(seed=61, n=1, d_in=256, d_out=384, n_adapters=1, ranks=[32])
    table = upload_table(ctx, c)
    W = to_dev(workloads.make_W(256, 384))
    assert L.lora_tune_shape(ctx, table, L.KIND_MERGE, np.zeros(1, np.int32), W, W, iters=3) > 0
    p = workloads.small(seed=62, n=512, d_in=256, d_out=256, n_adapters=2, ranks=[16, 32],
                        ids=np.repeat(np.array([0, 1], np.int32), 256))
    tp = upload_table(ctx, p)
    assert L.lora_tune_shape(ctx, tp, L.KIND_TILE_FUSED, p["ids"], to_dev(p["x"]),
                             to_dev(p["y"]), iters=3) > 0
    assert ctx.tiles_count() == 2
    y = to_dev(p["y"])
    L.lora_fused(ctx, tp, p["ids"], to_dev(p["x"]), y)
    ctx.sync_status()
    ref = oracle.fused(oracle.Table.from_case(p), p["ids"], p["x"], p["y"], nthreads=8)
    assert_parity(from_dev(y), ref, REL_FROB, MAX_ABS_RMS, "tuned tiles")
    ctx.close()


def test_lora_tune_reads_a_shape_file_and_writes_the_table(tmp_path):
    """The C driver of the offline search: one latency shape and one throughput shape
    from a file, the table written with a comment per shape, and a fresh context that
    loads it finds the tuned shapes (lora_tile_status LORA_OK) and stays exact."""
    shapes = tmp_path / "s.shapes"
    shapes.write_text("rows 16 256 256 8 4\nrows 64 256 256 8 4 0 throughput\n")
    out = tmp_path / "t.tbl"
    ctx = L.Context(0, max_rows=4096, max_rank=64)
    ctx.tune(str(shapes), str(out))
    text = out.read_text()
    assert ctx.tiles_count() == 2 and text.count("# tuned:") == 2
    fresh = L.Context(0, max_rows=4096, max_rank=64)
    c = workloads.make("tiny_decode", seed=5)             # 16 rows, d=256, 4 rank-8 adapters
    t = upload_table(fresh, c)
    y = to_dev(c["y"])
    L.lora_fused(fresh, t, c["ids"], to_dev(c["x"]), y)
    assert fresh.tile_status() == "LORA_E_NOTUNED"        # empty table: the default shape
    fresh.tiles_load(str(out))
    y = to_dev(c["y"])
    L.lora_fused(fresh, t, c["ids"], to_dev(c["x"]), y)
    fresh.sync_status()
    if len(np.unique(c["ids"])) == 4:                     # the tuned key (4 distinct adapters)
        assert fresh.tile_status() == "LORA_OK"
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"])
    assert_parity(from_dev(y), ref, REL_FROB, MAX_ABS_RMS, "after lora_tune")
    fresh.close()
    ctx.close()

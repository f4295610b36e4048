"""lora_fused_device_ids: adapter ids in device memory, planned on the GPU.  Checked
against lora_fused on the same ids (bit for bit, with both calls given the same
row-kernel cluster width, which fixes the order of every sum) and against the
oracle; captured in a CUDA graph and replayed with ids rewritten in place; bad ids
leave their rows alone and surface at sync_status."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_parity
from tests.conftest import MAX_ABS_RMS, REL_FROB

L = pytest.importorskip("adapter_sgmv_bgmv_gb300")
from tests.gpu_util import from_dev, to_dev, upload_table  # noqa: E402

pytestmark = pytest.mark.gpu


def _bucket(m: int) -> int:
    b = 1
    while b < m:
        b <<= 1
    return b


MODES = [0, 1]   # LORA_OPT_DEVICE_PLAN: one row per cluster / a plan kernel first


def _context(tmp_path, c, ids, mode=0, cluster=4, rows=2):
    """A context whose tile table gives the host-planned call (keyed by its active
    rows, distinct adapters and their largest rank) and the device-planned call
    (keyed by n, min(n, adapters) and the table's largest rank) the same shape."""
    ids = np.asarray(ids)
    act = ids[ids >= 0]
    present = np.unique(act)
    n = len(ids)
    d_in, d_out = c["d_in"], c["d_out"]
    lines = [f"0 {_bucket(len(act))} {_bucket(len(present))} {d_in} {d_out} "
             f"{int(c['rank'][present].max())} {cluster} {rows} 0 0",
             f"0 {_bucket(n)} {_bucket(min(n, len(c['rank'])))} {d_in} {d_out} "
             f"{int(c['rank'].max())} {cluster} {rows} 0 0"]
    path = tmp_path / "same_shape.tbl"
    path.write_text("# kind m_bucket s_bucket d_in d_out rank cfg0 cfg1 cfg2 cfg3\n" +
                    "\n".join(lines) + "\n")
    ctx = L.Context(0, max_rows=4096, max_rank=64)
    ctx.tiles_load(str(path))
    ctx.set_option(L.OPT_TILE_PATH, 0)
    ctx.set_option(L.OPT_DEVICE_PLAN, mode)
    return ctx


def _both(ctx, table, c, ids):
    x = to_dev(c["x"])
    y_host, y_dev = to_dev(c["y"]), to_dev(c["y"])
    L.lora_fused(ctx, table, ids, x, y_host)
    L.lora_fused_device_ids(ctx, table, torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda(),
                            x, y_dev)
    ctx.sync_status()
    return from_dev(y_host), from_dev(y_dev)


CASES = {
    "tiny_decode": lambda: (workloads.make("tiny_decode", seed=3), None),
    "llama7b_decode_het": lambda: (workloads.make("llama7b_decode_het", seed=3), None),
    "llama7b_decode_hom": lambda: (workloads.make("llama7b_decode_hom", seed=3), None),
    "lorazor_step_57": lambda: (lambda c: (c, workloads.lorazor_ids(c, 57)))(
        workloads.make("lorazor_decode", seed=0, step=57)),
    "small_mixed_ranks_released": lambda: (workloads.small(
        seed=71, n=300, d_in=512, d_out=384, n_adapters=6, ranks=[8, 16, 24, 32, 64, 16],
        paged=True, release_frac=0.3), None),
}


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", sorted(CASES))
def test_device_ids_match_host_ids_bit_for_bit(tmp_path, name, mode):
    c, ids = CASES[name]()
    ids = c["ids"] if ids is None else ids
    ctx = _context(tmp_path, c, ids, mode)
    table = upload_table(ctx, c)
    got_host, got_dev = _both(ctx, table, c, ids)
    np.testing.assert_array_equal(got_dev, got_host)
    rel = ids < 0
    np.testing.assert_array_equal(got_dev[rel], c["y"][rel])
    if c["n"] * c["d_in"] <= 300 * 512:              # small enough for the full oracle
        ref = oracle.fused(oracle.Table.from_case(c), ids, c["x"], c["y"], nthreads=8)
        assert_parity(got_dev, ref, REL_FROB, MAX_ABS_RMS, name)
    ctx.close()


@pytest.mark.parametrize("early", [0, 1])
@pytest.mark.parametrize("mode", MODES)
def test_device_ids_in_a_cuda_graph_replayed_with_new_ids(tmp_path, mode, early):
    c = workloads.make("llama7b_decode_het", seed=4)
    rng = np.random.default_rng(72)
    id_sets = [c["ids"]] + [rng.integers(-1, len(c["rank"]), c["n"]).astype(np.int32) for _ in range(3)]
    ctx = _context(tmp_path, c, c["ids"], mode)
    ctx.set_option(L.OPT_EARLY_PAGES, early)   # the ids are rewritten by a copy, not a kernel
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    y0 = to_dev(c["y"])
    y = y0.clone()
    ids_buf = torch.from_numpy(id_sets[0].copy()).cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    L.lora_fused_device_ids(ctx, table, ids_buf, x, y, s)      # outside capture: kernel set-up
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.lora_fused_device_ids(ctx, table, ids_buf, x, y, s)
    for ids in id_sets:
        ids_buf.copy_(torch.from_numpy(ids))
        y.copy_(y0)
        g.replay()
        torch.cuda.synchronize()
        ctx.sync_status()
        got = from_dev(y)
        ref = oracle.fused(oracle.Table.from_case(c), ids, c["x"], c["y"], nthreads=8)
        assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, "graph replay")
        rel = ids < 0
        np.testing.assert_array_equal(got[rel], c["y"][rel])
    ctx.close()


@pytest.mark.parametrize("mode", MODES)
def test_bad_device_ids_leave_their_rows_and_surface_at_sync(tmp_path, mode):
    c = workloads.small(seed=73, n=64, d_in=256, d_out=256, n_adapters=4, ranks=[8, 16, 8, 16])
    ids = c["ids"].copy()
    bad = ids.copy()
    bad[5] = 4                                        # past the table
    bad[9] = -7                                       # below -1
    ctx = _context(tmp_path, c, ids, mode)
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    y = to_dev(c["y"])
    L.lora_fused_device_ids(ctx, table, torch.from_numpy(bad).cuda(), x, y)
    with pytest.raises(L.LoraError) as e:
        ctx.sync_status()
    assert e.value.name == "LORA_E_ADAPTER"
    got = from_dev(y)
    np.testing.assert_array_equal(got[[5, 9]], c["y"][[5, 9]])
    clean = np.where((bad < -1) | (bad >= 4), -1, bad).astype(np.int32)
    ref = oracle.fused(oracle.Table.from_case(c), clean, c["x"], c["y"], nthreads=8)
    assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, "rows beside bad ids")
    y2 = to_dev(c["y"])                               # the word was cleared: a clean call is clean
    L.lora_fused_device_ids(ctx, table, torch.from_numpy(ids).cuda(), x, y2)
    ctx.sync_status()
    with pytest.raises(ValueError):
        L.lora_fused_device_ids(ctx, table, torch.from_numpy(ids.astype(np.int64)).cuda(), x, y2)
    with pytest.raises(L.LoraError) as e:             # more rows than the context holds
        L.lora_fused_device_ids(ctx, table, torch.zeros(5000, dtype=torch.int32, device="cuda"),
                                to_dev(np.zeros((5000, 256), np.uint16)),
                                to_dev(np.zeros((5000, 256), np.uint16)))
    assert e.value.name == "LORA_E_INVAL"
    ctx.close()

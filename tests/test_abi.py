"""The C ABI without a GPU: the library loads, exports every function include/lora.h
declares, and its host-only parts (status strings, plan, tile-table files) work."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_]+)\s*\(", text)))


def test_header_declares_the_calls():
    names = declared_functions()
    for required in ("lora_shrink", "lora_expand", "lora_fused", "lora_merge", "lora_unmerge",
                     "lora_table_create", "lora_plan_build", "lora_tiles_load"):
        assert required in names


def test_library_exports_every_declared_symbol():
    import adapter_sgmv_bgmv_gb300 as L
    lib = ctypes.CDLL(L.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert lib.lora_version() >= 1


def test_status_strings_and_no_gpu_context():
    import adapter_sgmv_bgmv_gb300 as L
    assert L._L.lora_strerror(0) == b"ok"
    for code in range(-12, 0):
        assert L._L.lora_strerror(code) != b"unknown status"
    if not torch.cuda.is_available():
        with pytest.raises(L.LoraError):
            L.Context(0)


def _host_table(n_adapters=6, ranks=(8, 16, 8, 24, 8, 8), pw=64):
    import adapter_sgmv_bgmv_gb300 as L
    ctx = L.Context(-1, max_rows=4096, max_rank=64)
    mr = 32
    ap = np.full((n_adapters, mr), -1, np.int32)
    bp = np.full((n_adapters, mr), -1, np.int32)
    nxt = 0
    for k, r in enumerate(ranks):
        ap[k, :r] = np.arange(nxt, nxt + r)
        bp[k, :r] = np.arange(nxt + r, nxt + 2 * r)
        nxt += 2 * r
    pool = torch.zeros((nxt, pw), dtype=torch.bfloat16)
    t = L.AdapterTable(ctx, pool, pool, np.array(ranks, np.int32),
                       np.full(n_adapters, 2.0, np.float32), ap, bp)
    return ctx, t


def _numpy_plan(ids, n_adapters):
    active = np.flatnonzero(ids >= 0).astype(np.int32)
    perm = active[np.argsort(ids[active], kind="stable")].astype(np.int32)
    counts = np.bincount(ids[active], minlength=n_adapters)
    seg_adapter = np.flatnonzero(counts).astype(np.int32)
    seg_offsets = np.concatenate([[0], np.cumsum(counts[seg_adapter])]).astype(np.int32)
    return active, perm, seg_offsets, seg_adapter


@pytest.mark.parametrize("seed", range(8))
def test_library_plan_is_bit_exact_against_numpy(seed):
    import adapter_sgmv_bgmv_gb300 as L
    ctx, t = _host_table()
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(0, 2000))
    ids = rng.integers(-1, 6, n).astype(np.int32)
    if seed == 3:
        ids[:] = -1
    if seed == 5:
        ids[:] = 2
    if seed == 6:
        ids[50:400] = 1                        # one long run among short ones
    p = L.lora_plan_build(ctx, t, ids)
    a, pm, so, sa = _numpy_plan(ids, 6)
    np.testing.assert_array_equal(p["active_rows"], a)
    np.testing.assert_array_equal(p["perm"], pm)
    np.testing.assert_array_equal(p["seg_offsets"], so)
    np.testing.assert_array_equal(p["seg_adapter"], sa)
    R = p["rows_per_item"]
    assert 1 <= R <= 64
    # independent item count: runs of consecutive rows inside each segment that are
    # at least tile_min_run long become 128-row tiles, the rest R-row items
    m = p["tile_min_run"]
    n_tiles = n_rows = 0
    for s in range(len(sa)):
        seg = pm[so[s]:so[s + 1]]
        breaks = np.flatnonzero(np.diff(seg) != 1) + 1
        runs = np.split(seg, breaks)
        pending = 0
        for run in runs:
            if m > 0 and len(run) >= m:
                n_rows += (pending + R - 1) // R
                pending = 0
                n_tiles += (len(run) + 127) // 128
            else:
                pending += len(run)
        n_rows += (pending + R - 1) // R
    assert p["tile_items"] == n_tiles and p["row_items"] == n_rows
    # page accounting of the table: adapter k holds 2 r_k pages, r_k (d_in + d_out) values
    ranks = np.array([8, 16, 8, 24, 8, 8])
    assert (t.a_pages >= 0).sum(axis=1).tolist() == ranks.tolist()
    assert ((t.a_pages >= 0).sum(axis=1) + (t.b_pages >= 0).sum(axis=1)).tolist() == (2 * ranks).tolist()


def test_page_in_checks_its_arguments_before_anything_else():
    """lora_page_in on a host-only context: argument errors first, then
    LORA_E_UNSUPPORTED (no device, nothing launched)."""
    import adapter_sgmv_bgmv_gb300 as L
    ctx, t = _host_table()
    a = np.zeros((8, 64), np.uint16)
    b = np.zeros((8, 64), np.uint16)

    def call(adapter, d_in, d_out):
        rc = L._L.lora_page_in(ctx.handle, t.handle, adapter, a.ctypes.data, d_in,
                               b.ctypes.data, d_out, None)
        return L.ERROR_NAMES[rc]

    assert call(99, 64, 64) == "LORA_E_ADAPTER"
    assert call(-1, 64, 64) == "LORA_E_ADAPTER"
    assert call(0, 12, 64) == "LORA_E_INVAL"      # not a multiple of 8
    assert call(0, 64, 72) == "LORA_E_INVAL"      # wider than a page
    assert call(0, 0, 64) == "LORA_E_INVAL"
    assert call(0, 64, 64) == "LORA_E_UNSUPPORTED"
    with pytest.raises(ValueError):               # the binding wants page-locked tensors
        L.lora_page_in(ctx, t, 0, torch.zeros((8, 64), dtype=torch.int16),
                       torch.zeros((8, 64), dtype=torch.int16))


def test_device_ids_call_checks_its_arguments_on_the_host():
    """lora_fused_device_ids never reads the ids on the host; its own arguments are
    still checked before anything else, and a host-only context launches nothing."""
    import adapter_sgmv_bgmv_gb300 as L
    ctx, t = _host_table()
    ids = np.zeros(4, np.int32)
    x = np.zeros((4, 64), np.uint16)
    y = np.zeros((4, 64), np.uint16)

    def call(n, ids_ptr=ids.ctypes.data, ld=64, d=64):
        rc = L._L.lora_fused_device_ids(ctx.handle, t.handle, ids_ptr, n, x.ctypes.data, ld, d,
                                        y.ctypes.data, ld, d, None)
        return L.ERROR_NAMES[rc]

    assert call(4, ids_ptr=None) == "LORA_E_INVAL"
    assert call(4, ids_ptr=ids.ctypes.data + 2) == "LORA_E_INVAL"   # misaligned ids
    assert call(5000) == "LORA_E_INVAL"                              # > max_rows
    assert call(-1) == "LORA_E_INVAL"
    assert call(0) == "LORA_OK"                                      # nothing to do
    assert call(4, d=72) == "LORA_E_INVAL"                           # wider than a page
    assert call(4) == "LORA_E_UNSUPPORTED"                           # no device
    assert L.ERROR_NAMES[L._L.lora_selftest_timeout(ctx.handle, 0, None)] == "LORA_E_INVAL"
    assert L.ERROR_NAMES[L._L.lora_selftest_timeout(ctx.handle, 10, None)] == "LORA_E_UNSUPPORTED"


def test_argument_block_calls_check_like_the_calls_they_stand_for():
    """lora_fused_args_call / lora_fused_device_ids_args_call: a null block is
    refused, and a filled block gives the codes of the eleven-argument calls (here on
    a host-only context: argument errors first, then no device)."""
    import ctypes

    import adapter_sgmv_bgmv_gb300 as L
    from adapter_sgmv_bgmv_gb300 import _lib
    ctx, t = _host_table()
    ids = np.zeros(4, np.int32)
    x = np.zeros((4, 64), np.uint16)
    y = np.zeros((4, 64), np.uint16)
    for name, plain in (("lora_fused_args_call", "lora_fused"),
                        ("lora_fused_device_ids_args_call", "lora_fused_device_ids")):
        fn = getattr(L._L, name)
        assert L.ERROR_NAMES[fn(None)] == "LORA_E_INVAL"
        for n, d in ((4, 64), (5000, 64), (4, 72), (0, 64), (4, 64)):
            blk = _lib.FusedArgs(ctx=ctx.handle, table=t.handle, ids=ids.ctypes.data, n=n,
                                 x=x.ctypes.data, ldx=64, y=y.ctypes.data, ldy=64, d_in=d,
                                 d_out=d, stream=None)
            a = L.ERROR_NAMES[fn(ctypes.byref(blk))]
            b = L.ERROR_NAMES[getattr(L._L, plain)(ctx.handle, t.handle, ids.ctypes.data, n,
                                                   x.ctypes.data, 64, d, y.ctypes.data, 64, d,
                                                   None)]
            assert a == b, (name, n, d, a, b)


def test_library_plan_errors_on_host():
    import adapter_sgmv_bgmv_gb300 as L
    ctx, t = _host_table()
    with pytest.raises(L.LoraError) as e:
        L.lora_plan_build(ctx, t, np.array([0, 6], np.int32))
    assert e.value.name == "LORA_E_ADAPTER"
    with pytest.raises(L.LoraError) as e:
        L.lora_plan_build(ctx, t, np.zeros(5000, np.int32))
    assert e.value.name == "LORA_E_CAPACITY"
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    with pytest.raises((L.LoraError, TypeError)):
        L.lora_fused(ctx, t, np.zeros(4, np.int32), x, x)   # host-only: no launches


def test_library_plan_over_many_adapters_and_after_a_refused_call():
    """The plan visits only the adapters in use (a bitmap, 64 adapters a word): ids
    at the word boundaries, half-released batches (short ones grouped row by row,
    long ones run by run) and a call refused for an id out of range (which must leave
    no count behind) all give the numpy grouping."""
    import adapter_sgmv_bgmv_gb300 as L
    na = 300
    ctx, t = _host_table(na, (8,) * na, pw=16)
    rng = np.random.default_rng(7)
    edges = np.array([0, 62, 63, 64, 65, 127, 128, 191, 192, 255, 256, 299], np.int32)
    for trial in range(12):
        # row by row up to 1024 rows, run by run beyond (runs of one id)
        n = 700 if trial < 6 else 3000
        ids = rng.choice(np.concatenate([edges, rng.integers(0, na, 40)]), n).astype(np.int32)
        if n > 1024:
            ids = np.repeat(ids[: n // 25], 25)[:n]
        ids[rng.random(n) < 0.5] = -1
        if trial % 2:
            bad = ids.copy()
            bad[rng.integers(0, n)] = na if trial % 4 == 1 else -2
            with pytest.raises(L.LoraError) as e:
                L.lora_plan_build(ctx, t, bad)
            assert e.value.name == "LORA_E_ADAPTER"
        p = L.lora_plan_build(ctx, t, ids)
        a, pm, so, sa = _numpy_plan(ids, na)
        np.testing.assert_array_equal(p["active_rows"], a)
        np.testing.assert_array_equal(p["perm"], pm)
        np.testing.assert_array_equal(p["seg_offsets"], so)
        np.testing.assert_array_equal(p["seg_adapter"], sa)


def test_tile_table_file_round_trip(tmp_path):
    import adapter_sgmv_bgmv_gb300 as L
    ctx, _ = _host_table()
    f = tmp_path / "tiles.tbl"
    # one line with the adapter bucket, one without it (nine fields: bucket 0), and
    # the same row shape again for a different number of adapters (a separate key)
    f.write_text("# comment\n0 64 64 4096 4096 16 8 1 0 0\n4 4096 4096 11008 64 2 0 0 0\n"
                 "0 64 1 4096 4096 16 16 4 0 0\n\n")
    ctx.tiles_load(str(f))
    assert ctx.tiles_count() == 3
    out = tmp_path / "out.tbl"
    ctx.tiles_save(str(out))
    rows = sorted(l for l in out.read_text().splitlines() if not l.startswith("#"))
    assert rows == ["0 64 1 4096 4096 16 16 4 0 0", "0 64 64 4096 4096 16 8 1 0 0",
                    "4 4096 0 4096 11008 64 2 0 0 0"]
    bad = tmp_path / "bad.tbl"
    bad.write_text("0 64 4096\n")
    with pytest.raises(L.LoraError):
        ctx.tiles_load(str(bad))
    with pytest.raises(L.LoraError):
        ctx.tiles_load(str(tmp_path / "missing.tbl"))


def test_shape_file_of_the_offline_search_is_checked_before_anything_runs(tmp_path):
    """lora_tune reads its shape file in full first: a missing file is LORA_E_IO, a
    malformed line LORA_E_INVAL; a well-formed file on a host-only context parses
    and stops at LORA_E_UNSUPPORTED (no launches), with no output file written."""
    import adapter_sgmv_bgmv_gb300 as L
    ctx = L.Context(-1, max_rows=4096, max_rank=64)
    out = tmp_path / "out.tbl"
    good = tmp_path / "good.shapes"
    good.write_text("# kind n d_in d_out rank adapters run objective\n"
                    "rows 64 4096 4096 16 64 0 throughput\n"
                    "tiles 16896 4096 11008 64 4 1056\n\n"
                    "merge 1 4096 11008 64 1   # merge ignores n\n")
    with pytest.raises(L.LoraError) as e:
        ctx.tune(str(good), str(out))
    assert e.value.name == "LORA_E_UNSUPPORTED" and not out.exists()
    with pytest.raises(L.LoraError) as e:
        ctx.tune(str(tmp_path / "missing.shapes"), str(out))
    assert e.value.name == "LORA_E_IO"
    bad_lines = ["rows 64 4096 4096 16",                     # too few fields
                 "conv 64 4096 4096 16 4",                   # unknown kind
                 "rows 64 4096 4100 16 4",                   # width not a multiple of 8
                 "rows 64 4096 4096 12 4",                   # rank not a multiple of 8
                 "rows 64 4096 4096 128 4",                  # rank above the context's max
                 "rows 64 4096 4096 16 4 0 fastest",         # unknown objective
                 "tiles 512 4096 4096 16 4 128 throughput",  # throughput is for rows only
                 "rows 6x4 4096 4096 16 4"]                  # not an integer
    for line in bad_lines:
        bad = tmp_path / "bad.shapes"
        bad.write_text("rows 16 256 256 8 4\n" + line + "\n")
        with pytest.raises(L.LoraError) as e:
            ctx.tune(str(bad), str(out))
        assert e.value.name == "LORA_E_INVAL", line
    assert not out.exists()
    assert ctx.tile_status() == "LORA_OK"
    ctx.close()

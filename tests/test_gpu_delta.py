"""GPU parity of lora_fused / lora_shrink / lora_expand against the CPU oracle,
through the C ABI.  Bar: relative Frobenius error <= 5e-3 and max abs error
<= 2e-2 * rms(y_ref) (bf16 inputs, fp32 accumulation); released rows, canaries and
zero-delta cases bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_parity, f64
from tests.conftest import MAX_ABS_RMS, REL_FROB

pytestmark = pytest.mark.gpu

L = pytest.importorskip("adapter_sgmv_bgmv_gb300")
from tests.gpu_util import from_dev, sample_rows, to_dev, upload_table  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    c = L.Context(0, max_rows=1 << 15, max_rank=64)
    yield c
    c.close()


def run_fused(ctx, case, ids=None, y=None):
    table = upload_table(ctx, case)
    ids = case["ids"] if ids is None else ids
    x = to_dev(case["x"])
    yd = to_dev(case["y"] if y is None else y)
    L.lora_fused(ctx, table, ids, x, yd)
    ctx.sync_status()
    return from_dev(yd)


SMALL_CASES = {
    "ragged": dict(seed=31, n=37, d_in=40, d_out=24, n_adapters=3, ranks=[8, 16, 8],
                   release_frac=0.25),
    "paged_mixed_rank": dict(seed=32, n=70, d_in=264, d_out=136, n_adapters=5,
                             ranks=[8, 16, 24, 32, 64], paged=True, page_width=272,
                             release_frac=0.1),
    "wide_out": dict(seed=33, n=19, d_in=64, d_out=1032, n_adapters=2, ranks=[16, 8]),
    "one_adapter_many_rows": dict(seed=34, n=300, d_in=512, d_out=512, n_adapters=1,
                                  ranks=[32]),
    "y_zero": dict(seed=35, n=48, d_in=128, d_out=256, n_adapters=4, ranks=[8, 8, 16, 16],
                   y_mode="zero"),
}


@pytest.mark.parametrize("name", sorted(SMALL_CASES))
def test_fused_small_cases_match_oracle(ctx, name):
    c = workloads.small(**SMALL_CASES[name])
    got = run_fused(ctx, c)
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=4)
    assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, name)
    rel = c["ids"] < 0
    np.testing.assert_array_equal(got[rel], c["y"][rel])


@pytest.mark.parametrize("name", ["tiny_decode", "llama7b_decode_het", "llama7b_decode_hom"])
@pytest.mark.parametrize("seed", [0, 1])
def test_fused_decode_configs_full(ctx, name, seed):
    c = workloads.make(name, seed=seed)
    got = run_fused(ctx, c)
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=8)
    assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, name)


@pytest.mark.parametrize("name", ["slora_prefill", "valora_prefill"])
def test_fused_prefill_configs_sampled(ctx, name):
    c = workloads.make(name, seed=0)
    got = run_fused(ctx, c)
    rows = sample_rows(c, k=96)
    ref = oracle.fused_rows(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], rows,
                            nthreads=8)
    assert_parity(got[rows], ref, REL_FROB, MAX_ABS_RMS, name)
    # property at full size: rows of one adapter with identical inputs agree, and
    # every active row moved
    assert (got != c["y"]).any(axis=1).all()


@pytest.mark.parametrize("step", [0, 57, 99])
def test_lorazor_active_rows(ctx, step):
    c = workloads.make("lorazor_decode", seed=0, step=step)
    ids = workloads.lorazor_ids(c, step)
    assert (ids < 0).sum() == 128 + step
    got = run_fused(ctx, c, ids=ids)
    rel = ids < 0
    np.testing.assert_array_equal(got[rel], c["y"][rel])        # released: bit-exact
    act = np.flatnonzero(~rel)
    ref = oracle.fused_rows(oracle.Table.from_case(c), ids, c["x"], c["y"], act, nthreads=8)
    assert_parity(got[act], ref, REL_FROB, MAX_ABS_RMS, f"lorazor step {step}")


def test_shrink_and_expand_match_oracle(ctx):
    c = workloads.small(seed=36, n=45, d_in=200, d_out=96, n_adapters=4,
                        ranks=[8, 16, 32, 64], paged=True, release_frac=0.2)
    table = upload_table(ctx, c)
    t = oracle.Table.from_case(c)
    v_ref = oracle.shrink(t, c["ids"], c["x"])
    v = torch.full((c["n"], 64), float("nan"), device="cuda")
    L.lora_shrink(ctx, table, c["ids"], to_dev(c["x"]), v)
    ctx.sync_status()
    vg = v.cpu().numpy()
    np.testing.assert_array_equal(np.isnan(vg), np.isnan(v_ref))   # same cells written
    m = ~np.isnan(v_ref)
    assert np.abs(vg[m] - v_ref[m]).max() <= 1e-4 * np.sqrt(np.mean(v_ref[m] ** 2)) * 64
    # expand from the oracle's v: same v on both sides
    v0 = np.where(np.isnan(v_ref), 0, v_ref).astype(np.float32)
    y = to_dev(c["y"])
    L.lora_expand(ctx, table, c["ids"], torch.from_numpy(v0).cuda(), y)
    ctx.sync_status()
    assert_parity(from_dev(y), oracle.expand(t, c["ids"], v0, c["y"]), REL_FROB, MAX_ABS_RMS,
                  "expand")


def test_zero_B_and_released_rows_bit_exact_with_canaries(ctx):
    c = workloads.small(seed=37, n=40, d_in=64, d_out=48, n_adapters=3, ranks=[8, 16, 8],
                        release_frac=0.3)
    zero_b = dict(c, b_pool=np.zeros_like(c["b_pool"]))
    table = upload_table(ctx, zero_b)
    # y lives inside a wider buffer: the columns past d_out are canaries
    big = np.full((c["n"], 64), 0x7FC1, np.uint16)
    big[:, :48] = c["y"]
    yd = to_dev(big)
    L.lora_fused(ctx, table, c["ids"], to_dev(c["x"]), yd[:, :48])
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(yd), big)


def test_empty_and_fully_released_batches_touch_nothing(ctx):
    c = workloads.make("tiny_decode", seed=3)
    table = upload_table(ctx, c)
    y = to_dev(c["y"])
    L.lora_fused(ctx, table, np.zeros(0, np.int32), to_dev(c["x"][:0]), y[:0])
    L.lora_fused(ctx, table, np.full(c["n"], -1, np.int32), to_dev(c["x"]), y)
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(y), c["y"])
    assert ctx.last_path() == (0, 0)        # nothing launched


def test_repeat_runs_are_bit_identical(ctx):
    c = workloads.make("llama7b_decode_het", seed=2)
    a = run_fused(ctx, c)
    b = run_fused(ctx, c)
    np.testing.assert_array_equal(a, b)


def test_host_side_errors_launch_nothing(ctx):
    c = workloads.small(seed=38, n=12, d_in=64, d_out=64, n_adapters=4, ranks=[8, 8, 8, 8])
    ap = c["a_pages"].copy()
    ap[2, 3] = -1                     # adapter 2 not resident
    bp = c["b_pages"].copy()
    bp[3, 0] = 10_000                 # adapter 3 points past the pool
    bad = dict(c, a_pages=ap, b_pages=bp)
    table = upload_table(ctx, bad)
    x, y = to_dev(c["x"]), to_dev(c["y"])
    cases = [(np.array([0, 2], np.int32), "LORA_E_NOT_RESIDENT"),
             (np.array([3, 0], np.int32), "LORA_E_PAGE"),
             (np.array([0, 4], np.int32), "LORA_E_ADAPTER"),
             (np.array([-2, 0], np.int32), "LORA_E_ADAPTER")]
    for ids, name in cases:
        with pytest.raises(L.LoraError) as e:
            L.lora_fused(ctx, table, ids, x[:2], y[:2])
        assert e.value.name == name
    with pytest.raises(L.LoraError) as e:   # misaligned x (odd element offset)
        flat = to_dev(np.zeros(2 * 64 + 8, np.uint16))
        L.lora_fused(ctx, table, np.array([0, 1], np.int32), flat[1:129].view(2, 64), y[:2])
    assert e.value.name == "LORA_E_INVAL"
    small_ctx = L.Context(0, max_rows=4, max_rank=64)
    t2 = upload_table(small_ctx, c)
    with pytest.raises(L.LoraError) as e:
        L.lora_fused(small_ctx, t2, c["ids"], x, y)
    assert e.value.name == "LORA_E_CAPACITY"
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(y), c["y"])
    rank_bad = dict(c, rank=np.array([8, 12, 8, 8], np.int32))
    t3 = upload_table(ctx, rank_bad)
    with pytest.raises(L.LoraError) as e:
        L.lora_fused(ctx, t3, np.array([1], np.int32), x[:1], y[:1])
    assert e.value.name == "LORA_E_RANK"


# ------------------------------------------------------------------ tensor-core tiles

TILE_CASES = {
    # one adapter, 300 consecutive rows: tiles of 128, 128 and 44 rows; d_in not a
    # multiple of the 64-wide K block, d_out not a multiple of the 128-wide N chunk
    "ragged_single_run": dict(seed=51, n=300, d_in=200, d_out=136, n_adapters=1, ranks=[24],
                              ids=np.zeros(300, np.int32)),
    # runs of several adapters cut by released rows, mixed ranks (pads 8 -> 16, 40 -> 48)
    "runs_with_releases": dict(seed=52, n=700, d_in=256, d_out=384, n_adapters=3,
                               ranks=[8, 40, 64], paged=True,
                               ids=np.concatenate([np.full(150, 0), np.full(3, -1),
                                                   np.full(260, 2), np.full(17, 1),
                                                   np.full(200, 1), np.full(70, 0)]).astype(np.int32)),
}


def _tile_check(ctx, c, tile_path: bool):
    ctx.set_option(L.OPT_TILE_PATH, 1 if tile_path else 0)
    try:
        got = run_fused(ctx, c)
        path, launches = ctx.last_path()
    finally:
        ctx.set_option(L.OPT_TILE_PATH, 1)
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=8)
    assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, f"tile_path={tile_path}")
    rel = c["ids"] < 0
    np.testing.assert_array_equal(got[rel], c["y"][rel])
    return path


@pytest.mark.parametrize("name", sorted(TILE_CASES))
def test_tile_kernels_match_oracle(ctx, name):
    c = workloads.small(**TILE_CASES[name])
    assert _tile_check(ctx, c, True) & 2          # the tensor-core tiles ran
    assert _tile_check(ctx, c, False) == 1        # row-gather only


def test_tile_kernels_rank_128():
    big = L.Context(0, max_rows=4096, max_rank=128)
    c = workloads.small(seed=53, n=256, d_in=320, d_out=512, n_adapters=2, ranks=[128, 96],
                        ids=np.repeat(np.array([0, 1], np.int32), 128))
    assert _tile_check(big, c, True) & 2
    big.close()


def test_tile_kernels_eight_way_k_split(ctx):
    # nine tiles at d_in = 4096: the fused shrink splits K eight ways (the launcher
    # doubles the split while tiles x split stays within one CTA per SM and each CTA
    # keeps at least four 64-wide K blocks), so the expand sums eight partials per
    # tile, two batches of four shares; ragged last tiles (88 and 16 rows) and a
    # ragged last column chunk (d_out = 384 + 72)
    c = workloads.small(seed=55, n=1000, d_in=4096, d_out=456, n_adapters=2, ranks=[64, 16],
                        ids=np.repeat(np.array([0, 1], np.int32), [600, 400]))
    assert _tile_check(ctx, c, True) & 2


def test_tile_shrink_and_expand_match_oracle(ctx):
    c = workloads.small(seed=54, n=400, d_in=192, d_out=256, n_adapters=2, ranks=[32, 16],
                        ids=np.repeat(np.array([1, 0], np.int32), 200))
    table = upload_table(ctx, c)
    t = oracle.Table.from_case(c)
    v_ref = oracle.shrink(t, c["ids"], c["x"])
    v = torch.full((c["n"], v_ref.shape[1]), float("nan"), device="cuda")
    L.lora_shrink(ctx, table, c["ids"], to_dev(c["x"]), v)
    ctx.sync_status()
    assert ctx.last_path()[0] & 2
    vg = v.cpu().numpy()
    np.testing.assert_array_equal(np.isnan(vg), np.isnan(v_ref))
    m = ~np.isnan(v_ref)
    assert np.abs(vg[m] - v_ref[m]).max() <= 1e-3 * np.sqrt(np.mean(v_ref[m] ** 2))
    v0 = np.where(np.isnan(v_ref), 0, v_ref).astype(np.float32)
    y = to_dev(c["y"])
    L.lora_expand(ctx, table, c["ids"], torch.from_numpy(v0).cuda(), y)
    ctx.sync_status()
    assert ctx.last_path()[0] & 2
    assert_parity(from_dev(y), oracle.expand(t, c["ids"], v0, c["y"]), REL_FROB, MAX_ABS_RMS,
                  "tile expand")


def test_prepared_fused_matches_lora_fused_and_reads_a_rewritten_ids_buffer(ctx):
    """PreparedFused reuses its converted arguments when handed the same ids array
    again: the array's new contents (rows released in place) must still be used."""
    c = workloads.small(seed=81, n=48, d_in=256, d_out=384, n_adapters=3, ranks=[8, 16, 32])
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    y_ref, y_got = to_dev(c["y"]), to_dev(c["y"])
    call = L.PreparedFused(ctx, table, x, y_got)
    ids = np.ascontiguousarray(c["ids"], np.int32).copy()
    for step in range(3):
        if step == 2:
            ids[::3] = -1                       # the same buffer, rewritten in place
        L.lora_fused(ctx, table, ids.copy(), x, y_ref)
        call(ids)
        ctx.sync_status()
        np.testing.assert_array_equal(from_dev(y_got), from_dev(y_ref))


def test_prepared_calls_over_a_ring_of_ids_objects(ctx):
    """PreparedFused and PreparedFusedDeviceIds keep the arguments of the last 256
    ids objects they were handed: a ring of three arrays (one rewritten in place
    between its turns) and then 300 fresh ones (past the 256 kept, so the oldest are
    dropped) give what lora_fused / lora_fused_device_ids give, call for call."""
    c = workloads.small(seed=83, n=40, d_in=128, d_out=256, n_adapters=4, ranks=[8, 16, 8, 32])
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    rng = np.random.default_rng(5)
    ring = [rng.integers(-1, 4, 40).astype(np.int32) for _ in range(3)]
    y_ref, y_got = to_dev(c["y"]), to_dev(c["y"])
    yd_ref, yd_got = to_dev(c["y"]), to_dev(c["y"])
    call = L.PreparedFused(ctx, table, x, y_got)
    call_d = L.PreparedFusedDeviceIds(ctx, table, x, yd_got)
    ring_d = [torch.from_numpy(r.copy()).cuda() for r in ring]
    for step in range(9):
        k = step % 3
        if step == 6:
            ring[k][::2] = -1                   # rewritten in place, host and device
            ring_d[k].copy_(torch.from_numpy(ring[k]))
        L.lora_fused(ctx, table, ring[k].copy(), x, y_ref)
        call(ring[k])
        L.lora_fused_device_ids(ctx, table, ring_d[k].clone(), x, yd_ref)
        call_d(ring_d[k])
    fresh = [rng.integers(-1, 4, 40).astype(np.int32) for _ in range(300)]
    for ids in fresh + fresh[:5]:
        L.lora_fused(ctx, table, ids.copy(), x, y_ref)
        call(ids)
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(y_got), from_dev(y_ref))
    np.testing.assert_array_equal(from_dev(yd_got), from_dev(yd_ref))


@pytest.mark.parametrize("name", ["llama7b_decode_het", "llama7b_decode_hom"])
def test_early_page_copies_change_nothing(ctx, name):
    """LORA_OPT_EARLY_PAGES only moves the adapter-page copies ahead of the wait for
    the previous kernel: results are bit-identical with the option off, and within
    the bar of the oracle."""
    c = workloads.make(name, seed=5)
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    got = {}
    for early in (0, 1):
        ctx.set_option(L.OPT_EARLY_PAGES, early)
        try:
            y = to_dev(c["y"])
            for _ in range(3):          # back to back, so the overlap actually happens
                y.copy_(to_dev(c["y"]))
                L.lora_fused(ctx, table, c["ids"], x, y)
            ctx.sync_status()
            got[early] = from_dev(y)
        finally:
            ctx.set_option(L.OPT_EARLY_PAGES, 0)
    np.testing.assert_array_equal(got[1], got[0])
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=8)
    assert_parity(got[1], ref, REL_FROB, MAX_ABS_RMS, name)


def test_early_staging_changes_nothing(ctx):
    """With LORA_OPT_EARLY_PAGES the tile path's copy of scattered adapters into dense
    rows runs before the wait for the previous kernel, into the scratch half that the
    previous staged call does not read.  Back-to-back calls on two adapter sets (so
    the halves alternate and hold different adapters) give bit-identical results with
    the option off, and the first call is within the bar of the oracle."""
    c1 = workloads.small(**TILE_CASES["runs_with_releases"])
    c2 = workloads.small(**dict(TILE_CASES["runs_with_releases"], seed=57))
    t1, t2 = upload_table(ctx, c1), upload_table(ctx, c2)
    x1, x2 = to_dev(c1["x"]), to_dev(c2["x"])
    got = {}
    for early in (0, 1):
        ctx.set_option(L.OPT_EARLY_PAGES, early)
        try:
            y1, y2 = to_dev(c1["y"]), to_dev(c2["y"])
            L.lora_fused(ctx, t1, c1["ids"], x1, y1)
            ctx.sync_status()
            first = from_dev(y1)
            for _ in range(3):
                L.lora_fused(ctx, t2, c2["ids"], x2, y2)
                assert ctx.last_path()[0] & 2
                L.lora_fused(ctx, t1, c1["ids"], x1, y1)
            ctx.sync_status()
            got[early] = (first, from_dev(y1), from_dev(y2))
        finally:
            ctx.set_option(L.OPT_EARLY_PAGES, 0)
    for a, b in zip(got[1], got[0]):
        np.testing.assert_array_equal(a, b)
    ref = oracle.fused(oracle.Table.from_case(c1), c1["ids"], c1["x"], c1["y"], nthreads=8)
    assert_parity(got[1][0], ref, REL_FROB, MAX_ABS_RMS, "early staging")


@pytest.mark.parametrize("name", ["valora_prefill", "runs_with_releases", "llama7b_decode_het",
                                  "llama7b_decode_hom", "lorazor_decode", "llama7b_decode_het:dev"])
def test_early_input_changes_nothing(ctx, name):
    """LORA_OPT_EARLY_INPUT lets the tensor-core shrink load x and run its MMAs before
    the previous kernel ends (the expand of a fused call loads its first y tiles
    before its shrink ends), and the row-gather kernel load x, shrink, exchange and
    compute its expand term before the wait, reading y only after it.  Four calls back
    to back that accumulate into the same y (each call reads what the previous one
    wrote) give bit-identical results with the options off, and one call is within
    the bar of the oracle."""
    wl, _, mode = name.partition(":")
    if wl in TILE_CASES:
        c = workloads.small(**TILE_CASES[wl])
    else:
        c = workloads.make(wl, seed=3)
    ids = workloads.lorazor_ids(c, 0) if wl == "lorazor_decode" else c["ids"]
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    ids_dev = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()

    def call(y):
        if mode == "dev":
            L.lora_fused_device_ids(ctx, table, ids_dev, x, y)
        else:
            L.lora_fused(ctx, table, ids, x, y)

    tile = wl in ("valora_prefill",) or wl in TILE_CASES
    got = {}
    for early in (0, 1):
        ctx.set_option(L.OPT_EARLY_PAGES, early)
        ctx.set_option(L.OPT_EARLY_INPUT, early)
        try:
            y = to_dev(c["y"])
            call(y)
            ctx.sync_status()
            assert bool(ctx.last_path()[0] & 2) == tile
            first = from_dev(y)
            for _ in range(4):
                call(y)
            ctx.sync_status()
            got[early] = (first, from_dev(y))
        finally:
            ctx.set_option(L.OPT_EARLY_PAGES, 0)
            ctx.set_option(L.OPT_EARLY_INPUT, 0)
    for a_, b_ in zip(got[1], got[0]):
        np.testing.assert_array_equal(a_, b_)
    if wl == "valora_prefill":
        rows = sample_rows(c, k=48)
        ref = oracle.fused_rows(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], rows,
                                nthreads=8)
        assert_parity(got[1][0][rows], ref, REL_FROB, MAX_ABS_RMS, name)
    else:
        ref = oracle.fused(oracle.Table.from_case(c), ids, c["x"], c["y"], nthreads=8)
        assert_parity(got[1][0], ref, REL_FROB, MAX_ABS_RMS, name)


B_OVER_A_CASES = {
    # cluster 1 (no wider split of d = 136), A's slice larger than B's, released rows
    "ragged_c1": dict(seed=91, n=37, d_in=200, d_out=136, n_adapters=3, ranks=[8, 16, 24],
                      release_frac=0.25),
    # cluster 2, B's slice larger than A's, ranks past one warp of page lanes
    "wide_out_rank96": dict(seed=92, n=40, d_in=256, d_out=1032, n_adapters=3,
                            ranks=[96, 40, 16], paged=True, page_width=1040),
}


@pytest.mark.parametrize("name", ["lorazor_decode", "lorazor_decode:dev", "llama7b_decode_het",
                                  "ragged_c1", "wide_out_rank96"])
def test_b_over_a_changes_nothing(ctx, name):
    """LORA_OPT_ROWS_B_OVER_A has the row-gather kernel copy B's page slices into the
    shared memory A's slices used, once the shrink has read them.  Forced on, forced
    off and left to the library (which takes it for the LoRazor step-0 batch: 752 CTAs,
    more than the GPU holds with both slices staged), with early input off and on (y
    rows staged, or read after the wait), four calls accumulating into one y give the
    same bits, and the first call is within the bar of the oracle."""
    wl, _, mode = name.partition(":")
    big = None
    if wl in B_OVER_A_CASES:
        c = workloads.small(**B_OVER_A_CASES[wl])
        big = L.Context(0, max_rows=1024, max_rank=128)
        cx = big
    else:
        c = workloads.make(wl, seed=5)
        cx = ctx
    ids = workloads.lorazor_ids(c, 0) if wl == "lorazor_decode" else c["ids"]
    try:
        table = upload_table(cx, c)
        x = to_dev(c["x"])
        ids_dev = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
        got = {}
        for early in (0, 1):
            for over in (-1, 0, 1):
                cx.set_option(L.OPT_EARLY_PAGES, early)
                cx.set_option(L.OPT_EARLY_INPUT, early)
                cx.set_option(L.OPT_ROWS_B_OVER_A, over)
                try:
                    y = to_dev(c["y"])
                    for it in range(5):
                        if mode == "dev":
                            L.lora_fused_device_ids(cx, table, ids_dev, x, y)
                        else:
                            L.lora_fused(cx, table, ids, x, y)
                        if it == 0:
                            cx.sync_status()
                            assert cx.last_path()[0] == 1
                            first = from_dev(y)
                    cx.sync_status()
                    got[(early, over)] = (first, from_dev(y))
                finally:
                    cx.set_option(L.OPT_EARLY_PAGES, 0)
                    cx.set_option(L.OPT_EARLY_INPUT, 0)
                    cx.set_option(L.OPT_ROWS_B_OVER_A, 0)
        for key, val in got.items():
            for a_, b_ in zip(val, got[(0, -1)]):
                np.testing.assert_array_equal(a_, b_, err_msg=str(key))
        ref = oracle.fused(oracle.Table.from_case(c), ids, c["x"], c["y"], nthreads=8)
        assert_parity(got[(1, 1)][0], ref, REL_FROB, MAX_ABS_RMS, name)
        rel = np.asarray(ids) < 0
        np.testing.assert_array_equal(got[(1, 1)][1][rel], c["y"][rel])
    finally:
        if big is not None:
            big.close()


def test_early_options_keep_a_mixed_chain_of_calls_in_order(ctx):
    """With early pages and early input on, one stream runs, back to back: a tile-path
    delta (y1), the base projection (writes y2), a row-gather delta (y3), a merge (W2),
    a tile-path delta on y2 (reads what the base projection wrote, two calls back), a
    shrink into v and an expand of v (y4).  Every result matches the oracle applied
    in the same order, so no early read crosses a dependency between calls."""
    t = workloads.small(seed=81, n=700, d_in=256, d_out=384, n_adapters=3, ranks=[16, 32, 64],
                        ids=np.repeat(np.array([0, 2, 1], np.int32), [300, 260, 140]))
    d = workloads.small(seed=82, n=48, d_in=256, d_out=384, n_adapters=3, ranks=[16, 32, 64])
    W = workloads.make_W(256, 384, seed=3)
    W2 = workloads.make_W(256, 384, seed=4)
    tab_t, tab_d = upload_table(ctx, t), upload_table(ctx, d)
    xt, xd = to_dev(t["x"]), to_dev(d["x"])
    y1, y3, y4 = to_dev(t["y"]), to_dev(d["y"]), to_dev(t["y"])
    y2 = to_dev(np.zeros((t["n"], 384), np.uint16))
    Wd, W2d = to_dev(W), to_dev(W2)
    v = torch.zeros((t["n"], 64), dtype=torch.float32, device="cuda")
    ctx.set_option(L.OPT_EARLY_PAGES, 1)
    ctx.set_option(L.OPT_EARLY_INPUT, 1)
    try:
        L.lora_fused(ctx, tab_t, t["ids"], xt, y1)
        assert ctx.last_path()[0] & 2
        L.lora_base_fused(ctx, tab_t, t["ids"], xt, Wd, y2)
        L.lora_fused(ctx, tab_d, d["ids"], xd, y3)
        assert ctx.last_path()[0] == 1
        L.lora_merge(ctx, tab_d, 1, W2d)
        L.lora_fused(ctx, tab_t, t["ids"], xt, y2)
        L.lora_shrink(ctx, tab_t, t["ids"], xt, v)
        L.lora_expand(ctx, tab_t, t["ids"], v, y4)
        ctx.sync_status()
    finally:
        ctx.set_option(L.OPT_EARLY_PAGES, 0)
        ctx.set_option(L.OPT_EARLY_INPUT, 0)
    T, D = oracle.Table.from_case(t), oracle.Table.from_case(d)
    assert_parity(from_dev(y1), oracle.fused(T, t["ids"], t["x"], t["y"], nthreads=8),
                  REL_FROB, MAX_ABS_RMS, "tile delta")
    base = oracle.base_fused(T, t["ids"], t["x"], W, nthreads=8)
    assert_parity(from_dev(y2), oracle.fused(T, t["ids"], t["x"], from_dev(
        to_dev(base)), nthreads=8), REL_FROB, MAX_ABS_RMS, "delta on the base projection")
    assert_parity(from_dev(y3), oracle.fused(D, d["ids"], d["x"], d["y"], nthreads=8),
                  REL_FROB, MAX_ABS_RMS, "row-gather delta")
    assert_parity(from_dev(W2d), oracle.merge(D, 1, W2, +1), REL_FROB, MAX_ABS_RMS, "merge")
    vh = v.cpu().numpy()
    assert_parity(from_dev(y4), oracle.expand(T, t["ids"], vh, t["y"], nthreads=8),
                  REL_FROB, MAX_ABS_RMS, "expand of the shrink's v")


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable(ctx):
    """Failure detection without a fault: a bounded wait on a barrier nothing arrives
    on gives up after 10 ms, the status word records it, sync_status reports
    LORA_E_TIMEOUT once, and the next call on the same context is exact."""
    ctx.sync_status()
    ctx.selftest_timeout(10000)
    with pytest.raises(L.LoraError) as e:
        ctx.sync_status()
    assert e.value.name == "LORA_E_TIMEOUT"
    ctx.sync_status()                                 # the word was cleared
    c = workloads.make("tiny_decode", seed=9)
    got = run_fused(ctx, c)
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=8)
    assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, "after a timed-out wait")


def test_repeated_ids_over_new_buffers_reuse_the_launch_and_stay_exact(ctx):
    """A decode step applies one ids array to every layer, each with its own adapter
    pools: the library keeps the launch of a row-gather call and, when a table with
    the same ranks and scales, the same shape and the same ids come back, patches
    the pools, x and y and launches.  Results must be bit-identical to a context
    that plans every call -- across layers (each its own tables and x / y),
    alternation between two batches, an option change and a tile-table reload in
    between, and ids rewritten in place -- and a table that cannot serve an adapter
    of the plan is refused, not served from the cache."""
    import os
    fresh = L.Context(0, max_rows=1 << 15, max_rank=64)
    try:
        rng = np.random.default_rng(5)
        ids_het = np.ascontiguousarray(workloads.make("llama7b_decode_het", seed=11)["ids"],
                                       np.int32).copy()
        ids_hom = np.zeros(64, np.int32)
        for layer in range(6):
            # this layer's adapters: the same ranks and scales, new weights
            het = workloads.make("llama7b_decode_het", seed=20 + layer)
            hom = workloads.make("llama7b_decode_hom", seed=20 + layer)
            xs = workloads.to_bf16_bits(rng.standard_normal((64, 4096), dtype=np.float32))
            for case, ids_c in ((het, ids_het), (hom, ids_hom)):
                t, f = upload_table(ctx, case), upload_table(fresh, case)
                x = to_dev(xs)
                y_a, y_b = to_dev(case["y"]), to_dev(case["y"])
                L.lora_fused(ctx, t, ids_c, x, y_a)          # cached after the first layer
                fresh.set_option(L.OPT_TILE_PATH, 1)         # clears the fresh context's cache
                L.lora_fused(fresh, f, ids_c, x, y_b)
                ctx.sync_status()
                fresh.sync_status()
                np.testing.assert_array_equal(from_dev(y_a), from_dev(y_b))
                if layer in (0, 5):
                    ref = oracle.fused(oracle.Table.from_case(case), ids_c, xs, case["y"], nthreads=8)
                    assert_parity(from_dev(y_a), ref, REL_FROB, MAX_ABS_RMS, f"layer {layer}")
            # both contexts always run the same configuration (a different cluster
            # width would change the split-K summation order)
            if layer == 2:
                for c_ in (ctx, fresh):
                    c_.set_option(L.OPT_EARLY_PAGES, 1)
            if layer == 3:
                tbl = os.path.join(os.path.dirname(L.__file__), "tiles.tbl")
                if os.path.exists(tbl):
                    for c_ in (ctx, fresh):
                        c_.tiles_load(tbl)
            if layer == 4:
                ids_het[::5] = -1                            # the same buffer, new contents
        # same ranks and scales, but adapter ids_hom[0] = 0 is not resident here
        bad = workloads.make("llama7b_decode_hom", seed=99)
        ap = bad["a_pages"].copy()
        ap[0, 0] = -1
        tb = upload_table(ctx, dict(bad, a_pages=ap))
        y = to_dev(bad["y"])
        with pytest.raises(L.LoraError) as e:
            L.lora_fused(ctx, tb, ids_hom, to_dev(bad["x"]), y)
        assert e.value.name == "LORA_E_NOT_RESIDENT"
        ctx.sync_status()
        np.testing.assert_array_equal(from_dev(y), bad["y"])
    finally:
        ctx.set_option(L.OPT_EARLY_PAGES, 0)
        fresh.close()


def test_scattered_adapters_are_copied_once_and_again_after_their_pages_change(ctx):
    """S-LoRA's unified pool holds the adapters in scattered pages; the table keeps a
    dense copy of them for the tensor-core kernels.  The first prefill call copies
    them (three launches), later calls do not (two) and give the same bits; after a
    page-in of new weights, and after lora_table_invalidate for pages written behind
    the library's back, the next call copies again and matches the oracle on the new
    weights."""
    c = workloads.make("slora_prefill", seed=2)
    table = upload_table(ctx, c)
    x = to_dev(c["x"])
    outs, launches = [], []
    for _ in range(3):
        y = to_dev(c["y"])
        L.lora_fused(ctx, table, c["ids"], x, y)
        launches.append(ctx.last_path()[1])
        ctx.sync_status()
        outs.append(from_dev(y))
    assert launches[0] == launches[1] + 1 and launches[1] == launches[2] == 2, launches
    np.testing.assert_array_equal(outs[1], outs[0])
    np.testing.assert_array_equal(outs[2], outs[0])
    rows = sample_rows(c, k=64)
    ref = oracle.fused_rows(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], rows, nthreads=8)
    assert_parity(outs[0][rows], ref, REL_FROB, MAX_ABS_RMS, "first call")
    # new weights for the first request's adapter, through lora_page_in
    k = int(c["ids"][0])
    r = int(c["rank"][k])
    rng = np.random.default_rng(7)
    new_a = workloads.to_bf16_bits(rng.standard_normal((r, 4096), dtype=np.float32) / 64)
    new_b = workloads.to_bf16_bits(rng.standard_normal((r, 4096), dtype=np.float32) / 4)
    ha = torch.from_numpy(new_a.view(np.int16)).pin_memory()
    hb = torch.from_numpy(new_b.view(np.int16)).pin_memory()
    L.lora_page_in(ctx, table, k, ha, hb)
    c2 = dict(c, a_pool=c["a_pool"].copy())
    c2["a_pool"][c["a_pages"][k, :r], :4096] = new_a
    c2["a_pool"][c["b_pages"][k, :r], :4096] = new_b
    c2["b_pool"] = c2["a_pool"]
    y = to_dev(c["y"])
    L.lora_fused(ctx, table, c["ids"], x, y)
    assert ctx.last_path()[1] == 3                           # copied again
    ctx.sync_status()
    ref2 = oracle.fused_rows(oracle.Table.from_case(c2), c["ids"], c["x"], c["y"], rows, nthreads=8)
    assert_parity(from_dev(y)[rows], ref2, REL_FROB, MAX_ABS_RMS, "after page-in")
    # pages written by the caller: back to the original weights, then invalidate
    table.a_pool.copy_(to_dev(c["a_pool"]))
    table.invalidate(k)
    y = to_dev(c["y"])
    L.lora_fused(ctx, table, c["ids"], x, y)
    assert ctx.last_path()[1] == 3
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(y), outs[0])

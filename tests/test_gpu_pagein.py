"""Adapter page-in (lora_page_in) on the GPU: bit-exact pages, the delta over
paged-in adapters against the oracle, overlap with compute on another stream, and
the same-stream ordering with early page copies on."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import assert_parity
from tests.conftest import MAX_ABS_RMS, REL_FROB

L = pytest.importorskip("adapter_sgmv_bgmv_gb300")
from tests.gpu_util import from_dev, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    c = L.Context(0, max_rows=4096, max_rank=128)
    yield c
    c.close()


def _pinned(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).pin_memory()


def _host_rows(c, k):
    """Adapter k's A and B as the rows its pages hold (row j = page j)."""
    r = int(c["rank"][k])
    pool = c["a_pool"]
    a = pool[c["a_pages"][k, :r], :c["d_in"]]
    b = c["b_pool"][c["b_pages"][k, :r], :c["d_out"]]
    return _pinned(a), _pinned(b)


def _empty_table(ctx, c):
    """The case's page tables over a zeroed pool of the same shape."""
    pool = torch.zeros(c["a_pool"].shape, dtype=torch.bfloat16, device="cuda")
    t = L.AdapterTable(ctx, pool, pool, c["rank"], c["scale"], c["a_pages"], c["b_pages"])
    return t, pool


def _case(seed=61, n=600):
    ranks = [8, 16, 32, 64]
    ids = np.repeat(np.arange(4, dtype=np.int32), n // 4)        # runs long enough for tiles
    ids[::7] = (ids[::7] + 1) % 4                               # and short runs for the rows path
    return workloads.small(seed=seed, n=n, d_in=256, d_out=384, n_adapters=4, ranks=ranks,
                           paged=True, ids=ids)


def test_page_in_fills_the_pages_bit_exactly_and_the_delta_matches_the_oracle(ctx):
    c = _case()
    t, pool = _empty_table(ctx, c)
    hosts = [_host_rows(c, k) for k in range(4)]
    for k in range(4):
        L.lora_page_in(ctx, t, k, *hosts[k])
        assert ctx.last_path() == (8, 1)
    ctx.sync_status()
    got = from_dev(pool)
    used = np.zeros(got.shape[0], bool)
    for k in range(4):
        r = int(c["rank"][k])
        pa, pb = c["a_pages"][k, :r], c["b_pages"][k, :r]
        np.testing.assert_array_equal(got[pa, :c["d_in"]], c["a_pool"][pa, :c["d_in"]])
        np.testing.assert_array_equal(got[pb, :c["d_out"]], c["b_pool"][pb, :c["d_out"]])
        np.testing.assert_array_equal(got[pa, c["d_in"]:], 0)    # the rest of a page untouched
        used[pa] = used[pb] = True
    np.testing.assert_array_equal(got[~used], 0)
    y = to_dev(c["y"])
    L.lora_fused(ctx, t, c["ids"], to_dev(c["x"]), y)
    ctx.sync_status()
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=8)
    assert_parity(from_dev(y), ref, REL_FROB, MAX_ABS_RMS, "after page-in")


def test_page_in_overlaps_compute_on_another_stream(ctx):
    """Adapter 3 is paged in on a side stream while a call over adapters 0-2 runs;
    the call that uses adapter 3 is ordered after the page-in by an event."""
    c = _case(seed=62)
    t, _ = _empty_table(ctx, c)
    hosts = [_host_rows(c, k) for k in range(4)]
    for k in range(3):
        L.lora_page_in(ctx, t, k, *hosts[k])
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    ids_a = np.where(c["ids"] == 3, -1, c["ids"]).astype(np.int32)
    x = to_dev(c["x"])
    y1 = to_dev(c["y"])
    side.wait_stream(main)
    L.lora_fused(ctx, t, ids_a, x, y1, main)
    L.lora_page_in(ctx, t, 3, *hosts[3], stream=side)
    done = torch.cuda.Event()
    done.record(side)
    main.wait_event(done)
    y2 = to_dev(c["y"])
    L.lora_fused(ctx, t, c["ids"], x, y2, main)
    ctx.sync_status()
    tab = oracle.Table.from_case(c)
    assert_parity(from_dev(y1), oracle.fused(tab, ids_a, c["x"], c["y"], nthreads=8), REL_FROB,
                  MAX_ABS_RMS, "call beside the page-in")
    assert_parity(from_dev(y2), oracle.fused(tab, c["ids"], c["x"], c["y"], nthreads=8), REL_FROB,
                  MAX_ABS_RMS, "call after the page-in")


def test_page_in_then_delta_on_the_same_stream_with_early_page_copies(ctx):
    """A page-in writes the pools, so the delta call right after it on the same
    stream takes no early page copies: alternating two versions of every adapter,
    each call sees the version paged in just before it."""
    c1 = _case(seed=63)
    c2 = dict(c1)
    rng = np.random.default_rng(64)
    pool2 = c1["a_pool"].copy()
    used = np.concatenate([c1["a_pages"][c1["a_pages"] >= 0], c1["b_pages"][c1["b_pages"] >= 0]])
    pool2[used] = workloads._normal(rng, (used.size, pool2.shape[1]), 0.05)
    c2["a_pool"] = c2["b_pool"] = pool2
    t, _ = _empty_table(ctx, c1)
    hosts = {v: [_host_rows(cv, k) for k in range(4)] for v, cv in ((1, c1), (2, c2))}
    x = to_dev(c1["x"])
    ctx.set_option(L.OPT_EARLY_PAGES, 1)
    try:
        outs = []
        for v in (1, 2, 1, 2):
            for k in range(4):
                L.lora_page_in(ctx, t, k, *hosts[v][k])
            y = to_dev(c1["y"])
            L.lora_fused(ctx, t, c1["ids"], x, y)
            outs.append((v, y))
        ctx.sync_status()
    finally:
        ctx.set_option(L.OPT_EARLY_PAGES, 0)
    refs = {v: oracle.fused(oracle.Table.from_case(cv), cv["ids"], cv["x"], cv["y"], nthreads=8)
            for v, cv in ((1, c1), (2, c2))}
    for v, y in outs:
        assert_parity(from_dev(y), refs[v], REL_FROB, MAX_ABS_RMS, f"version {v}")


def test_cached_decode_launch_is_not_reused_right_after_a_page_in(ctx):
    """With early pages and early input on, a decode-only call is kept in the launch
    cache laid out for early input (y read after the wait, no y rows in shared
    memory).  A page-in just before a call turns early input off for that call, so
    the cached launch must not be reused then.  Alternating two versions of every
    adapter (a page-in before the first of two calls), each call sees the version
    paged in before it."""
    c1 = _case(seed=66, n=64)
    c1["ids"] = (np.arange(64) % 4).astype(np.int32)          # runs of one row: row-gather only
    c2 = dict(c1)
    rng = np.random.default_rng(67)
    pool2 = c1["a_pool"].copy()
    used = np.concatenate([c1["a_pages"][c1["a_pages"] >= 0], c1["b_pages"][c1["b_pages"] >= 0]])
    pool2[used] = workloads._normal(rng, (used.size, pool2.shape[1]), 0.05)
    c2["a_pool"] = c2["b_pool"] = pool2
    t, _ = _empty_table(ctx, c1)
    hosts = {v: [_host_rows(cv, k) for k in range(4)] for v, cv in ((1, c1), (2, c2))}
    x = to_dev(c1["x"])
    ctx.set_option(L.OPT_EARLY_PAGES, 1)
    ctx.set_option(L.OPT_EARLY_INPUT, 1)
    try:
        outs = []
        for v in (1, 2, 1, 2):
            for k in range(4):
                L.lora_page_in(ctx, t, k, *hosts[v][k])
            for _ in range(2):
                y = to_dev(c1["y"])
                L.lora_fused(ctx, t, c1["ids"], x, y)
                assert ctx.last_path()[0] == 1
                outs.append((v, y))
        ctx.sync_status()
    finally:
        ctx.set_option(L.OPT_EARLY_PAGES, 0)
        ctx.set_option(L.OPT_EARLY_INPUT, 0)
    refs = {v: oracle.fused(oracle.Table.from_case(cv), cv["ids"], cv["x"], cv["y"], nthreads=8)
            for v, cv in ((1, c1), (2, c2))}
    for v, y in outs:
        assert_parity(from_dev(y), refs[v], REL_FROB, MAX_ABS_RMS, f"version {v}")


def test_page_in_refuses_bad_buffers_and_arguments(ctx):
    c = _case(seed=65)
    t, pool = _empty_table(ctx, c)
    ha, hb = _host_rows(c, 1)
    with pytest.raises(ValueError):                  # not page-locked
        L.lora_page_in(ctx, t, 1, ha.clone(), hb)
    with pytest.raises(ValueError):                  # rows != rank
        L.lora_page_in(ctx, t, 1, _pinned(np.zeros((8, 256), np.uint16)), hb)
    # the C layer refuses pageable memory by itself (nothing launched)
    plain = np.zeros((16, 256), np.uint16)
    rc = L._L.lora_page_in(ctx.handle, t.handle, 1, plain.ctypes.data, 256, hb.data_ptr(), 384,
                           torch.cuda.current_stream().cuda_stream)
    assert L.ERROR_NAMES[rc] == "LORA_E_INVAL"
    wide = _pinned(np.zeros((16, c["a_pool"].shape[1] + 8), np.uint16))
    with pytest.raises(L.LoraError) as e:            # wider than a page
        L.lora_page_in(ctx, t, 1, wide, hb)
    assert e.value.name == "LORA_E_INVAL"
    with pytest.raises(L.LoraError) as e:
        L.lora_page_in(ctx, t, 9, ha, hb)
    assert e.value.name == "LORA_E_ADAPTER"
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(pool), 0)   # nothing was written


def test_page_in_bandwidth_report(ctx):
    """32 rank-64 adapters at d = 4096 (32 MB) paged in back to back: report the
    rate (no bar: it depends on the host link) and check one adapter's pages."""
    n_ad, r, d = 32, 64, 4096
    rng = np.random.default_rng(66)
    n_pages = 2 * r * n_ad
    order = rng.permutation(n_pages).astype(np.int32)
    ap = order[: r * n_ad].reshape(n_ad, r)
    bp = order[r * n_ad:].reshape(n_ad, r)
    pool = torch.zeros((n_pages, d), dtype=torch.bfloat16, device="cuda")
    big = L.Context(0, max_rows=64, max_rank=64)
    t = L.AdapterTable(big, pool, pool, np.full(n_ad, r, np.int32), np.ones(n_ad, np.float32), ap, bp)
    ha = [_pinned(rng.integers(0, 1 << 16, (r, d), dtype=np.uint16)) for _ in range(n_ad)]
    hb = [_pinned(rng.integers(0, 1 << 16, (r, d), dtype=np.uint16)) for _ in range(n_ad)]
    for k in range(n_ad):                            # warm-up
        L.lora_page_in(big, t, k, ha[k], hb[k])
    torch.cuda.synchronize()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    # device time: the launches queue up behind a short sleep kernel, so the host's
    # per-call cost stays out of the timed region
    torch.cuda._sleep(4_000_000)
    e0.record()
    for k in range(n_ad):
        L.lora_page_in(big, t, k, ha[k], hb[k])
    e1.record()
    torch.cuda.synchronize()
    # issue-bound: the same launches as the host issues them
    e2.record()
    for k in range(n_ad):
        L.lora_page_in(big, t, k, ha[k], hb[k])
    e3 = torch.cuda.Event(enable_timing=True)
    e3.record()
    torch.cuda.synchronize()
    nbytes = 2 * n_ad * r * d * 2
    dev_ms, host_ms = e0.elapsed_time(e1), e2.elapsed_time(e3)
    print(f"\npage-in: {nbytes / 1e6:.1f} MB in {n_ad} launches; device {dev_ms * 1e3:.1f} us = "
          f"{nbytes / (dev_ms * 1e-3) / 1e9:.1f} GB/s; as issued from Python {host_ms * 1e3:.1f} us = "
          f"{nbytes / (host_ms * 1e-3) / 1e9:.1f} GB/s")
    got = from_dev(pool)
    np.testing.assert_array_equal(got[ap[7]], ha[7].numpy().view(np.uint16))
    np.testing.assert_array_equal(got[bp[7]], hb[7].numpy().view(np.uint16))
    big.close()

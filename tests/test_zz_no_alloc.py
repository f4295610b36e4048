"""lora_fused_noalloc: the fused delta for callers that must not allocate device or
pinned memory while it runs (its scratch is a fixed array inside the library).
It must give the same results as lora_fused, call after call, and leave the GPU's
free memory unchanged.  Collected last on purpose: a failure here comes after every
other test has run."""
import numpy as np
import pytest
import torch

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


def test_noalloc_matches_fused_on_two_calls_and_allocates_nothing():
    ctx = L.Context(0, max_rows=4096, max_rank=64)
    cases = [_case(71), _case(72)]
    tables = [upload_table(ctx, c) for c in cases]
    xs = [to_dev(c["x"]) for c in cases]
    y_ref = [to_dev(c["y"]) for c in cases]
    y_got = [to_dev(c["y"]) for c in cases]
    warm = to_dev(cases[0]["y"])
    for c, t, x, y in zip(cases, tables, xs, y_ref):      # the existing entry point
        L.lora_fused(ctx, t, c["ids"], x, y)
    L.lora_fused_noalloc(ctx, tables[0], cases[0]["ids"], xs[0], warm)   # first-call set-up
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for c, t, x, y in zip(cases, tables, xs, y_got):      # two calls in a row
        L.lora_fused_noalloc(ctx, t, c["ids"], x, y)
        assert ctx.last_path()[0] == 3                    # tiles and row-gather both ran
    ctx.sync_status()
    assert torch.cuda.mem_get_info()[0] == free_before
    for k in range(2):
        assert_parity(from_dev(y_got[k]), from_dev(y_ref[k]), REL_FROB, MAX_ABS_RMS, f"call {k}")
        rel = cases[k]["ids"] < 0
        np.testing.assert_array_equal(from_dev(y_got[k])[rel], cases[k]["y"][rel])
    ctx.close()


def test_noalloc_rejects_batches_beyond_its_fixed_scratch():
    ctx = L.Context(0, max_rows=1 << 15, max_rank=64)
    c = workloads.small(seed=73, n=65 * 128, d_in=64, d_out=64, n_adapters=1, ranks=[8],
                        ids=np.zeros(65 * 128, np.int32))
    t = upload_table(ctx, c)
    y = to_dev(c["y"])
    with pytest.raises(L.LoraError) as e:
        L.lora_fused_noalloc(ctx, t, c["ids"], to_dev(c["x"]), y)
    assert e.value.name == "LORA_E_CAPACITY"
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(y), c["y"])
    ctx.close()

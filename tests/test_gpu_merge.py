"""GPU parity of lora_merge / lora_unmerge (W +/- s A B in place) against the oracle."""
import numpy as np
import pytest

import oracle
import workloads
from tests._helpers import adapter_mats, assert_parity, bf16_ulp, f64
from tests.conftest import MAX_ABS_RMS, REL_FROB

pytestmark = pytest.mark.gpu

L = pytest.importorskip("adapter_sgmv_bgmv_gb300")
from tests.gpu_util import from_dev, to_dev, upload_table  # noqa: E402


@pytest.fixture(scope="module")
def ctx():
    c = L.Context(0, max_rows=1 << 12, max_rank=64)
    yield c
    c.close()


@pytest.mark.parametrize("kernel", [0, 1], ids=["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("shape", [(96, 80, [16, 8]), (200, 264, [64, 32]), (128, 256, [8, 24])])
def test_merge_small_full(ctx, shape, kernel):
    ctx.set_option(L.OPT_MERGE_KERNEL, kernel)
    try:
        _merge_small_full(ctx, shape)
    finally:
        ctx.set_option(L.OPT_MERGE_KERNEL, 0)


def _merge_small_full(ctx, shape):
    d_in, d_out, ranks = shape
    c = workloads.small(seed=41, n=1, d_in=d_in, d_out=d_out, n_adapters=len(ranks),
                        ranks=ranks, paged=True)
    W = workloads.make_W(d_in, d_out, seed=4)
    table = upload_table(ctx, c)
    t = oracle.Table.from_case(c)
    for k in range(len(ranks)):
        Wd = to_dev(W)
        L.lora_merge(ctx, table, k, Wd)
        ctx.sync_status()
        got = from_dev(Wd)
        ref = oracle.merge(t, k, W, +1)
        assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, f"merge k={k}")
        L.lora_unmerge(ctx, table, k, Wd)
        ctx.sync_status()
        back = from_dev(Wd)
        A, B = adapter_mats(c, k)
        mag = np.maximum(np.abs(f64(W)), np.abs(f64(W) + float(c["scale"][k]) * (A @ B)))
        assert (np.abs(f64(back) - f64(W)) <= 2 * bf16_ulp(mag)).all()


def test_merge_valora_full_size_sampled(ctx):
    c = workloads.make("valora_merge", seed=0)
    W = c["W"]
    table = upload_table(ctx, c)
    Wd = to_dev(W)
    k = c["merge_adapter"]
    L.lora_merge(ctx, table, k, Wd)
    ctx.sync_status()
    got = from_dev(Wd)
    rows = np.unique(np.concatenate([np.arange(0, 4096, 97), [0, 127, 128, 4095]]))
    ref = oracle.merge(oracle.Table.from_case(c), k, W, +1, nthreads=8, rows=rows)
    assert_parity(got[rows], ref, REL_FROB, MAX_ABS_RMS, "valora merge")
    # every element is within one bf16 step of the oracle's
    assert (np.abs(f64(got[rows]) - f64(ref)) <= bf16_ulp(f64(ref)) + 1e-30).mean() > 0.999
    L.lora_unmerge(ctx, table, k, Wd)
    ctx.sync_status()
    back = from_dev(Wd)
    A, B = adapter_mats(c, k)
    mag = np.maximum(np.abs(f64(W[rows])),
                     np.abs(f64(W[rows]) + float(c["scale"][k]) * (A[rows] @ B)))
    assert (np.abs(f64(back[rows]) - f64(W[rows])) <= 2 * bf16_ulp(mag)).all()


def test_merge_rejects_bad_arguments(ctx):
    c = workloads.small(seed=42, n=1, d_in=64, d_out=64, n_adapters=2, ranks=[8, 8])
    table = upload_table(ctx, c)
    W = to_dev(workloads.make_W(64, 64))
    with pytest.raises(L.LoraError) as e:
        L.lora_merge(ctx, table, 5, W)
    assert e.value.name == "LORA_E_ADAPTER"
    with pytest.raises(L.LoraError) as e:
        L.lora_merge(ctx, table, 0, to_dev(workloads.make_W(72, 64)))   # d_in > page width
    assert e.value.name == "LORA_E_INVAL"

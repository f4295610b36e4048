"""GPU parity of lora_base_fused -- the base projection with the adapter term in one
tensor-core GEMM, y = bf16(x W + s_k (x A_k) B_k), x W alone for released rows --
against the oracle (x W as a float64 matmul plus the adapter term in double, one
rounding), through the C ABI, on every output element.  Bar: the benchmark spec's
(relative Frobenius <= 5e-3, every element within max(2e-2 rms, one bf16 step), the
one-step allowance on at most 1e-3 of the elements)."""
import os

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

NCPU = os.cpu_count() or 4


@pytest.fixture(scope="module")
def ctx():
    c = L.Context(0, max_rows=1 << 15, max_rank=128)
    yield c
    c.close()


def _run(ctx, case, W, ids=None, canary=True):
    ids = case["ids"] if ids is None else ids
    table = upload_table(ctx, case)
    n, d_out = case["n"], W.shape[1]
    # y starts as NaN bit patterns: every element must be overwritten
    y = to_dev(np.full((n, d_out), 0x7FC1 if canary else 0, np.uint16))
    L.lora_base_fused(ctx, table, ids, to_dev(case["x"]), to_dev(W), y)
    ctx.sync_status()
    path = ctx.last_path()[0]
    return from_dev(y), path


def _report(stats):
    print(f"\n[parity] {stats['what']}: rel_frob={stats['rel_frob']:.3e} "
          f"max_abs/rms={stats['max_abs_over_rms']:.3e} one-step={stats['one_step']}"
          f"/{stats['elements']} (cap {stats['one_step_cap']})")


SMALL = {
    # two 256-row pair blocks (the second one 44 rows, so its second CTA's half lies
    # wholly past n), d_in not a multiple of the 64-wide K block, d_out = 256 + 136
    # (a ragged second column block whose second CTA holds 8 valid columns), mixed
    # ranks with a padded one, paged adapters, released rows, blocks holding several
    # adapters
    "ragged_mixed": dict(seed=201, n=300, d_in=200, d_out=392, n_adapters=4,
                         ranks=[8, 24, 64, 128], paged=True, release_frac=0.15),
    # long runs of one adapter: blocks with a single term (no masked rows)
    "runs": dict(seed=202, n=512, d_in=256, d_out=512, n_adapters=2, ranks=[64, 16],
                 ids=np.repeat(np.array([1, 0, -1, 1], np.int32), 128)),
    # 16 x 10 = 160 tiles over at most 76 CTA pairs, so a pair runs two or three tiles
    # in a row (both accumulators, the stage ring wrapping across tiles), with 16 K
    # blocks per tile -- more than the ring holds -- before each block's adapter
    # stages; runs of several lengths, released rows, blocks with one to three
    # adapters, and blocks whose two halves hold different adapters
    "multi_tile": dict(seed=206, n=4096, d_in=1024, d_out=2560, n_adapters=3,
                       ranks=[16, 64, 32], paged=True,
                       ids=np.repeat(np.array([0, 1, -1, 2, 1, 0, 2, -1, 1, 2], np.int32),
                                     [700, 300, 57, 900, 441, 128, 1000, 3, 300, 267])),
    # the first CTA's half of the pair released, the second's all one adapter: the
    # term's stages carry rows in one half only
    "second_half_only": dict(seed=207, n=256, d_in=192, d_out=512, n_adapters=2, ranks=[32, 16],
                             ids=np.repeat(np.array([-1, 1], np.int32), 128)),
    # one row per adapter (a decode-like block with many terms, all in the first
    # CTA's half of the pair)
    "many_terms": dict(seed=203, n=40, d_in=128, d_out=256, n_adapters=40, ranks=[16] * 40,
                       ids=np.arange(40, dtype=np.int32)),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_match_the_oracle(ctx, name):
    c = workloads.small(**SMALL[name])
    W = workloads.make_W(c["d_in"], c["d_out"], seed=7)
    got, path = _run(ctx, c, W)
    assert path & 16
    ref = oracle.base_fused(oracle.Table.from_case(c), c["ids"], c["x"], W, nthreads=NCPU)
    _report(assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, name))


def test_every_row_released_is_the_plain_gemm(ctx):
    c = workloads.small(seed=204, n=260, d_in=320, d_out=640, n_adapters=2, ranks=[16, 16])
    W = workloads.make_W(320, 640, seed=8)
    ids = np.full(260, -1, np.int32)
    got, path = _run(ctx, c, W, ids=ids)
    assert path == 16                               # no shrink: nothing to add
    ref = oracle.base_fused(oracle.Table.from_case(c), ids, c["x"], W, nthreads=NCPU)
    _report(assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, "all released"))


def test_zero_base_leaves_the_delta_alone(ctx):
    """W = 0: the GEMM's base part vanishes and y is the adapter term alone, the
    strictest check of the term stages (compared with the fused oracle on y_in = 0)."""
    c = workloads.small(**dict(SMALL["ragged_mixed"], y_mode="zero"))
    W = np.zeros((c["d_in"], c["d_out"]), np.uint16)
    got, _ = _run(ctx, c, W)
    ref = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"], nthreads=NCPU)
    _report(assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, "W = 0"))
    rel = c["ids"] < 0
    assert (got[rel] == 0).all()                    # released rows: x 0 = 0 exactly


@pytest.fixture(scope="module")
def valora():
    c = workloads.make("valora_prefill", seed=0)
    W = workloads.make_W(c["d_in"], c["d_out"], seed=0)
    return c, W


def test_valora_every_element(ctx, valora):
    """16,896 x 4096 -> 11008 with four rank-64 adapters: all rows and columns."""
    c, W = valora
    got, path = _run(ctx, c, W)
    assert path & 16
    ref = oracle.base_fused(oracle.Table.from_case(c), c["ids"], c["x"], W, nthreads=NCPU)
    _report(assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, "valora base + delta"))


def test_valora_delta_part_alone(ctx, valora):
    c, _ = valora
    cz = dict(c, y=np.zeros_like(c["y"]))
    got, _ = _run(ctx, cz, np.zeros((c["d_in"], c["d_out"]), np.uint16))
    ref = oracle.fused(oracle.Table.from_case(cz), c["ids"], c["x"], cz["y"], nthreads=NCPU)
    _report(assert_parity(got, ref, REL_FROB, MAX_ABS_RMS, "valora, W = 0"))


def test_bad_arguments_launch_nothing(ctx):
    c = workloads.small(seed=205, n=16, d_in=64, d_out=64, n_adapters=2, ranks=[8, 8])
    table = upload_table(ctx, c)
    y = to_dev(c["y"])
    x = to_dev(c["x"])
    Wbad = to_dev(np.zeros(64 * 64 + 8, np.uint16))[1:1 + 64 * 64].view(64, 64)   # misaligned
    with pytest.raises(L.LoraError) as e:
        L.lora_base_fused(ctx, table, c["ids"], x, Wbad, y)
    assert e.value.name == "LORA_E_INVAL" and ctx.last_path() == (0, 0)
    with pytest.raises(L.LoraError) as e:
        L.lora_base_fused(ctx, table, np.full(16, 5, np.int32), x, to_dev(workloads.make_W(64, 64)), y)
    assert e.value.name == "LORA_E_ADAPTER"
    ctx.sync_status()
    np.testing.assert_array_equal(from_dev(y), c["y"])

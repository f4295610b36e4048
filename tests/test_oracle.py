"""Pins for the CPU oracle, each against something other than the oracle itself:
hand-worked values, float64 brute force with numpy matmul, closed forms, the
dense-GEMM reduction, merged == unmerged inference, and torch's bf16 conversion."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests._helpers import (adapter_mats, assert_nearest_bf16, assert_parity, bf16_ulp,
                            exact_delta, f64, parity_values, to_bf16_bits)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_delta.txt")


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_round_hand_patterns():
    cases = {1.0: 0x3F80, -2.0: 0xC000, 1 + 2 ** -8: 0x3F80,        # tie -> even (down)
             1 + 3 * 2 ** -8: 0x3F82,                                 # tie -> even (up)
             1 + 2 ** -8 + 2 ** -30: 0x3F81,                          # just above the tie
             2.0 ** -133: 0x0001, 2.0 ** -134: 0x0000, 3 * 2.0 ** -134: 0x0002,
             3.3895313892515355e38: 0x7F7F, 3.4e38: 0x7F80, -0.0: 0x8000,
             float("inf"): 0x7F80, float("-inf"): 0xFF80}
    for v, bits in cases.items():
        assert oracle.bf16_round(v) == bits, (v, hex(oracle.bf16_round(v)), hex(bits))
    assert oracle.bf16_round(float("nan")) & 0x7F80 == 0x7F80
    assert oracle.bf16_value(0x3F80) == 1.0 and oracle.bf16_value(0xC0A0) == -5.0


def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, 4000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    vals = np.concatenate([vals, rng.standard_normal(2000).astype(np.float32),
                           (rng.standard_normal(500) * 1e-39).astype(np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_bf16_round_is_nearest_for_doubles():
    rng = np.random.default_rng(2)
    vals = rng.standard_normal(3000) * np.exp(rng.uniform(-20, 20, 3000))
    got = np.array([oracle.bf16_round(float(v)) for v in vals], np.uint16)
    assert_nearest_bf16(got, vals, slack=0.0)


# ---------------------------------------------------------------- hand-worked values

def _golden():
    rows = {}
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, rest = line.split(None, 1)
            rows[key] = [[float(t) for t in part.split()] for part in rest.split("|")]
    return rows


def _golden_case():
    g = _golden()
    d_in, d_out = int(g["d_in"][0][0]), int(g["d_out"][0][0])
    a_pool = to_bf16_bits(np.array(g["a0_cols"] + g["a1_cols"], np.float32))
    b_pool = to_bf16_bits(np.array(g["b0_rows"] + g["b1_rows"], np.float32))
    case = dict(d_in=d_in, d_out=d_out, a_pool=a_pool, b_pool=b_pool,
                rank=np.array([2, 2], np.int32), scale=np.array(g["scale"][0], np.float32),
                a_pages=np.array([[0, 1], [2, 3]], np.int32),
                b_pages=np.array([[0, 1], [2, 3]], np.int32),
                ids=np.array(g["ids"][0], np.int32),
                x=to_bf16_bits(np.array(g["x"], np.float32)),
                y=to_bf16_bits(np.array(g["y_in"], np.float32)), n=3)
    return case, g


def test_golden_hand_delta():
    case, g = _golden_case()
    t = oracle.Table.from_case(case)
    y = oracle.fused(t, case["ids"], case["x"], case["y"])
    np.testing.assert_array_equal(f64(y), np.array(g["y_out"]))
    v = oracle.shrink(t, case["ids"], case["x"])
    np.testing.assert_array_equal(v[[0, 2]], np.array([g["v_rows"][0], g["v_rows"][2]]))
    assert np.isnan(v[1]).all()                      # released row: v untouched
    y2 = oracle.expand(t, case["ids"], v, case["y"])
    np.testing.assert_array_equal(f64(y2), np.array(g["y_out"]))
    W = to_bf16_bits(np.array(g["W_in"], np.float32))
    Wm = oracle.merge(t, 0, W, +1)
    np.testing.assert_array_equal(f64(Wm), np.array(g["W_merged"]))
    np.testing.assert_array_equal(oracle.merge(t, 0, Wm, -1), W)   # exact here
    p = oracle.plan(case["ids"], 2)
    assert p["active_rows"].tolist() == [0, 2] and p["perm"].tolist() == [0, 2]
    assert p["seg_offsets"].tolist() == [0, 1, 2] and p["seg_adapter"].tolist() == [0, 1]


# ---------------------------------------------------------------- brute force

SMALL = [
    dict(seed=3, n=9, d_in=40, d_out=24, n_adapters=3, ranks=[8, 16, 8]),
    dict(seed=4, n=12, d_in=64, d_out=64, n_adapters=2, ranks=[8, 24], paged=True,
         release_frac=0.3),
    dict(seed=5, n=7, d_in=16, d_out=48, n_adapters=4, ranks=[8, 8, 16, 32],
         release_frac=0.5, y_mode="zero"),
]


@pytest.mark.parametrize("kw", SMALL)
def test_fused_is_nearest_bf16_of_exact(kw):
    c = workloads.small(**kw)
    t = oracle.Table.from_case(c)
    y = oracle.fused(t, c["ids"], c["x"], c["y"])
    exact = f64(c["y"]) + exact_delta(c)
    assert_nearest_bf16(y, exact)
    rel = c["ids"] < 0
    np.testing.assert_array_equal(y[rel], c["y"][rel])


@pytest.mark.parametrize("kw", SMALL)
def test_shrink_expand_brute_force(kw):
    c = workloads.small(**kw)
    t = oracle.Table.from_case(c)
    v = oracle.shrink(t, c["ids"], c["x"])
    X = f64(c["x"])
    for i, k in enumerate(c["ids"]):
        if k < 0:
            assert np.isnan(v[i]).all()
            continue
        A, _ = adapter_mats(c, int(k))
        r = A.shape[1]
        np.testing.assert_allclose(v[i, :r], X[i] @ A, rtol=1e-6, atol=1e-6)
        assert np.isnan(v[i, r:]).all()                  # columns >= rank untouched
    v0 = np.where(np.isnan(v), 0, v).astype(np.float32)
    y = oracle.expand(t, c["ids"], v0, c["y"])
    exact = f64(c["y"]).copy()
    for i, k in enumerate(c["ids"]):
        if k >= 0:
            _, B = adapter_mats(c, int(k))
            exact[i] += float(c["scale"][k]) * (v0[i, :B.shape[0]].astype(np.float64) @ B)
    assert_nearest_bf16(y, exact)
    # shrink then expand (v rounded to fp32) against the fused definition
    assert_parity(y, oracle.fused(t, c["ids"], c["x"], c["y"]), 1e-5, 1e-4, "decomposition")


def test_merge_brute_force_and_row_subset():
    c = workloads.small(seed=6, n=1, d_in=48, d_out=40, n_adapters=2, ranks=[8, 16],
                        paged=True)
    W = workloads.make_W(48, 40, seed=1)
    t = oracle.Table.from_case(c)
    for k, sign in ((0, +1), (1, -1)):
        A, B = adapter_mats(c, k)
        got = oracle.merge(t, k, W, sign)
        assert_nearest_bf16(got, f64(W) + sign * float(c["scale"][k]) * (A @ B))
        rows = np.array([0, 5, 47, 13])
        np.testing.assert_array_equal(oracle.merge(t, k, W, sign, rows=rows), got[rows])


# ---------------------------------------------------------------- closed forms

def _tiny():
    return workloads.make("tiny_decode", seed=7)


def test_zero_B_and_zero_scale_leave_y_bit_exact():
    c = _tiny()
    for mutate in ("B", "s"):
        d = dict(c)
        if mutate == "B":
            d["b_pool"] = np.zeros_like(c["b_pool"])
        else:
            d["scale"] = np.zeros_like(c["scale"])
        y = oracle.fused(oracle.Table.from_case(d), d["ids"], d["x"], d["y"])
        np.testing.assert_array_equal(y, c["y"])


def test_released_and_zero_x_rows_unchanged():
    c = _tiny()
    ids = c["ids"].copy()
    ids[::3] = -1
    x = c["x"].copy()
    x[1] = 0
    y = oracle.fused(oracle.Table.from_case(c), ids, x, c["y"])
    np.testing.assert_array_equal(y[::3], c["y"][::3])
    np.testing.assert_array_equal(y[1], c["y"][1])
    assert (y[ids >= 0] != c["y"][ids >= 0]).any()


def test_one_hot_adapter_moves_one_value():
    c = _tiny()
    d_in, d_out = c["d_in"], c["d_out"]
    p_idx, q_idx = 37, 201
    a_pool = np.zeros_like(c["a_pool"])
    b_pool = np.zeros_like(c["b_pool"])
    a_pool[0, p_idx] = to_bf16_bits(np.array([1.0], np.float32))[0]   # A_0[:,0] = e_p
    b_pool[0, q_idx] = to_bf16_bits(np.array([1.0], np.float32))[0]   # B_0[0,:] = e_q
    d = dict(c, a_pool=a_pool, b_pool=b_pool)
    ids = np.zeros(c["n"], np.int32)
    y = oracle.fused(oracle.Table.from_case(d), ids, c["x"], c["y"])
    s = float(c["scale"][0])
    assert s == 2.0
    expect = c["y"].copy()
    col = f64(c["y"][:, q_idx]) + s * f64(c["x"][:, p_idx])
    expect[:, q_idx] = to_bf16_bits(col.astype(np.float32))   # exact in fp32 here
    np.testing.assert_array_equal(y, expect)


def test_single_adapter_batch_is_one_dense_gemm():
    c = workloads.small(seed=8, n=33, d_in=96, d_out=80, n_adapters=1, ranks=[16],
                        y_mode="zero")
    A, B = adapter_mats(c, 0)
    dense = float(c["scale"][0]) * (f64(c["x"]) @ (A @ B))   # one GEMM with Delta W
    y = oracle.fused(oracle.Table.from_case(c), c["ids"], c["x"], c["y"])
    assert_nearest_bf16(y, dense, slack=1e-6)


def test_merged_equals_unmerged_inference():
    """x.(W + s A B) with the merged weight and x.W + s (x A) B through the delta both
    land within the parity bar of the exact float64 value (each carries only bf16
    rounding); a transposed or sign-flipped Delta W would miss by O(1)."""
    c = workloads.small(seed=9, n=24, d_in=128, d_out=96, n_adapters=1, ranks=[16],
                        y_mode="zero")
    W = workloads.make_W(128, 96, seed=2)
    t = oracle.Table.from_case(c)
    A, B = adapter_mats(c, 0)
    X = f64(c["x"])
    exact = X @ f64(W) + float(c["scale"][0]) * ((X @ A) @ B)
    Wm = oracle.merge(t, 0, W, +1)
    merged = X @ f64(Wm)                                   # x . merge(W)
    base = to_bf16_bits((X @ f64(W)).astype(np.float32))
    unmerged = f64(oracle.fused(t, c["ids"], c["x"], base))  # x.W + s (x A) B
    for name, got in (("merged", merged), ("unmerged", unmerged)):
        rel, mx = parity_values(got, exact)
        assert rel <= 5e-3 and mx <= 2e-2, (name, rel, mx)
    rel, _ = parity_values(merged, unmerged)
    assert rel <= 5e-3


def test_merge_then_unmerge_restores_W_within_two_ulps():
    c = workloads.small(seed=10, n=1, d_in=64, d_out=64, n_adapters=1, ranks=[32])
    W = workloads.make_W(64, 64, seed=3)
    t = oracle.Table.from_case(c)
    W2 = oracle.merge(t, 0, oracle.merge(t, 0, W, +1), -1)
    A, B = adapter_mats(c, 0)
    mag = np.maximum(np.abs(f64(W)), np.abs(f64(W) + float(c["scale"][0]) * (A @ B)))
    assert (np.abs(f64(W2) - f64(W)) <= 2 * bf16_ulp(mag)).all()


def test_fused_same_result_any_thread_count():
    c = workloads.small(seed=11, n=50, d_in=64, d_out=72, n_adapters=5,
                        ranks=[8, 16, 24, 8, 32], release_frac=0.2)
    t = oracle.Table.from_case(c)
    y1 = oracle.fused(t, c["ids"], c["x"], c["y"], nthreads=1)
    y4 = oracle.fused(t, c["ids"], c["x"], c["y"], nthreads=4)
    np.testing.assert_array_equal(y1, y4)


# ---------------------------------------------------------------- plan bookkeeping

def _numpy_plan(ids, n_adapters):
    ids = np.asarray(ids)
    active = np.flatnonzero(ids >= 0).astype(np.int32)
    perm = active[np.argsort(ids[active], kind="stable")].astype(np.int32)
    counts = np.bincount(ids[active], minlength=n_adapters)
    seg_adapter = np.flatnonzero(counts).astype(np.int32)
    seg_offsets = np.concatenate([[0], np.cumsum(counts[seg_adapter])]).astype(np.int32)
    return active, perm, seg_offsets, seg_adapter


@pytest.mark.parametrize("seed", range(6))
def test_plan_matches_independent_numpy(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(0, 300))
    na = int(rng.integers(1, 40))
    ids = rng.integers(-1, na, n).astype(np.int32)
    if seed == 4:
        ids[:] = -1
    p = oracle.plan(ids, na)
    a, pm, so, sa = _numpy_plan(ids, na)
    np.testing.assert_array_equal(p["active_rows"], a)
    np.testing.assert_array_equal(p["perm"], pm)
    np.testing.assert_array_equal(p["seg_offsets"], so)
    np.testing.assert_array_equal(p["seg_adapter"], sa)
    assert sorted(p["perm"].tolist()) == p["active_rows"].tolist()
    for s in range(len(sa)):
        assert (ids[p["perm"][so[s]:so[s + 1]]] == sa[s]).all()


def test_plan_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.plan(np.array([0, 5], np.int32), 3)
    with pytest.raises(ValueError):
        oracle.plan(np.array([-2], np.int32), 3)


# ---------------------------------------------------------------- base projection + delta

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_base_fused_is_nearest_bf16_of_float64_brute_force(seed):
    """x W + s (x A) B per row by numpy float64 matmuls on gathered matrices (x W alone
    for released rows): the oracle's output is the nearest bf16 of it."""
    c = workloads.small(seed=90 + seed, n=11, d_in=48, d_out=40, n_adapters=3,
                        ranks=[8, 16, 24], paged=bool(seed % 2), release_frac=0.25)
    W = workloads.make_W(48, 40, seed=seed)
    y = oracle.base_fused(oracle.Table.from_case(c), c["ids"], c["x"], W)
    exact = f64(c["x"]) @ f64(W) + exact_delta(c)
    assert_nearest_bf16(y, exact, slack=1e-6)


def test_base_fused_closed_form_one_hot_adapter():
    """x = [1, 2]; W = [[0.5, 1], [1, -1]] so x W = [2.5, -1]; a rank-8 adapter whose
    A column 0 is e_1 (v_0 = x_1 = 2) and B row 0 is [1, 0.25], all else zero, s = 2:
    the adapter term is 2 * 2 * [1, 0.25] = [4, 1], so y = [6.5, 0] exactly; a released
    row gets x W alone."""
    bf = lambda a: to_bf16_bits(np.asarray(a, np.float32))
    a_pool = np.zeros((8, 2), np.uint16)
    a_pool[0] = bf([0.0, 1.0])
    b_pool = np.zeros((8, 2), np.uint16)
    b_pool[0] = bf([1.0, 0.25])
    pages = np.arange(8, dtype=np.int32).reshape(1, 8)
    t = oracle.Table(a_pool, b_pool, np.array([8], np.int32), np.array([2.0], np.float32),
                     pages, pages)
    x = bf([[1.0, 2.0], [1.0, 2.0]])
    W = bf([[0.5, 1.0], [1.0, -1.0]])
    y = oracle.base_fused(t, np.array([0, -1], np.int32), x, W)
    np.testing.assert_array_equal(f64(y), [[6.5, 0.0], [2.5, -1.0]])


def test_base_fused_with_zero_base_is_the_delta_alone():
    """W = 0: the base projection vanishes and the result is bit for bit the fused
    delta on y_in = 0 (both round s (x A) B once)."""
    c = workloads.small(seed=95, n=13, d_in=64, d_out=48, n_adapters=4, ranks=[8, 16, 32, 8],
                        paged=True, release_frac=0.2, y_mode="zero")
    t = oracle.Table.from_case(c)
    y = oracle.base_fused(t, c["ids"], c["x"], np.zeros((64, 48), np.uint16))
    np.testing.assert_array_equal(y, oracle.fused(t, c["ids"], c["x"], c["y"]))


def test_base_fused_with_every_row_released_is_the_dense_product():
    c = workloads.small(seed=96, n=9, d_in=56, d_out=32, n_adapters=2, ranks=[8, 8])
    W = workloads.make_W(56, 32, seed=3)
    y = oracle.base_fused(oracle.Table.from_case(c), np.full(9, -1, np.int32), c["x"], W)
    assert_nearest_bf16(y, f64(c["x"]) @ f64(W), slack=1e-6)


def test_base_fused_equals_merged_inference():
    """Unmerged x W + s (x A) B against merged x (W + s A B) (VaLoRA blog, section 4.4:
    the two modes compute the same layer)."""
    c = workloads.small(seed=97, n=24, d_in=96, d_out=80, n_adapters=2, ranks=[16, 8],
                        ids=np.ones(24, np.int32))
    W = workloads.make_W(96, 80, seed=4)
    t = oracle.Table.from_case(c)
    y = oracle.base_fused(t, c["ids"], c["x"], W)
    merged = f64(c["x"]) @ f64(oracle.merge(t, 1, W, +1))
    assert_parity(y, to_bf16_bits(merged.astype(np.float32)), 5e-3, 2e-2, "merged vs unmerged")

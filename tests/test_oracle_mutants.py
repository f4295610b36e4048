"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that the
pins catch each one: a pin that cannot fail pins nothing."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads
from tests._helpers import adapter_mats, exact_delta, f64, parity_values

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "fused_sign": ("bf16_to_double(*yo) + s_fused * term[o]", "bf16_to_double(*yo) - s_fused * term[o]"),
    "dropped_last_input_term": ("for (int64_t col = 0; col < d_in; ++col)",
                                "for (int64_t col = 0; col < d_in - 1; ++col)"),
    "dropped_last_rank_term": ("acc += v[j] * B_at(t, k, j, o);",
                               "if (j < r - 1) acc += v[j] * B_at(t, k, j, o);"),
    "transposed_B_index": ("acc += v[j] * B_at(t, k, j, o);",
                           "acc += v[j] * B_at(t, k, (int)(o % r), (int64_t)j);"),
    "truncating_round": ("double units = rint(ldexp(a, -q));",
                         "double units = floor(ldexp(a, -q));"),
    "merge_ignores_sign": ("(sign < 0 ? -1.0 : 1.0)", "(sign < 0 ? 1.0 : 1.0)"),
    "unstable_grouping": ("int32_t row = active_rows[q];\n        perm",
                          "int32_t row = active_rows[na - 1 - q];\n        perm"),
    "scale_dropped": ("const double s_fused = (double)c->t.scale[k];",
                      "const double s_fused = 1.0;"),
    "base_delta_scale_dropped": ("dst[o] *= s_delta;", "dst[o] *= 1.0;"),
    "base_delta_on_released_rows": ("            dst[o] = 0.0;\n        return;",
                                    "            dst[o] = 1.0;\n        return;"),
}


def _pins_hold() -> bool:
    """A compact subset of the pins in test_oracle.py; True when all hold."""
    try:
        c = workloads.small(seed=21, n=10, d_in=40, d_out=32, n_adapters=3,
                            ranks=[8, 16, 8], release_frac=0.2)
        t = oracle.Table.from_case(c)
        y = oracle.fused(t, c["ids"], c["x"], c["y"])
        rel, _ = parity_values(f64(y), f64(c["y"]) + exact_delta(c))
        if rel > 5e-3:
            return False
        v = oracle.shrink(t, c["ids"], c["x"])
        k0 = int(c["ids"][c["ids"] >= 0][0])
        i0 = int(np.flatnonzero(c["ids"] == k0)[0])
        A, B = adapter_mats(c, k0)
        if not np.allclose(v[i0, :A.shape[1]], f64(c["x"][i0]) @ A, rtol=1e-5, atol=1e-5):
            return False
        W = workloads.make_W(40, 32, seed=5)
        for sign in (+1, -1):
            Wm = oracle.merge(t, 0, W, sign)
            A0, B0 = adapter_mats(c, 0)
            r2, _ = parity_values(f64(Wm), f64(W) + sign * float(c["scale"][0]) * (A0 @ B0))
            if r2 > 5e-3:
                return False
        if oracle.bf16_round(1 + 3 * 2 ** -8) != 0x3F82 or oracle.bf16_round(1.9999) != 0x4000:
            return False
        yb = oracle.base_fused(t, c["ids"], c["x"], W[:40, :32])
        rb, _ = parity_values(f64(yb), f64(c["x"]) @ f64(W[:40, :32]) + exact_delta(c))
        if rb > 5e-3:
            return False
        ids = np.array([2, 0, 2, -1, 0, 1, 2], np.int32)
        if oracle.plan(ids, 3)["perm"].tolist() != [1, 4, 5, 0, 2, 6]:
            return False
        return True
    except Exception:
        return False


def test_pins_hold_on_the_real_oracle():
    assert _pins_hold()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so),
                           str(path), "-lm", "-lpthread"])
    monkeypatch.setattr(oracle, "_lib", oracle.bind(str(so)))
    assert not _pins_hold(), f"planted mistake '{name}' went unnoticed"

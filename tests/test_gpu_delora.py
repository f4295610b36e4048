"""Mixture inference (VaLoRA blog, section 4.4.2, deLoRA): with adapter 1 merged into
W, a request for adapter x is served as x.(W_merge - W_deLoRA1 + W_LoRAx), i.e. the
merged adapter is taken out again by a delta with the opposite scale and the target
adapter's delta is added -- here two lora_fused calls on the merged base output, the
first through a table entry that shares adapter 1's pages with scale -s_1."""
import numpy as np
import pytest

import oracle
import workloads
from tests._helpers import bf16_ulp, f64, parity_values, to_bf16_bits
from tests.conftest import MAX_ABS_RMS, REL_FROB

pytestmark = pytest.mark.gpu

L = pytest.importorskip("adapter_sgmv_bgmv_gb300")
from tests.gpu_util import from_dev, to_dev, upload_table  # noqa: E402


def test_delora_mixture_equals_target_adapter_alone():
    ctx = L.Context(0, max_rows=4096, max_rank=64)
    c = workloads.small(seed=81, n=96, d_in=256, d_out=192, n_adapters=2, ranks=[16, 32],
                        y_mode="zero", ids=np.ones(96, np.int32))
    # entry 2 = adapter 0's pages with the opposite scale (the "deLoRA" of adapter 0)
    mix = dict(c, rank=np.append(c["rank"], c["rank"][0]).astype(np.int32),
               scale=np.append(c["scale"], -c["scale"][0]).astype(np.float32),
               a_pages=np.vstack([c["a_pages"], c["a_pages"][:1]]),
               b_pages=np.vstack([c["b_pages"], c["b_pages"][:1]]))
    table = upload_table(ctx, mix)
    W = workloads.make_W(256, 192, seed=9)
    Wd = to_dev(W)
    L.lora_merge(ctx, table, 0, Wd)                      # W_merge = W + s_0 A_0 B_0
    X = f64(c["x"])
    base_merged = to_bf16_bits((X @ f64(from_dev(Wd))).astype(np.float32))
    y = to_dev(base_merged)
    x = to_dev(c["x"])
    L.lora_fused(ctx, table, np.full(96, 2, np.int32), x, y)   # - s_0 (x A_0) B_0
    L.lora_fused(ctx, table, np.full(96, 1, np.int32), x, y)   # + s_1 (x A_1) B_1
    ctx.sync_status()
    # reference: the target adapter alone on the unmerged base
    base = to_bf16_bits((X @ f64(W)).astype(np.float32))
    ref = f64(oracle.fused(oracle.Table.from_case(c), np.ones(96, np.int32), c["x"], base))
    got = f64(from_dev(y))
    rel, _ = parity_values(got, ref)
    assert rel <= REL_FROB, rel
    # the two paths differ by up to four bf16 roundings (merged W, merged base output,
    # and one more output rounding per call) on top of the kernels' own error
    rms = np.sqrt(np.mean(ref * ref))
    assert (np.abs(got - ref) <= MAX_ABS_RMS * rms + 4 * bf16_ulp(ref)).all()
    ctx.close()

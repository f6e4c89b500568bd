"""The benchmark's bookkeeping without a GPU: the FLOP count of a block against the per-block
figures of the workload table (GEMM + attention GFLOP), the algorithmic work of the labelled
library steps, and the committed-traffic lookup's source check."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from diffusion_transformer_flux_gb300 import synth  # noqa: E402


@pytest.mark.parametrize("B,S,gflop", [(1, 4608, 1304.6), (4, 1536, 1507.5), (2, 4608, 2609.2), (1, 16896, 7334.7)])
def test_block_flops_match_the_workload_table(B, S, gflop):
    # per-block totals of the 535M-shaped, 12B @512 px, 12B @1024 px and 12B @2048 px workloads
    assert bench.block_flops(B, S, 3072, 12288, 24) / 1e9 == pytest.approx(gflop, abs=0.05)


def test_kernel_work_of_labelled_steps():
    wl = synth.WORKLOADS["flux535m_bf16"]
    bound, amount, unit = bench.kernel_work("double.fc1", wl)
    assert (bound, unit) == ("tensor", "FLOP") and amount / 1e9 == pytest.approx(347.9, abs=0.05)
    # the image stream's QKV alone: 4096 rows
    assert bench.kernel_work("double.qkv.img", wl)[1] == 2.0 * 4096 * 3072 * 9216
    assert bench.kernel_work("single.attention", wl)[1] == 4.0 * 4608 * 4608 * 128 * 24
    model = synth.WORKLOADS["flux12b_512px_model"]
    bound, amount, unit = bench.kernel_work("modulation.batched", model)
    assert (bound, unit) == ("hbm", "B")
    assert amount / 1e9 == pytest.approx(8.61, abs=0.01)  # 76 streams x 6D x D bf16 weights
    assert bench.kernel_work("no.such.step", wl)[0] == "unknown"
    # the FP8 casts: bf16 in and E4M3 out (3 B per element), or under MXFP8 the represented values
    # out in bf16 (4 B)
    f8 = synth.WORKLOADS["flux12b_2048px_fp8"]
    rows = f8.batch * (f8.seq_img + f8.seq_txt)
    assert bench.kernel_work("single.fp8_cast_u", f8) == ("hbm", 3.0 * rows * f8.mlp_hidden, "B")
    assert bench.kernel_work("double.fp8_cast_h1", f8, "mxfp8")[1] == 4.0 * rows * f8.hidden
    assert bench.kernel_work("double.fp8_cast_w", f8, "mxfp8")[1] == 2 * 4.0 * (4 * 3072 ** 2 + 2 * 12288 * 3072)


def test_committed_traffic_is_used_only_on_the_sources_it_was_taken_on(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    label, value = next(iter(t["workloads"]["flux535m_bf16"].items()))
    monkeypatch.setattr(bench, "source_digest", lambda: t["source_digest"])
    assert bench.committed_traffic(label, "flux535m_bf16") == float(value)
    assert bench.committed_traffic(label, "no_such_workload") is None
    monkeypatch.setattr(bench, "source_digest", lambda: "0" * 16)
    assert bench.committed_traffic(label, "flux535m_bf16") is None

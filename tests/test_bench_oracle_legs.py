"""The bench's oracle legs on the CPU: the parity task and its summary (fed the
oracle's own output, which must pass with no flips, and a corrupted output, which
must fail), and the reference arm's JSON line with a measured step time."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_parity_task_passes_the_oracle_and_fails_a_corruption():
    import synth
    from oracle import moe
    lay, _ = bench._oracle_layer(0, 0, 1792, 0.0)
    x = synth.tokens_bf16(5, 2, 2560)
    out = moe.layer_forward(lay, x, want=("idx",))
    y = moe.f64_to_bf16(out["y"])
    good = bench.oracle_task(("layer", 0, 0, 1792, 0.0, x, y, out["idx"]))
    assert good["flips"] == 0 and good["bad"] == 0 and good["rel_l2"] < 5e-3
    bad_y = y.copy()
    bad_y[1, :100] = moe.f64_to_bf16(-moe.bf16_to_f64(y[1, :100]))
    bad = bench.oracle_task(("layer", 0, 0, 1792, 0.0, x, bad_y, out["idx"]))
    s_good, s_bad = bench.parity_summary([good]), bench.parity_summary([bad])
    assert s_good["pass"] and not s_bad["pass"]
    # another expert list beyond a near-tie counts as a routing failure
    other = out["idx"].copy()
    other[0, 0] = [e for e in range(512) if e not in other[0]][0]
    wrong = bench.oracle_task(("layer", 0, 0, 1792, 0.0, x, y, other))
    assert wrong["bad"] == 1 and not bench.parity_summary([wrong])["pass"]


def test_reference_arm_times_its_steps():
    import argparse
    args = argparse.Namespace(steps=2, warmup=3)
    wl = dict(bench.WORKLOADS["layer145b_t1"], name="layer145b_t1")
    line = bench.reference_arm(args, wl, bench.config_of("layer145b_t1", wl, 1))
    assert line["impl"] == "reference" and line["e2e"]["h2d_bytes_per_step"] == 0
    # value is the sample's tokens over the measured step time
    assert np.isclose(line["value"], 1e3 * wl["T"] / line["ms_per_step"], rtol=2e-3)
    assert line["config"]["sample_tokens_per_step"] == 1

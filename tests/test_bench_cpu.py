"""The bench's roofline arithmetic on the CPU: algorithmic bytes and FLOPs
of each workload, checked against sizes counted independently here, tensor
by tensor (x, offsets, mask, weight, bias and out moved once; the
contraction's 2 * P * O * K FLOPs)."""

import bench
from deformable_convolution_vision_gb300.inputs import (ATTN_WORKLOADS, MSDA_WORKLOADS,
                                                        WORKLOADS)


def _conv_bytes(B, C, H, W, O, k, pad, mask=True, bias=True, es=2):
    Ho, Wo = H + 2 * pad - k + 1, W + 2 * pad - k + 1
    return (B * H * W * C * es                      # x
            + B * 2 * k * k * Ho * Wo * 4             # offsets, fp32
            + (B * k * k * Ho * Wo * 4 if mask else 0)
            + O * C * k * k * es                      # weight
            + (O * 4 if bias else 0)
            + B * Ho * Wo * O * es)                   # out


def test_convolution_bytes_and_flops():
    cases = {
        "decoder3x3": (1, 64, 128, 128, 64, 3, 1),
        "aspp7x7": (1, 64, 256, 256, 64, 7, 3),
        "backbone3x3": (8, 256, 64, 64, 256, 3, 1),
        "boundary5x5": (2, 128, 160, 224, 128, 5, 2),
    }
    for name, (B, C, H, W, O, k, pad) in cases.items():
        wl = WORKLOADS[name]
        assert bench.algorithmic_bytes(wl) == _conv_bytes(B, C, H, W, O, k, pad), name
        Ho, Wo = H + 2 * pad - k + 1, W + 2 * pad - k + 1
        assert wl.flops == 2 * B * Ho * Wo * O * k * k * C, name
    # the headline workload: 55.7 MB and 26.3 GFLOP per step
    wl = WORKLOADS["aspp7x7"]
    assert bench.algorithmic_bytes(wl) == 55_714_048
    assert wl.flops == 26_306_674_688


def test_msda_bytes():
    for m in MSDA_WORKLOADS.values():
        S = sum(h * w for h, w in m.shapes)
        pts = m.B * m.Q * m.G * len(m.shapes) * m.K
        value = m.B * S * m.G * m.D * 2
        out = m.B * m.Q * m.G * m.D * 2
        assert bench.msda_bytes(m, 2) == value + pts * 2 * 4 + pts * 4 + out, m.name
        # backward: value and grad_out read, the fp32 value gradient zeroed and
        # written, locations and weights read, their gradients written
        assert bench.msda_backward_bytes(m, 2) == (value + 2 * m.B * S * m.G * m.D * 4 + out
                                                   + 2 * (pts * 2 * 4 + pts * 4)), m.name


def test_single_scale_bytes():
    for a in ATTN_WORKLOADS.values():
        Ho, Wo = a.out_size()
        K = a.kernel[0] * a.kernel[1]
        rows = a.B * Ho * Wo * a.G
        value = a.B * a.H * a.W * a.G * a.D * 2
        out = rows * a.D * 2
        assert bench.attn_bytes(a, 2) == value + rows * K * 8 + rows * K * 4 + out, a.name
        assert bench.attn_backward_bytes(a, 2) == (value + 2 * a.B * a.H * a.W * a.G * a.D * 4
                                                   + out + 2 * (rows * K * 8 + rows * K * 4)), a.name


def test_reference_arm_stays_within_its_budget():
    """The reference arm (the oracle on the host cores) sizes its per-step
    sample so that any --steps/--warmup finishes within the budget."""
    import argparse
    for steps, warmup in [(20, 3), (2000, 10), (1, 0), (100000, 100)]:
        a = argparse.Namespace(steps=steps, warmup=warmup, reference_step_seconds=2.0,
                               reference_budget_seconds=120.0)
        per = bench.reference_step_seconds(a)
        assert 0.0 < per <= 2.0
        assert per * (steps + 0.25 * warmup) <= 120.0 + 1e-9
    # few steps keep the full per-step sample
    a = argparse.Namespace(steps=20, warmup=3, reference_step_seconds=2.0, reference_budget_seconds=120.0)
    assert bench.reference_step_seconds(a) == 2.0


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line in the bench contract's form, on the same workload
    description and metric as the GPU arm."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "decoder3x3",
                        "--steps", "2", "--warmup", "3", "--reference-budget-seconds", "1"],
                       cwd=root, capture_output=True, text=True, timeout=300,
                       env={k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE")})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    wl = WORKLOADS["decoder3x3"]
    assert d["config"] == bench.config_dict(wl, bench.L2_NOTE)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}

"""bench.py's oracle arm (--impl reference) on CPU: each workload family
prints one JSON line with the contract's keys, its own metric and unit, and
a positive value.  The default workload's arm needs the full 2M-token prompt
and is left to the benchmark itself."""
import json
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.mark.parametrize("workload,unit", [("gdn_f32_h32_r4096_g8", "tokens/s"),
                                           ("prefill_bf16_p32k", "TFLOP/s")])
def test_reference_arm_prints_one_contract_line(workload, unit):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                          "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == unit and line["value"] > 0
    assert line["config"]["workload"] == workload
    # the same config object the GPU arm prints for this workload and rank count
    sys.path.insert(0, str(ROOT))
    import bench

    cfg = bench.gdn_config(workload, 1) if workload in bench.GDN_WORKLOADS else \
        bench.prefill_config(workload, 1)
    assert line["config"] == cfg
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0

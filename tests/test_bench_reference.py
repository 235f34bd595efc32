"""bench.py's reference arm on the block-sparse and FP8 lines: the oracle (the
block-mask oracle, and the float64 model of the FP8 forward) timed on the
host cores, one JSON line each (no GPU needed)."""
import json

import pytest


@pytest.mark.parametrize("workload", ["sparse8k", "fp8_8k"])
def test_reference_arm_line(workload, capsys):
    import bench
    rc = bench.main(["--impl", "reference", "--workload", workload, "--steps", "1",
                     "--warmup", "0"])
    assert rc == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOPS" and line["value"] > 0
    assert line["dtype"] == "f64" and line["config"]["workload"] == workload
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0

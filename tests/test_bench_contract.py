"""The benchmark's JSON line, on the CPU: the reference arm (the fp64 oracle on the
host cores) prints the contract's keys with values of the right kind, and the
GPU arm refuses to run without a CUDA device instead of falling back to the CPU."""

import json

import pytest
import torch


def _line(capsys, argv):
    import bench

    bench.main(argv)
    out = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(out) == 1, out
    return json.loads(out[0])


@pytest.mark.timeout(300)
@pytest.mark.parametrize("workload", ["tiny_fp32", "ec_e16"])
def test_reference_arm_line(capsys, workload):
    d = _line(capsys, ["--impl", "reference", "--steps", "1", "--warmup", "0",
                       "--workload", workload])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["unit"] == "tokens/s" and d["dtype"] == "f64"
    assert d["config"]["workload"].startswith(workload)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == d["unit"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device behaviour")
def test_gpu_arm_refuses_without_a_device():
    import bench

    with pytest.raises(Exception):
        bench.main(["--steps", "1", "--warmup", "3", "--no-cpu-baseline", "--workload", "tiny_fp32"])

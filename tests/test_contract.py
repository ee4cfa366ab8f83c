"""Host-side contract checks: the reference arm's JSON line (run here on the CPU, a bounded oracle sample) and
the binding's refusal to run anything when the CUDA library is missing (there is no fallback)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_complete_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config",
                          "tiny_decode", "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "tiny_decode"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_binding_refuses_without_the_library(monkeypatch):
    from continuous_batching_paged_ragged_gb300 import pkv
    missing = os.path.join(ROOT, "continuous_batching_paged_ragged_gb300", "no-such-dir", "libpkv.so")
    assert not os.path.exists(missing)
    monkeypatch.setattr(pkv, "LIB_PATH", missing)
    monkeypatch.setattr(pkv, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        pkv.load()
    with pytest.raises(RuntimeError):
        pkv.pkv_pool_bytes(pkv.pkv_config(1, 4, 2, 64, 16, 64, 0))

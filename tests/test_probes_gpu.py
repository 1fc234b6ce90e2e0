"""The GB300 probe program (tiled_attention_flashattention_gb300/probes) builds,
runs with every wait inside its bound, and reports the figures the kernels'
design rests on within broad bands: 32-wide-per-cycle ex2, 64-cycle
M128 N128 K16 tensor-core MMAs, and mbarrier waits of well under a microsecond."""
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu


def test_probes_run_and_report_plausible_rates():
    r = subprocess.run([sys.executable, "-m", "tiled_attention_flashattention_gb300.probes"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    out = r.stdout
    ex2 = float(re.search(r"ex2\.approx\.ftz\.f32\s+([\d.]+) per cycle", out).group(1))
    assert 8 <= ex2 <= 128
    ss = float(re.search(r"SS M128 N128 K16\s+([\d.]+) cycles per MMA issued", out).group(1))
    assert 32 <= ss <= 160
    wait = int(re.search(r"bounded wait on a completed mbarrier phase\s+(\d+)", out).group(1))
    assert 0 < wait < 2000
    assert "status 0" in out

"""The phase-traced build (libverify_trace.so) records a sane timeline: run the trace tool on a small
pass in a child process (the traced library replaces libverify.so there) and check that every phase
kind appears with non-negative, ordered times."""
import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_phase_trace_tool_reports_every_phase_kind():
    out = subprocess.run([sys.executable, "-m", "weight_streaming_gb300.phase_trace", "--layers", "4", "--passes", "2"],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    rows = {}
    for line in out.stdout.splitlines():
        m = re.match(r"^(mixer in|mixer out|gate\+up|down|head)\s+(\d+)\s+(.*)$", line)
        if m:
            rows[m.group(1)] = (int(m.group(2)), m.group(3).split())
    assert set(rows) == {"mixer in", "mixer out", "gate+up", "down", "head"}, out.stdout
    for kind, (n, vals) in rows.items():
        assert n == (1 if kind == "head" else 4)
        nums = [float(v) for v in vals if v != "-"]
        assert all(0.0 <= v < 5e4 for v in nums), (kind, vals)
        # columns: stage-ld, staging, stream med, stream max, fixup tail, x-slice, release, phase
        stage_ld, staging, med, mx = (float(v) for v in vals[:4])
        assert stage_ld <= staging and med <= mx
    total = float(re.search(r"last phase done: ([\d.]+) us", out.stdout).group(1))
    assert total > 0.0

"""A bounded device wait runs out, and the library reports it instead of hanging.

The wait-test build of the library (libverify_waittest.so: every bounded wait gives up after
milliseconds, and a workspace hook word can make one CTA leave its first grid-barrier arrival out)
runs a small verify pass in a child process three times: normally, with CTA 0's arrival left out
(every other CTA's barrier wait runs out: the call returns and the workspace's status word reads
VP_ERR_TIMEOUT), and again after vp_workspace_init (the results equal the first run's bit for bit).

Source: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "The megakernel is per
layer, not per step" (a bounded spin on the grid barrier that writes an error code, which the host
raises)."""
import importlib
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_barrier_wait_runs_out_and_reports_timeout():
    build = importlib.import_module("weight_streaming_gb300.build")
    lib = build.build(variant="waittest")
    env = dict(os.environ, VP_LIBVERIFY=lib)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "wait_child.py")], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-3000:]
    got = dict(line.rsplit(" ", 1) for line in out.stdout.strip().splitlines())
    from weight_streaming_gb300 import _lib as V
    assert int(got["normal status"]) == V.VP_OK
    assert int(got["skipped-arrival status"]) == V.VP_ERR_TIMEOUT
    assert int(got["after-init status"]) == V.VP_OK
    assert got["after-init equal"] == "1"

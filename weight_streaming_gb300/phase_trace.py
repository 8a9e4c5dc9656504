"""Phase timeline of a verify pass: where the time of each phase kind goes.

Builds the phase-traced library (libverify_trace.so: the same kernels with globaltimer stamps at each
phase start, end of staging, end of each warp's units and fixups, and the grid barrier; see
csrc/trace.cuh), runs verify passes of a synthetic model on one GPU and prints, per phase kind, the
mean over the last pass's phases of (us):

  stage-ld       phase start -> the staging's loads and row statistics done (slowest CTA)
  staging        phase start -> activations staged (slowest CTA)
  stream med/max staging done -> a warp's units done (median / slowest warp)
  fixup tail     last warp's units done -> last warp's row blocks finished within its CTA
  x-slice        (K-sliced phases) -> grid barrier and the cross-slice sums done (slowest CTA)
  release        last of those done -> first CTA past the grid barrier
  phase          phase start -> next phase start

  python -m weight_streaming_gb300.phase_trace [--layers 16] [--M 8] [--save timeline.npy]

The stamps cost a few global stores per phase and CTA; the traced pass runs within ~2 % of the
untraced one.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

KINDS = ("mixer in", "mixer out", "gate+up", "down")
COLS = ("stage-ld", "staging", "stream med", "stream max", "fixup tail", "x-slice", "release", "phase")


def phase_stats(T: np.ndarray, last_of_launch: set) -> dict:
    """Per phase kind, the list of per-phase figures (ns) from stamps T[phase][CTA][slot]: slot 0
    phase start, 1 staging done, 2..17 each warp's units done, 18..33 each warp's fixups within the
    CTA done, 34 barrier exit, 35 cross-slice sums done (K-sliced phases; 0 elsewhere).  The last phase of a launch has no barrier after it (no release / phase figure)."""
    n_ph = T.shape[0]
    stats = {}
    for gp in range(n_ph):
        kind = "head" if gp == n_ph - 1 else KINDS[gp % 4]
        S = T[gp]
        t0, t1, t2, t3, t4, t5 = S[:, 0], S[:, 1], S[:, 2:18], S[:, 18:34], S[:, 34], S[:, 35]
        d = {"stage-ld": (S[:, 36] - t0).max(), "staging": (t1 - t0).max(), "stream med": np.median(t2 - t1[:, None]),
             "stream max": (t2 - t1[:, None]).max(), "fixup tail": t3.max() - t2.max()}
        done = t3.max()
        if (t5 > 0).all():  # a K-sliced phase: grid barrier, then the cross-slice sums
            d["x-slice"] = t5.max() - t3.max()
            done = t5.max()
        if gp not in last_of_launch:
            d["release"] = t4.min() - done
            d["phase"] = T[gp + 1][:, 0].min() - t0.min()
        stats.setdefault(kind, []).append(d)
    return stats


def report(T: np.ndarray, last_of_launch: set, layers: int, M: int) -> list:
    """The printed table: the mean of each figure per phase kind, in us."""
    stats = phase_stats(T, last_of_launch)
    lines = [f"verify pass, {layers} layers, M = {M}: mean per phase kind (us)",
             f"{'phase kind':12s} {'n':>4s} " + " ".join(f"{c:>11s}" for c in COLS)]
    for kind in KINDS + ("head",):
        lst = stats.get(kind, [])
        if not lst:
            continue
        vals = []
        for c in COLS:
            v = [x[c] for x in lst if c in x]
            vals.append(f"{np.mean(v) / 1e3:11.2f}" if v else f"{'-':>11s}")
        lines.append(f"{kind:12s} {len(lst):4d} " + " ".join(vals))
    total = (T[-1][:, 18:34].max() - T[0][:, 0].min()) / 1e3
    lines.append(f"first phase start -> last phase done: {total:.1f} us")
    return lines


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=16)
    ap.add_argument("--M", type=int, default=8)
    ap.add_argument("--passes", type=int, default=5)
    ap.add_argument("--save", default=None, help="write the last pass's stamps [phase][CTA][slot] (.npy)")
    args = ap.parse_args(argv)

    from .build import build
    os.environ["VP_LIBVERIFY"] = build(trace=True)
    import torch

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import synth
    from . import _lib as V
    from .model import Geometry, SyntheticModel

    M = args.M
    geom = Geometry(n_layers=args.layers)
    sm = SyntheticModel(geom, seed=0)
    H = geom.hidden
    x0 = torch.from_numpy(synth.normal_bf16(0, synth.stream_id(0, synth.T_X0), (M, H)).view(np.int16))
    x0 = x0.cuda().view(torch.bfloat16)
    t = synth.uniform_ints(0, synth.stream_id(0, synth.T_PENDING) + 7, 0, M, geom.vocab)
    pending, _ = synth.planted_pending(0, t, geom.vocab)
    pend = torch.from_numpy(pending).cuda()
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    ws = sm.workspace(M)
    for _ in range(args.passes):
        sm.run(x0, pend, am, nc, cm, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK

    n_ph = 4 * args.layers + 1
    per_launch = 160
    launches = (n_ph + per_launch - 1) // per_launch
    buf = np.zeros((2, per_launch, 256, 37), np.uint64)  # kTraceSlots stamps per phase and CTA
    done = V.vp_trace_read(M, buf)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    rows = []  # the last pass: launch l holds phases [l * n / launches, (l + 1) * n / launches)
    last_of_launch = set()
    for l in range(launches):
        p0, p1 = l * n_ph // launches, (l + 1) * n_ph // launches
        par = (done - launches + l) & 1
        for p in range(p1 - p0):
            rows.append(buf[par, p, :G, :].astype(np.int64))
        last_of_launch.add(p1 - 1)
    T = np.stack(rows)
    if args.save:
        np.save(args.save, T)

    print("\n".join(report(T, last_of_launch, args.layers, M)))

if __name__ == "__main__":
    main()

"""The phase timeline's arithmetic on hand-made stamps (no GPU): staging is the slowest CTA's
staging, the stream figures are per warp from its CTA's staging end, the fixup tail runs from the
last warp's units to the last warp's fixups, release from there to the first CTA past the barrier,
and the last phase of a launch has no release or phase figure."""
import numpy as np

from weight_streaming_gb300.phase_trace import phase_stats, report


def stamps(n_ph=5, G=3):
    T = np.zeros((n_ph, G, 37), np.int64)
    for p in range(n_ph):
        base = 100_000 * p
        for c in range(G):
            T[p, c, 0] = base + 10 * c                      # phase start
            T[p, c, 36] = base + 400 + 100 * c              # loads and statistics done
            T[p, c, 1] = base + 1_000 + 100 * c             # staged: CTA 2 slowest (1,200 after its start 20)
            T[p, c, 2:18] = T[p, c, 1] + 5_000 + np.arange(16) * 10 + 1_000 * (c == 1) * (np.arange(16) == 3)
            T[p, c, 18:34] = T[p, c, 2:18] + 2_000
            T[p, c, 34] = base + 60_000 + c
    return T


def test_phase_stats_figures():
    T = stamps()
    st = phase_stats(T, last_of_launch={4})
    assert set(st) == {"mixer in", "mixer out", "gate+up", "down", "head"}
    d = st["mixer in"][0]
    assert d["staging"] == 1_180  # CTA 2: 1,200 - 20
    assert d["stage-ld"] == 580
    assert d["stream max"] == 6_030  # CTA 1, warp 3: 5,000 + 30 + 1,000 after its own staging end
    assert d["stream med"] == np.median(T[0, :, 2:18] - T[0, :, 1:2])
    assert d["fixup tail"] == T[0, :, 18:34].max() - T[0, :, 2:18].max() == 2_000
    assert d["release"] == T[0, :, 34].min() - T[0, :, 18:34].max()
    assert d["phase"] == 100_000
    assert "release" not in st["head"][0] and "phase" not in st["head"][0]


def test_report_lists_every_kind_once():
    lines = report(stamps(), {4}, layers=1, M=8)
    assert lines[0].startswith("verify pass, 1 layers, M = 8")
    kinds = [ln.split()[0] for ln in lines[2:-1]]
    assert kinds == ["mixer", "mixer", "gate+up", "down", "head"]
    assert lines[-1].startswith("first phase start -> last phase done:")
    head = lines[-2].split()
    assert head[-3:] == ["-", "-", "-"]


def test_k_sliced_phase_reports_its_cross_slice_step():
    """A phase with cross-slice sums (slot 35 stamped in every CTA) reports them from the last
    in-CTA fixup to the slowest CTA's sums, and its release from there."""
    T = stamps()
    T[1, :, 35] = T[1, :, 18:34].max() + 3_000 + np.arange(T.shape[1]) * 100
    st = phase_stats(T, last_of_launch={4})
    d = st["mixer out"][0]
    assert d["x-slice"] == 3_000 + 100 * (T.shape[1] - 1)
    assert d["release"] == T[1, :, 34].min() - T[1, :, 35].max()
    assert "x-slice" not in st["mixer in"][0]

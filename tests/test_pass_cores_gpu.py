"""The verify pass with the real mixer cores (vp_verify_pass_cores) through the C ABI, against the
oracle's Gated DeltaNet and attention blocks (oracle/gdn_layer.py, oracle/attn_layer.py), at small
widths and at the pages' own (hidden 5120, 16 q/k and 48 v heads of 128, 24 query and 4 key-value
heads of 256).

A 2-layer model (layer 0 Gated DeltaNet, layer 1 attention) runs the whole pass with its trace on.
Every block is checked against the oracle's block computed from the device's own input to it:
the residual after each mixer block within the block's budget (the cores' output, rounded to bf16
on both sides, may differ by a few ulps of its head's scale, carried through the out-projection), the
MLP blocks as in the surrogate pass; and the state the pass leaves behind: the delta-rule state after
the 8 rows, the convolution history, the keys and values appended to the cache.

Sources: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "The megakernel is
per layer, not per step" (the two layer graphs) and "What one token costs the bus" (the recurrent
state); "Beating Splash on an M5 Max" -- "What actually moved the needle" (parity buffers)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import REL, dev_bf16, dev_i32, host_bf16_bits, workspace
from oracle.attn_layer import attn_block
from oracle.gdn_layer import gdn_block
from passutil import DELTA, DeviceModel, make_head, make_layer, mlp_block_ref, prop_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


SMALL = dict(hidden=256, inter=512, n_qk=2, n_v=4, Hq=4, Hkv=2, vocab=2064)
PAGES = dict(hidden=5120, inter=17408, n_qk=16, n_v=48, Hq=24, Hkv=4, vocab=2064)
D_GDN, D_ATT = 128, 256


def bfr(x):
    return oracle.bf16_round(np.asarray(x, np.float64))


def bfv(bits):
    return oracle.bf16_value(bits)


def build(V, cfg, lanes, cap, seed):
    H, nqk, nv, Hq, Hkv = cfg["hidden"], cfg["n_qk"], cfg["n_v"], cfg["Hq"], cfg["Hkv"]
    G = oracle.geom(n_layers=2, hidden=H, inter=cfg["inter"], vocab=cfg["vocab"], period=2,
                    gdn_in=(2 * nqk + 2 * nv) * D_GDN, gdn_z=nv * D_GDN, attn_q=2 * Hq * D_ATT, attn_kv=2 * Hkv * D_ATT,
                    attn_z=Hq * D_ATT)
    layers = [make_layer(G, seed, 0, (0.75, 1.0, 1.25, 0.625, 1.125, 0.875)),
              make_layer(G, seed, 1, (1.25, 0.5, 0.875, 1.0625, 0.75, 1.375))]
    head = make_head(G, seed, 0.5)
    rng = np.random.default_rng(seed)
    C = (2 * nqk + nv) * D_GDN

    def exact32(x):  # fp32 values that bf16 holds exactly: the same numbers on both sides
        return bfv(bfr(x)).astype(np.float32)

    gd = {"A": bfr(rng.standard_normal((nv, H)) / np.sqrt(H)), "B": bfr(rng.standard_normal((nv, H)) / np.sqrt(H)),
          "taps": bfr(rng.uniform(-0.6, 0.6, (C, 4))), "A_log": exact32(rng.uniform(-2.0, 0.0, nv)),
          "dt_bias": exact32(rng.uniform(-1.0, 1.0, nv)), "w_norm": exact32(rng.uniform(0.5, 1.5, D_GDN)),
          "state": (0.1 * rng.standard_normal((lanes, nv, D_GDN, D_GDN))).astype(np.float32),
          "window": bfr(rng.standard_normal((lanes, 3, C)))}
    at = {"q_norm": exact32(rng.uniform(0.5, 1.5, D_ATT)), "k_norm": exact32(rng.uniform(0.5, 1.5, D_ATT)),
          "k_cache": bfr(rng.standard_normal((lanes, Hkv, cap, D_ATT))),
          "v_cache": bfr(rng.standard_normal((lanes, Hkv, cap, D_ATT)))}
    dm = DeviceModel(V, G, layers, head)
    keep = []

    def dev(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
        if dtype is not None:
            t = t.view(dtype)
        keep.append(t)
        return t

    dg = {"A": dev(gd["A"].view(np.int16)), "B": dev(gd["B"].view(np.int16)), "taps": dev(gd["taps"].view(np.int16)),
          "A_log": dev(gd["A_log"]), "dt_bias": dev(gd["dt_bias"]), "w_norm": dev(gd["w_norm"]),
          "state_a": dev(gd["state"]), "state_b": dev(np.zeros_like(gd["state"])),
          "window": dev(gd["window"].view(np.int16)), "hist": dev(np.zeros((lanes, 11, C), np.int16))}
    da = {"q_norm": dev(at["q_norm"]), "k_norm": dev(at["k_norm"]), "k_cache": dev(at["k_cache"].view(np.int16)),
          "v_cache": dev(at["v_cache"].view(np.int16))}
    c0 = V.vp_core_desc(w_a=dg["A"].data_ptr(), w_b=dg["B"].data_ptr(), conv_taps=dg["taps"].data_ptr(),
                        a_log=dg["A_log"].data_ptr(), dt_bias=dg["dt_bias"].data_ptr(), norm_w=dg["w_norm"].data_ptr(),
                        state_a=dg["state_a"].data_ptr(), state_b=dg["state_b"].data_ptr(),
                        window_a=dg["window"].data_ptr(), conv_hist=dg["hist"].data_ptr())
    c1 = V.vp_core_desc(q_norm=da["q_norm"].data_ptr(), k_norm=da["k_norm"].data_ptr(),
                        k_cache=da["k_cache"].data_ptr(), v_cache=da["v_cache"].data_ptr())
    V.vp_model_set_cores(dm.model, V.vp_core_geom(nqk, nv, D_GDN, Hq, Hkv, D_ATT, cap), [c0, c1])
    torch.cuda.synchronize()
    return G, layers, head, gd, at, dm, dg, da, keep


def core_budget(on_bits, w, s, hidden, h_ref, d, ulps):
    """Budget of a mixer block whose core output (the out-projection's input, bf16) may differ from
    the oracle's by a few ulps of its head's scale: ulps * 2^-8 (|on| + the head's root mean square),
    carried through the out-projection (its sum |x w| over those differences), plus the projection's
    own tolerance and one bf16 ulp of the new residual.  The attention core sees each of its bf16
    inputs once (4 ulps); the delta-rule output of row j carries the one-ulp input differences of rows
    0..j through the state, so the Gated DeltaNet core gets 8."""
    on = bfv(on_bits)
    M, K = on.shape
    rms = np.sqrt((on.reshape(M, K // d, d) ** 2).mean(axis=2))
    dz = ulps * 2.0 ** -8 * (np.abs(on) + np.repeat(rms, d, axis=1))
    _, a_y = oracle.linear(oracle.FP8, on_bits, w, None, s, hidden)
    prop = prop_bound(oracle.FP8, dz, w, None, s, hidden)
    dy = REL * (a_y + prop) + prop
    return dy + DELTA * (np.abs(bfv(h_ref)) + dy)


def within(got_bits, ref_bits, budget, what):
    err = np.abs(bfv(got_bits) - bfv(ref_bits))
    bad = ~(err <= budget)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside budget, max err/budget " \
                          f"{float(np.max(err / budget)):.3g}"


@pytest.mark.parametrize("cfg,lanes,cap,ctx", [(SMALL, 1, 64, [17]), (SMALL, 2, 300, [0, 255]),
                                               (PAGES, 1, 1024, [513]), (PAGES, 4, 2048, [0, 77, 1030, 2040])])
def test_cores_pass_matches_oracle_blocks(V, cfg, lanes, cap, ctx):
    M = 8 * lanes
    G, layers, head, gd, at, dm, dg, da, keep = build(V, cfg, lanes, cap, seed=51 + lanes)
    H, nqk, nv, Hq, Hkv = cfg["hidden"], cfg["n_qk"], cfg["n_v"], cfg["Hq"], cfg["Hkv"]
    x0 = synth.normal_bf16(80 + M, synth.stream_id(0, synth.T_X0), (M, H))
    pending = np.zeros(M, np.int32)
    ctx = np.asarray(ctx, np.int32)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(lanes, dtype=torch.int32, device="cuda")
    cm = torch.empty((lanes, 8), dtype=torch.int32, device="cuda")
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    trace = torch.empty((4, M, H), dtype=torch.bfloat16, device="cuda")
    ws = workspace(V.vp_pass_cores_workspace_bytes(dm.model, M))
    V.vp_verify_pass_cores(dm.model, dev_bf16(x0), M, dev_i32(ctx), 0, dev_i32(pending), am, nc, cm, trace, lg, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    tr = host_bf16_bits(trace)

    # block 0: Gated DeltaNet, lane by lane from x0
    d0 = layers[0]
    g = {"hidden": H, "n_qk": nqk, "n_v": nv, "d": D_GDN}
    wts = {"in": d0["in"], "s_in": d0["s_in"], "out": d0["out"], "s_out": d0["s_out"], "A": gd["A"], "B": gd["B"],
           "taps": bfv(gd["taps"]), "A_log": gd["A_log"].astype(np.float64),
           "dt_bias": gd["dt_bias"].astype(np.float64), "w_norm": gd["w_norm"].astype(np.float64)}
    state_b = dg["state_b"].cpu().numpy()
    hist = dg["hist"].cpu().numpy().view(np.uint16)
    for l in range(lanes):
        rows = slice(8 * l, 8 * l + 8)
        on = []
        h_ref, st, win, _ = gdn_block(x0[rows], g, wts, gd["state"][l].astype(np.float64), bfv(gd["window"][l]),
                                      core_out=on)
        within(tr[0][rows], h_ref, core_budget(on[0], d0["out"], d0["s_out"], H, h_ref, D_GDN, 8), f"GDN block, lane {l}")
        tol = 2.0 ** -6 * np.abs(st).max()
        assert np.abs(state_b[l] - st).max() <= tol, ("state after 8 rows", l, np.abs(state_b[l] - st).max(), tol)
        assert np.array_equal(hist[l, :3], gd["window"][l])  # the window the pass read
        # the window after 8 rows: the in-projection's q, k, v outputs of rows 5..7 (bf16), each within
        # the linear tolerance of the oracle's plus one bf16 ulp
        _, a_u = oracle.linear(oracle.FP8, oracle.rmsnorm(x0[rows][5:8], G.eps), d0["in"], None, d0["s_in"],
                               (2 * nqk + nv) * D_GDN)
        hw = bfv(hist[l, 8:11])
        assert np.all(np.abs(hw - win) <= REL * a_u + 2.0 ** -7 * np.abs(win) + 1e-30), ("window after 8 rows", l)
    # block 1: the MLP of layer 0
    h_ref, budget = mlp_block_ref(G, d0, tr[0])
    within(tr[1], h_ref, budget, "MLP block 1")
    # block 2: attention over the caches as they were before the pass
    d1 = layers[1]
    ga = {"hidden": H, "Hq": Hq, "Hkv": Hkv, "D": D_ATT}
    wa = {"q": d1["in"], "s_q": d1["s_in"], "kv": d1["kv"], "s_kv": d1["s_kv"], "o": d1["out"], "s_o": d1["s_out"],
          "q_norm": at["q_norm"].astype(np.float64), "k_norm": at["k_norm"].astype(np.float64)}
    ob = []
    h_ref, (kb, vb), _ = attn_block(tr[1], ga, wa, at["k_cache"], at["v_cache"], ctx, core_out=ob)
    within(tr[2], h_ref, core_budget(ob[0], d1["out"], d1["s_out"], H, h_ref, D_ATT, 4), "attention block")
    kc = da["k_cache"].cpu().numpy().view(np.uint16)
    vc = da["v_cache"].cpu().numpy().view(np.uint16)
    for l in range(lanes):
        for j in range(8):
            p = ctx[l] + j
            for got, ref in ((kc[l, :, p], kb[8 * l + j]), (vc[l, :, p], vb[8 * l + j])):
                # one bf16 ulp of the row's scale: the keys are normalised and rotated, the values the
                # projection's outputs (both rounded once on each side)
                rv = bfv(ref)
                scale = np.sqrt((rv ** 2).mean(axis=-1, keepdims=True))
                assert np.all(np.abs(bfv(got) - rv) <= 2.0 ** -7 * (np.abs(rv) + scale)), ("appended row", l, j)
        untouched = np.ones(cap, bool)
        untouched[ctx[l]:ctx[l] + 8] = False
        assert np.array_equal(kc[l][:, untouched], at["k_cache"][l][:, untouched])
    # block 3: the MLP of layer 1
    h_ref, budget = mlp_block_ref(G, d1, tr[2])
    within(tr[3], h_ref, budget, "MLP block 3")
    # the head on the device's last residual: its own argmax and acceptance
    am, lg = am.cpu().numpy(), lg.cpu().numpy()
    assert np.array_equal(am, np.argmax(lg, axis=1))
    nc_o, cm_o = oracle.accept(am, pending)
    assert np.array_equal(nc.cpu().numpy(), nc_o) and np.array_equal(cm.cpu().numpy(), cm_o)


def test_cores_pass_is_deterministic(V):
    """Two passes from the same state (state_a, window_a and the cache rows before ctx unchanged)
    give the same bits."""
    lanes, cap = 2, 128
    M = 8 * lanes
    G, layers, head, gd, at, dm, dg, da, keep = build(V, SMALL, lanes, cap, seed=9)
    x0 = dev_bf16(synth.normal_bf16(3, synth.stream_id(0, synth.T_X0), (M, SMALL["hidden"])))
    ctx = dev_i32(np.array([5, 40], np.int32))
    pend = dev_i32(np.zeros(M, np.int32))
    outs = []
    for _ in range(2):
        am = torch.empty(M, dtype=torch.int32, device="cuda")
        nc = torch.empty(lanes, dtype=torch.int32, device="cuda")
        cm = torch.empty((lanes, 8), dtype=torch.int32, device="cuda")
        lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
        ws = workspace(V.vp_pass_cores_workspace_bytes(dm.model, M))
        V.vp_verify_pass_cores(dm.model, x0, M, ctx, 0, pend, am, nc, cm, None, lg, ws)
        torch.cuda.synchronize()
        outs.append((lg.clone(), dg["state_b"].clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("cfg,lanes,cap,ctx,keep", [(SMALL, 2, 64, [5, 40], [3, 8]),
                                                   (PAGES, 4, 1100, [0, 77, 1030, 500], [1, 8, 5, 2])])
def test_cores_commit_then_next_pass(V, cfg, lanes, cap, ctx, keep):
    """A pass of parity 0, the commit of `keep` rows per lane, then a pass of parity 1 at ctx + keep."""
    M = 8 * lanes
    G, layers, head, gd, at, dm, dg, da, _ = build(V, cfg, lanes, cap, seed=71 + lanes)
    H, nqk, nv = cfg["hidden"], cfg["n_qk"], cfg["n_v"]
    g = {"hidden": H, "n_qk": nqk, "n_v": nv, "d": D_GDN}
    d0 = layers[0]
    wts = {"in": d0["in"], "s_in": d0["s_in"], "out": d0["out"], "s_out": d0["s_out"], "A": gd["A"], "B": gd["B"],
           "taps": bfv(gd["taps"]), "A_log": gd["A_log"].astype(np.float64),
           "dt_bias": gd["dt_bias"].astype(np.float64), "w_norm": gd["w_norm"].astype(np.float64)}
    ws = workspace(V.vp_pass_cores_workspace_bytes(dm.model, M))
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(lanes, dtype=torch.int32, device="cuda")
    cm = torch.empty((lanes, 8), dtype=torch.int32, device="cuda")
    pend = dev_i32(np.zeros(M, np.int32))
    x0 = synth.normal_bf16(90 + M, synth.stream_id(0, synth.T_X0), (M, H))
    V.vp_verify_pass_cores(dm.model, dev_bf16(x0), M, dev_i32(np.asarray(ctx, np.int32)), 0, pend, am, nc, cm, None,
                           None, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    state_a0 = dg["state_a"].clone()
    sb_pass = dg["state_b"].cpu().numpy()
    hist = dg["hist"].cpu().numpy().view(np.uint16)
    V.vp_commit_cores(dm.model, M, dev_i32(np.asarray(keep, np.int32)), 0, ws)
    torch.cuda.synchronize()
    assert torch.equal(dg["state_a"], state_a0)  # the intact buffer
    sb = dg["state_b"].cpu().numpy()
    win = dg["window"].cpu().numpy().view(np.uint16)
    for l in range(lanes):
        n = keep[l]
        assert np.array_equal(win[l], hist[l, n:n + 3]), ("window", l)
        if n == 8:
            assert np.array_equal(sb[l], sb_pass[l]), ("a full commit reproduces the pass's state", l)
        _, st, wref, _ = gdn_block(x0[8 * l:8 * l + 8], g, wts, gd["state"][l].astype(np.float64),
                                   bfv(gd["window"][l]), rows=n)
        tol = 2.0 ** -6 * np.abs(st).max()
        assert np.abs(sb[l] - st).max() <= tol, ("state after the committed rows", l, n)
        _, a_u = oracle.linear(oracle.FP8, oracle.rmsnorm(x0[8 * l:8 * l + 8], G.eps), d0["in"], None, d0["s_in"],
                               (2 * nqk + nv) * D_GDN)
        rows_w = [r - 3 for r in range(n, n + 3) if r >= 3]  # window rows that come from the pass's u
        if rows_w:
            ww = bfv(win[l][3 - len(rows_w):])
            wr = wref[3 - len(rows_w):]
            bound = REL * a_u[rows_w] + 2.0 ** -7 * np.abs(wr) + 1e-30
            assert np.all(np.abs(ww - wr) <= bound), ("window against the oracle", l)
    # the next pass, parity 1: reads state_b and the new window, writes state_a
    sb_t = dg["state_b"].clone()
    ctx1 = np.asarray(ctx, np.int32) + np.asarray(keep, np.int32)
    x1 = synth.normal_bf16(95 + M, synth.stream_id(0, synth.T_X0), (M, H))
    trace = torch.empty((4, M, H), dtype=torch.bfloat16, device="cuda")
    V.vp_verify_pass_cores(dm.model, dev_bf16(x1), M, dev_i32(ctx1), 1, pend, am, nc, cm, trace, None, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    assert torch.equal(dg["state_b"], sb_t)  # read only at parity 1
    tr = host_bf16_bits(trace)
    sa = dg["state_a"].cpu().numpy()
    for l in range(lanes):
        rows = slice(8 * l, 8 * l + 8)
        on = []
        h_ref, st, _, _ = gdn_block(x1[rows], g, wts, sb[l].astype(np.float64), bfv(win[l]), core_out=on)
        within(tr[0][rows], h_ref, core_budget(on[0], d0["out"], d0["s_out"], H, h_ref, D_GDN, 8),
               f"GDN block of the parity-1 pass, lane {l}")
        assert np.abs(sa[l] - st).max() <= 2.0 ** -6 * np.abs(st).max(), ("state after the parity-1 pass", l)

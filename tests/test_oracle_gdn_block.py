"""Pins of the Gated DeltaNet mixer-block oracle (oracle/gdn_layer.py) to library routines (torch's
conv1d, normalize, softplus, sigmoid, rms_norm), closed forms and an independent torch composition
of the whole block."""
import numpy as np
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import gdn_layer as gl

G = {"hidden": 256, "n_qk": 2, "n_v": 4, "d": 16}


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_short_conv_matches_torch_conv1d():
    rng = np.random.default_rng(70)
    T, C = 8, 24
    x, win, taps = rng.standard_normal((T, C)), rng.standard_normal((3, C)), rng.standard_normal((C, 4))
    y, e = gl.short_conv_silu(x, win, taps)
    inp = torch.from_numpy(np.concatenate([win, x]).T[None])  # [1][C][3 + T]
    ref = F.silu(F.conv1d(inp, torch.from_numpy(taps)[:, None, :], groups=C))[0].T.numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-14)
    assert np.array_equal(e[-3:], x[-3:])


def test_short_conv_closed_forms_and_window_carry():
    rng = np.random.default_rng(71)
    T, C = 8, 10
    x, win = rng.standard_normal((T, C)), rng.standard_normal((3, C))
    taps = np.zeros((C, 4))
    taps[:, 3] = 1.0  # the current token only
    y, _ = gl.short_conv_silu(x, win, taps)
    np.testing.assert_allclose(y, x / (1 + np.exp(-x)), rtol=1e-15)
    taps = np.zeros((C, 4))
    taps[:, 0] = 1.0  # three tokens back: the window for the first three rows
    y, _ = gl.short_conv_silu(x, win, taps)
    np.testing.assert_allclose(y[:3], win / (1 + np.exp(-win)), rtol=1e-15)
    np.testing.assert_allclose(y[3:], x[:5] / (1 + np.exp(-x[:5])), rtol=1e-15)
    # rows 0..n-1, then n..7 from the carried window, equal the 8 rows at once
    taps = rng.standard_normal((C, 4))
    full, _ = gl.short_conv_silu(x, win, taps)
    for n in range(1, 8):
        a, e = gl.short_conv_silu(x[:n], win, taps)
        b, _ = gl.short_conv_silu(x[n:], e[n:n + 3], taps)
        np.testing.assert_array_equal(np.concatenate([a, b]), full)


def test_l2norm_gates_and_gated_norm_match_torch():
    rng = np.random.default_rng(72)
    x = rng.standard_normal((8, 4 * 16)) * 3
    n = gl.l2norm_heads(x, 16)
    ref = F.normalize(torch.from_numpy(x.reshape(8, 4, 16)), dim=-1, eps=1e-30).numpy().reshape(8, 64)
    np.testing.assert_allclose(n, ref, rtol=1e-6)  # eps 1e-6 inside the root vs none
    np.testing.assert_allclose((n.reshape(8, 4, 16) ** 2).sum(-1), 1.0, rtol=1e-6)
    a, b = rng.standard_normal((8, 4)), rng.standard_normal((8, 4))
    A_log, dt = rng.standard_normal(4), rng.standard_normal(4)
    al, be = gl.gates(a, b, A_log, dt)
    t = torch.from_numpy
    np.testing.assert_allclose(al, torch.exp(-torch.exp(t(A_log)) * F.softplus(t(a + dt))).numpy(), rtol=1e-14)
    np.testing.assert_allclose(be, torch.sigmoid(t(b)).numpy(), rtol=1e-15)
    assert np.all((al > 0) & (al < 1)) and np.all((be > 0) & (be < 1))
    # softplus(0) = ln 2: alpha = 2^(-exp(A_log)); sigmoid(0) = 1/2
    al0, be0 = gl.gates(np.zeros((1, 4)), np.zeros((1, 4)), A_log, np.zeros(4))
    np.testing.assert_allclose(al0[0], 2.0 ** -np.exp(A_log), rtol=1e-14)
    assert np.all(be0 == 0.5)
    o, z, w = rng.standard_normal((8, 4, 16)), rng.standard_normal((8, 4, 16)), rng.standard_normal(16)
    ref = F.rms_norm(t(o), (16,), weight=t(w), eps=1e-6) * F.silu(t(z))
    np.testing.assert_allclose(gl.gated_rmsnorm(o, z, w), ref.numpy(), rtol=1e-13, atol=1e-14)


def block_case(seed=73):
    rng = np.random.default_rng(seed)
    H, nqk, nv, d = G["hidden"], G["n_qk"], G["n_v"], G["d"]
    cin, cc = (2 * nqk + 2 * nv) * d, (2 * nqk + nv) * d
    w = {"in": synth.fp8_matrix(seed, 0, synth.T_IN, cin, H), "s_in": 0.05,
         "out": synth.fp8_matrix(seed, 0, synth.T_OUT, H, nv * d), "s_out": 0.05,
         "A": bf16_bits(rng.standard_normal((nv, H)) * 0.05), "B": bf16_bits(rng.standard_normal((nv, H)) * 0.05),
         "taps": bf16_vals(bf16_bits(rng.standard_normal((cc, 4)) * 0.5)),
         "A_log": rng.uniform(-3, 0, nv), "dt_bias": rng.uniform(-1, 1, nv), "w_norm": rng.uniform(0.5, 1.5, d)}
    h = synth.normal_bf16(seed, synth.stream_id(0, synth.T_X0), (8, H))
    state = rng.standard_normal((nv, d, d)) * 0.1
    window = bf16_vals(bf16_bits(rng.standard_normal((3, cc))))
    return h, w, state, window


def torch_block(h, w, state, window, rows):
    """The same block written independently with torch ops (fp64, bf16 casts at the same points)."""
    H, nqk, nv, d = G["hidden"], G["n_qk"], G["n_v"], G["d"]
    cq, cv = nqk * d, nv * d
    bf = lambda x: x.to(torch.bfloat16).double()  # noqa: E731
    fp8 = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).double()  # noqa: E731
    hv = torch.from_numpy(bf16_vals(h))
    r = bf(hv / torch.sqrt((hv * hv).mean(-1, keepdim=True) + 1e-6))
    u = r @ (fp8(w["in"]) * w["s_in"]).T
    qkv, z = bf(u[:, :2 * cq + cv]), bf(u[:, 2 * cq + cv:])
    a = r @ torch.from_numpy(bf16_vals(w["A"])).T
    b = r @ torch.from_numpy(bf16_vals(w["B"])).T
    e = torch.cat([torch.from_numpy(window), qkv])
    y = F.silu(F.conv1d(e.T[None], torch.from_numpy(w["taps"])[:, None, :], groups=e.shape[1])[0].T)
    def unit(x):  # each head over its L2 norm (eps inside the root)
        x = x.reshape(8, nqk, d)
        return x / torch.sqrt((x ** 2).sum(-1, keepdim=True) + 1e-6)
    q, k = bf(unit(y[:, :cq])), bf(unit(y[:, cq:2 * cq]))
    v = bf(y[:, 2 * cq:].reshape(8, nv, d))
    q, k = q.repeat_interleave(nv // nqk, dim=1), k.repeat_interleave(nv // nqk, dim=1)
    al = torch.exp(-torch.exp(torch.from_numpy(w["A_log"])) * F.softplus(a + torch.from_numpy(w["dt_bias"])))
    be = torch.sigmoid(b)
    S = torch.from_numpy(state.copy())
    outs, S_rows = [], None
    eye = torch.eye(d, dtype=torch.float64)
    for t in range(8):
        S = torch.stack([S[i] @ (al[t, i] * (eye - be[t, i] * torch.outer(k[t, i], k[t, i])))
                         + be[t, i] * torch.outer(v[t, i], k[t, i]) for i in range(nv)])
        outs.append(torch.stack([S[i] @ q[t, i] for i in range(nv)]))
        if t + 1 == rows:
            S_rows = S.clone()
    o = torch.stack(outs)
    on = bf(F.rms_norm(o, (d,), weight=torch.from_numpy(w["w_norm"]), eps=1e-6) * F.silu(z.reshape(8, nv, d)))
    yo = on.reshape(8, cv) @ (fp8(w["out"]) * w["s_out"]).T
    return bf(hv + yo).numpy(), S_rows.numpy(), e[rows:rows + 3].numpy()


def test_block_matches_independent_torch_composition():
    h, w, state, window = block_case()
    for rows in (8, 3, 1):
        h_new, st, win, _ = gl.gdn_block(h, G, w, state, window, rows)
        ref_h, ref_st, ref_win = torch_block(h, w, state, window, rows)
        got = bf16_vals(h_new)
        # a bf16 rounding point may fall either side between two fp64 summation orders: one ulp
        assert np.all(np.abs(got - ref_h) <= np.abs(ref_h) * 2.0 ** -7 + 1e-30), rows
        assert np.mean(got == ref_h) > 0.97, rows
        np.testing.assert_allclose(st, ref_st, rtol=1e-6, atol=1e-9)
        np.testing.assert_array_equal(win, ref_win)


def test_block_window_and_state_after_a_partial_accept():
    """After n committed rows the state equals the verify scan's state after n rows (the re-scan of
    the commit), and with nothing committed the window is unchanged."""
    h, w, state, window = block_case(74)
    _, _, _, (q, k, v, al, be) = gl.gdn_block(h, G, w, state, window, 8)
    for n in range(0, 9):
        _, st, win, _ = gl.gdn_block(h, G, w, state, window, n)
        ref, _ = oracle.gdn_scan(state[None], q, k, v, al, be, np.array([n], np.int32), want_out=False)
        np.testing.assert_array_equal(st, ref[0])
        if n == 0:
            np.testing.assert_array_equal(win, window)

"""The Gated DeltaNet mixer block with its real core, in fp64: TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the bench's CPU-baseline leg may use this module; the
product path never imports it.  It shares nothing with the CUDA library.

Sources (web pages, cited by title and section):
 - "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max", section "The megakernel is
   per layer, not per step" (the block's graph: RMSNorm; the QKV and Z projections in FP8 and the
   A/B projections in BF16; the core -- a short convolution, Q/K normalisation, the gates and the
   delta recurrence against the recurrent state; gated RMSNorm with SiLU of Z; the FP8 output
   projection with the residual), and section "What one token costs the bus" (the A/B
   projections, norms and convolution are small BF16 tensors outside the FP8 / NVFP4 stream).
 - "144 tok/s needs 502 GB/s", section "The engine hard-codes the model" (4-tap convolutions,
   decays and time biases are bf16 / fp32 vectors; the recurrent state is fp32, 48 heads of
   128 x 128 per layer).
 - "Beating Splash on an M5 Max", section "What actually moved the needle" (the recurrent state
   and the convolution window are both double-buffered; a partial accept re-scans the committed
   rows, and the state and window after every possible kept count must match a reference scan).

The pages name the steps; the formulas below are readings (the plainest ones the names support):
 - in-projection rows: q (n_qk heads), k (n_qk heads), v (n_v heads), then z (n_v heads), each
   head d wide; the A and B projections give one value per v head;
 - short convolution: causal and depthwise over q, k and v, 4 taps, tap 3 on the current token and
   taps 0..2 on the three tokens before it (the window carries those across passes), then SiLU;
 - Q/K normalisation: each head of q and k divided by its L2 norm (eps 1e-6 inside the root);
 - gates: beta = sigmoid(b) and alpha = exp(-exp(A_log) * softplus(a + dt_bias)) per v head
   (A_log is the layer's decay, dt_bias its time bias);
 - q / k head i serves v heads i * (n_v / n_qk) ... (i + 1) * (n_v / n_qk) - 1;
 - the recurrence is the gated delta rule of oracle.gdn_scan;
 - gated RMSNorm per v head: o / sqrt(mean(o^2) + 1e-6) * w_norm * silu(z);
 - bf16 rounding points: the in-projection outputs, q, k, v after the convolution and norm (the
   recurrence's inputs), the gated-norm output, the new residual.
"""
from __future__ import annotations

import numpy as np

from . import FP8, bf16_round, bf16_value, gdn_scan, linear, rmsnorm

EPS = 1e-6


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def short_conv_silu(x: np.ndarray, window: np.ndarray, taps: np.ndarray):
    """Causal depthwise 4-tap convolution, then SiLU.  x: fp64 [T][C] (the rows in order), window:
    fp64 [3][C] (the three rows before x, oldest first), taps: fp64 [C][4].
    y[t][c] = silu(sum_j taps[c][j] * e[t + j][c]) with e = window rows then x rows.
    Returns (y [T][C], e [T + 3][C]); the window after the first n rows is e[n : n + 3]."""
    T = x.shape[0]
    e = np.concatenate([window, x], axis=0)
    y = np.zeros_like(x)
    for t in range(T):
        acc = np.zeros(x.shape[1])
        for j in range(4):
            acc += taps[:, j] * e[t + j]
        y[t] = silu(acc)
    return y, e


def l2norm_heads(x: np.ndarray, d: int) -> np.ndarray:
    """Each d-wide head of the rows of x divided by sqrt(sum of squares + EPS)."""
    shp = x.shape
    h = x.reshape(shp[0], -1, d)
    return (h / np.sqrt((h * h).sum(axis=-1, keepdims=True) + EPS)).reshape(shp)


def gates(a: np.ndarray, b: np.ndarray, A_log: np.ndarray, dt_bias: np.ndarray):
    """(alpha, beta) per row and v head: alpha = exp(-exp(A_log) softplus(a + dt_bias)),
    beta = sigmoid(b)."""
    sp = np.logaddexp(0.0, a + dt_bias)
    return np.exp(-np.exp(A_log) * sp), 1.0 / (1.0 + np.exp(-b))


def gated_rmsnorm(o: np.ndarray, z: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Per head (last axis d): o / sqrt(mean(o^2) + EPS) * w * silu(z)."""
    return o / np.sqrt((o * o).mean(axis=-1, keepdims=True) + EPS) * w * silu(z)


def gdn_block(h_bf16: np.ndarray, g: dict, wts: dict, state: np.ndarray, window: np.ndarray, rows: int = 8,
              core_out: list | None = None):
    """One lane's Gated DeltaNet mixer block over its 8 verify rows.

    h_bf16: uint16 [8][hidden] (the residual); g: {"hidden", "n_qk", "n_v", "d"}; wts: "in" FP8
    codes [(2 n_qk + 2 n_v) d][hidden] with scale "s_in", "out" FP8 codes [hidden][n_v d] with
    "s_out", "A" / "B" bf16 bits [n_v][hidden], "taps" fp64 [(2 n_qk + n_v) d][4] (bf16 values),
    "A_log" / "dt_bias" fp64 [n_v], "w_norm" fp64 [d]; state: fp64 [n_v][d][d] (parity buffer A);
    window: fp64 [3][(2 n_qk + n_v) d].  The outputs (and so the new residual) are the verify scan's
    over all 8 rows; the returned state and window are those after the first `rows` rows (8 after a
    full accept, n_commit for the re-scan after a partial one).
    Returns (new residual uint16 [8][hidden], state after `rows` rows, window after `rows` rows,
    the recurrence's inputs (q, k, v bf16 bits [8][n_v][d], alpha, beta [8][n_v])).  core_out: when a
    list, the out-projection's input (the gated norm's bf16 bits [8][n_v d]) is appended to it."""
    H, nqk, nv, d = g["hidden"], g["n_qk"], g["n_v"], g["d"]
    cq, cv = nqk * d, nv * d
    r = rmsnorm(h_bf16)
    u = linear(FP8, r, wts["in"], None, wts["s_in"], 2 * cq + 2 * cv, with_abs=False)
    qkv = bf16_value(bf16_round(u[:, :2 * cq + cv]))
    z = bf16_value(bf16_round(u[:, 2 * cq + cv:]))
    rv = bf16_value(r)
    a = rv @ bf16_value(wts["A"]).T
    b = rv @ bf16_value(wts["B"]).T
    y, e = short_conv_silu(qkv, window, wts["taps"])
    q = bf16_round(l2norm_heads(y[:, :cq], d)).reshape(8, nqk, d)
    k = bf16_round(l2norm_heads(y[:, cq:2 * cq], d)).reshape(8, nqk, d)
    v = bf16_round(y[:, 2 * cq:]).reshape(8, nv, d)
    rep = nv // nqk
    qe, ke = np.repeat(q, rep, axis=1), np.repeat(k, rep, axis=1)
    alpha, beta = gates(a, b, wts["A_log"], wts["dt_bias"])
    st, o = gdn_scan(state[None], qe, ke, v, alpha, beta, np.array([8], np.int32))  # the verify scan
    if rows != 8:  # the commit re-scan: the state after the committed rows only
        st, _ = gdn_scan(state[None], qe, ke, v, alpha, beta, np.array([rows], np.int32), want_out=False)
    on = bf16_round(gated_rmsnorm(o, z.reshape(8, nv, d), wts["w_norm"]).reshape(8, cv))
    if core_out is not None:
        core_out.append(on)
    y_out = linear(FP8, on, wts["out"], None, wts["s_out"], H, with_abs=False)
    h_new = bf16_round(bf16_value(h_bf16) + y_out)
    return h_new, st[0], e[rows:rows + 3], (qe, ke, v, alpha, beta)

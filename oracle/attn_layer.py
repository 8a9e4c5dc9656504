"""The gated-attention mixer block with its real core, in fp64: TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the bench's CPU-baseline leg may use this module; the
product path never imports it.  It shares nothing with the CUDA library.

Sources (web pages, cited by title and section):
 - "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max", section "The megakernel is
   per layer, not per step" (the block's graph: RMSNorm; FP8 QKV and gate projections; the core --
   Q/K RMSNorm, RoPE, causal q k^T softmax weighting V over a read-and-appended KV cache; the
   partials merged and multiplied by the sigmoid of the gate; the FP8 output projection with the
   residual).
 - "144 tok/s needs 502 GB/s", section "The engine hard-codes the model" (24 query heads, 4 KV
   heads of 256; the attention in-projection is queries, keys, values and an output gate,
   6144 + 1024 + 1024 + 6144 rows; norms are small bf16 vectors).

The pages name the steps; the formulas below are readings (the plainest ones the names support):
 - the q projection's rows are the queries (Hq heads) then the gate (Hq heads); the kv
   projection's rows are the keys (Hkv heads) then the values (Hkv heads);
 - Q/K RMSNorm: each head of q and k over its root mean square (eps 1e-6), times a per-dimension
   weight shared by the heads;
 - RoPE: the published rotary embedding (Su et al., "RoFormer", 2021) over the whole head, pairs
   (2i, 2i + 1) rotated by pos * base^(-2i / D), base 10000, pos = the row's cache position
   (ctx + j for verify row j);
 - the core is oracle.attention_verify (the causal softmax over the cache and the lane's own rows,
   times sigmoid(gate));
 - bf16 rounding points: the projection outputs, q and k after norm and RoPE (the core's inputs),
   the core's output, the new residual.
"""
from __future__ import annotations

import numpy as np

from . import FP8, attention_verify, bf16_round, bf16_value, linear, rmsnorm

EPS = 1e-6
ROPE_BASE = 10000.0


def head_rmsnorm(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x: [..., D]; each head over sqrt(mean(x^2) + EPS), times w [D]."""
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + EPS) * w


def rope(x: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """x: [M][heads][D], pos: [M]; pairs (2i, 2i + 1) rotated by pos * base^(-2i / D)."""
    D = x.shape[-1]
    theta = ROPE_BASE ** (-np.arange(0, D, 2) / D)  # [D / 2]
    ang = pos[:, None, None] * theta[None, None, :]
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def attn_block(h_bf16: np.ndarray, g: dict, wts: dict, k_cache: np.ndarray, v_cache: np.ndarray,
               ctx: np.ndarray, core_out: list | None = None):
    """The attention mixer block for M = 8 * lanes verify rows.

    h_bf16: uint16 [M][hidden]; g: {"hidden", "Hq", "Hkv", "D"}; wts: "q" FP8 codes [2 Hq D][hidden]
    with scale "s_q", "kv" FP8 codes [2 Hkv D][hidden] with "s_kv", "o" FP8 codes [hidden][Hq D] with
    "s_o", "q_norm" / "k_norm" fp64 [D]; k_cache / v_cache: bf16 bits [lanes][Hkv][cap][D] holding
    ctx[l] positions per lane.  Returns (new residual uint16 [M][hidden], the rows' keys and values
    as appended (bf16 bits [M][Hkv][D]), the core's q and gate inputs (bf16 bits [M][Hq][D])).  core_out:
    when a list, the o-projection's input (the core's bf16 output bits [M][Hq D]) is appended to it."""
    H, Hq, Hkv, D = g["hidden"], g["Hq"], g["Hkv"], g["D"]
    M = h_bf16.shape[0]
    r = rmsnorm(h_bf16)
    qg = bf16_value(bf16_round(linear(FP8, r, wts["q"], None, wts["s_q"], 2 * Hq * D, with_abs=False)))
    kv = bf16_value(bf16_round(linear(FP8, r, wts["kv"], None, wts["s_kv"], 2 * Hkv * D, with_abs=False)))
    q, gate = qg[:, :Hq * D].reshape(M, Hq, D), qg[:, Hq * D:].reshape(M, Hq, D)
    k, v = kv[:, :Hkv * D].reshape(M, Hkv, D), kv[:, Hkv * D:].reshape(M, Hkv, D)
    pos = (np.repeat(np.asarray(ctx, np.float64), 8) + np.tile(np.arange(8.0), M // 8))
    qb = bf16_round(rope(head_rmsnorm(q, wts["q_norm"]), pos))
    kb = bf16_round(rope(head_rmsnorm(k, wts["k_norm"]), pos))
    vb, gb = bf16_round(v), bf16_round(gate)
    core = attention_verify(qb, kb, vb, k_cache, v_cache, ctx, gb, with_abs=False)
    ob = bf16_round(core.reshape(M, Hq * D))
    if core_out is not None:
        core_out.append(ob)
    y = linear(FP8, ob, wts["o"], None, wts["s_o"], H, with_abs=False)
    return bf16_round(bf16_value(h_bf16) + y), (kb, vb), (qb, gb)

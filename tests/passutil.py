"""Helpers for the verify-pass tests: synthetic canonical weights on the host, the same weights
packed on the device, and the per-block error budget used to compare one GPU block with the
oracle from the oracle's own block input."""
from __future__ import annotations

import numpy as np

import oracle
import synth
from helpers import REL, dev_u8

DELTA = 2.0 ** -7  # one bf16 ulp, relative to the value (a rounding step may flip by one ulp)


def make_layer(G, seed, l, scales=None):
    """Canonical weights of layer l (the seeded recipe; the same bits as the device fills of
    weight_streaming_gb300.model.SyntheticModel).  scales: the six per-tensor scales, default 1."""
    attn = (l % G.period) == G.period - 1
    n_in = G.attn_q if attn else G.gdn_in
    kz = G.attn_z if attn else G.gdn_z
    d = {"attn": attn, "n_in": n_in, "kz": kz,
         "in": synth.fp8_matrix(seed, l, synth.T_IN, n_in, G.hidden),
         "kv": synth.fp8_matrix(seed, l, synth.T_KV, G.attn_kv, G.hidden) if attn else None,
         "out": synth.fp8_matrix(seed, l, synth.T_OUT, G.hidden, kz)}
    d["gate_c"], d["gate_s"] = synth.nvfp4_matrix(seed, l, synth.T_GATE_C, synth.T_GATE_S, G.inter, G.hidden)
    d["up_c"], d["up_s"] = synth.nvfp4_matrix(seed, l, synth.T_UP_C, synth.T_UP_S, G.inter, G.hidden)
    d["down_c"], d["down_s"] = synth.nvfp4_matrix(seed, l, synth.T_DOWN_C, synth.T_DOWN_S, G.hidden, G.inter)
    for i, k in enumerate(("s_in", "s_kv", "s_out", "ts_gate", "ts_up", "ts_down")):
        d[k] = 1.0 if scales is None else float(scales[i])
    return d


def make_head(G, seed, ts=1.0):
    hc, hs = synth.nvfp4_matrix(seed, synth.HEAD_LAYER, synth.T_HEAD_C, synth.T_HEAD_S, G.vocab, G.hidden)
    return hc, hs, float(ts)


def make_layers(G, seed, unit_scales=False):
    rng = np.random.default_rng(seed + 777)
    layers = []
    for l in range(G.n_layers):
        sc = [1.0 if unit_scales else float(rng.uniform(0.5, 1.5)) for _ in range(6)]
        layers.append(make_layer(G, seed, l, sc))
    head = make_head(G, seed, 1.0 if unit_scales else float(rng.uniform(0.5, 1.5)))
    return layers, head


class DeviceModel:
    """The same canonical weights packed on the device, behind a vp_model handle."""

    def __init__(self, V, G, layers, head):
        import torch
        self.keep = []
        descs = []

        def pk8(w):
            p = torch.empty(V.vp_packed_bytes_fp8(*w.shape), dtype=torch.uint8, device="cuda")
            V.vp_pack_fp8(dev_u8(w), w.shape[0], w.shape[1], p)
            self.keep.append(p)
            return p.data_ptr()

        def pk4(c, s):
            n, k = c.shape[0], 2 * c.shape[1]
            p = torch.empty(V.vp_packed_bytes_nvfp4(n, k), dtype=torch.uint8, device="cuda")
            V.vp_pack_nvfp4(dev_u8(c), dev_u8(s), n, k, p)
            self.keep.append(p)
            return p.data_ptr()

        for d in layers:
            ld = V.vp_layer_desc()
            ld.kind = V.VP_LAYER_ATTN if d["attn"] else V.VP_LAYER_GDN
            ld.w_in, ld.s_in, ld.n_in = pk8(d["in"]), d["s_in"], d["n_in"]
            if d["attn"]:
                ld.w_kv, ld.s_kv, ld.n_kv = pk8(d["kv"]), d["s_kv"], d["kv"].shape[0]
            ld.w_out, ld.s_out, ld.k_out = pk8(d["out"]), d["s_out"], d["kz"]
            ld.w_gate, ld.ts_gate = pk4(d["gate_c"], d["gate_s"]), d["ts_gate"]
            ld.w_up, ld.ts_up = pk4(d["up_c"], d["up_s"]), d["ts_up"]
            ld.w_down, ld.ts_down = pk4(d["down_c"], d["down_s"]), d["ts_down"]
            descs.append(ld)
        hp = pk4(head[0], head[1])
        self.model = V.vp_model(G.hidden, G.inter, G.eps, descs, V.vp_head_desc(hp, head[2], G.vocab))
        torch.cuda.synchronize()


# ------------------------------------------------------------------ error budget of one block

def prop_bound(fmt, dx, codes, scales, ts, N):
    """An upper bound of sum_k dx[m][k] |w[n][k]| (dx >= 0): the oracle's sum |x w| over dx rounded
    up to bf16.  bf16 keeps 8 significant bits, so rounding dx (1 + 2^-7) to nearest stays above dx;
    the bound is at most 2^-6 above the exact sum."""
    v = np.maximum(np.asarray(dx, np.float64), 0.0) * (1.0 + 2.0 ** -7)
    _, a = oracle.linear(fmt, oracle.bf16_round(v), codes, scales, ts, N)
    return a


def mixer_block_ref(G, d, h_in_bits):
    """Oracle output of one mixer block and its per-element error budget for a device block that
    starts from the same input.  Budget terms: the fp32-accumulation tolerance REL * sum|x w| of
    each linear, at most one bf16 ulp of difference in every rounded intermediate (RMSNorm output,
    z, the residual sum), and the propagation of those differences through the next linear."""
    r = oracle.rmsnorm(h_in_bits, G.eps)
    u, a_u = oracle.linear(oracle.FP8, r, d["in"], None, d["s_in"], d["n_in"])
    kz = d["kz"]
    z_bits = oracle.bf16_round(u[:, :kz])
    z = oracle.bf16_value(z_bits)
    du = (REL + DELTA) * a_u[:, :kz]
    dz = du + DELTA * (np.abs(z) + du)
    y, a_y = oracle.linear(oracle.FP8, z_bits, d["out"], None, d["s_out"], G.hidden)
    prop = prop_bound(oracle.FP8, dz, d["out"], None, d["s_out"], G.hidden)
    dy = REL * (a_y + prop) + prop
    h_out = oracle.bf16_round(oracle.bf16_value(h_in_bits) + y)
    hv = oracle.bf16_value(h_out)
    return h_out, dy + DELTA * (np.abs(hv) + dy)


def mlp_block_ref(G, d, h_in_bits):
    r = oracle.rmsnorm(h_in_bits, G.eps)
    g, a_g = oracle.linear(oracle.NVFP4, r, d["gate_c"], d["gate_s"], d["ts_gate"], G.inter)
    u, a_u = oracle.linear(oracle.NVFP4, r, d["up_c"], d["up_s"], d["ts_up"], G.inter)
    s = oracle.silu_mul(g, u)
    a_bits = oracle.bf16_round(s)
    av = oracle.bf16_value(a_bits)
    dg = (REL + DELTA) * a_g
    du = (REL + DELTA) * a_u
    silu_g = oracle.silu_mul(g, np.ones_like(g))
    ds = 1.1 * dg * (np.abs(u) + du) + (np.abs(silu_g) + 1.1 * dg) * du + 1e-6 * np.abs(s)
    da = ds + DELTA * (np.abs(av) + ds)
    y, a_y = oracle.linear(oracle.NVFP4, a_bits, d["down_c"], d["down_s"], d["ts_down"], G.hidden)
    prop = prop_bound(oracle.NVFP4, da, d["down_c"], d["down_s"], d["ts_down"], G.hidden)
    dy = REL * (a_y + prop) + prop
    h_out = oracle.bf16_round(oracle.bf16_value(h_in_bits) + y)
    hv = oracle.bf16_value(h_out)
    return h_out, dy + DELTA * (np.abs(hv) + dy)

"""Pins the fp64 oracle to facts that do not come from the oracle itself.

Each test checks one oracle function against values the pages print, a closed form, an independent
library routine (torch / numpy), or brute force on tiny inputs.  A plausible slip in the oracle
(a dropped term, a wrong nibble, sign or index, a transposed operand) fails at least one of them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))


# ------------------------------------------------------------------ independent decoders

def e4m3_torch(codes):
    """E4M3 values from torch's float8_e4m3fn conversion (a library routine)."""
    t = torch.as_tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def e2m1_formula(code):
    """Generic minifloat decode: sign bit 3, 2-bit exponent (bias 1), 1-bit mantissa."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = (m / 2.0) if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -v if s else v


def dequant_nvfp4_indep(codes, scales, ts):
    """Dequantizes canonical NVFP4 with torch's E4M3 and the formula decode (not the oracle)."""
    lo = codes & 15
    hi = codes >> 4
    N, K2 = codes.shape
    q = np.empty((N, 2 * K2), np.int64)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    lut = np.array([e2m1_formula(c) for c in range(16)])
    sv = np.repeat(e4m3_torch(scales), 16, axis=1)
    return lut[q] * sv * ts


def bf16_vals_torch(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def rand_bf16(rng, shape, scale=1.0):
    x = torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ formats

def test_e2m1_value_set_matches_page():
    t = oracle.e2m1_table()
    assert sorted(set(t.tolist())) == sorted(set(GOLD["e2m1_value_set"]["values"]))
    assert t[8] == 0.0 and math.copysign(1.0, t[8]) == -1.0  # code 8 is -0


def test_e2m1_bit_layout_matches_minifloat_formula():
    t = oracle.e2m1_table()
    for c in range(16):
        assert t[c] == e2m1_formula(c), c
    # codes 8..15 are the negatives of 0..7, and each half is increasing in magnitude
    assert np.all(t[8:] == -t[:8])
    assert np.all(np.diff(t[:8]) > 0)


def test_e4m3_table_matches_torch_and_page_max():
    t = oracle.e4m3_table()
    ref = e4m3_torch(np.arange(256))
    nan_o = np.isnan(t)
    assert np.array_equal(nan_o, np.isnan(ref))
    assert np.array_equal(np.flatnonzero(nan_o), [0x7F, 0xFF])
    assert np.array_equal(t[~nan_o], ref[~nan_o])
    assert np.nanmax(t) == GOLD["e4m3_block_scale_max"]["value"] == t[0x7E]
    assert t[0x01] == 2.0 ** -9  # smallest subnormal
    assert t[0x08] == 2.0 ** -6 and t[0x38] == 1.0


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-40, 38, 20000),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 3.4e38, 1e-40, -1e-41, 9.2e-41]),
    ]).astype(np.float32)
    # exact ties between two bf16 neighbours (round half to even)
    base = rng.integers(0, 0x7F00, 2000).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    v = np.concatenate([v, ties]).astype(np.float32)
    ours = oracle.bf16_round(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_round_is_single_rounding_from_fp64():
    # x = 1 + 2^-8 + 2^-40: just above the bf16 tie 1 + 2^-8, so it must round UP to 1 + 2^-7.
    # Rounding through fp32 first would land exactly on the tie and round down to 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    bits = int(oracle.bf16_round(np.array([x]))[0])
    assert Fraction(float(bf16_vals_torch([bits])[0])) == 1 + Fraction(1, 128)
    # brute force: nearest bf16 by exact rational distance over a neighbourhood
    rng = np.random.default_rng(1)
    xs = rng.standard_normal(300) * 2.0 ** rng.integers(-20, 20, 300)
    got = oracle.bf16_round(xs)
    for x, b in zip(xs, got):
        cands = [int(b) + d for d in (-1, 0, 1)]
        dist = [abs(Fraction(float(bf16_vals_torch([c & 0xFFFF])[0])) - Fraction(float(x))) for c in cands]
        assert dist[1] <= min(dist), (x, b)


# ------------------------------------------------------------------ linear layers

def test_nvfp4_one_hot_probes_cover_all_codes_and_scales():
    """x = e_k reproduces w[n][k] = e2m1(code) * e4m3(scale) * ts exactly, for all 16 codes and all
    127 finite non-negative scale codes 0x00..0x7E."""
    N, G = 16, 128
    K = 16 * G
    codes = np.zeros((N, K // 2), np.uint8)
    for n in range(N):
        codes[n, :] = n | (n << 4)
    scales = np.tile(np.arange(G, dtype=np.uint8), (N, 1))
    scales[:, 127] = 0x7E  # 0x7F is NaN; keep the last group finite
    ts = 0.75
    M = G
    x = np.zeros((M, K), np.uint16)
    for m in range(M):
        x[m, 16 * m + (m % 16)] = 0x3F80  # bf16 1.0
    y, a = oracle.linear(oracle.NVFP4, x, codes, scales, ts, N)
    val = np.array(GOLD["e2m1_value_set"]["values"])  # noqa: F841 (the set is pinned above)
    for m in range(M):
        sc = e4m3_torch([scales[0, m]])[0]
        for n in range(N):
            assert y[m, n] == e2m1_formula(n) * sc * ts
            assert a[m, n] == abs(e2m1_formula(n) * sc * ts)


def test_nvfp4_dyadic_inputs_match_integer_matmul():
    """Integer x and power-of-two scales make every product an integer multiple of 2^-10, so the
    exact result is an int64 matmul (numpy) scaled by 2^-10."""
    rng = np.random.default_rng(2)
    M, N, K = 5, 24, 128
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    pow2_codes = np.array([0x30, 0x38, 0x40, 0x28], np.uint8)  # 0.5, 1, 2, 0.25
    scales = pow2_codes[rng.integers(0, 4, (N, K // 16))]
    xi = rng.integers(-3, 4, (M, K))
    x = torch.from_numpy(xi.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = oracle.linear(oracle.NVFP4, x, codes, scales, 1.0, N, with_abs=False)
    w = dequant_nvfp4_indep(codes, scales, 1.0)
    wi = np.rint(w * 1024).astype(np.int64)
    assert np.array_equal(wi / 1024.0, w)
    exact = (xi.astype(np.int64) @ wi.T) / 1024.0
    assert np.array_equal(y, exact)


def test_nvfp4_matches_numpy_matmul_random():
    rng = np.random.default_rng(3)
    M, N, K = 7, 40, 256
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (N, K // 16), dtype=np.uint8)
    x = rand_bf16(rng, (M, K))
    ts = 1.3
    y, a = oracle.linear(oracle.NVFP4, x, codes, scales, ts, N)
    w = dequant_nvfp4_indep(codes, scales, ts)
    xv = bf16_vals_torch(x)
    np.testing.assert_allclose(y, xv @ w.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a, np.abs(xv) @ np.abs(w).T, rtol=1e-12, atol=1e-12)
    rows = np.array([39, 0, 17], np.int32)
    y2, a2 = oracle.linear(oracle.NVFP4, x, codes, scales, ts, N, rows=rows)
    assert np.array_equal(y2, y[:, rows]) and np.array_equal(a2, a[:, rows])


def test_nvfp4_nibble_order_low_first():
    """Element 2j is the low nibble: a code byte 0x10 (low 0, high 1 = 0.5) only reaches x[2j+1]."""
    K = 32
    codes = np.zeros((1, K // 2), np.uint8)
    codes[0, 3] = 0x10
    scales = np.full((1, K // 16), 0x38, np.uint8)
    x = np.zeros((2, K), np.uint16)
    x[0, 6] = 0x3F80
    x[1, 7] = 0x3F80
    y = oracle.linear(oracle.NVFP4, x, codes, scales, 1.0, 1, with_abs=False)
    assert y[0, 0] == 0.0 and y[1, 0] == 0.5


def test_fp8_matches_numpy_matmul_random():
    rng = np.random.default_rng(4)
    M, N, K = 9, 33, 96
    w8 = rng.integers(0, 256, (N, K), dtype=np.uint8)
    w8[(w8 & 0x7F) == 0x7F] = 0x11  # no NaN codes
    x = rand_bf16(rng, (M, K))
    s = 0.37
    y, a = oracle.linear(oracle.FP8, x, w8, None, s, N)
    w = e4m3_torch(w8) * s
    xv = bf16_vals_torch(x)
    np.testing.assert_allclose(y, xv @ w.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a, np.abs(xv) @ np.abs(w).T, rtol=1e-12, atol=1e-12)


def test_linear_rejects_bad_arguments():
    x = np.zeros((2, 16), np.uint16)
    with pytest.raises(ValueError):
        oracle.linear(oracle.NVFP4, x, np.zeros((4, 8), np.uint8), np.zeros((4, 1), np.uint8), 1.0, 4,
                      rows=np.array([4], np.int32))


# ------------------------------------------------------------------ glue

def test_silu_mul_matches_torch_and_closed_forms():
    rng = np.random.default_rng(5)
    g = rng.standard_normal(1000) * 20
    u = rng.standard_normal(1000) * 5
    out = oracle.silu_mul(g, u)
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-300)
    z = oracle.silu_mul(np.array([0.0, 50.0, -50.0]), np.array([3.0, 1.0, 1.0]))
    assert z[0] == 0.0 and abs(z[1] - 50.0) < 1e-18 and abs(z[2]) < 1e-19
    # silu(-x) = silu(x) - x
    xs = rng.standard_normal(50)
    np.testing.assert_allclose(oracle.silu_mul(-xs, np.ones(50)), oracle.silu_mul(xs, np.ones(50)) - xs,
                               rtol=1e-12, atol=1e-14)


def _round_bf16_numpy(v):
    """Independent fp64 -> bf16 RNE (numpy frexp/rint), values only."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)
    q = np.maximum(e - 8, -133).astype(np.float64)
    return np.rint(v / 2.0 ** q) * 2.0 ** q


def test_rmsnorm_matches_torch_formula():
    rng = np.random.default_rng(6)
    h = rand_bf16(rng, (6, 320), 7.0)
    r = oracle.rmsnorm(h, 1e-6)
    hv = torch.from_numpy(bf16_vals_torch(h))
    ref = torch.nn.functional.rms_norm(hv, (320,), eps=1e-6).numpy()
    assert np.array_equal(bf16_vals_torch(r), _round_bf16_numpy(ref))
    # closed form: a constant row c maps to c / sqrt(c^2 + eps)
    c = np.full((1, 64), 0x4040, np.uint16)  # 3.0
    rc = bf16_vals_torch(oracle.rmsnorm(c, 1e-6))
    assert np.all(rc == _round_bf16_numpy(3.0 / math.sqrt(9.0 + 1e-6)))


def test_argmax_lowest_index_ties_and_nan():
    rng = np.random.default_rng(7)
    for _ in range(200):
        v = rng.integers(-3, 4, 50).astype(np.float64)
        assert oracle.argmax(v) == int(np.argmax(v))  # numpy returns the first maximum
    assert oracle.argmax(np.array([-0.0, 0.0, -1.0])) == 0
    assert oracle.argmax(np.array([0.0, -0.0])) == 0
    assert oracle.argmax(np.array([-1.0, np.nan, 2.0, 2.0])) == 2
    assert oracle.argmax(np.array([np.nan, -1.0])) == 1
    assert oracle.argmax(np.array([np.nan, np.nan])) == 0
    assert oracle.argmax(np.array([-np.inf, -np.inf])) == 0


# ------------------------------------------------------------------ acceptance

def _accept_by_definition(t, drafts):
    """1 + length of the longest common prefix of drafts[0..6] and t[0..6]."""
    n = 0
    for a, b in zip(t[:7], drafts):
        if a != b:
            break
        n += 1
    return n + 1


def test_accept_brute_force_binary_vocab():
    # every target pattern (8 tokens) x every draft pattern (7 tokens) over V = 2
    tp = np.array(list(itertools.product([0, 1], repeat=8)), np.int32)
    dp = np.array(list(itertools.product([0, 1], repeat=7)), np.int32)
    T = np.repeat(tp, len(dp), axis=0)
    D = np.tile(dp, (len(tp), 1))
    anchor = np.full((T.shape[0], 1), 5, np.int32)
    pending = np.concatenate([anchor, D], axis=1)
    nc, cm = oracle.accept(T.reshape(-1), pending.reshape(-1))
    eq = (T[:, :7] == D)
    lcp = np.cumprod(eq, axis=1).sum(axis=1)
    assert np.array_equal(nc, lcp + 1)
    lo, hi = GOLD["accept_commit_range"]["min"], GOLD["accept_commit_range"]["max"]
    assert nc.min() == lo and nc.max() == hi
    j = np.arange(8)[None, :]
    expect = np.where(j <= lcp[:, None], T, -1)
    assert np.array_equal(cm, expect)


def test_accept_random_vocab3_against_definition():
    rng = np.random.default_rng(8)
    n = 20000
    T = rng.integers(0, 3, (n, 8)).astype(np.int32)
    D = rng.integers(0, 3, (n, 7)).astype(np.int32)
    pending = np.concatenate([rng.integers(0, 3, (n, 1)).astype(np.int32), D], axis=1)
    nc, cm = oracle.accept(T.reshape(-1), pending.reshape(-1))
    for i in range(0, n, 97):
        assert nc[i] == _accept_by_definition(T[i], D[i])
        assert list(cm[i][:nc[i]]) == list(T[i][:nc[i]])
        assert all(v == -1 for v in cm[i][nc[i]:])


# ------------------------------------------------------------------ byte counts

def test_pass_bytes_match_page_table():
    g = GOLD["geometry"]
    G = oracle.geom(n_layers=g["layers"], hidden=g["hidden"], inter=g["intermediate"], vocab=g["vocab"],
                    period=g["full_attention_period"], attn_kv=2 * g["kv_heads"] * g["head_dim"])
    b = oracle.pass_bytes(G)
    pb = GOLD["pass_bytes_gb"]
    for i, key in enumerate(["mlp_codes", "mlp_scales", "gdn_fp8", "attn_fp8", "head"]):
        assert round(b[i] / 1e9, 3) == pb[key], key
    assert round(b[5] / 1e9, 3) == pb["weight_gemm_total"]
    assert b[5] == 17_555_292_160
    # 9 bytes per 16 NVFP4 weights
    assert (b[0] + b[1]) * 16 == 9 * (64 * 3 * 17408 * 5120)
    assert (b[4]) * 16 == 9 * (248320 * 5120)


def test_arithmetic_intensity_matches_page():
    ai = GOLD["arithmetic_intensity_flop_per_byte"]
    for M, key in ((8, "M8"), (32, "M32")):
        flop_per_byte = 2 * M / (GOLD["bytes_per_16_weights_nvfp4"]["value"] / 16)
        assert round(flop_per_byte) == ai[key]


# ------------------------------------------------------------------ the surrogate pass

def _tiny_model(seed=11, L=4, H=64, I=96, V=200, gdn_in=80, gdn_z=48, aq=72, akv=16, az=40):
    import synth
    rng = np.random.default_rng(seed)
    layers = []
    for l in range(L):
        attn = (l % 4) == 3
        d = {}
        n_in = aq if attn else gdn_in
        kz = az if attn else gdn_z
        d["in"] = synth.fp8_matrix(seed, l, synth.T_IN, n_in, H)
        d["kv"] = synth.fp8_matrix(seed, l, synth.T_KV, akv, H) if attn else None
        d["out"] = synth.fp8_matrix(seed, l, synth.T_OUT, H, kz)
        d["gate_c"], d["gate_s"] = synth.nvfp4_matrix(seed, l, synth.T_GATE_C, synth.T_GATE_S, I, H)
        d["up_c"], d["up_s"] = synth.nvfp4_matrix(seed, l, synth.T_UP_C, synth.T_UP_S, I, H)
        d["down_c"], d["down_s"] = synth.nvfp4_matrix(seed, l, synth.T_DOWN_C, synth.T_DOWN_S, H, I)
        d.update(s_in=float(rng.uniform(0.5, 1.5)), s_kv=1.0, s_out=float(rng.uniform(0.5, 1.5)),
                 ts_gate=float(rng.uniform(0.5, 1.5)), ts_up=float(rng.uniform(0.5, 1.5)),
                 ts_down=float(rng.uniform(0.5, 1.5)))
        layers.append(d)
    hc, hs = synth.nvfp4_matrix(seed, synth.HEAD_LAYER, synth.T_HEAD_C, synth.T_HEAD_S, V, H)
    G = oracle.geom(n_layers=L, hidden=H, inter=I, vocab=V, period=4, gdn_in=gdn_in, gdn_z=gdn_z,
                    attn_q=aq, attn_kv=akv, attn_z=az)
    return G, layers, (hc, hs, 0.9)


def test_verify_pass_matches_independent_torch_composition():
    """Re-composes the surrogate pass with torch fp64 ops, numpy RNE and the independent decoders,
    and compares every traced residual state and the final logits."""
    import synth
    G, layers, head = _tiny_model()
    M = 16
    x0 = synth.normal_bf16(3, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    pending = np.zeros(M, np.int32)
    out = oracle.verify_pass(G, layers, head, x0, pending, want_trace=True, want_logits=True)

    def fp8(codes, s):
        return torch.from_numpy(e4m3_torch(codes) * s)

    def rms(hv):
        return torch.from_numpy(_round_bf16_numpy(torch.nn.functional.rms_norm(hv, (G.hidden,), eps=1e-6).numpy()))

    h = torch.from_numpy(bf16_vals_torch(x0))
    for l, d in enumerate(layers):
        attn = (l % 4) == 3
        kz = G.attn_z if attn else G.gdn_z
        r = rms(h)
        u = r @ fp8(d["in"], d["s_in"]).T
        z = torch.from_numpy(_round_bf16_numpy(u[:, :kz].numpy()))
        h = torch.from_numpy(_round_bf16_numpy((h + z @ fp8(d["out"], d["s_out"]).T).numpy()))
        assert np.array_equal(h.numpy(), bf16_vals_torch(out["trace"][2 * l])), l
        r = rms(h)
        g = r @ torch.from_numpy(dequant_nvfp4_indep(d["gate_c"], d["gate_s"], d["ts_gate"])).T
        u = r @ torch.from_numpy(dequant_nvfp4_indep(d["up_c"], d["up_s"], d["ts_up"])).T
        a = torch.from_numpy(_round_bf16_numpy((torch.nn.functional.silu(g) * u).numpy()))
        dn = a @ torch.from_numpy(dequant_nvfp4_indep(d["down_c"], d["down_s"], d["ts_down"])).T
        h = torch.from_numpy(_round_bf16_numpy((h + dn).numpy()))
        assert np.array_equal(h.numpy(), bf16_vals_torch(out["trace"][2 * l + 1])), l
    r = rms(h)
    logits = (r @ torch.from_numpy(dequant_nvfp4_indep(head[0], head[1], head[2])).T).numpy()
    np.testing.assert_allclose(out["logits"], logits, rtol=1e-12, atol=1e-12)
    assert np.array_equal(out["argmax"], np.argmax(out["logits"], axis=1))


# ------------------------------------------------------------------ affine INT4 ("Q4")

def bf16_bits_of(values):
    """bf16 bit patterns (uint16) of values that bf16 holds exactly."""
    t = torch.tensor(np.asarray(values, np.float64)).to(torch.bfloat16)
    assert np.array_equal(t.to(torch.float64).numpy(), np.asarray(values, np.float64))
    return t.view(torch.int16).numpy().view(np.uint16)


def dequant_q4_indep(codes, scales, biases):
    """w = scale * q + bias per group of 64 along K, with torch's bf16 decoding (not the oracle)."""
    N, K2 = codes.shape
    q = np.empty((N, 2 * K2), np.float64)
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    sv = np.repeat(bf16_vals_torch(scales), 64, axis=1)
    bv = np.repeat(bf16_vals_torch(biases), 64, axis=1)
    return sv * q + bv, np.abs(sv * q) + np.abs(bv)


def test_q4_bytes_match_page_table():
    """Nine bytes per sixteen weights reproduce the page's byte table of the 4-bit checkpoint."""
    t = GOLD["q4_bytes_mb"]
    shapes = {"gdn_in_16640x5120": (16640, 5120), "gdn_out_5120x6144": (5120, 6144),
              "attn_in_14336x5120": (14336, 5120), "attn_out_5120x6144": (5120, 6144),
              "lm_head_248320x5120": (248320, 5120), "token_embedding_248320x5120": (248320, 5120)}
    for key, (n, k) in shapes.items():
        assert round(oracle.q4_bytes(n, k) / 1e6, 2) == t[key], key
        assert oracle.q4_bytes(n, k) * 16 == 9 * n * k
    g = GOLD["geometry"]
    mlp = 2 * oracle.q4_bytes(g["intermediate"], g["hidden"]) + oracle.q4_bytes(g["hidden"], g["intermediate"])
    assert round(mlp / 1e6, 2) == t["swiglu_gate_up_down_per_layer"]
    tot = GOLD["q4_target_total"]
    total = (tot["layers_gdn"] * (oracle.q4_bytes(16640, 5120) + oracle.q4_bytes(5120, 6144))
             + tot["layers_attention"] * (oracle.q4_bytes(14336, 5120) + oracle.q4_bytes(5120, 6144))
             + g["layers"] * mlp + 2 * oracle.q4_bytes(g["vocab"], g["hidden"]))
    assert round(total / 1e9 + tot["small_tensors_gb"], 3) == tot["gb"]


def test_q4_one_hot_probes_cover_all_codes():
    """x = e_k reproduces w[n][k] = scale * q + bias exactly: all 16 codes, scales and biases of both
    signs and very different magnitudes, and the group boundary (k = 63 | 64) of every group."""
    N, groups = 16, 6
    K = 64 * groups
    codes = np.zeros((N, K // 2), np.uint8)
    for n in range(N):
        codes[n, :] = n | (n << 4)
    sv = [0.0078125, -0.5, 3.0, 2.0 ** -20, 96.0, 0.1015625]
    bv = [-0.0546875, 1.25, -6.0, 2.0 ** -18, 0.0, -1000.0]
    scales = np.tile(bf16_bits_of(sv), (N, 1))
    biases = np.tile(bf16_bits_of(bv), (N, 1))
    probes = []
    for gi in range(groups):
        probes += [64 * gi, 64 * gi + 63, 64 * gi + 17]
    x = np.zeros((len(probes), K), np.uint16)
    for m, k in enumerate(probes):
        x[m, k] = 0x3F80  # bf16 1.0
    y, a = oracle.linear_q4(x, codes, scales, biases, N)
    for m, k in enumerate(probes):
        gi = k // 64
        for n in range(N):
            assert y[m, n] == sv[gi] * n + bv[gi], (m, n)
            assert a[m, n] == abs(sv[gi] * n) + abs(bv[gi])


def test_q4_group_sum_closed_form():
    """x = 1 on one whole group: y = scale * (sum of the group's codes) + 64 * bias."""
    rng = np.random.default_rng(11)
    N, K = 8, 256
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = bf16_bits_of(np.ldexp(1.0, rng.integers(-8, 2, (N, K // 64))))
    biases = bf16_bits_of(rng.integers(-40, 40, (N, K // 64)) / 8.0)
    x = np.zeros((K // 64, K), np.uint16)
    for gi in range(K // 64):
        x[gi, 64 * gi:64 * gi + 64] = 0x3F80
    y = oracle.linear_q4(x, codes, scales, biases, N, with_abs=False)
    q = np.empty((N, K), np.int64)
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    for gi in range(K // 64):
        for n in range(N):
            s = bf16_vals_torch(scales[n, gi:gi + 1])[0]
            b = bf16_vals_torch(biases[n, gi:gi + 1])[0]
            assert y[gi, n] == s * q[n, 64 * gi:64 * gi + 64].sum() + 64 * b


def test_q4_matches_numpy_matmul_random():
    rng = np.random.default_rng(12)
    M, N, K = 6, 24, 320
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = rand_bf16(rng, (N, K // 64), 0.05)
    biases = rand_bf16(rng, (N, K // 64), 0.4)
    x = rand_bf16(rng, (M, K))
    y, a = oracle.linear_q4(x, codes, scales, biases, N)
    w, wa = dequant_q4_indep(codes, scales, biases)
    xv = bf16_vals_torch(x)
    np.testing.assert_allclose(y, xv @ w.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a, np.abs(xv) @ wa.T, rtol=1e-12, atol=1e-12)
    rows = np.array([23, 1, 9], np.int32)
    y2, a2 = oracle.linear_q4(x, codes, scales, biases, N, rows=rows)
    assert np.array_equal(y2, y[:, rows]) and np.array_equal(a2, a[:, rows])


def test_q4_nibble_order_low_first():
    """Element 2j is the low nibble: a code byte 0x50 (low 0, high 5) only reaches x[2j + 1]."""
    K = 64
    codes = np.zeros((1, K // 2), np.uint8)
    codes[0, 4] = 0x50
    scales = bf16_bits_of([[0.5]])
    biases = bf16_bits_of([[0.0]])
    x = np.zeros((2, K), np.uint16)
    x[0, 8] = 0x3F80
    x[1, 9] = 0x3F80
    y = oracle.linear_q4(x, codes, scales, biases, 1, with_abs=False)
    assert y[0, 0] == 0.0 and y[1, 0] == 2.5


def test_q4_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.linear_q4(np.zeros((1, 96), np.uint16), np.zeros((1, 48), np.uint8), np.zeros((1, 1), np.uint16),
                         np.zeros((1, 1), np.uint16), 1)


# ------------------------------------------------------------------ sampled acceptance

def test_target_dist_top_p_truncation_closed_form():
    """Probabilities 0.5 / 0.3 / 0.2 (+ a negligible fourth): top_k = 3, top_p = 0.7 keeps two and
    renormalises them to 0.625 / 0.375; top_p = 1 keeps all three."""
    lg = np.log(np.array([0.3, 0.5, 1e-12, 0.2]))
    tok, p, _ = oracle.target_dist(lg, 1.0, 3, 0.7)
    assert tok.tolist() == [1, 0] and np.allclose(p, [0.625, 0.375], rtol=1e-14)
    tok, p, mg = oracle.target_dist(lg, 1.0, 3, 1.0)
    assert tok.tolist() == [1, 0, 3] and np.allclose(p, [0.5, 0.3, 0.2], rtol=1e-14) and mg == np.inf


def test_target_dist_temperature_and_softmax():
    rng = np.random.default_rng(21)
    lg = rng.standard_normal(500) * 3
    for T, k in ((0.6, 20), (1.0, 32), (1.7, 5)):
        tok, p, _ = oracle.target_dist(lg, T, k, 1.0)
        order = np.lexsort((np.arange(lg.size), -lg))[:k]  # larger logit first, lower index among equals
        assert tok.tolist() == order.tolist()
        ref = torch.softmax(torch.tensor(lg[order] / T, dtype=torch.float64), 0).numpy()
        np.testing.assert_allclose(p, ref, rtol=1e-13)
        assert math.isclose(p[0] / p[1], math.exp((lg[order[0]] - lg[order[1]]) / T), rel_tol=1e-12)


def test_target_dist_ties_and_top1():
    lg = np.array([1.0, 3.0, 3.0, -2.0, 3.0])
    tok, p, _ = oracle.target_dist(lg, 1.0, 4, 1.0)
    assert tok.tolist() == [1, 2, 4, 0]
    tok, p, _ = oracle.target_dist(lg, 0.5, 1, 0.9)
    assert tok.tolist() == [oracle.argmax(lg)] and p.tolist() == [1.0]


def test_sample_accept_top1_point_mass_is_greedy_acceptance():
    """top_k = 1 with point-mass drafts is greedy decoding: the result equals the greedy acceptance
    rule on the rows' argmax, whatever the uniforms."""
    rng = np.random.default_rng(22)
    L, V = 6, 50
    lg = rng.standard_normal((8 * L, V))
    t = np.array([oracle.argmax(r) for r in lg], np.int32)
    pending = rng.integers(0, V, 8 * L).astype(np.int32)
    for l in range(L):  # planted prefixes of length l
        pending[8 * l + 1:8 * l + 1 + l] = t[8 * l:8 * l + l]
    u = rng.random((8 * L, 2))
    nc, cm, _ = oracle.sample_accept(lg, 0.8, 1, 1.0, pending, None, None, u)
    nc2, cm2 = oracle.accept(t, pending)
    assert np.array_equal(nc, nc2) and np.array_equal(cm, cm2)


@pytest.mark.parametrize("point_mass", [False, True])
def test_sample_accept_preserves_target_distribution(point_mass):
    """Speculative sampling leaves the committed token distributed as the target's: over a grid of
    the two uniforms and every draft token d (weighted by q(d)), the first committed token of a lane
    follows row 0's target distribution p, up to the grid's resolution."""
    V, G = 6, 160
    lg_row = np.log(np.array([0.05, 0.3, 0.1, 0.25, 0.2, 0.1]))
    p_tok, p_prob, _ = oracle.target_dist(lg_row, 1.0, 5, 0.95)  # token 0 falls outside top_k
    p_t = np.zeros(V)
    p_t[p_tok] = p_prob
    if point_mass:
        qs = {d: (1.0 if d == 3 else 0.0) for d in range(V)}
    else:
        qv = np.array([0.3, 0.1, 0.2, 0.15, 0.05, 0.2])
        qs = {d: qv[d] for d in range(V)}
    uu = (np.arange(G) + 0.5) / G
    U = np.stack(np.meshgrid(uu, uu, indexing="ij"), -1).reshape(-1, 2)  # (u0, u1) pairs
    L = U.shape[0]
    lg = np.tile(lg_row, (8 * L, 1))
    uni = np.zeros((8 * L, 2))
    uni[0::8] = U
    dist = np.zeros(V)
    for d, qd in qs.items():
        if qd == 0.0:
            continue
        pending = np.zeros(8 * L, np.int32)
        pending[1::8] = d
        if point_mass:
            dt = dp = None
        else:
            dt = np.tile(np.arange(16, dtype=np.int32), (8 * L, 1))
            dp = np.zeros((8 * L, 16))
            dp[:, :V] = np.array([qs[i] for i in range(V)])
        nc, cm, _ = oracle.sample_accept(lg, 1.0, 5, 0.95, pending, dt, dp, uni)
        first = cm[:, 0]
        dist += qd * np.bincount(first, minlength=V)[:V] / L
    np.testing.assert_allclose(dist, p_t, atol=3.0 / G)
    assert dist[0] == 0.0  # outside the target's candidates


def test_sample_accept_rejects_bad_arguments():
    lg = np.zeros((8, 10))
    pend = np.zeros(8, np.int32)
    u = np.zeros((8, 2))
    for T, k, p in ((0.0, 5, 1.0), (1.0, 33, 1.0), (1.0, 11, 1.0), (1.0, 5, 0.0)):
        with pytest.raises(ValueError):
            oracle.sample_accept(lg, T, k, p, pend, None, None, u)


# ------------------------------------------------------------------ verify attention

def attn_case(rng, L=1, Hq=6, Hkv=1, D=32, cap=40, ctx=None):
    M = 8 * L
    q = rand_bf16(rng, (M, Hq, D))
    kn = rand_bf16(rng, (M, Hkv, D))
    vn = rand_bf16(rng, (M, Hkv, D))
    kc = rand_bf16(rng, (L, Hkv, cap, D))
    vc = rand_bf16(rng, (L, Hkv, cap, D))
    gate = rand_bf16(rng, (M, Hq, D))
    ctx = np.array(ctx if ctx is not None else rng.integers(0, cap - 8, L), np.int32)
    return q, kn, vn, kc, vc, ctx, gate


def test_attention_matches_torch_sdpa():
    """Against torch's scaled_dot_product_attention (fp64) with the causal verify mask and the
    sigmoid gate applied afterwards."""
    rng = np.random.default_rng(31)
    L, Hq, Hkv, D, cap = 2, 6, 2, 32, 40
    q, kn, vn, kc, vc, ctx, gate = attn_case(rng, L, Hq, Hkv, D, cap, ctx=[13, 0])
    out, a = oracle.attention_verify(q, kn, vn, kc, vc, ctx, gate)
    f = lambda x: torch.from_numpy(bf16_vals_torch(x))  # noqa: E731
    for l in range(L):
        n = ctx[l] + 8
        K = torch.cat([f(kc[l][:, :ctx[l]]), f(kn[8 * l:8 * l + 8]).permute(1, 0, 2)], 1)  # [Hkv][n][D]
        Vv = torch.cat([f(vc[l][:, :ctx[l]]), f(vn[8 * l:8 * l + 8]).permute(1, 0, 2)], 1)
        Q = f(q[8 * l:8 * l + 8]).permute(1, 0, 2)  # [Hq][8][D]
        K = K.repeat_interleave(Hq // Hkv, 0)
        Vv = Vv.repeat_interleave(Hq // Hkv, 0)
        mask = torch.arange(n)[None, :] <= (ctx[l] + torch.arange(8))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, attn_mask=mask)
        o = o * torch.sigmoid(f(gate[8 * l:8 * l + 8]).permute(1, 0, 2))
        np.testing.assert_allclose(out[8 * l:8 * l + 8], o.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    assert np.all(a >= np.abs(out) - 1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(32)
    q, kn, vn, kc, vc, ctx, gate = attn_case(rng, ctx=[0])
    out = oracle.attention_verify(q, kn, vn, kc, vc, ctx, None, with_abs=False)
    # an empty cache: row 0 sees only its own key, so its output is its own value
    assert np.array_equal(out[0], np.repeat(bf16_vals_torch(vn[0]), 6, 0))
    # identical keys: uniform weights, the output is the mean of the visible values
    kn2 = np.tile(kn[:1], (8, 1, 1))
    out2 = oracle.attention_verify(q, kn2, vn, kc, vc, ctx, None, with_abs=False)
    vv = bf16_vals_torch(vn)[:, 0]
    for j in range(8):
        np.testing.assert_allclose(out2[j], np.tile(vv[:j + 1].mean(0), (6, 1)), rtol=1e-12, atol=1e-14)
    # a zero gate halves the output
    zero = np.zeros_like(gate)
    out3 = oracle.attention_verify(q, kn, vn, kc, vc, ctx, zero, with_abs=False)
    np.testing.assert_allclose(out3, out / 2, rtol=1e-15)


def test_attention_causal_and_grouped():
    rng = np.random.default_rng(33)
    q, kn, vn, kc, vc, ctx, gate = attn_case(rng, Hq=6, Hkv=2, ctx=[20])
    out = oracle.attention_verify(q, kn, vn, kc, vc, ctx, gate, with_abs=False)
    kn2, vn2 = kn.copy(), vn.copy()
    kn2[5:] ^= 0x0040  # perturb the keys / values of rows 5..7
    vn2[5:] ^= 0x0040
    out2 = oracle.attention_verify(q, kn2, vn2, kc, vc, ctx, gate, with_abs=False)
    assert np.array_equal(out[:5], out2[:5]) and not np.array_equal(out[5:], out2[5:])
    # heads 0..2 read kv head 0, heads 3..5 kv head 1: equal queries and gates give equal outputs
    q2, g2 = q.copy(), gate.copy()
    q2[:, 1], g2[:, 1] = q2[:, 0], g2[:, 0]
    q2[:, 4], g2[:, 4] = q2[:, 0], g2[:, 0]
    out3 = oracle.attention_verify(q2, kn, vn, kc, vc, ctx, g2, with_abs=False)
    assert np.array_equal(out3[:, 0], out3[:, 1]) and not np.array_equal(out3[:, 0], out3[:, 4])


# ------------------------------------------------------------------ Gated DeltaNet verify scan

def gdn_case(rng, L=1, H=2, d=16):
    M = 8 * L
    st = rng.standard_normal((L, H, d, d)) * 0.3
    q = rand_bf16(rng, (M, H, d))
    k = rand_bf16(rng, (M, H, d), 0.25)
    v = rand_bf16(rng, (M, H, d))
    a = rng.uniform(0.8, 1.0, (M, H))
    b = rng.uniform(0.0, 1.0, (M, H))
    return st, q, k, v, a, b


def test_gdn_matches_matrix_form_of_the_delta_rule():
    """Against the gated delta rule written as matrix products in torch:
    S_t = S_{t-1} alpha (I - beta k k^T) + beta v k^T, o_t = S_t q_t."""
    rng = np.random.default_rng(41)
    st, q, k, v, a, b = gdn_case(rng, L=2)
    rows = np.array([8, 5], np.int32)
    so, out = oracle.gdn_scan(st, q, k, v, a, b, rows)
    f = lambda x: torch.from_numpy(bf16_vals_torch(x))  # noqa: E731
    for l in range(2):
        for h in range(2):
            S = torch.from_numpy(st[l, h].copy())
            for j in range(rows[l]):
                r = 8 * l + j
                kv, vv, qv = f(k[r, h]), f(v[r, h]), f(q[r, h])
                eye = torch.eye(kv.numel(), dtype=torch.float64)
                S = S @ (a[r, h] * (eye - b[r, h] * torch.outer(kv, kv))) + b[r, h] * torch.outer(vv, kv)
                np.testing.assert_allclose(out[r, h], (S @ qv).numpy(), rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(so[l, h], S.numpy(), rtol=1e-11, atol=1e-12)


def test_gdn_closed_forms():
    rng = np.random.default_rng(42)
    st, q, k, v, a, b = gdn_case(rng)
    # no rows: the state passes through unchanged
    so, _ = oracle.gdn_scan(st, q, k, v, a, b, [0])
    assert np.array_equal(so, st)
    # beta = 0: pure decay by the product of the alphas
    so, _ = oracle.gdn_scan(st, q, k, v, a, np.zeros_like(b), [8])
    np.testing.assert_allclose(so[0], st[0] * np.prod(a, axis=0)[:, None, None], rtol=1e-13)
    # alpha = beta = 1 and k = e_c: the delta rule overwrites column c of S with v
    k1 = np.zeros_like(k)
    k1[:, :, 3] = 0x3F80  # bf16 1.0
    so, _ = oracle.gdn_scan(st, q, k1, v, np.ones_like(a), np.ones_like(b), [1])
    expect = st[0].copy()
    expect[:, :, 3] = bf16_vals_torch(v[0])
    np.testing.assert_allclose(so[0], expect, rtol=0, atol=1e-15)


def test_gdn_retrieves_the_written_value():
    """The delta rule's defining property: after one step with a unit-norm key k, the state maps k to
    (1 - beta) * alpha * S k + beta * v (with beta = 1 the memory returns exactly v for k), and the
    output for q = k is that vector.  The key (0.5 on four coordinates) has k^T k = 1 exactly."""
    rng = np.random.default_rng(44)
    st, q, k, v, a, b = gdn_case(rng)
    ku = np.zeros_like(k)
    ku[:, :, [1, 4, 9, 14]] = 0x3F00  # bf16 0.5
    kval = bf16_vals_torch(ku[0, 0])
    assert float(kval @ kval) == 1.0
    for beta in (b, np.ones_like(b)):
        so, out = oracle.gdn_scan(st, ku, ku, v, a, beta, [1])
        for h in range(st.shape[1]):
            want = (1 - beta[0, h]) * a[0, h] * (st[0, h] @ kval) + beta[0, h] * bf16_vals_torch(v[0, h])
            np.testing.assert_allclose(so[0, h] @ kval, want, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(out[0, h], want, rtol=1e-12, atol=1e-13)


def test_gdn_scan_composes_row_by_row():
    """The re-scan invariant: scanning n rows at once equals n one-row scans in sequence."""
    rng = np.random.default_rng(43)
    st, q, k, v, a, b = gdn_case(rng)
    for n in range(9):
        full, _ = oracle.gdn_scan(st, q, k, v, a, b, [n])
        cur = st
        for j in range(n):
            sh = lambda x: np.roll(x, -j, axis=0)  # noqa: E731  (row j first)
            cur, _ = oracle.gdn_scan(cur, sh(q), sh(k), sh(v), sh(a), sh(b), [1])
        np.testing.assert_array_equal(full, cur)


# ------------------------------------------------------------------ decode loop pieces

def test_lookup_drafts_worked_examples():
    """Hand-worked continuations: the longest earlier match of the history's suffix wins, the most
    recent among equals; the continuation is copied while it lasts, then its last token repeats; no
    match repeats the anchor."""
    cases = [
        ([5, 6, 7, 8, 5, 6], [6, 7, 8, 5, 6, 6, 6, 6]),
        ([1, 2, 9, 2, 3, 1, 2], [2, 9, 2, 3, 1, 2, 2, 2]),  # "1 2" (length 2) beats "2" at position 4
        ([4, 7, 4, 8, 4], [4, 8, 4, 4, 4, 4, 4, 4]),        # two length-1 matches: the later one
        ([1, 2, 3], [3, 3, 3, 3, 3, 3, 3, 3]),              # no earlier occurrence of 3
        ([9], [9] * 8),
    ]
    cap = 16
    hist = np.zeros((len(cases), cap), np.int32)
    hl = np.zeros(len(cases), np.int32)
    for i, (h, _) in enumerate(cases):
        hist[i, :len(h)] = h
        hl[i] = len(h)
    out = oracle.lookup_drafts(hist, hl).reshape(-1, 8)
    for i, (_, want) in enumerate(cases):
        assert out[i].tolist() == want, (i, out[i].tolist())


def test_lookup_drafts_match_cap():
    """With max_match = 1 only the last token is matched: the most recent earlier occurrence wins."""
    hist = np.array([[1, 2, 9, 2, 3, 1, 2, 0, 0, 0]], np.int32)
    out = oracle.lookup_drafts(hist, np.array([7], np.int32), max_match=1)
    assert out.tolist() == [2, 3, 1, 2, 2, 2, 2, 2]


def test_embed_nvfp4_is_the_rounded_table_row():
    """Row t of the table equals column t of the NVFP4 linear with one-hot activations, rounded once
    to bf16 (by the single-rounding conversion pinned above)."""
    rng = np.random.default_rng(51)
    V, K = 40, 256
    codes = rng.integers(0, 256, (V, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, (V, K // 16), dtype=np.uint8)
    toks = np.array([0, 39, 7, 7, 21], np.int32)
    ts = 0.6
    emb = oracle.embed_nvfp4(codes, scales, ts, toks)
    x = np.zeros((K, K), np.uint16)
    x[np.arange(K), np.arange(K)] = 0x3F80
    w = oracle.linear(oracle.NVFP4, x, codes, scales, ts, V, with_abs=False)  # w[k][t] = W[t][k]
    # (values compared, -0 == +0: code 8 is E2M1's -0, which the row keeps and a sum does not)
    assert np.array_equal(oracle.bf16_value(emb), oracle.bf16_value(oracle.bf16_round(w[:, toks].T.copy())))
    # with ts = 1 every product is exact in bf16 (<= 5 significant bits): torch's conversion agrees
    emb1 = oracle.embed_nvfp4(codes, scales, 1.0, toks)
    w1 = oracle.linear(oracle.NVFP4, x, codes, scales, 1.0, V, with_abs=False)
    ref1 = torch.from_numpy(w1[:, toks].T.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_value(emb1), oracle.bf16_value(ref1))


def test_commit_append_and_full_history():
    hist = np.zeros((2, 10), np.int32)
    hl = np.array([3, 8], np.int32)
    hist[0, :3] = [1, 2, 3]
    nc = np.array([2, 3], np.int32)
    cm = np.array([[7, 8, -1, -1, -1, -1, -1, -1], [4, 5, 6, -1, -1, -1, -1, -1]], np.int32)
    assert oracle.commit_append(hist, hl, nc, cm) == -1  # lane 1 would overflow: left as it was
    assert hist[0, :5].tolist() == [1, 2, 3, 7, 8] and hl.tolist() == [5, 8]


# ------------------------------------------------------------------ wider verify (R rows per lane)
# "mlx-dspark" -- "Lookup drafts": deep lookup matches verify 16-32 rows; the acceptance rule is the
# same longest prefix over R - 1 drafts.

@pytest.mark.parametrize("R", [1, 2, 3, 4, 5])
def test_accept_rows_brute_force_binary_vocab(R):
    """Every target pattern (R tokens) x every draft pattern (R - 1 tokens) over V = 2, against the
    definition: 1 + the length of the longest common prefix of the drafts and the first R - 1
    targets, the committed row the targets up to it and -1 after."""
    tp = np.array(list(itertools.product([0, 1], repeat=R)), np.int32)
    drafts = list(itertools.product([0, 1], repeat=R - 1))
    dp = np.array(drafts, np.int32).reshape(len(drafts), R - 1)
    T = np.repeat(tp, len(dp), axis=0)
    D = np.tile(dp, (len(tp), 1))
    pending = np.concatenate([np.full((T.shape[0], 1), 7, np.int32), D], axis=1)
    nc, cm = oracle.accept(T.reshape(-1), pending.reshape(-1), rows=R)
    for i in range(T.shape[0]):
        lcp = next((j for j in range(R - 1) if T[i, j] != D[i, j]), R - 1)
        assert nc[i] == lcp + 1
        assert cm[i].tolist() == [int(T[i, j]) if j <= lcp else -1 for j in range(R)]
    assert nc.min() == 1 and nc.max() == R


@pytest.mark.parametrize("R", [16, 32])
def test_accept_rows_planted_prefixes(R):
    """Random targets with every prefix length 0 .. R - 1 planted once per lane (the draft after the
    prefix differs): n_commit is the planted length + 1; R = 8 equals the 8-row function."""
    rng = np.random.default_rng(R)
    L = R
    T = rng.integers(0, 1000, (L, R)).astype(np.int32)
    D = rng.integers(0, 1000, (L, R - 1)).astype(np.int32)
    for l in range(L):
        n = l % R
        D[l, :n] = T[l, :n]
        if n < R - 1:
            D[l, n] = (T[l, n] + 1) % 1000
    pending = np.concatenate([np.zeros((L, 1), np.int32), D], axis=1)
    nc, cm = oracle.accept(T.reshape(-1), pending.reshape(-1), rows=R)
    assert nc.tolist() == [l % R + 1 for l in range(L)]
    T8 = T[:, :8].copy()
    P8 = pending[:, :8].copy()
    assert [np.array_equal(a, b) for a, b in zip(oracle.accept(T8.reshape(-1), P8.reshape(-1), rows=8),
                                                   oracle.accept(T8.reshape(-1), P8.reshape(-1)))] == [True, True]


def test_lookup_drafts_rows_worked_examples():
    """16-row lookups of the worked examples above: the continuation copied while it lasts, then its
    last token repeated to fill 15 drafts; the first 8 entries equal the 8-row lookup."""
    cases = [
        ([5, 6, 7, 8, 5, 6], [6, 7, 8, 5, 6] + [6] * 11),
        ([1, 2, 9, 2, 3, 1, 2], [2, 9, 2, 3, 1, 2] + [2] * 10),
        ([1, 2, 3], [3] * 16),
    ]
    cap = 16
    hist = np.zeros((len(cases), cap), np.int32)
    hl = np.zeros(len(cases), np.int32)
    for i, (h, _) in enumerate(cases):
        hist[i, :len(h)] = h
        hl[i] = len(h)
    out = oracle.lookup_drafts(hist, hl, rows=16).reshape(-1, 16)
    out8 = oracle.lookup_drafts(hist, hl).reshape(-1, 8)
    for i, (_, want) in enumerate(cases):
        assert out[i].tolist() == want, (i, out[i].tolist())
        assert out[i, :8].tolist() == out8[i].tolist()


def test_commit_append_rows():
    hist = np.zeros((2, 40), np.int32)
    hl = np.array([2, 0], np.int32)
    hist[0, :2] = [9, 9]
    cm = np.full((2, 16), -1, np.int32)
    cm[0, :11] = np.arange(11)
    cm[1, :1] = [42]
    assert oracle.commit_append(hist, hl, np.array([11, 1], np.int32), cm) == 0
    assert hist[0, :13].tolist() == [9, 9] + list(range(11)) and hist[1, :1].tolist() == [42]
    assert hl.tolist() == [13, 1]

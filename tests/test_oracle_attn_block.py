"""Pins of the gated-attention mixer-block oracle (oracle/attn_layer.py): RoPE against its complex
form and its relative-position property, the per-head RMSNorm against torch, and the whole block
against an independent torch composition (scaled_dot_product_attention for the core)."""
import numpy as np
import torch
import torch.nn.functional as F

import synth
from oracle import attn_layer as al

G = {"hidden": 256, "Hq": 4, "Hkv": 2, "D": 16}


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_rope_is_a_complex_rotation_and_relative():
    rng = np.random.default_rng(80)
    x = rng.standard_normal((5, 3, 16))
    pos = np.array([0.0, 1.0, 7.0, 100.0, 32775.0])
    y = al.rope(x, pos)
    # pairs as complex numbers times exp(i pos theta_i)
    zc = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * pos[:, None, None] * 10000.0 ** (-np.arange(0, 16, 2) / 16))
    np.testing.assert_allclose(y[..., 0::2], zc.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[..., 1::2], zc.imag, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(al.rope(x[:1], np.zeros(1)), x[:1])  # position 0: identity
    # the score of rotated q and k depends only on the position difference
    q, k = rng.standard_normal((1, 1, 16)), rng.standard_normal((1, 1, 16))
    s1 = (al.rope(q, np.array([10.0])) * al.rope(k, np.array([3.0]))).sum()
    s2 = (al.rope(q, np.array([1007.0])) * al.rope(k, np.array([1000.0]))).sum()
    np.testing.assert_allclose(s1, s2, rtol=1e-9)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)


def test_head_rmsnorm_matches_torch():
    rng = np.random.default_rng(81)
    x, w = rng.standard_normal((8, 4, 16)) * 5, rng.uniform(0.5, 1.5, 16)
    ref = F.rms_norm(torch.from_numpy(x), (16,), weight=torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(al.head_rmsnorm(x, w), ref, rtol=1e-13)


def case(seed=82, L=2, cap=40):
    rng = np.random.default_rng(seed)
    H, Hq, Hkv, D = G["hidden"], G["Hq"], G["Hkv"], G["D"]
    w = {"q": synth.fp8_matrix(seed, 3, synth.T_IN, 2 * Hq * D, H), "s_q": 0.05,
         "kv": synth.fp8_matrix(seed, 3, synth.T_KV, 2 * Hkv * D, H), "s_kv": 0.05,
         "o": synth.fp8_matrix(seed, 3, synth.T_OUT, H, Hq * D), "s_o": 0.05,
         "q_norm": rng.uniform(0.5, 1.5, D), "k_norm": rng.uniform(0.5, 1.5, D)}
    h = synth.normal_bf16(seed, synth.stream_id(3, synth.T_X0), (8 * L, H))
    kc = bf16_bits(rng.standard_normal((L, Hkv, cap, D)))
    vc = bf16_bits(rng.standard_normal((L, Hkv, cap, D)))
    ctx = np.array([0, 17][:L], np.int32)
    return h, w, kc, vc, ctx


def torch_block(h, w, kc, vc, ctx):
    H, Hq, Hkv, D = G["hidden"], G["Hq"], G["Hkv"], G["D"]
    M = h.shape[0]
    bf = lambda x: x.to(torch.bfloat16).double()  # noqa: E731
    fp8 = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).double()  # noqa: E731
    hv = torch.from_numpy(bf16_vals(h))
    r = bf(hv / torch.sqrt((hv * hv).mean(-1, keepdim=True) + 1e-6))
    qg = bf(r @ (fp8(w["q"]) * w["s_q"]).T)
    kv = bf(r @ (fp8(w["kv"]) * w["s_kv"]).T)
    q, gate = qg[:, :Hq * D].reshape(M, Hq, D), qg[:, Hq * D:].reshape(M, Hq, D)
    k, v = kv[:, :Hkv * D].reshape(M, Hkv, D), kv[:, Hkv * D:].reshape(M, Hkv, D)

    def rot(x, pos):  # RoPE through complex multiplication
        xc = torch.complex(x[..., 0::2], x[..., 1::2])
        th = 10000.0 ** (-torch.arange(0, D, 2, dtype=torch.float64) / D)
        yc = xc * torch.polar(torch.ones_like(th), pos[:, None, None] * th)
        return torch.stack([yc.real, yc.imag], dim=-1).reshape(x.shape)
    pos = torch.tensor([float(ctx[r // 8] + r % 8) for r in range(M)], dtype=torch.float64)
    qn = bf(rot(F.rms_norm(q, (D,), weight=torch.from_numpy(w["q_norm"]), eps=1e-6), pos))
    kn = bf(rot(F.rms_norm(k, (D,), weight=torch.from_numpy(w["k_norm"]), eps=1e-6), pos))
    out = torch.zeros(M, Hq, D, dtype=torch.float64)
    for l in range(M // 8):
        c = int(ctx[l])
        K = torch.cat([torch.from_numpy(bf16_vals(kc[l, :, :c])), kn[8 * l:8 * l + 8].transpose(0, 1)], dim=1)
        Vv = torch.cat([torch.from_numpy(bf16_vals(vc[l, :, :c])), bf(v[8 * l:8 * l + 8]).transpose(0, 1)], dim=1)
        K, Vv = K.repeat_interleave(Hq // Hkv, dim=0), Vv.repeat_interleave(Hq // Hkv, dim=0)
        mask = torch.arange(c + 8)[None, :] <= (c + torch.arange(8))[:, None]
        o = F.scaled_dot_product_attention(qn[8 * l:8 * l + 8].transpose(0, 1), K, Vv, attn_mask=mask)
        out[8 * l:8 * l + 8] = o.transpose(0, 1) * torch.sigmoid(gate[8 * l:8 * l + 8])
    y = bf(out.reshape(M, Hq * D)) @ (fp8(w["o"]) * w["s_o"]).T
    return bf(hv + y).numpy()


def test_block_matches_independent_torch_composition():
    h, w, kc, vc, ctx = case()
    h_new, (kb, vb), _ = al.attn_block(h, G, w, kc, vc, ctx)
    ref = torch_block(h, w, kc, vc, ctx)
    got = bf16_vals(h_new)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-30)  # one bf16 ulp at most
    assert np.mean(got == ref) > 0.97
    assert kb.shape == (16, 2, 16) and vb.shape == (16, 2, 16)

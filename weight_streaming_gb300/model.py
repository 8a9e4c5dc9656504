"""Device-resident packed weights and the verify-pass model handle.

Canonical weights (NVFP4 codes [N][K/2] + E4M3 scales [N][K/16], or FP8 E4M3 [N][K]) are packed on
the device by vp_pack_nvfp4 / vp_pack_fp8 into the layout the kernels stream, then described to
vp_model_create.  `SyntheticModel` fills the canonical tensors with the seeded synthetic recipe
(synth) directly in HBM, one tensor at a time, so a full 17.6 GB pass fits next to a single
canonical scratch tensor.
"""
from __future__ import annotations

import torch

from . import _lib as V
from .geometry import Geometry  # noqa: F401  (re-exported)


def pack_nvfp4(codes: torch.Tensor, scales: torch.Tensor, stream=None) -> torch.Tensor:
    N, K2 = codes.shape
    K = 2 * K2
    out = torch.empty(V.vp_packed_bytes_nvfp4(N, K), dtype=torch.uint8, device=codes.device)
    V.vp_pack_nvfp4(codes, scales, N, K, out, stream)
    return out


def pack_fp8(w: torch.Tensor, stream=None) -> torch.Tensor:
    N, K = w.shape
    out = torch.empty(V.vp_packed_bytes_fp8(N, K), dtype=torch.uint8, device=w.device)
    V.vp_pack_fp8(w, N, K, out, stream)
    return out


class SyntheticModel:
    """A verify-pass model whose weights come from the seeded synthetic recipe:
    NVFP4 code bytes uniform, E4M3 block scales 2^U(-6,0), FP8 weights E4M3(N(0,1)); tensor scales
    are drawn uniformly in [0.5, 1.5] (``unit_scales=True`` sets them all to 1)."""

    def __init__(self, geom: Geometry, seed: int = 0, device="cuda", unit_scales: bool = True):
        import numpy as np

        import synth
        self.geom, self.seed = geom, seed
        H, I = geom.hidden, geom.inter
        rng = np.random.default_rng(seed + 12345)
        self.scales = []
        self.packed = []
        layers = []

        def sc():
            return 1.0 if unit_scales else float(rng.uniform(0.5, 1.5))

        def fp8(l, t, N, K):
            w = torch.empty((N, K), dtype=torch.uint8, device=device)
            synth.gpu_fp8_normal_codes(w, seed, synth.stream_id(l, t))
            p = pack_fp8(w)
            del w
            self.packed.append(p)
            return p

        def nvfp4(l, tc, ts, N, K):
            c = torch.empty((N, K // 2), dtype=torch.uint8, device=device)
            s = torch.empty((N, K // 16), dtype=torch.uint8, device=device)
            synth.gpu_uniform_bytes(c, seed, synth.stream_id(l, tc))
            synth.gpu_scale_codes(s, seed, synth.stream_id(l, ts))
            p = pack_nvfp4(c, s)
            del c, s
            self.packed.append(p)
            return p

        for l in range(geom.n_layers):
            attn = geom.is_attn(l)
            d = V.vp_layer_desc()
            d.kind = V.VP_LAYER_ATTN if attn else V.VP_LAYER_GDN
            n_in = geom.attn_q if attn else geom.gdn_in
            kz = geom.attn_z if attn else geom.gdn_z
            d.w_in = fp8(l, synth.T_IN, n_in, H).data_ptr()
            d.s_in, d.n_in = sc(), n_in
            if attn:
                d.w_kv = fp8(l, synth.T_KV, geom.attn_kv, H).data_ptr()
                d.s_kv, d.n_kv = sc(), geom.attn_kv
            else:
                d.w_kv, d.s_kv, d.n_kv = None, 1.0, 0
            d.w_out = fp8(l, synth.T_OUT, H, kz).data_ptr()
            d.s_out, d.k_out = sc(), kz
            d.w_gate = nvfp4(l, synth.T_GATE_C, synth.T_GATE_S, I, H).data_ptr()
            d.ts_gate = sc()
            d.w_up = nvfp4(l, synth.T_UP_C, synth.T_UP_S, I, H).data_ptr()
            d.ts_up = sc()
            d.w_down = nvfp4(l, synth.T_DOWN_C, synth.T_DOWN_S, H, I).data_ptr()
            d.ts_down = sc()
            self.scales.append(dict(s_in=d.s_in, s_kv=d.s_kv, s_out=d.s_out, ts_gate=d.ts_gate, ts_up=d.ts_up,
                                    ts_down=d.ts_down))
            layers.append(d)
        hp = nvfp4(synth.HEAD_LAYER, synth.T_HEAD_C, synth.T_HEAD_S, geom.vocab, H)
        self.head_ts = sc()
        head = V.vp_head_desc(hp.data_ptr(), self.head_ts, geom.vocab)
        torch.cuda.synchronize()
        self.model = V.vp_model(H, I, geom.eps, layers, head)

    def attach_cores(self, lanes: int, cap: int, seed: int = 7):
        """Attaches the real mixer cores with synthetic parameters and state, all drawn on the device
        from one seeded generator: A and B ~ N(0,1)/sqrt(hidden) (bf16), convolution taps U(-0.6, 0.6),
        A_log U(-2, 0), dt_bias U(-1, 1), the norm weights U(0.5, 1.5), delta-rule states 0.1 N(0,1),
        convolution windows and cached keys / values N(0,1).  Caches hold `cap` positions per lane."""
        g = self.geom
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        H, C = g.hidden, (2 * g.n_qk + g.n_v) * g.d
        self.core_tensors = []

        def keep(t):
            self.core_tensors.append(t)
            return t.data_ptr()

        def normal(shape, std=1.0, dtype=torch.bfloat16):
            return (torch.randn(shape, generator=gen, device="cuda") * std).to(dtype)

        def uniform(shape, lo, hi, dtype=torch.float32):
            return (torch.rand(shape, generator=gen, device="cuda") * (hi - lo) + lo).to(dtype)

        descs = []
        for l in range(g.n_layers):
            c = V.vp_core_desc()
            if g.is_attn(l):
                c.q_norm = keep(uniform(g.D, 0.5, 1.5))
                c.k_norm = keep(uniform(g.D, 0.5, 1.5))
                c.k_cache = keep(normal((lanes, g.Hkv, cap, g.D)))
                c.v_cache = keep(normal((lanes, g.Hkv, cap, g.D)))
            else:
                c.w_a = keep(normal((g.n_v, H), H ** -0.5))
                c.w_b = keep(normal((g.n_v, H), H ** -0.5))
                c.conv_taps = keep(uniform((C, 4), -0.6, 0.6, torch.bfloat16))
                c.a_log = keep(uniform(g.n_v, -2.0, 0.0))
                c.dt_bias = keep(uniform(g.n_v, -1.0, 1.0))
                c.norm_w = keep(uniform(g.d, 0.5, 1.5))
                c.state_a = keep(normal((lanes, g.n_v, g.d, g.d), 0.1, torch.float32))
                c.state_b = keep(torch.zeros((lanes, g.n_v, g.d, g.d), device="cuda"))
                c.window_a = keep(normal((lanes, 3, C)))
                c.conv_hist = keep(torch.zeros((lanes, 11, C), dtype=torch.bfloat16, device="cuda"))
            descs.append(c)
        torch.cuda.synchronize()
        V.vp_model_set_cores(self.model, V.vp_core_geom(g.n_qk, g.n_v, g.d, g.Hq, g.Hkv, g.D, cap), descs)

    def cores_workspace(self, M: int) -> torch.Tensor:
        return torch.zeros(V.vp_pass_cores_workspace_bytes(self.model, M), dtype=torch.uint8, device="cuda")

    def run_cores(self, x0, ctx, pending, argmax, n_commit, committed, ws, parity=0, trace=None, logits=None,
                  stream=None):
        M = x0.shape[0]
        V.vp_verify_pass_cores(self.model, x0, M, ctx, parity, pending, argmax, n_commit, committed, trace, logits,
                               ws, stream)

    def commit_cores(self, M, n_commit, parity, ws, stream=None):
        V.vp_commit_cores(self.model, M, n_commit, parity, ws, stream)

    def workspace(self, M: int) -> torch.Tensor:
        n = V.vp_pass_workspace_bytes(self.model, M)
        return torch.zeros(n, dtype=torch.uint8, device="cuda")

    def launch_count(self) -> int:
        return V.vp_pass_launch_count(self.model)

    def run(self, x0, pending, argmax, n_commit, committed, ws, trace=None, logits=None, stream=None):
        M = x0.shape[0]
        V.vp_verify_pass(self.model, x0, M, pending, argmax, n_commit, committed, trace, logits, ws, stream)

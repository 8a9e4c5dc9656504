"""Shape constants of the verify pass: the 64-layer hybrid target's projection widths, the attention
period and the per-pass weight bytes.  Plain Python with no library import, so that code which only
needs the shapes (the oracle arm of the bench, tests on the CPU) never loads libverify.so.

Source: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "What one token costs
the bus" (the NVFP4 / FP8 weight groups and their bytes); "144 tok/s needs 502 GB/s" -- "The engine
hard-codes the model" (hidden 5120, intermediate 17408, vocabulary 248320, every fourth layer full
attention).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass
class Geometry:
    n_layers: int = 64
    hidden: int = 5120
    inter: int = 17408
    vocab: int = 248320
    period: int = 4          # every `period`-th layer (index % period == period - 1) is attention
    gdn_in: int = 16384
    gdn_z: int = 6144
    attn_q: int = 12288
    attn_kv: int = 2048
    attn_z: int = 6144
    eps: float = 1e-6
    # the mixer cores: Gated DeltaNet q/k heads, v heads and head width; attention query and
    # key-value heads and head width (gdn_in = (2 n_qk + 2 n_v) d, attn_q = 2 Hq D, attn_kv = 2 Hkv D)
    n_qk: int = 16
    n_v: int = 48
    d: int = 128
    Hq: int = 24
    Hkv: int = 4
    D: int = 256

    def is_attn(self, l: int) -> bool:
        return (l % self.period) == self.period - 1

    def pass_bytes(self) -> int:
        H, I = self.hidden, self.inter
        b = 0
        for l in range(self.n_layers):
            if self.is_attn(l):
                b += self.attn_q * H + self.attn_kv * H + H * self.attn_z
            else:
                b += self.gdn_in * H + H * self.gdn_z
            b += (2 * I * H + H * I) * 9 // 16
        b += self.vocab * H * 9 // 16
        return b

    def kv_bytes(self, ctx: int) -> int:
        """Bytes of the key and value cache rows one lane's attention cores read at context ctx (the
        cached rows and the 8 new ones), over all attention layers."""
        n_attn = sum(self.is_attn(l) for l in range(self.n_layers))
        return n_attn * 2 * self.Hkv * (ctx + 8) * self.D * 2

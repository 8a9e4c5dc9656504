"""GPU parity of the verify attention over a BF16 KV cache (vp_attention_verify) against the fp64
oracle, through the C ABI: one and several 1,024-key partitions, the pages' 24 / 4 head geometry,
ragged context lengths per lane, a group of 8 heads, the cache append, an out-of-range length
reported through the status word, bit-reproducibility, and values across bf16's whole range."""
import numpy as np
import pytest
import torch

import oracle
from helpers import workspace

pytestmark = pytest.mark.gpu

D = 256


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


def bf16(rng, shape, scale=1.0):
    t = torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def case(seed, L, Hq, Hkv, cap, ctx, gate=True):
    rng = np.random.default_rng(seed)
    M = 8 * L
    return dict(q=bf16(rng, (M, Hq, D)), kn=bf16(rng, (M, Hkv, D)), vn=bf16(rng, (M, Hkv, D)),
                kc=bf16(rng, (L, Hkv, cap, D)), vc=bf16(rng, (L, Hkv, cap, D)),
                gate=bf16(rng, (M, Hq, D)) if gate else None, ctx=np.array(ctx, np.int32))


def run(V, c, ws=None):
    M, Hq = c["q"].shape[:2]
    L, Hkv, cap = c["kc"].shape[:3]
    kc, vc = dev(c["kc"]), dev(c["vc"])
    out = torch.empty((M, Hq, D), dtype=torch.int16, device="cuda")
    if ws is None:
        ws = workspace(V.vp_workspace_bytes(V.VP_OP_ATTN, M, Hkv, cap))
    V.vp_attention_verify(dev(c["q"]), dev(c["kn"]), dev(c["vn"]), kc, vc, torch.from_numpy(c["ctx"]).cuda(), cap,
                          dev(c["gate"]) if c["gate"] is not None else None, out, M, Hq, Hkv, D, ws)
    torch.cuda.synchronize()
    st = V.vp_read_status(ws)
    return out.cpu().numpy().view(np.uint16), kc.cpu().numpy().view(np.uint16), vc.cpu().numpy().view(np.uint16), st


def assert_close(out_bits, ref, a, what):
    got = torch.from_numpy(out_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    bound = 2e-3 * a + 2.0 ** -8 * np.abs(ref) + 1e-6  # the tolerance plus the output's bf16 rounding
    bad = ~(np.abs(got - ref) <= bound)
    assert not bad.any(), (what, int(bad.sum()), np.argwhere(bad)[:3].tolist())


@pytest.mark.parametrize("L,Hq,Hkv,cap,ctx", [
    (1, 6, 1, 64, [0]),              # empty cache: the rows see only themselves
    (1, 6, 1, 200, [37]),            # one partition, a ragged last tile
    (2, 24, 4, 3072, [1000, 2100]),  # the pages' heads; one and three partitions
    (1, 8, 1, 2056, [2048]),         # a group of 8 heads; the verify rows start a new partition
    (4, 24, 4, 1300, [0, 5, 1023, 1292]),
])
def test_attention_matches_oracle(V, L, Hq, Hkv, cap, ctx):
    c = case(sum(ctx) + Hq + L, L, Hq, Hkv, cap, ctx)
    out, kc, vc, st = run(V, c)
    assert st == V.VP_OK
    ref, a = oracle.attention_verify(c["q"], c["kn"], c["vn"], c["kc"], c["vc"], c["ctx"], c["gate"])
    assert_close(out, ref, a, f"attention L={L} Hq={Hq} ctx={ctx}")
    for l in range(L):  # the verify rows were appended; nothing else in the cache changed
        n = ctx[l]
        assert np.array_equal(kc[l][:, n:n + 8], c["kn"][8 * l:8 * l + 8].transpose(1, 0, 2))
        assert np.array_equal(vc[l][:, n:n + 8], c["vn"][8 * l:8 * l + 8].transpose(1, 0, 2))
        assert np.array_equal(kc[l][:, :n], c["kc"][l][:, :n]) and np.array_equal(kc[l][:, n + 8:], c["kc"][l][:, n + 8:])


def test_attention_without_gate_and_deterministic(V):
    c = case(5, 2, 24, 4, 2600, [2500, 7], gate=False)
    out1, _, _, _ = run(V, c)
    out2, _, _, _ = run(V, c)
    assert np.array_equal(out1, out2)
    ref, a = oracle.attention_verify(c["q"], c["kn"], c["vn"], c["kc"], c["vc"], c["ctx"], None)
    assert_close(out1, ref, a, "no gate")


def test_attention_out_of_range_context_is_reported(V):
    """A lane whose 8 new positions do not fit the cache is skipped by the kernels' own check: zero
    output for it, the other lane computed, VP_ERR_SHAPE in the status word."""
    c = case(6, 2, 6, 1, 100, [95, 10])
    out, kc, _, st = run(V, c)
    assert st == V.VP_ERR_SHAPE
    assert np.all(out[:8] == 0)
    assert np.array_equal(kc[0], c["kc"][0])  # nothing written for the bad lane
    ref, a = oracle.attention_verify(c["q"][8:], c["kn"][8:], c["vn"][8:], c["kc"][1:], c["vc"][1:], c["ctx"][1:],
                                     c["gate"][8:])
    assert_close(out[8:], ref, a, "good lane")


def test_attention_values_over_bf16_range(V):
    """The cache is BF16: values far outside half precision's range (up to ~1e30 here, half's
    largest finite is 65504) and tiny ones (~1e-30, below half's smallest subnormal) must pass
    through the weighted sum exactly as bf16 holds them.  Each key-value head's values get their own
    scale; queries and keys stay N(0,1) so the softmax weights are ordinary."""
    c = case(11, 2, 24, 4, 1100, [1000, 37])
    for name in ("vn", "vc"):
        x = torch.from_numpy(c[name].view(np.int16)).view(torch.bfloat16).double()
        axis = 1  # the key-value head axis: [M][Hkv][D] and [L][Hkv][cap][D]
        scale = torch.tensor([1e30, 1e6, 1e-30, 3.0], dtype=torch.float64)
        shape = [1] * x.dim()
        shape[axis] = 4
        c[name] = (x * scale.view(shape)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out, _, _, st = run(V, c)
    assert st == V.VP_OK
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.all(np.isfinite(got))
    ref, a = oracle.attention_verify(c["q"], c["kn"], c["vn"], c["kc"], c["vc"], c["ctx"], c["gate"])
    assert_close(out, ref, a, "values over the bf16 range")

"""GPU parity of the verify pass at the pages' own shapes (hidden 5120, intermediate 17408, Gated
DeltaNet in 16384 / z 6144, attention q 12288 / kv 2048 / z 6144, vocabulary 248320), through the
C ABI, at every width the bench times.

At these shapes the executor takes paths that the small-geometry tests never reach: K-sliced
phases (the interleaved gate + up cut into K slices at 2+ token tiles), RMSNorm staging that takes
its row statistic from the producer's row-block sums of squares, and a head in which each warp
folds several row blocks into its running argmax.

* Blocks: a 2-layer model (one Gated DeltaNet layer, one attention layer) runs all four blocks in
  one vp_verify_blocks call with the trace on, so that every phase after the first reads what the
  previous phase produced (row-block sums included).  Each block's output is checked against the
  oracle's block computed from the device's own input to that block, within the block's budget.
* Head: vp_head_argmax_accept over the full 248320 x 5120 NVFP4 head, logits against the fp64
  oracle element by element, argmax bit-exact against the oracle's argmax of the device's own
  logits, and against the oracle's fp64 argmax where that is unique; acceptance bit-exact.
* Pass: the bench's 64-layer synthetic model at M = 8 (vp_verify_pass with trace and logits):
  internal consistency, the first, a middle and the last two blocks teacher-forced from the
  device's own trace, and the head from the device's last residual.

Sources: "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "Formats, and what
runs where" (NVFP4 / FP8 numerics, BF16 activations, fp32 accumulation) and "The megakernel is per
layer, not per step" (greedy acceptance); "Beating Splash on an M5 Max" -- "The bugs a second
reviewer found" (one argmax tie rule)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import ABS, REL, dev_bf16, dev_i32, dev_u8, host_bf16_bits, workspace
from passutil import DeviceModel, make_head, make_layer, mixer_block_ref, mlp_block_ref

pytestmark = pytest.mark.gpu

PAGES = dict(hidden=5120, inter=17408, gdn_in=16384, gdn_z=6144, attn_q=12288, attn_kv=2048, attn_z=6144)


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


@pytest.fixture(scope="module")
def two_layers(V):
    """Layer 0 Gated DeltaNet, layer 1 attention, at the pages' widths; per-tensor scales != 1."""
    G = oracle.geom(n_layers=2, vocab=2064, period=2, **PAGES)
    layers = [make_layer(G, 31, 0, (0.75, 1.0, 1.25, 0.625, 1.125, 0.875)),
              make_layer(G, 31, 1, (1.25, 0.5, 0.875, 1.0625, 0.75, 1.375))]
    head = make_head(G, 31, 0.5)
    dm = DeviceModel(V, G, layers, head)
    return G, layers, head, dm


def check_block(G, layers, b, h_in, got, what):
    d = layers[b // 2]
    h_ref, budget = (mixer_block_ref if b % 2 == 0 else mlp_block_ref)(G, d, h_in)
    err = np.abs(oracle.bf16_value(got) - oracle.bf16_value(h_ref))
    bad = ~(err <= budget)
    assert not bad.any(), f"{what} block {b}: {int(bad.sum())} of {bad.size} outside budget, max err/budget " \
                          f"{float(np.max(err / budget)):.3g}"


@pytest.mark.parametrize("M", [1, 8, 13, 16, 24, 32])
def test_blocks_at_page_shapes_chain(V, two_layers, M):
    G, layers, head, dm = two_layers
    x0 = synth.normal_bf16(40 + M, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    h = dev_bf16(x0)
    trace = torch.empty((4, M, G.hidden), dtype=torch.bfloat16, device="cuda")
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    V.vp_verify_blocks(dm.model, h, M, 0, 4, trace, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    tr = host_bf16_bits(trace)
    assert np.array_equal(tr[-1], host_bf16_bits(h))
    h_in = x0
    for b in range(4):
        check_block(G, layers, b, h_in, tr[b], f"M={M}")
        h_in = tr[b]


@pytest.fixture(scope="module")
def full_head(V):
    G = oracle.geom(n_layers=1, vocab=248320, **PAGES)
    hc, hs, _ = make_head(G, 0)
    packed = torch.empty(V.vp_packed_bytes_nvfp4(G.vocab, G.hidden), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(dev_u8(hc), dev_u8(hs), G.vocab, G.hidden, packed)
    torch.cuda.synchronize()
    return G, hc, hs, packed


def check_head(ref, a, pending, am, nc, cm, lg, rel=REL):
    """Device head results (argmax, n_commit, committed, fp32 logits) against the oracle's fp64 logits
    `ref` and their scale a = sum |x w|.  rel: the tolerance per unit of a (REL for an exact bf16
    input; REL plus one bf16 ulp when the device rounded the head input itself)."""
    M = ref.shape[0]
    err = np.abs(lg.astype(np.float64) - ref)
    bad = ~(err <= rel * a + ABS)
    assert not bad.any(), f"head logits: {int(bad.sum())} of {bad.size} outside tolerance"
    # bit-exact on the same logits: the lowest index among the largest values of each device row
    for m in range(M):
        assert am[m] == oracle.argmax(lg[m].astype(np.float64)), m
    # against the fp64 logits wherever the oracle's winner is unique within the tolerance
    tol = rel * a + ABS
    top = np.argmax(ref, axis=1)
    lead = ref[np.arange(M), top][:, None] - ref
    lead[np.arange(M), top] = np.inf
    clear = np.all(lead > 2 * (tol + tol[np.arange(M), top][:, None]), axis=1)
    assert np.array_equal(am[clear], top[clear])
    # elsewhere the device's choice must be a valid one: within both tolerances of the exact maximum
    rows = np.arange(M)
    assert np.all(ref[rows, am] >= ref[rows, top] - (tol[rows, am] + tol[rows, top]))
    # acceptance: bit-exact given the device's argmax, and equal to the oracle's where every row is clear
    nc_o, cm_o = oracle.accept(am, pending)
    assert np.array_equal(nc, nc_o) and np.array_equal(cm, cm_o)
    nc_r, _ = oracle.accept(top.astype(np.int32), pending)
    lanes_clear = clear.reshape(-1, 8).all(axis=1)
    assert np.array_equal(nc[lanes_clear], nc_r[lanes_clear])
    return top


@pytest.mark.parametrize("M", [8, 32])
def test_full_head_against_oracle(V, full_head, M):
    G, hc, hs, packed = full_head
    ts = 0.8125
    x = synth.normal_bf16(60 + M, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    ref, a = oracle.linear(oracle.NVFP4, x, hc, hs, ts, G.vocab)
    pending, _ = synth.planted_pending(M, np.argmax(ref, axis=1), G.vocab)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_HEAD, M, G.vocab, G.hidden))
    V.vp_head_argmax_accept(packed, ts, dev_bf16(x), M, G.vocab, G.hidden, dev_i32(pending), am, nc, cm, lg, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    check_head(ref, a, pending, am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy(), lg.cpu().numpy())


def test_full_pass_m8_teacher_forced(V):
    """The bench's 64-layer model at M = 8: the device's own trace, block by block, against the
    oracle's blocks from the same inputs, and the fused head against the oracle from the device's
    last residual."""
    from weight_streaming_gb300.geometry import Geometry
    from weight_streaming_gb300.model import SyntheticModel
    geom = Geometry()
    G = oracle.geom()
    M = 8
    sm = SyntheticModel(geom, seed=0)
    x0 = synth.normal_bf16(0, synth.stream_id(0, synth.T_X0), (M, geom.hidden))
    t = synth.uniform_ints(0, synth.stream_id(0, synth.T_PENDING) + 7, 0, M, geom.vocab)
    pending, _ = synth.planted_pending(0, t, geom.vocab)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(1, dtype=torch.int32, device="cuda")
    cm = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    lg = torch.empty((M, geom.vocab), dtype=torch.float32, device="cuda")
    trace = torch.empty((2 * geom.n_layers, M, geom.hidden), dtype=torch.bfloat16, device="cuda")
    ws = sm.workspace(M)
    sm.run(dev_bf16(x0), dev_i32(pending), am, nc, cm, ws, trace=trace, logits=lg)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    tr = host_bf16_bits(trace)
    del sm
    torch.cuda.empty_cache()
    lay = [None] * G.n_layers
    for b in (0, 1, 63, 126, 127):
        if lay[b // 2] is None:
            lay[b // 2] = make_layer(G, 0, b // 2)
        check_block(G, lay, b, x0 if b == 0 else tr[b - 1], tr[b], "64-layer pass")
    hc, hs, ts = make_head(G, 0)
    ref, a = oracle.linear(oracle.NVFP4, oracle.rmsnorm(tr[-1], G.eps), hc, hs, ts, G.vocab)
    # the device rounds RMSNorm(h) to bf16 itself: one ulp may flip per element (2^-7 of |r w|)
    check_head(ref, a, pending, am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy(), lg.cpu().numpy(),
               rel=REL + 2.0 ** -7)

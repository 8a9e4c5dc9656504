"""GPU parity of the verify pass (vp_verify_blocks / vp_verify_pass) against the oracle.

Per block: the device runs one block from the oracle's own input to that block (the oracle's trace),
and its output must lie within the block's error budget (passutil).  End to end: the device pass and
the oracle pass start from the same x0; over several layers near-equal bf16 roundings may go either
way, so the end-to-end check is on what is unique: clear-margin argmax rows, the device's internal
consistency (argmax of its own logits, acceptance of its own argmax) and a bounded drift."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_bf16, dev_i32, host_bf16_bits, workspace
from passutil import DeviceModel, make_layers, mixer_block_ref, mlp_block_ref

pytestmark = pytest.mark.gpu

SMALL = dict(n_layers=4, hidden=256, inter=512, vocab=2064, period=4, gdn_in=512, gdn_z=384, attn_q=384, attn_kv=128,
             attn_z=256)


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


@pytest.fixture(scope="module")
def small(V):
    G = oracle.geom(**SMALL)
    layers, head = make_layers(G, seed=21)
    dm = DeviceModel(V, G, layers, head)
    return G, layers, head, dm


def run_blocks(V, dm, h_bits, b0, b1):
    M = h_bits.shape[0]
    h = dev_bf16(h_bits)
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    V.vp_verify_blocks(dm.model, h, M, b0, b1, None, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    return host_bf16_bits(h)


@pytest.mark.parametrize("M", [8, 32])
def test_each_block_matches_oracle_from_oracle_input(V, small, M):
    G, layers, head, dm = small
    x0 = synth.normal_bf16(5, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    ref = oracle.verify_pass(G, layers, head, x0, np.zeros(M, np.int32), want_trace=True)
    h_in = x0
    for b in range(2 * G.n_layers):
        d = layers[b // 2]
        h_ref, budget = (mixer_block_ref if b % 2 == 0 else mlp_block_ref)(G, d, h_in)
        assert np.array_equal(h_ref, ref["trace"][b])  # the block reference is the oracle's own chain
        got = oracle.bf16_value(run_blocks(V, dm, h_in, b, b + 1))
        err = np.abs(got - oracle.bf16_value(h_ref))
        bad = ~(err <= budget)
        assert not bad.any(), f"block {b}: {int(bad.sum())} elements outside budget, max err/budget " \
                              f"{float(np.max(err / budget)):.3g}"
        h_in = ref["trace"][b]


def test_blocks_compose_into_the_pass(V, small):
    """vp_verify_blocks over all blocks leaves the same residual stream as vp_verify_pass's trace."""
    G, layers, head, dm = small
    M = 16
    x0 = synth.normal_bf16(6, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    h_all = run_blocks(V, dm, x0, 0, 2 * G.n_layers)
    trace = torch.empty((2 * G.n_layers, M, G.hidden), dtype=torch.bfloat16, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    V.vp_verify_pass(dm.model, dev_bf16(x0), M, dev_i32(np.zeros(M, np.int32)), am, nc, cm, trace, None, ws)
    torch.cuda.synchronize()
    assert np.array_equal(host_bf16_bits(trace[-1]), h_all)


@pytest.mark.parametrize("M", [8, 16, 24, 32])
def test_pass_end_to_end(V, small, M):
    G, layers, head, dm = small
    x0 = synth.normal_bf16(7 + M, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    ref0 = oracle.verify_pass(G, layers, head, x0, np.zeros(M, np.int32), want_logits=True)
    pending, _ = synth.planted_pending(M, ref0["argmax"], G.vocab)
    ref = oracle.verify_pass(G, layers, head, x0, pending, want_trace=True, want_logits=True)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    trace = torch.empty((2 * G.n_layers, M, G.hidden), dtype=torch.bfloat16, device="cuda")
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    V.vp_verify_pass(dm.model, dev_bf16(x0), M, dev_i32(pending), am, nc, cm, trace, lg, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    am, nc, cm, lg = am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy(), lg.cpu().numpy()
    # device consistency: argmax of its own logits; acceptance of its own argmax
    assert np.array_equal(am, np.argmax(lg, axis=1))
    for l in range(M // 8):
        acc = 0
        while acc < 7 and am[8 * l + acc] == pending[8 * l + acc + 1]:
            acc += 1
        assert nc[l] == acc + 1
        assert list(cm[l]) == [int(am[8 * l + j]) if j <= acc else -1 for j in range(8)]
    # drift of the residual stream stays small
    tr = oracle.bf16_value(host_bf16_bits(trace))
    rt = oracle.bf16_value(ref["trace"])
    rel = np.abs(tr - rt).max(axis=2) / np.sqrt((rt ** 2).mean(axis=2))
    assert rel.max() < 0.05, rel.max()
    # rows whose exact top-1 leads clearly must agree
    rl = ref["logits"]
    srt = np.sort(rl, axis=1)
    clear = (srt[:, -1] - srt[:, -2]) > 0.02 * np.abs(rl).max(axis=1)
    assert np.array_equal(am[clear], ref["argmax"][clear])
    assert clear.mean() > 0.5
    lanes_clear = clear.reshape(-1, 8).all(axis=1)
    assert np.array_equal(nc[lanes_clear], ref["n_commit"][lanes_clear])


def test_pass_is_deterministic_and_graph_capturable(V, small):
    G, layers, head, dm = small
    M = 8
    x0 = dev_bf16(synth.normal_bf16(8, synth.stream_id(0, synth.T_X0), (M, G.hidden)))
    pend = dev_i32(np.zeros(M, np.int32))
    outs = []
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(1, dtype=torch.int32, device="cuda")
    cm = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    for _ in range(2):
        V.vp_verify_pass(dm.model, x0, M, pend, am, nc, cm, None, lg, ws)
        torch.cuda.synchronize()
        outs.append((am.clone(), lg.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    lg.zero_()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            V.vp_verify_pass(dm.model, x0, M, pend, am, nc, cm, None, lg, ws, stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(am, outs[0][0]) and torch.equal(lg, outs[0][1])

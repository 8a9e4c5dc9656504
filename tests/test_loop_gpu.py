"""GPU parity of the device-resident decode loop's pieces against the oracle (embedding gather, lookup
drafts, history append: bit for bit) and of vp_decode_steps, which runs rounds with no host in the
loop, against the same rounds driven from the host one call at a time (the same GPU pass, the
oracle's lookup and append on the host): identical histories; the loop also replays from a CUDA
graph."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_u8, workspace
from passutil import DeviceModel, make_layers

pytestmark = pytest.mark.gpu

SMALL = dict(n_layers=4, hidden=256, inter=512, vocab=2064, period=4, gdn_in=512, gdn_z=384, attn_q=384, attn_kv=128,
             attn_z=256)


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def test_embed_matches_oracle(V):
    Vv, K = 2064, 5120
    codes, scales = synth.nvfp4_matrix(3, 900, synth.T_HEAD_C, synth.T_HEAD_S, Vv, K)
    toks = np.array([0, 2063, 17, 17, 1024, 5, 6, 7], np.int32)
    for ts in (1.0, 0.6875, 1.3):
        x = torch.empty((8, K), dtype=torch.int16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        V.vp_embed_nvfp4(dev_u8(codes), dev_u8(scales), ts, i32(toks), 8, Vv, K, x, st)
        torch.cuda.synchronize()
        ref = oracle.embed_nvfp4(codes, scales, float(np.float32(ts)), toks)
        assert np.array_equal(x.cpu().numpy().view(np.uint16), ref), ts
        assert st.item() == 0
    bad = toks.copy()
    bad[3] = Vv
    V.vp_embed_nvfp4(dev_u8(codes), dev_u8(scales), 1.0, i32(bad), 8, Vv, K, x, st)
    torch.cuda.synchronize()
    assert st.item() == V.VP_ERR_SHAPE and np.all(x.cpu().numpy()[3] == 0)


def test_lookup_and_append_match_oracle(V):
    rng = np.random.default_rng(61)
    L, cap = 4, 3000
    hist = np.zeros((L, cap), np.int32)
    hl = np.array([1, 40, 1500, 2991], np.int32)
    for l in range(L):  # repetitive text: a small alphabet with copied spans
        base = rng.integers(0, 50, hl[l])
        for s0 in range(0, hl[l] - 20, 97):
            base[s0 + 10:s0 + 20] = base[s0:s0 + 10]
        hist[l, :hl[l]] = base
    for mm in (1, 4, 8):
        pend = torch.empty(8 * L, dtype=torch.int32, device="cuda")
        V.vp_lookup_drafts(i32(hist), i32(hl), L, cap, mm, pend)
        torch.cuda.synchronize()
        assert np.array_equal(pend.cpu().numpy(), oracle.lookup_drafts(hist, hl, mm)), mm
    nc = np.array([3, 8, 1, 10], np.int32)
    nc[3] = 8  # lane 3: 2991 + 8 > 2998? no: cap 3000 -> overflow at +10 only; keep 8 = fits
    cm = rng.integers(0, 50, (L, 8)).astype(np.int32)
    h_d, hl_d, st = i32(hist), i32(hl), torch.zeros(1, dtype=torch.int32, device="cuda")
    V.vp_commit_append(h_d, hl_d, L, cap, i32(nc), i32(cm), st)
    torch.cuda.synchronize()
    h2, hl2 = hist.copy(), hl.copy()
    assert oracle.commit_append(h2, hl2, nc, cm) == 0
    assert np.array_equal(h_d.cpu().numpy(), h2) and np.array_equal(hl_d.cpu().numpy(), hl2) and st.item() == 0
    V.vp_commit_append(h_d, hl_d, L, cap, i32(nc), i32(cm), st)  # lane 3 is now full
    torch.cuda.synchronize()
    assert st.item() == V.VP_ERR_SHAPE and hl_d.cpu().numpy()[3] == hl2[3]


@pytest.fixture(scope="module")
def loop_model(V):
    G = oracle.geom(**SMALL)
    layers, head = make_layers(G, seed=31)
    dm = DeviceModel(V, G, layers, head)
    ec, es = synth.nvfp4_matrix(31, 901, synth.T_HEAD_C, synth.T_HEAD_S, G.vocab, G.hidden)
    return G, dm, ec, es


@pytest.mark.parametrize("lanes", [1, 4])
def test_decode_steps_equal_host_driven_rounds(V, loop_model, lanes):
    G, dm, ec, es = loop_model
    M, cap, steps, mm, ts = 8 * lanes, 400, 4, 8, 0.5
    rng = np.random.default_rng(62 + lanes)
    hist = np.zeros((lanes, cap), np.int32)
    hl = np.full(lanes, 60, np.int32)
    for l in range(lanes):
        base = rng.integers(0, 30, 60)
        base[30:60] = base[0:30]  # a copied span so that lookup finds continuations
        hist[l, :60] = base
    ecd, esd = dev_u8(ec), dev_u8(es)
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    x0 = torch.empty((M, G.hidden), dtype=torch.int16, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(lanes, dtype=torch.int32, device="cuda")
    cm = torch.empty((lanes, 8), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    # host-driven: the GPU embeds and verifies; the host looks up and appends (oracle)
    h_h, hl_h = hist.copy(), hl.copy()
    for _ in range(steps):
        pend = oracle.lookup_drafts(h_h, hl_h, mm)
        V.vp_embed_nvfp4(ecd, esd, ts, i32(pend), M, G.vocab, G.hidden, x0, st)
        V.vp_verify_pass(dm.model, x0, M, i32(pend), am, nc, cm, None, None, ws)
        torch.cuda.synchronize()
        assert oracle.commit_append(h_h, hl_h, nc.cpu().numpy(), cm.cpu().numpy()) == 0

    # device-resident: one call, every round on the device
    h_d, hl_d = i32(hist), i32(hl)
    pend_d = torch.empty(M, dtype=torch.int32, device="cuda")
    V.vp_lookup_drafts(h_d, hl_d, lanes, cap, mm, pend_d, st)
    V.vp_decode_steps(dm.model, steps, ecd, esd, ts, G.vocab, G.hidden, h_d, hl_d, cap, lanes, mm, pend_d, x0, am,
                      nc, cm, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(hl_d.cpu().numpy(), hl_h) and np.array_equal(h_d.cpu().numpy(), h_h)
    assert np.all(hl_h >= 60 + steps)  # every round commits at least one token

    # the same rounds captured in a CUDA graph and replayed from the initial state
    h_g, hl_g = i32(hist), i32(hl)
    pend_g = torch.empty(M, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            V.vp_lookup_drafts(h_g, hl_g, lanes, cap, mm, pend_g, st)
            V.vp_decode_steps(dm.model, steps, ecd, esd, ts, G.vocab, G.hidden, h_g, hl_g, cap, lanes, mm, pend_g,
                              x0, am, nc, cm, ws, st)
        h_g.copy_(i32(hist))
        hl_g.copy_(i32(hl))
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(h_g.cpu().numpy(), h_h) and np.array_equal(hl_g.cpu().numpy(), hl_h)

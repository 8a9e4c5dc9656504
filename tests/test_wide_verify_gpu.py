"""The wider verify through the C ABI: R verify rows per lane (anchor + R - 1 drafts; 1 lane of 16 or
32 rows, 2 lanes of 16, 8 lanes of 4; above 32 rows, runs of 32: 2 lanes of 32, 8 of 16), for the deep
lookup drafts of "Speculative decoding" (mlx-dspark), section "Lookup drafts" (drafts grow to 32
tokens, 16-32 rows verified in one pass).

- vp_argmax_accept_rows over given logits: argmax and acceptance bit-exact against the oracle's
  lowest-index argmax and its R-row acceptance, with every prefix length planted;
- vp_verify_pass_rows on a small model: the same logits and argmax as the 8-row pass at the same M
  (bit for bit), the acceptance equal to the oracle's over those tokens (drafts planted from them, so
  long prefixes are accepted);
- vp_lookup_drafts_rows / vp_commit_append_rows bit for bit against the oracle;
- vp_decode_steps_rows equal to the same rounds driven from the host."""
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


def planted(t, rows, rng, vocab):
    """Drafts per lane of `rows` rows: lane l copies the first (rows - 1 - 5 l) mod rows targets (lane 0
    all of them), then differs."""
    M = t.size
    pend = rng.integers(0, vocab, M).astype(np.int32)
    for l in range(M // rows):
        n = (rows - 1 - 5 * l) % rows
        base = rows * l
        pend[base + 1:base + 1 + n] = t[base:base + n]
        if n < rows - 1:
            pend[base + 1 + n] = (t[base + n] + 1) % vocab
    return pend


@pytest.mark.parametrize("M,rows", [(32, 32), (32, 16), (16, 16), (32, 4), (24, 8), (64, 32), (128, 16)])
def test_argmax_accept_rows_matches_oracle(V, M, rows):
    rng = np.random.default_rng(M + rows)
    Vv = 5003
    lg = rng.standard_normal((M, Vv)).astype(np.float32)
    lg[3, 17] = lg[3, 4000] = 50.0  # a tie: the lower index wins
    t = np.array([oracle.argmax(r) for r in lg], np.int32)
    pend = planted(t, rows, rng, Vv)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // rows, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // rows, rows), dtype=torch.int32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_ARGMAX, min(M, 32), Vv, 0))
    V.vp_argmax_accept_rows(torch.from_numpy(lg).cuda(), M, Vv, rows, i32(pend), am, nc, cm, ws)
    torch.cuda.synchronize()
    assert np.array_equal(am.cpu().numpy(), t)
    nc_o, cm_o = oracle.accept(t, pend, rows=rows)
    assert np.array_equal(nc.cpu().numpy(), nc_o) and np.array_equal(cm.cpu().numpy(), cm_o)


@pytest.fixture(scope="module")
def small_model(V):
    G = oracle.geom(**SMALL)
    layers, head = make_layers(G, seed=41)
    dm = DeviceModel(V, G, layers, head)
    ec, es = synth.nvfp4_matrix(41, 901, synth.T_HEAD_C, synth.T_HEAD_S, G.vocab, G.hidden)
    return G, dm, ec, es


@pytest.mark.parametrize("M,rows", [(32, 32), (32, 16), (16, 16), (32, 4)])
def test_verify_pass_rows(V, small_model, M, rows):
    G, dm, _, _ = small_model
    rng = np.random.default_rng(100 + M + rows)
    x0 = torch.from_numpy(synth.normal_bf16(7 + M, synth.stream_id(0, synth.T_X0), (M, G.hidden)).view(np.int16)).cuda()
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    lg8 = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    am8 = torch.empty(M, dtype=torch.int32, device="cuda")
    nc8 = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm8 = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    V.vp_verify_pass(dm.model, x0, M, i32(np.zeros(M, np.int32)), am8, nc8, cm8, None, lg8, ws)
    torch.cuda.synchronize()
    t = am8.cpu().numpy()
    pend = planted(t, rows, rng, G.vocab)
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // rows, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // rows, rows), dtype=torch.int32, device="cuda")
    V.vp_verify_pass_rows(dm.model, x0, M, rows, i32(pend), am, nc, cm, None, lg, ws)
    torch.cuda.synchronize()
    assert torch.equal(lg, lg8) and np.array_equal(am.cpu().numpy(), t)
    nc_o, cm_o = oracle.accept(t, pend, rows=rows)
    assert np.array_equal(nc.cpu().numpy(), nc_o) and np.array_equal(cm.cpu().numpy(), cm_o)
    assert nc_o.max() > 8 or rows <= 8  # a lane commits more tokens than an 8-row verify can


@pytest.mark.parametrize("M,rows", [(64, 32), (128, 16), (96, 8)])
def test_verify_pass_rows_beyond_32_rows(V, small_model, M, rows):
    """Above 32 rows the call runs passes of 32 rows: logits and argmax equal to 8-row passes over the
    same 32-row slices, the acceptance equal to the oracle's over all lanes."""
    G, dm, _, _ = small_model
    rng = np.random.default_rng(200 + M + rows)
    x0 = torch.from_numpy(synth.normal_bf16(9 + M, synth.stream_id(0, synth.T_X0), (M, G.hidden)).view(np.int16)).cuda()
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    assert V.vp_pass_workspace_bytes(dm.model, M) == V.vp_pass_workspace_bytes(dm.model, 32)
    lg8 = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    am8 = torch.empty(M, dtype=torch.int32, device="cuda")
    nc8 = torch.empty(4, dtype=torch.int32, device="cuda")
    cm8 = torch.empty((4, 8), dtype=torch.int32, device="cuda")
    z = i32(np.zeros(32, np.int32))
    for r0 in range(0, M, 32):
        V.vp_verify_pass(dm.model, x0[r0:r0 + 32], 32, z, am8[r0:r0 + 32], nc8, cm8, None, lg8[r0:r0 + 32], ws)
    torch.cuda.synchronize()
    t = am8.cpu().numpy()
    pend = planted(t, rows, rng, G.vocab)
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // rows, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // rows, rows), dtype=torch.int32, device="cuda")
    V.vp_verify_pass_rows(dm.model, x0, M, rows, i32(pend), am, nc, cm, None, lg, ws)
    torch.cuda.synchronize()
    assert torch.equal(lg, lg8) and np.array_equal(am.cpu().numpy(), t)
    nc_o, cm_o = oracle.accept(t, pend, rows=rows)
    assert np.array_equal(nc.cpu().numpy(), nc_o) and np.array_equal(cm.cpu().numpy(), cm_o)


def test_lookup_and_append_rows_match_oracle(V):
    rng = np.random.default_rng(71)
    for L, rows in ((1, 32), (2, 16), (4, 8), (8, 4), (4, 32), (16, 8), (32, 4)):
        cap = 900
        hist = np.zeros((L, cap), np.int32)
        hl = rng.integers(1, 800, L).astype(np.int32)
        for l in range(L):
            base = rng.integers(0, 40, hl[l])
            for s0 in range(0, hl[l] - 40, 83):
                base[s0 + 20:s0 + 40] = base[s0:s0 + 20]
            hist[l, :hl[l]] = base
        for mm in (1, 8):
            pend = torch.empty(rows * L, dtype=torch.int32, device="cuda")
            V.vp_lookup_drafts_rows(i32(hist), i32(hl), L, rows, cap, mm, pend)
            torch.cuda.synchronize()
            assert np.array_equal(pend.cpu().numpy(), oracle.lookup_drafts(hist, hl, mm, rows=rows)), (L, rows, mm)
        nc = rng.integers(1, rows + 1, L).astype(np.int32)
        cm = rng.integers(0, 40, (L, rows)).astype(np.int32)
        h_d, hl_d, st = i32(hist), i32(hl), torch.zeros(1, dtype=torch.int32, device="cuda")
        V.vp_commit_append_rows(h_d, hl_d, L, rows, cap, i32(nc), i32(cm), st)
        torch.cuda.synchronize()
        h2, hl2 = hist.copy(), hl.copy()
        assert oracle.commit_append(h2, hl2, nc, cm) == 0
        assert np.array_equal(h_d.cpu().numpy(), h2) and np.array_equal(hl_d.cpu().numpy(), hl2) and st.item() == 0


@pytest.mark.parametrize("lanes,rows", [(1, 32), (2, 16), (2, 32), (8, 16)])
def test_decode_steps_rows_equal_host_driven_rounds(V, small_model, lanes, rows):
    G, dm, ec, es = small_model
    M, cap, steps, mm, ts = rows * lanes, 600, 3, 8, 0.5
    rng = np.random.default_rng(90 + rows)
    hist = np.zeros((lanes, cap), np.int32)
    hl = np.full(lanes, 80, np.int32)
    for l in range(lanes):
        base = rng.integers(0, 30, 80)
        base[40:80] = base[0:40]
        hist[l, :80] = base
    ecd, esd = dev_u8(ec), dev_u8(es)
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    x0 = torch.empty((M, G.hidden), dtype=torch.int16, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(lanes, dtype=torch.int32, device="cuda")
    cm = torch.empty((lanes, rows), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    h_h, hl_h = hist.copy(), hl.copy()
    for _ in range(steps):
        pend = oracle.lookup_drafts(h_h, hl_h, mm, rows=rows)
        V.vp_embed_nvfp4(ecd, esd, ts, i32(pend), M, G.vocab, G.hidden, x0, st)
        V.vp_verify_pass_rows(dm.model, x0, M, rows, i32(pend), am, nc, cm, None, None, ws)
        torch.cuda.synchronize()
        assert oracle.commit_append(h_h, hl_h, nc.cpu().numpy(), cm.cpu().numpy()) == 0
    h_d, hl_d = i32(hist), i32(hl)
    pend_d = torch.empty(M, dtype=torch.int32, device="cuda")
    V.vp_lookup_drafts_rows(h_d, hl_d, lanes, rows, cap, mm, pend_d, st)
    V.vp_decode_steps_rows(dm.model, steps, rows, ecd, esd, ts, G.vocab, G.hidden, h_d, hl_d, cap, lanes, mm, pend_d,
                           x0, am, nc, cm, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(hl_d.cpu().numpy(), hl_h) and np.array_equal(h_d.cpu().numpy(), h_h)
    assert np.all(hl_h >= 80 + steps)

"""The verify pass with sampled acceptance (vp_verify_pass_sampled) through the C ABI: its logits and
argmax are those of the greedy pass bit for bit, and its acceptance is the oracle's sampled
acceptance over those logits -- exactly on every lane whose decisions clear the rounding margin,
valid on the rest; with top_k = 1 and point-mass drafts it is the greedy acceptance.

Sources: "144 tok/s needs 502 GB/s" (Splash) -- "Exact, up to top-32" (speculative sampling over
the top-32 target candidates); "Beating Splash on an M5 Max" -- "What actually moved the needle"
(one GPU kernel over the verify logits samples and accepts)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import dev_bf16, dev_i32, workspace
from passutil import DeviceModel, make_layers

pytestmark = pytest.mark.gpu

SMALL = dict(n_layers=4, hidden=256, inter=512, vocab=2064, period=4, gdn_in=512, gdn_z=384, attn_q=384, attn_kv=128,
             attn_z=256)
MARGIN = 1e-4  # fp32 against fp64 on probabilities of order one


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


@pytest.fixture(scope="module")
def small(V):
    G = oracle.geom(**SMALL)
    layers, head = make_layers(G, seed=29)
    return G, DeviceModel(V, G, layers, head)


def greedy(V, dm, G, x0, pending):
    M = x0.shape[0]
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))
    V.vp_verify_pass(dm.model, dev_bf16(x0), M, dev_i32(pending), am, nc, cm, None, lg, ws)
    torch.cuda.synchronize()
    return am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy(), lg.cpu().numpy()


def sampled(V, dm, G, x0, pending, T, k, p, dt, dp, u, want_logits=True):
    M = x0.shape[0]
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.full((M // 8,), -7, dtype=torch.int32, device="cuda")
    cm = torch.full((M // 8, 8), -7, dtype=torch.int32, device="cuda")
    lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda") if want_logits else None
    ws = workspace(V.vp_pass_sampled_workspace_bytes(dm.model, M))
    V.vp_verify_pass_sampled(dm.model, dev_bf16(x0), M, dev_i32(pending), T, k, p,
                             dev_i32(dt) if dt is not None else None,
                             torch.from_numpy(dp).cuda() if dp is not None else None,
                             torch.from_numpy(u).cuda(), am, nc, cm, lg, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    return am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy(), lg.cpu().numpy() if want_logits else None


def drafts_from(lg, seed):
    """Drafts and their 16-candidate distributions built around each row's leading candidates, so that
    acceptance is often possible: row r's draft (pending[r + 1]) is one of its 4 largest logits."""
    rng = np.random.default_rng(seed)
    M, Vv = lg.shape
    pending = rng.integers(0, Vv, M).astype(np.int32)
    dt = np.zeros((M, 16), np.int32)
    dp = np.zeros((M, 16), np.float32)
    for r in range(M):
        if r % 8 == 7:
            continue
        top = np.argsort(-lg[r], kind="stable")[:10]
        cands = np.concatenate([top, rng.integers(0, Vv, 6)])
        dt[r] = cands
        dp[r] = rng.dirichlet(np.ones(16)).astype(np.float32)
        pending[r + 1] = cands[rng.integers(0, 4)]
    return pending, dt, dp


@pytest.mark.parametrize("M,T,k,p", [(8, 1.0, 20, 0.95), (32, 0.7, 32, 0.9), (16, 0.05, 8, 1.0)])
def test_sampled_pass_matches_oracle_over_its_logits(V, small, M, T, k, p):
    G, dm = small
    x0 = synth.normal_bf16(70 + M, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    _, _, _, lg0 = greedy(V, dm, G, x0, np.zeros(M, np.int32))
    pending, dt, dp = drafts_from(lg0, M)
    am_g, _, _, lg_g = greedy(V, dm, G, x0, pending)
    u = np.random.default_rng(M + 1).random((M, 2)).astype(np.float32)
    am, nc, cm, lg = sampled(V, dm, G, x0, pending, T, k, p, dt, dp, u)
    assert np.array_equal(lg, lg_g) and np.array_equal(am, am_g)  # the same pass, the same bits
    nc_r, cm_r, mg = oracle.sample_accept(lg.astype(np.float64), T, k, p, pending, dt, dp.astype(np.float64),
                                          u.astype(np.float64))
    clear = mg > MARGIN
    assert clear.any()
    assert np.array_equal(nc[clear], nc_r[clear]) and np.array_equal(cm[clear], cm_r[clear])
    for l in range(M // 8):  # every lane: a valid result
        assert 1 <= nc[l] <= 8
        a = nc[l] - 1
        assert np.array_equal(cm[l, :a], pending[8 * l + 1:8 * l + 1 + a])
        assert 0 <= cm[l, a] < G.vocab and np.all(cm[l, a + 1:] == -1)


def test_sampled_pass_top1_point_mass_is_greedy(V, small):
    """top_k = 1 makes the target a point mass on the argmax; point-mass drafts are accepted exactly
    when they equal it: the greedy rule, bit for bit (logits not requested: they stay in the workspace)."""
    G, dm = small
    M = 24
    x0 = synth.normal_bf16(91, synth.stream_id(0, synth.T_X0), (M, G.hidden))
    am0, _, _, _ = greedy(V, dm, G, x0, np.zeros(M, np.int32))
    pending, _ = synth.planted_pending(91, am0, G.vocab)
    am_g, nc_g, cm_g, _ = greedy(V, dm, G, x0, pending)
    u = np.random.default_rng(5).random((M, 2)).astype(np.float32)
    am, nc, cm, _ = sampled(V, dm, G, x0, pending, 1.0, 1, 1.0, None, None, u, want_logits=False)
    assert np.array_equal(am, am_g) and np.array_equal(nc, nc_g) and np.array_equal(cm, cm_g)

"""GPU parity of the sampled acceptance over verify logits (vp_sample_accept) against the fp64 oracle,
through the C ABI.  Decisions are compared exactly on every lane whose decisions clear the rounding
margin (the oracle reports, per lane, the smallest distance of an acceptance test, a draw or a top_p
cut to its boundary); lanes inside the margin are checked for validity only."""
import numpy as np
import pytest
import torch

import oracle
from helpers import dev_i32, workspace

pytestmark = pytest.mark.gpu

MARGIN = 1e-4  # fp32 against fp64 on probabilities of order one


@pytest.fixture(scope="module")
def V_():
    from weight_streaming_gb300 import _lib
    return _lib


def make_case(seed, M, V, n_boost=12):
    """Logits with a few dominant tokens per row (so that drafts are often accepted) and drafts
    taken from those tokens, with draft distributions over 16 candidates that include the draft."""
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((M, V)).astype(np.float32)
    boost = np.zeros((M, n_boost), np.int64)
    for r in range(M):
        boost[r] = rng.choice(V, n_boost, replace=False)
        lg[r, boost[r]] += rng.uniform(4.0, 9.0, n_boost).astype(np.float32)
    pending = rng.integers(0, V, M).astype(np.int32)
    dt = np.zeros((M, 16), np.int32)
    dp = np.zeros((M, 16), np.float32)
    for r in range(M):
        if r % 8 == 7:
            continue
        cands = np.concatenate([boost[r][:10], rng.integers(0, V, 6)])
        w = rng.dirichlet(np.ones(16)).astype(np.float32)
        dt[r] = cands
        dp[r] = w
        pending[r + 1] = cands[rng.integers(0, 4)]  # the draft checked at row r
    u = rng.random((M, 2)).astype(np.float32)
    return lg, pending, dt, dp, u


def run_gpu(V_, lg, T, k, p, pending, dt, dp, u):
    M, V = lg.shape
    nc = torch.full((M // 8,), -7, dtype=torch.int32, device="cuda")
    cm = torch.full((M // 8, 8), -7, dtype=torch.int32, device="cuda")
    ws = workspace(V_.vp_workspace_bytes(V_.VP_OP_SAMPLE, M, V, 0))
    dtd = dev_i32(dt) if dt is not None else None
    dpd = torch.from_numpy(dp).cuda() if dp is not None else None
    V_.vp_sample_accept(torch.from_numpy(lg).cuda(), M, V, T, k, p, dev_i32(pending), dtd, dpd,
                        torch.from_numpy(u).cuda(), nc, cm, ws)
    torch.cuda.synchronize()
    return nc.cpu().numpy(), cm.cpu().numpy()


def check(V_, lg, T, k, p, pending, dt, dp, u):
    """Runs both sides; returns the number of lanes compared exactly."""
    nc, cm = run_gpu(V_, lg, T, k, p, pending, dt, dp, u)
    nc_r, cm_r, mg = oracle.sample_accept(lg.astype(np.float64), T, k, p, pending, dt,
                                          dp.astype(np.float64) if dp is not None else None, u.astype(np.float64))
    clear = mg > MARGIN
    assert np.array_equal(nc[clear], nc_r[clear]), (nc, nc_r, mg)
    assert np.array_equal(cm[clear], cm_r[clear]), (cm, cm_r, mg)
    for l in range(nc.size):  # every lane: a valid result
        assert 1 <= nc[l] <= 8
        a = nc[l] - 1
        assert np.array_equal(cm[l, :a], pending[8 * l + 1:8 * l + 1 + a])
        assert 0 <= cm[l, a] < lg.shape[1] and np.all(cm[l, a + 1:] == -1)
    return int(clear.sum())


@pytest.mark.parametrize("M,V,T,k,p", [
    (8, 1000, 1.0, 20, 0.95),
    (16, 4096, 0.7, 32, 0.9),
    (32, 5000, 1.3, 8, 1.0),
    (32, 248320, 0.6, 20, 0.95),   # the vocabulary of the pages' target, Qwen's default top_k
    (8, 20, 1.0, 20, 1.0),         # V below one chunk and below 32
])
def test_sample_accept_matches_oracle(V_, M, V, T, k, p):
    compared = 0
    for seed in range(4):
        lg, pending, dt, dp, u = make_case(1000 * seed + M + V, M, V, n_boost=min(12, V))
        compared += check(V_, lg, T, k, p, pending, dt, dp, u)
    assert compared >= M // 8 * 2  # most lanes clear the margin


def test_sample_accept_point_mass_drafts(V_):
    lg, pending, _, _, u = make_case(77, 32, 248320)
    assert check(V_, lg, 0.8, 20, 0.95, pending, None, None, u) >= 2


def test_sample_accept_top1_point_mass_is_greedy(V_):
    """top_k = 1 with point-mass drafts: equals the greedy argmax + accept call on the same logits."""
    M, V = 32, 248320
    lg, pending, _, _, u = make_case(78, M, V)
    nc, cm = run_gpu(V_, lg, 1.0, 1, 1.0, pending, None, None, u)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc2 = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm2 = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    ws = workspace(V_.vp_workspace_bytes(V_.VP_OP_ARGMAX, M, V, 0))
    V_.vp_argmax_accept(torch.from_numpy(lg).cuda(), M, V, dev_i32(pending), am, nc2, cm2, ws)
    torch.cuda.synchronize()
    assert np.array_equal(nc, nc2.cpu().numpy()) and np.array_equal(cm, cm2.cpu().numpy())


def test_sample_accept_ties_and_nan(V_):
    """Equal logits across the top_k boundary (the lower index wins on both sides) and NaN logits
    (counted as -inf)."""
    M, V = 8, 9000
    lg, pending, dt, dp, u = make_case(79, M, V)
    for r in range(M):
        top = np.argsort(-lg[r])[:30]
        lg[r, top[15:25]] = lg[r, top[15]]  # a run of ties around k = 20
        lg[r, top[25]] = np.nan
    check(V_, lg, 1.0, 20, 1.0, pending, dt, dp, u)


def test_sample_accept_acceptance_rate_matches_definition(V_):
    """Over many lanes with point-mass drafts on the rows' most likely token, the accepted fraction
    of the first draft follows p(d): E[accept] = mean over lanes of p_row(d)."""
    M, V = 32, 3000
    rng = np.random.default_rng(80)
    acc, expect = [], []
    for seed in range(40):
        lg, pending, _, _, u = make_case(200 + seed, M, V)
        for l in range(M // 8):
            tok, p, _ = oracle.target_dist(lg[8 * l].astype(np.float64), 1.0, 20, 1.0)
            pending[8 * l + 1] = tok[0]
            expect.append(p[0])
        u[:, 0] = rng.random(M).astype(np.float32)
        nc, _ = run_gpu(V_, lg, 1.0, 20, 1.0, pending, None, None, u)
        acc += list(nc >= 2)
    acc, expect = np.array(acc, float), np.array(expect)
    se = np.sqrt(np.sum(expect * (1 - expect))) / acc.size
    assert abs(acc.mean() - expect.mean()) < 4 * se + 1e-3

"""GPU parity of the vocabulary head fused with argmax and greedy acceptance.

vp_argmax_accept runs the device reduction + acceptance code on given fp32 logits, so it must match
the oracle bit for bit (both decide on the same fp32 values).  The fused head computes its own
logits; there the argmax must (a) be the lowest-index maximum of the device's own logits and
(b) be one of the oracle's valid choices: tokens whose exact logit is within the tolerance bound of
the exact maximum (several answers are correct at near-ties)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import REL, ABS, assert_linear_close, dev_bf16, dev_i32, dev_u8, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


def run_argmax(V, logits32: np.ndarray, pending: np.ndarray):
    M, Vv = logits32.shape
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_ARGMAX, M, Vv, 0))
    V.vp_argmax_accept(torch.from_numpy(logits32).cuda(), M, Vv, dev_i32(pending), am, nc, cm, ws)
    torch.cuda.synchronize()
    return am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy()


@pytest.mark.parametrize("M,Vv", [(8, 1), (8, 100), (16, 20000), (32, 248320)])
def test_argmax_accept_bit_exact(V, M, Vv):
    rng = np.random.default_rng(M + Vv)
    lg = rng.standard_normal((M, Vv)).astype(np.float32)
    if Vv >= 100:
        # planted ties of the maximum at several indices (lowest must win)
        for m in range(0, M, 3):
            idx = np.sort(rng.choice(Vv, 4, replace=False))
            lg[m, idx] = 50.0
        lg[1, :] = 0.0
        lg[1, 7] = -0.0
        lg[1, 3] = -0.0  # all zeros: index 0 wins (-0 == +0)
        lg[2, :] = np.nan
        lg[2, Vv - 1] = -np.inf  # all NaN / -inf: index 0
        lg[4, 10] = np.inf
        lg[4, 5] = np.inf
        lg[5, ::2] = np.nan  # NaN never wins
        lg[6, :] = -np.inf
    t_ref = np.array([oracle.argmax(lg[m].astype(np.float64)) for m in range(M)], np.int32)
    pending, planted = synth.planted_pending(3, t_ref, Vv, prefix=[(l * 3) % 8 for l in range(M // 8)])
    am, nc, cm = run_argmax(V, lg, pending)
    assert np.array_equal(am, t_ref)
    nc_ref, cm_ref = oracle.accept(t_ref, pending)
    assert np.array_equal(nc, nc_ref) and np.array_equal(cm, cm_ref)
    if Vv > 1:
        assert np.array_equal(nc - 1, planted)


def test_argmax_accept_all_acceptance_lengths(V):
    M, Vv = 32, 4096
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((M, Vv)).astype(np.float32)
    t_ref = np.argmax(lg, axis=1).astype(np.int32)
    for prefix in ([0, 1, 2, 3], [4, 5, 6, 7]):
        pending, planted = synth.planted_pending(9, t_ref, Vv, prefix=prefix)
        am, nc, cm = run_argmax(V, lg, pending)
        nc_ref, cm_ref = oracle.accept(t_ref, pending)
        assert np.array_equal(nc, nc_ref) and np.array_equal(cm, cm_ref)
        assert list(nc - 1) == prefix


def run_head(V, codes, scales, ts, x, pending):
    Vv, K = codes.shape[0], codes.shape[1] * 2
    M = x.shape[0]
    packed = torch.empty(V.vp_packed_bytes_nvfp4(Vv, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(dev_u8(codes), dev_u8(scales), Vv, K, packed)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    lg = torch.empty((M, Vv), dtype=torch.float32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_HEAD, M, Vv, K))
    V.vp_head_argmax_accept(packed, ts, dev_bf16(x), M, Vv, K, dev_i32(pending), am, nc, cm, lg, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    # again without the logits output: identical decisions
    am2 = torch.empty_like(am)
    nc2 = torch.empty_like(nc)
    cm2 = torch.empty_like(cm)
    V.vp_head_argmax_accept(packed, ts, dev_bf16(x), M, Vv, K, dev_i32(pending), am2, nc2, cm2, None, ws)
    torch.cuda.synchronize()
    assert torch.equal(am, am2) and torch.equal(nc, nc2) and torch.equal(cm, cm2)
    return am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy(), lg.cpu().numpy()


def check_head(am, nc, cm, lg, y_ref, a_ref, pending, what):
    M = am.size
    assert_linear_close(lg, y_ref, a_ref, what)
    # (a) the device argmax is the lowest-index maximum of its own logits
    assert np.array_equal(am, np.argmax(lg, axis=1))
    # (b) it is a valid choice against the exact logits
    tol = REL * a_ref + ABS
    t_ref = np.argmax(y_ref, axis=1)
    unique = np.zeros(M, bool)
    for m in range(M):
        best = y_ref[m, t_ref[m]]
        assert y_ref[m, am[m]] >= best - tol[m, am[m]] - tol[m, t_ref[m]], (what, m)
        others = np.delete(y_ref[m] + tol[m], t_ref[m])
        unique[m] = best - tol[m, t_ref[m]] > others.max()
        if unique[m]:
            assert am[m] == t_ref[m]
    # acceptance: equal to the oracle's wherever every row of the lane is decided uniquely
    nc_ref, cm_ref = oracle.accept(t_ref.astype(np.int32), pending)
    for l in range(M // 8):
        if unique[8 * l:8 * l + 8].all():
            assert nc[l] == nc_ref[l] and np.array_equal(cm[l], cm_ref[l])
        assert 1 <= nc[l] <= 8
    return unique


@pytest.mark.parametrize("M,Vv,K", [(8, 5136, 1024), (16, 4096, 768), (32, 2064, 2048), (8, 2048, 5120)])
def test_head_matches_oracle(V, M, Vv, K):
    codes = synth.uniform_bytes(M + Vv, 1, 0, Vv * K // 2).reshape(Vv, K // 2)
    scales = synth.scale_codes(M + Vv, 2, 0, Vv * K // 16).reshape(Vv, K // 16)
    x = synth.normal_bf16(M + Vv, 3, (M, K))
    ts = 0.8
    y_ref, a_ref = oracle.linear(oracle.NVFP4, x, codes, scales, ts, Vv)
    t_ref = np.argmax(y_ref, axis=1).astype(np.int32)
    pending, planted = synth.planted_pending(M, t_ref, Vv)
    am, nc, cm, lg = run_head(V, codes, scales, ts, x, pending)
    unique = check_head(am, nc, cm, lg, y_ref, a_ref, pending, f"head {M}x{Vv}x{K}")
    assert unique.mean() >= 0.5


def test_head_workspace_reused_with_new_inputs(V):
    """The fused head at M = 32, K = 5120 (a phase cut into K slices) called three times on one
    workspace with different hidden states: each call's logits match the oracle's for its own
    input (a barrier left counted by the previous call would let the slices' sums read stale
    partials)."""
    M, Vv, K = 32, 2064, 5120
    codes = synth.uniform_bytes(77, 1, 0, Vv * K // 2).reshape(Vv, K // 2)
    scales = synth.scale_codes(77, 2, 0, Vv * K // 16).reshape(Vv, K // 16)
    packed = torch.empty(V.vp_packed_bytes_nvfp4(Vv, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(dev_u8(codes), dev_u8(scales), Vv, K, packed)
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_HEAD, M, Vv, K))
    for i in range(3):
        x = synth.normal_bf16(300 + i, 3, (M, K))
        y_ref, a_ref = oracle.linear(oracle.NVFP4, x, codes, scales, 0.8, Vv)
        pending, _ = synth.planted_pending(i, np.argmax(y_ref, axis=1).astype(np.int32), Vv)
        am = torch.empty(M, dtype=torch.int32, device="cuda")
        nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
        cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
        lg = torch.empty((M, Vv), dtype=torch.float32, device="cuda")
        V.vp_head_argmax_accept(packed, 0.8, dev_bf16(x), M, Vv, K, dev_i32(pending), am, nc, cm, lg, ws)
        torch.cuda.synchronize()
        assert V.vp_read_status(ws) == V.VP_OK
        assert_linear_close(lg.cpu().numpy(), y_ref, a_ref, f"head call {i}")
        check_head(am.cpu().numpy(), nc.cpu().numpy(), cm.cpu().numpy(), lg.cpu().numpy(), y_ref, a_ref, pending,
                   f"head call {i}")

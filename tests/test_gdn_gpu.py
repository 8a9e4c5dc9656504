"""GPU parity of the Gated DeltaNet verify scan (vp_gdn_scan) against the fp64 oracle, through the C
ABI, and the pages' rollback property: from the intact parity buffer A, a re-scan of the n committed
rows reproduces, bit for bit, the state of a one-row-at-a-time reference scan for every n in 0..8."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DK = DV = 128


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


def bf16(rng, shape, scale=1.0):
    return torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def case(seed, L, H):
    rng = np.random.default_rng(seed)
    M = 8 * L
    st = (rng.standard_normal((L, H, DV, DK)) * 0.1).astype(np.float32)
    q = bf16(rng, (M, H, DK))
    k = bf16(rng, (M, H, DK), 1.0 / np.sqrt(DK))  # about unit norm, as after the layer's normalisation
    v = bf16(rng, (M, H, DV))
    a = rng.uniform(0.85, 1.0, (M, H)).astype(np.float32)
    b = rng.uniform(0.05, 0.95, (M, H)).astype(np.float32)
    return st, q, k, v, a, b


def d16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def run(V, st, q, k, v, a, b, rows, want_out=True, st_dev=None):
    L, H = st.shape[:2]
    M = 8 * L
    sin = torch.from_numpy(st).cuda() if st_dev is None else st_dev
    sout = torch.full_like(sin, float("nan"))
    out = torch.full((M, H, DV), float("nan"), device="cuda") if want_out else None
    V.vp_gdn_scan(sin, sout, d16(q), d16(k), d16(v), torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(),
                  torch.from_numpy(np.asarray(rows, np.int32)).cuda(), M, H, DK, DV, out)
    torch.cuda.synchronize()
    return sin, sout, out


def tol(ref, scale):
    return 2e-5 * scale + 1e-6  # fp32 dot products of 128 terms, 8 sequential steps


@pytest.mark.parametrize("L,H,rows", [(1, 4, [8]), (2, 48, [8, 3]), (4, 6, [0, 1, 7, 8])])
def test_gdn_matches_oracle(V, L, H, rows):
    st, q, k, v, a, b = case(L * 100 + H, L, H)
    sin, sout, out = run(V, st, q, k, v, a, b, rows)
    ref_s, ref_o = oracle.gdn_scan(st.astype(np.float64), q, k, v, a.astype(np.float64), b.astype(np.float64), rows)
    s_gpu = sout.cpu().numpy().astype(np.float64)
    scale = np.abs(ref_s).max()
    assert np.abs(s_gpu - ref_s).max() <= tol(ref_s, scale)
    o_gpu = out.cpu().numpy().astype(np.float64)
    for l in range(L):
        n = rows[l]
        got, ref = o_gpu[8 * l:8 * l + n], ref_o[8 * l:8 * l + n]
        assert np.abs(got - ref).max(initial=0.0) <= tol(ref, np.abs(ref).max(initial=1.0) * 4)
        assert np.all(np.isnan(o_gpu[8 * l + n:8 * l + 8]))  # rows past the scan are untouched
    assert np.array_equal(sin.cpu().numpy(), st)  # parity buffer A is intact


def test_gdn_rescan_is_bitwise_the_reference_scan(V):
    """For every number n of kept rows: the re-scan of n rows from A equals, bit for bit, n one-row
    scans applied in sequence (the reference scan), and the verify scan's outputs of rows < n."""
    L, H = 1, 8
    st, q, k, v, a, b = case(7, L, H)
    _, s8, o8 = run(V, st, q, k, v, a, b, [8])
    for n in range(9):
        _, sn, on = run(V, st, q, k, v, a, b, [n])
        cur = torch.from_numpy(st).cuda()
        for j in range(n):
            sh = lambda x: np.ascontiguousarray(np.roll(x, -j, axis=0))  # noqa: E731  (row j first)
            _, cur, _ = run(V, st, sh(q), sh(k), sh(v), sh(a), sh(b), [1], want_out=False, st_dev=cur)
        assert torch.equal(sn, cur), n
        assert torch.equal(on[:n], o8[:n])
    assert torch.equal(run(V, st, q, k, v, a, b, [8])[1], s8)  # deterministic


def test_gdn_in_place_and_no_output(V):
    st, q, k, v, a, b = case(8, 2, 3)
    _, ref, _ = run(V, st, q, k, v, a, b, [5, 8])
    buf = torch.from_numpy(st).cuda()
    V.vp_gdn_scan(buf, buf, d16(q), d16(k), d16(v), torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(),
                  torch.tensor([5, 8], dtype=torch.int32, device="cuda"), 16, 3, DK, DV, None)
    torch.cuda.synchronize()
    assert torch.equal(buf, ref)

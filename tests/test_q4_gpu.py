"""GPU parity of the affine 4-bit ("Q4", group 64) linear layer (vp_pack_q4, vp_linear_q4) against
the fp64 oracle, through the C ABI: the packed layout byte for byte, shapes spanning several row
blocks, split-K, ragged M, one to four n-tiles and K slices, exactness on dyadic inputs, and the
MLP shapes of the pages' 4-bit checkpoint on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_linear_close, dev_bf16, dev_u8, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


def dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).cuda()


def q4_case(seed, M, N, K):
    codes = synth.uniform_bytes(seed, 21, 0, N * K // 2).reshape(N, K // 2)
    sc, bi = synth.q4_scales_biases(seed, 22, 0, N * K // 64)
    x = synth.normal_bf16(seed, 23, (M, K))
    return codes, sc.reshape(N, K // 64), bi.reshape(N, K // 64), x


def pack(V, codes, scales, biases):
    N, K = codes.shape[0], codes.shape[1] * 2
    packed = torch.empty(V.vp_packed_bytes_q4(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_q4(dev_u8(codes), dev_u16(scales), dev_u16(biases), N, K, packed)
    return packed


def run_q4(V, codes, scales, biases, x, packed=None):
    N, K = codes.shape[0], codes.shape[1] * 2
    M = x.shape[0]
    if packed is None:
        packed = pack(V, codes, scales, biases)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_Q4, M, N, K))
    V.vp_linear_q4(packed, dev_bf16(x), y, M, N, K, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    return y.cpu().numpy()


def expected_packed_q4(codes, scales, biases):
    """The documented packed layout, built independently in numpy: per 16-row block, 256-wide chunk
    and 8-row strip, for half h, row g and quarter c four words, word w holding the codes of steps
    s = 8h + 2w and s + 1 (k = 16 s + 4 c .. + 3) in nibble order (s,0) (s+1,0) (s,2) (s+1,2) (s,1)
    (s+1,1) (s,3) (s+1,3); then per row the chunk's four (scale | bias << 16) words."""
    N, K = codes.shape[0], codes.shape[1] * 2
    q = np.empty((N, K), np.uint32)
    q[:, 0::2] = codes & 15
    q[:, 1::2] = codes >> 4
    out = []
    for rb in range(N // 16):
        for kc in range(K // 256):
            for t in range(2):
                r0 = 16 * rb + 8 * t
                blk = q[r0:r0 + 8, 256 * kc:256 * kc + 256].reshape(8, 2, 4, 2, 4, 4)  # [g][h][w][d][c][e]
                blk = blk.transpose(1, 0, 4, 2, 3, 5)  # [h][g][c][w][d][e]
                order = [(0, 0), (1, 0), (0, 2), (1, 2), (0, 1), (1, 1), (0, 3), (1, 3)]  # (d, e) per nibble
                words = np.zeros(blk.shape[:4], np.uint32)
                for nib, (d, e) in enumerate(order):
                    words |= blk[..., d, e] << np.uint32(4 * nib)
                out.append(words.reshape(-1).view(np.uint8))
                sw = (scales[r0:r0 + 8, 4 * kc:4 * kc + 4].astype(np.uint32)
                      | (biases[r0:r0 + 8, 4 * kc:4 * kc + 4].astype(np.uint32) << np.uint32(16)))
                out.append(np.ascontiguousarray(sw).reshape(-1).view(np.uint8))
    return np.concatenate(out)


def test_pack_q4_layout(V):
    N, K = 48, 512
    codes, sc, bi, _ = q4_case(31, 1, N, K)
    packed = pack(V, codes, sc, bi)
    torch.cuda.synchronize()
    exp = expected_packed_q4(codes, sc, bi)
    assert exp.size == N * K * 9 // 16
    assert np.array_equal(packed.cpu().numpy(), exp)


SHAPES = [
    (8, 1024, 1024),   # one slice, several row blocks per CTA
    (1, 16, 256),      # smallest: one row block, one chunk
    (3, 272, 256),     # odd M, odd row-block count
    (13, 1040, 1024),  # ragged M in the second n-tile
    (24, 528, 768),    # three n-tiles
    (32, 4096, 512),   # four n-tiles
    (32, 256, 4096),   # K slices at four n-tiles
    (16, 512, 8192),   # K slices at two n-tiles
    (8, 4112, 2048),   # fewer units than warps
    (8, 512, 17408),   # MLP-down width: K slices at one n-tile
    (8, 256, 5120),    # hidden width at one n-tile: two slices of the Q4 staging width
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_q4_matches_oracle(V, M, N, K):
    codes, sc, bi, x = q4_case(400 + M + N + K, M, N, K)
    y = run_q4(V, codes, sc, bi, x)
    y_ref, a_ref = oracle.linear_q4(x, codes, sc, bi, N)
    assert_linear_close(y, y_ref, a_ref, f"q4 {M}x{N}x{K}")


def test_linear_q4_dyadic_is_exact(V):
    """Integer activations, power-of-two scales and biases in eighths: every term is exact in fp32,
    so the GPU result equals the oracle bit for bit."""
    rng = np.random.default_rng(41)
    M, N, K = 8, 512, 512
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sv = np.ldexp(1.0, rng.integers(-1, 2, (N, K // 64)))
    bv = rng.integers(-40, 41, (N, K // 64)) / 8.0
    to_bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    sc, bi = to_bits(sv), to_bits(bv)
    xi = rng.integers(-4, 5, (M, K)).astype(np.float32)
    x = torch.from_numpy(xi).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = run_q4(V, codes, sc, bi, x)
    y_ref = oracle.linear_q4(x, codes, sc, bi, N, with_abs=False)
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_linear_q4_is_deterministic(V):
    codes, sc, bi, x = q4_case(42, 16, 2048, 2048)
    packed = pack(V, codes, sc, bi)
    assert np.array_equal(run_q4(V, codes, sc, bi, x, packed), run_q4(V, codes, sc, bi, x, packed))


def test_linear_q4_zero_and_scaled_rows(V):
    """A zero row gives exactly zero; rows scaled by 2^40 and 2^-40 keep their relative accuracy
    (the group sums are taken in the same row-scaled units as the tensor-core products)."""
    M, N, K = 8, 256, 1024
    codes, sc, bi, x = q4_case(43, M, N, K)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    xv[1] *= 2.0 ** 40
    xv[2] *= 2.0 ** -40
    xv[3] = 0.0
    x2 = xv.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = run_q4(V, codes, sc, bi, x2)
    y_ref, a_ref = oracle.linear_q4(x2, codes, sc, bi, N)
    assert_linear_close(y, y_ref, a_ref, "q4 dynamic range")
    assert np.all(y[3] == 0.0)


@pytest.mark.parametrize("M", [8, 32])
@pytest.mark.parametrize("N,K", [(17408, 5120), (5120, 17408)])
def test_linear_q4_mlp_shapes_sampled_rows(V, M, N, K):
    """The 4-bit checkpoint's MLP gate/up and down shapes, full size on the GPU; the oracle checks 96
    sampled output rows (every row block boundary class: first, last, and random rows)."""
    codes, sc, bi, x = q4_case(500 + M + N, M, N, K)
    y = run_q4(V, codes, sc, bi, x)
    rng = np.random.default_rng(N + M)
    rows = np.unique(np.concatenate([[0, 15, 16, N - 1], rng.integers(0, N, 92)])).astype(np.int32)
    y_ref, a_ref = oracle.linear_q4(x, codes, sc, bi, N, rows=rows)
    assert_linear_close(y[:, rows], y_ref, a_ref, f"q4 {M}x{N}x{K} sampled")


def test_linear_q4_workspace_reused_by_k_sliced_calls(V):
    """M = 32, K = 5120: the phase is cut into K slices that meet at a grid barrier; three calls
    with different activations on one workspace each match the oracle for their own input."""
    M, N, K = 32, 512, 5120
    codes, scales, biases, _ = q4_case(91, M, N, K)
    packed = pack(V, codes, scales, biases)
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_Q4, M, N, K))
    for i in range(3):
        x = synth.normal_bf16(400 + i, 23, (M, K))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        V.vp_linear_q4(packed, dev_bf16(x), y, M, N, K, ws)
        torch.cuda.synchronize()
        assert V.vp_read_status(ws) == V.VP_OK
        y_ref, a_ref = oracle.linear_q4(x, codes, scales, biases, N)
        assert_linear_close(y.cpu().numpy(), y_ref, a_ref, f"q4 call {i}")

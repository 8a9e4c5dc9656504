"""GPU parity of the skinny NVFP4 / FP8 linear layers (vp_linear_*) and the packers against the
fp64 oracle, through the C ABI.  Sizes span several 256-row groups, several CTAs per group
(split-K), ragged M, partial last groups and both activation-staging modes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import ABS, REL, assert_linear_close, dev_bf16, dev_u8, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


def nvfp4_case(seed, M, N, K):
    codes = synth.uniform_bytes(seed, 1, 0, N * K // 2).reshape(N, K // 2)
    scales = synth.scale_codes(seed, 2, 0, N * K // 16).reshape(N, K // 16)
    x = synth.normal_bf16(seed, 3, (M, K))
    return codes, scales, x


def fp8_case(seed, M, N, K):
    w = synth.fp8_normal_codes(seed, 4, 0, N * K).reshape(N, K)
    x = synth.normal_bf16(seed, 5, (M, K))
    return w, x


def run_nvfp4(V, codes, scales, x, ts):
    N, K = codes.shape[0], codes.shape[1] * 2
    M = x.shape[0]
    packed = torch.empty(V.vp_packed_bytes_nvfp4(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(dev_u8(codes), dev_u8(scales), N, K, packed)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_NVFP4, M, N, K))
    V.vp_linear_nvfp4(packed, ts, dev_bf16(x), y, M, N, K, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    return y.cpu().numpy()


def run_fp8(V, w, x, s):
    N, K = w.shape
    M = x.shape[0]
    packed = torch.empty(V.vp_packed_bytes_fp8(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_fp8(dev_u8(w), N, K, packed)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_FP8, M, N, K))
    V.vp_linear_fp8(packed, s, dev_bf16(x), y, M, N, K, ws)
    torch.cuda.synchronize()
    assert V.vp_read_status(ws) == V.VP_OK
    return y.cpu().numpy()


# ------------------------------------------------------------------ packers

def expected_packed_nvfp4(codes, scales):
    """The documented packed layout, built independently in numpy."""
    N, K = codes.shape[0], codes.shape[1] * 2
    nq = K // 64
    out = []
    for slab in range((N + 255) // 256):
        nrb = min(16, N // 16 - 16 * slab)
        for q in range(nq):
            for rbi in range(nrb):
                rb = 16 * slab + rbi
                blk = np.zeros(576, np.uint8)
                for L in range(32):
                    g, t = L // 4, L % 4
                    for j in range(4):
                        for i in range(4):
                            row = rb * 16 + g + 8 * (i & 1)
                            k = 64 * q + 16 * j + 2 * t + 8 * (i >> 1)
                            blk[16 * L + 4 * j + i] = codes[row, k // 2]
                for g in range(8):
                    for j in range(4):
                        for h in range(2):
                            blk[512 + 8 * g + 2 * j + h] = scales[rb * 16 + g + 8 * h, 4 * q + j]
                out.append(blk)
    return np.concatenate(out)


def test_pack_nvfp4_layout(V):
    N, K = 288, 128  # one full slab + a partial one
    codes, scales, _ = nvfp4_case(7, 1, N, K)
    packed = torch.empty(V.vp_packed_bytes_nvfp4(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(dev_u8(codes), dev_u8(scales), N, K, packed)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), expected_packed_nvfp4(codes, scales))


def test_pack_fp8_layout(V):
    N, K = 272, 128
    w, _ = fp8_case(8, 1, N, K)
    packed = torch.empty(V.vp_packed_bytes_fp8(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_fp8(dev_u8(w), N, K, packed)
    torch.cuda.synchronize()
    got = packed.cpu().numpy()
    nq = K // 64
    pos = 0
    for slab in range((N + 255) // 256):
        nrb = min(16, N // 16 - 16 * slab)
        for q in range(nq):
            for rbi in range(nrb):
                rb = 16 * slab + rbi
                for L in range(32):
                    g, t = L // 4, L % 4
                    for j in range(4):
                        for i in range(4):
                            for e in range(2):
                                row = rb * 16 + g + 8 * (i & 1)
                                k = 64 * q + 16 * j + 2 * t + 8 * (i >> 1) + e
                                assert got[pos + 32 * L + 8 * j + 2 * i + e] == w[row, k]
                pos += 1024
    assert pos == got.size


# ------------------------------------------------------------------ parity

SHAPES = [
    (8, 1024, 1024),   # tiny NVFP4 linear of the synthetic recipe
    (1, 16, 64),       # smallest
    (3, 272, 192),     # partial group, odd M
    (13, 1040, 1024),  # several groups + ragged last group
    (24, 528, 640),
    (32, 4096, 512),   # many groups, all K staged at once
    (32, 256, 4096),   # activation window larger than shared memory: staged in batches
    (8, 4112, 2048),   # split-K over many CTAs + ragged group
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_nvfp4_matches_oracle(V, M, N, K):
    codes, scales, x = nvfp4_case(100 + M + N + K, M, N, K)
    ts = 1.0 if (M, N, K) == (8, 1024, 1024) else 0.75
    y = run_nvfp4(V, codes, scales, x, ts)
    y_ref, a_ref = oracle.linear(oracle.NVFP4, x, codes, scales, ts, N)
    assert_linear_close(y, y_ref, a_ref, f"nvfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_linear_fp8_matches_oracle(V, M, N, K):
    w, x = fp8_case(200 + M + N + K, M, N, K)
    y = run_fp8(V, w, x, 0.625)
    y_ref, a_ref = oracle.linear(oracle.FP8, x, w, None, 0.625, N)
    assert_linear_close(y, y_ref, a_ref, f"fp8 {M}x{N}x{K}")


def test_linear_nvfp4_dyadic_is_exact(V):
    """Integer activations and power-of-two block scales: every partial sum is exact in fp32, so the
    GPU result equals the oracle bit for bit."""
    rng = np.random.default_rng(9)
    M, N, K = 8, 512, 256
    codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    scales = np.array([0x30, 0x38, 0x40], np.uint8)[rng.integers(0, 3, (N, K // 16))]
    xi = rng.integers(-4, 5, (M, K)).astype(np.float32)
    x = torch.from_numpy(xi).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = run_nvfp4(V, codes, scales, x, 1.0)
    y_ref = oracle.linear(oracle.NVFP4, x, codes, scales, 1.0, N, with_abs=False)
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_linear_fp8_dyadic_is_exact(V):
    rng = np.random.default_rng(10)
    M, N, K = 16, 256, 512
    w = np.array([0x38, 0xB8, 0x40, 0x30, 0x00, 0x48], np.uint8)[rng.integers(0, 6, (N, K))]  # +-1, 2, .5, 0, 4
    xi = rng.integers(-3, 4, (M, K)).astype(np.float32)
    x = torch.from_numpy(xi).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = run_fp8(V, w, x, 1.0)
    y_ref = oracle.linear(oracle.FP8, x, w, None, 1.0, N, with_abs=False)
    assert np.array_equal(y.astype(np.float64), y_ref)


def test_linear_is_deterministic(V):
    codes, scales, x = nvfp4_case(11, 16, 2048, 2048)
    y1 = run_nvfp4(V, codes, scales, x, 1.0)
    y2 = run_nvfp4(V, codes, scales, x, 1.0)
    assert np.array_equal(y1, y2)


def test_linear_wide_dynamic_range_rows(V):
    """Rows whose magnitudes differ by 2^60 and a zero row: the per-row power-of-two staging keeps
    each row's relative accuracy."""
    M, N, K = 8, 256, 1024
    codes, scales, x = nvfp4_case(12, M, N, K)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float()
    xv[1] *= 2.0 ** 60
    xv[2] *= 2.0 ** -60
    xv[3] = 0.0
    x2 = xv.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y = run_nvfp4(V, codes, scales, x2, 1.0)
    y_ref, a_ref = oracle.linear(oracle.NVFP4, x2, codes, scales, 1.0, N)
    assert_linear_close(y, y_ref, a_ref, "dynamic range")
    assert np.all(y[3] == 0.0)

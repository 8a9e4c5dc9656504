"""GPU parity of the skinny NVFP4 / FP8 linear layers (vp_linear_*) and the packers against the
fp64 oracle, through the C ABI.  Sizes span several 256-row groups, several CTAs per group
(split-K), ragged M, one to four n-tiles, and phases cut into K slices."""
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
    """The documented packed layout, built independently in numpy: 16-row blocks, 256-wide K chunks,
    two 8-row strips per chunk; a strip holds, for half h, row g and quarter c, the bytes of steps
    8h .. 8h+7 that cover k = 16s + 4c .. +3, then the rows' 16 block scales."""
    N, K = codes.shape[0], codes.shape[1] * 2
    out = []
    for rb in range(N // 16):
        for kc in range(K // 256):
            for t in range(2):
                r0 = 16 * rb + 8 * t
                c = codes[r0:r0 + 8, 128 * kc:128 * kc + 128].reshape(8, 2, 8, 4, 2)  # [g][h][ss][c][b]
                out.append(c.transpose(1, 0, 3, 2, 4).reshape(-1))
                out.append(scales[r0:r0 + 8, 16 * kc:16 * kc + 16].reshape(-1))
    return np.concatenate(out)


def expected_packed_fp8(w):
    N, K = w.shape
    out = []
    for rb in range(N // 16):
        for kc in range(K // 128):
            for t in range(2):
                r0 = 16 * rb + 8 * t
                q = w[r0:r0 + 8, 128 * kc:128 * kc + 128].reshape(8, 2, 4, 4, 4)  # [g][h][ss][c][b]
                out.append(q.transpose(1, 0, 3, 2, 4).reshape(-1))
    return np.concatenate(out)


def test_pack_nvfp4_layout(V):
    N, K = 48, 512  # three row blocks, two chunks
    codes, scales, _ = nvfp4_case(7, 1, N, K)
    packed = torch.empty(V.vp_packed_bytes_nvfp4(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(dev_u8(codes), dev_u8(scales), N, K, packed)
    torch.cuda.synchronize()
    exp = expected_packed_nvfp4(codes, scales)
    assert exp.size == N * K * 9 // 16
    assert np.array_equal(packed.cpu().numpy(), exp)


def test_pack_fp8_layout(V):
    N, K = 48, 384
    w, _ = fp8_case(8, 1, N, K)
    packed = torch.empty(V.vp_packed_bytes_fp8(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_fp8(dev_u8(w), N, K, packed)
    torch.cuda.synchronize()
    exp = expected_packed_fp8(w)
    assert exp.size == N * K
    assert np.array_equal(packed.cpu().numpy(), exp)


# ------------------------------------------------------------------ parity

SHAPES = [
    (8, 1024, 1024),   # tiny NVFP4 linear of the synthetic recipe
    (1, 16, 256),      # smallest: one row block, one chunk
    (3, 272, 256),     # odd M, odd row-block count
    (13, 1040, 1024),  # ragged M in the second n-tile
    (24, 528, 768),    # three n-tiles
    (32, 4096, 512),   # four n-tiles, many row blocks per warp
    (32, 256, 4096),   # activations wider than shared memory: three K slices
    (16, 512, 8192),   # the same with two n-tiles
    (8, 4112, 2048),   # fewer units than warps: row blocks split across warps
    (8, 512, 17408),   # MLP-down width at M = 8: three K slices
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


@pytest.mark.parametrize("M,N,K", [(5, 64, 384), (8, 1024, 6144)])
def test_linear_fp8_half_chunks(V, M, N, K):
    """FP8 reduction widths that are a multiple of 128 but not of 256 (mixer out-projection)."""
    w, x = fp8_case(300 + M + N + K, M, N, K)
    y = run_fp8(V, w, x, 1.25)
    y_ref, a_ref = oracle.linear(oracle.FP8, x, w, None, 1.25, N)
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


@pytest.mark.parametrize("fmt,M,N,K", [("nvfp4", 8, 2432, 5120), ("nvfp4", 16, 2432, 17408), ("nvfp4", 24, 2432, 5120),
                                         ("nvfp4", 32, 2432, 5120), ("fp8", 8, 2432, 6144), ("fp8", 16, 2432, 6144)])
def test_linear_dyadic_shared_row_blocks_exact(V, fmt, M, N, K):
    """Shapes whose row blocks are split among several warps of a CTA (one row block of 10 units per
    CTA over 10 warps at M = 8, K = 5120; pairs and triples of warps in K-sliced phases), so that the
    in-CTA fixups sum partials from warps of the same tensor-memory lane quarter and of other
    quarters, with one K slice and with several.  Integer activations and power-of-two scales make
    every partial sum exact in fp32: the result equals the oracle bit for bit."""
    rng = np.random.default_rng(M * 7 + K)
    if fmt == "nvfp4":
        codes = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
        scales = np.array([0x30, 0x38, 0x40], np.uint8)[rng.integers(0, 3, (N, K // 16))]
        xi = rng.integers(-4, 5, (M, K)).astype(np.float32)
    else:
        w = np.array([0x38, 0xB8, 0x40, 0x30, 0x00, 0x48], np.uint8)[rng.integers(0, 6, (N, K))]
        xi = rng.integers(-3, 4, (M, K)).astype(np.float32)
    x = torch.from_numpy(xi).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if fmt == "nvfp4":
        y = run_nvfp4(V, codes, scales, x, 1.0)
        y_ref = oracle.linear(oracle.NVFP4, x, codes, scales, 1.0, N, with_abs=False)
    else:
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


@pytest.mark.parametrize("fmt,M", [("fp8", 16), ("fp8", 32), ("nvfp4", 16), ("nvfp4", 32)])
def test_workspace_reused_by_k_sliced_calls(V, fmt, M):
    """One workspace serves several calls without a reset in between (the workspace contract).
    With K = 5120 at M > 8 the single phase is cut into K slices that meet at a grid barrier, so
    the barrier's counter must be back at zero when a call ends.  Each call gets different
    activations: a call whose barrier passed early would sum the previous call's partials."""
    N, K = 512, 5120
    if fmt == "fp8":
        w, _ = fp8_case(70 + M, M, N, K)
        packed = torch.empty(V.vp_packed_bytes_fp8(N, K), dtype=torch.uint8, device="cuda")
        V.vp_pack_fp8(dev_u8(w), N, K, packed)
        op, call, scale = V.VP_OP_FP8, V.vp_linear_fp8, 0.75
    else:
        codes, scales, _ = nvfp4_case(70 + M, M, N, K)
        packed = torch.empty(V.vp_packed_bytes_nvfp4(N, K), dtype=torch.uint8, device="cuda")
        V.vp_pack_nvfp4(dev_u8(codes), dev_u8(scales), N, K, packed)
        op, call, scale = V.VP_OP_NVFP4, V.vp_linear_nvfp4, 0.75
    ws = workspace(V.vp_workspace_bytes(op, M, N, K))
    for i in range(3):
        x = synth.normal_bf16(200 + 10 * M + i, 5, (M, K))
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        call(packed, scale, dev_bf16(x), y, M, N, K, ws)
        torch.cuda.synchronize()
        assert V.vp_read_status(ws) == V.VP_OK
        if fmt == "fp8":
            y_ref, a_ref = oracle.linear(oracle.FP8, x, w, None, scale, N)
        else:
            y_ref, a_ref = oracle.linear(oracle.NVFP4, x, codes, scales, scale, N)
        assert_linear_close(y.cpu().numpy(), y_ref, a_ref, f"{fmt} M={M} call {i}")

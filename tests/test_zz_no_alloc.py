"""The no-allocation linear call (vp_linear_nvfp4_noalloc) through the C ABI: on two calls in a row
it returns bit for bit what vp_linear_nvfp4 returns with a caller workspace (same kernel, same
reduction order) and reports a clean status word through vp_noalloc_read_status, and a shape whose
bookkeeping exceeds its fixed scratch is refused.  This file is
collected last so that it also runs after everything else has used the GPU."""
import numpy as np
import pytest
import torch

import synth
from helpers import dev_bf16, dev_u8, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import _lib
    return _lib


@pytest.mark.parametrize("M,N,K", [(8, 1024, 1024), (13, 2064, 2560)])
def test_noalloc_matches_workspace_call_twice(V, M, N, K):
    codes = synth.uniform_bytes(M + N + K, 1, 0, N * K // 2).reshape(N, K // 2)
    scales = synth.scale_codes(M + N + K, 2, 0, N * K // 16).reshape(N, K // 16)
    x = dev_bf16(synth.normal_bf16(M + N + K, 3, (M, K)))
    packed = torch.empty(V.vp_packed_bytes_nvfp4(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(dev_u8(codes), dev_u8(scales), N, K, packed)
    y_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = workspace(V.vp_workspace_bytes(V.VP_OP_NVFP4, M, N, K))
    V.vp_linear_nvfp4(packed, 0.75, x, y_ref, M, N, K, ws)
    torch.cuda.synchronize()
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        V.vp_linear_nvfp4_noalloc(packed, 0.75, x, y, M, N, K)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref)
        assert V.vp_noalloc_read_status() == V.VP_OK
    assert np.isfinite(y.cpu().numpy()).all()


def test_noalloc_refuses_oversized_shape(V):
    L = V.lib()
    fake = 0x10000000  # never dereferenced: the size check comes first
    st = L.vp_linear_nvfp4_noalloc(fake, 1.0, fake, fake, 32, 248320, 5120, None)
    assert st == V.VP_ERR_WORKSPACE

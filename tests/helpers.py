"""Shared test helpers: device transfer of host arrays and the parity checks."""
from __future__ import annotations

import numpy as np

# The linear-layer tolerance of the verify pass: |y - y_ref| <= REL * sum_k |x_k w_k| + ABS, per
# element, in fp32 (fp32 accumulation over K <= 17408 stays far inside it).
REL = 2e-3
ABS = 1e-6


def dev_u8(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def dev_i32(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_bf16_bits(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def workspace(nbytes: int):
    import torch
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")


def assert_linear_close(y_gpu: np.ndarray, y_ref: np.ndarray, a_ref: np.ndarray, what: str = ""):
    y_gpu = np.asarray(y_gpu, np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = REL * a_ref + ABS
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first {idx.tolist()}: "
                             f"gpu {y_gpu[tuple(idx[0])]!r} ref {y_ref[tuple(idx[0])]!r} "
                             f"bound {bound[tuple(idx[0])]!r}")
    return float((err / np.maximum(a_ref, 1e-30)).max())

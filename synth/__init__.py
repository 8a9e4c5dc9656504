"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds no arithmetic of the verify pass.  It only produces bytes with stated
distributions, from one counter-based generator that is implemented twice from its published
definition: here in numpy (host) and in ``synth.cu`` (device fill kernels, used to create the
17.6 GB weight set in HBM quickly).  Element ``i`` of stream ``s`` under seed ``seed`` is the
``i``-th output of a SplitMix64 generator (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) whose state starts at ``key(seed, s)``::

    key(seed, s) = mix64(seed * GOLDEN + s)
    word(seed, s, i) = mix64(key + (i + 1) * GOLDEN)          (all mod 2**64)
    mix64(z): z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB; z ^ z>>31

so any element can be regenerated on its own, on either side, bit for bit.

Distributions (the input recipe):

* ``uniform_bytes``: byte ``j`` = byte ``j % 8`` (little end first) of ``word(j // 8)``.  Used for
  NVFP4 code bytes: both nibbles are uniform over the 16 E2M1 codes.
* ``scale_codes``: E4M3 code of ``2**u`` rounded to nearest, ``u ~ U(-6, 0)``.  ``r = word(i) >> 32``
  maps to ``u = -6 + 6 (r + 1/2) / 2**32``; the code is found by comparing ``r`` with integer
  thresholds computed once on the host (fp64) from the E4M3 values that torch's float8_e4m3fn
  conversion reports, so the device only compares integers.
* ``fp8_normal_codes``: E4M3 code of ``x ~ N(0, 1)`` rounded to nearest, by the same integer
  threshold method on the normal CDF (inverse-CDF sampling).
* ``normal_bf16`` (host only): Box-Muller from two words, rounded to bf16 by torch.
* ``q4_scales_biases`` (host only): the affine 4-bit format's group scales and biases, bf16 (rounded
  by torch): scale = 2**u with u ~ U(-8, -4) from one word, bias = -scale * (7.5 + v) with
  v ~ U(-1/2, 1/2) from the next -- the group minimum that an affine quantiser of zero-centred
  weights stores, so that weights span about [-7.5, 7.5] scales.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
C1 = 0xBF58476D1CE4E5B9
C2 = 0x94D049BB133111EB
_M64 = (1 << 64) - 1

# Stream ids of the pass tensors: (layer + 1) << 8 | tensor.
T_IN, T_KV, T_OUT, T_GATE_C, T_GATE_S, T_UP_C, T_UP_S, T_DOWN_C, T_DOWN_S = range(1, 10)
T_HEAD_C, T_HEAD_S, T_X0, T_PENDING = 10, 11, 12, 13
HEAD_LAYER = 1000


def stream_id(layer: int, tensor: int) -> int:
    return ((layer + 1) << 8) | tensor


def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * C1) & _M64
    z = ((z ^ (z >> 27)) * C2) & _M64
    return z ^ (z >> 31)


def key(seed: int, stream: int) -> int:
    return _mix64_int(seed * GOLDEN + stream)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(C1)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(C2)
    return z ^ (z >> np.uint64(31))


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """uint64 words i = start .. start+count-1 of the stream (computed in blocks of 2^20 words, so
    that the temporaries of a large request stay small)."""
    k = np.uint64(key(seed, stream))
    out = np.empty(max(count, 0), np.uint64)
    blk = 1 << 20
    with np.errstate(over="ignore"):
        for b0 in range(0, count, blk):
            n = min(blk, count - b0)
            i = np.arange(start + b0 + 1, start + b0 + n + 1, dtype=np.uint64)
            out[b0:b0 + n] = _mix64(k + i * np.uint64(GOLDEN))
    return out


def uniform_bytes(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Bytes start .. start+count-1 of the byte stream (uniform over 0..255)."""
    if count <= 0:
        return np.zeros(0, np.uint8)
    w0 = start // 8
    w1 = (start + count + 7) // 8
    w = words(seed, stream, w0, w1 - w0)
    b = w.view(np.uint8) if np.little_endian else w.byteswap().view(np.uint8)
    off = start - 8 * w0
    return np.array(b[off:off + count], copy=True)


# ------------------------------------------------------------------ threshold tables

_tables = {}


def _e4m3_values() -> np.ndarray:
    """Values of the 256 E4M3 codes as reported by torch's float8_e4m3fn conversion."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def scale_thresholds():
    """(thresholds uint64 [48], codes uint8 [49]) for 2**U(-6,0) rounded to E4M3."""
    if "scale" not in _tables:
        v = _e4m3_values()
        codes = np.arange(0x08, 0x39, dtype=np.uint8)  # 2**-6 .. 1.0, increasing values
        vals = v[codes]
        thr = []
        for a, b in zip(vals[:-1], vals[1:]):
            bnd = math.log2((a + b) / 2.0)  # rounding boundary in u
            t = math.ceil((bnd + 6.0) / 6.0 * 2.0**32 - 0.5)
            thr.append(min(max(t, 0), 1 << 32))
        _tables["scale"] = (np.array(thr, np.uint64), codes)
    return _tables["scale"]


def fp8_normal_thresholds():
    """(thresholds uint64 [253], codes uint8 [254]) for N(0,1) rounded to E4M3 (no NaN codes)."""
    if "normal" not in _tables:
        v = _e4m3_values()
        neg = [c for c in range(0x81, 0xFF)]  # -2**-9 .. -448
        pos = [c for c in range(0x01, 0x7F)]  # 2**-9 .. 448
        order = sorted(neg, key=lambda c: v[c]) + [0x80, 0x00] + sorted(pos, key=lambda c: v[c])
        vals = [v[c] for c in order]
        thr = []
        for i in range(len(order) - 1):
            if order[i] == 0x80 and order[i + 1] == 0x00:
                bnd = 0.0
            else:
                bnd = (vals[i] + vals[i + 1]) / 2.0
            cdf = 0.5 * math.erfc(-bnd / math.sqrt(2.0))
            t = math.ceil(cdf * 2.0**32 - 0.5)
            thr.append(min(max(t, 0), 1 << 32))
        _tables["normal"] = (np.array(thr, np.uint64), np.array(order, np.uint8))
    return _tables["normal"]


def _threshold_codes(seed, stream, start, count, table) -> np.ndarray:
    """Code of word start + i: the number of thresholds <= its top 32 bits picks it.  Done in blocks
    of 2^20 words, so that the temporaries stay small (the same values as one whole-array pass)."""
    thr, codes = table
    out = np.empty(count, np.uint8)
    blk = 1 << 20
    for b0 in range(0, count, blk):
        n = min(blk, count - b0)
        r = words(seed, stream, start + b0, n) >> np.uint64(32)
        out[b0:b0 + n] = codes[np.searchsorted(thr, r, side="right")]
    return out


def scale_codes(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    return _threshold_codes(seed, stream, start, count, scale_thresholds())


def fp8_normal_codes(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    return _threshold_codes(seed, stream, start, count, fp8_normal_thresholds())


def normal_bf16(seed: int, stream: int, shape) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) samples, Box-Muller on two words per element."""
    import torch
    n = int(np.prod(shape))
    w = words(seed, stream, 0, 2 * n).reshape(n, 2)
    u1 = ((w[:, 0] >> np.uint64(11)).astype(np.float64) + 0.5) / 2.0**53
    u2 = ((w[:, 1] >> np.uint64(11)).astype(np.float64) + 0.5) / 2.0**53
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    t = torch.from_numpy(z).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).reshape(shape).copy()


def q4_scales_biases(seed: int, stream: int, start: int, count: int) -> tuple:
    """(scales, biases): bf16 bit patterns (uint16) of groups start .. start+count-1."""
    import torch
    w = words(seed, stream, 2 * start, 2 * count).reshape(count, 2)
    u = -8.0 + 4.0 * ((w[:, 0] >> np.uint64(11)).astype(np.float64) + 0.5) / 2.0**53
    v = ((w[:, 1] >> np.uint64(11)).astype(np.float64) + 0.5) / 2.0**53 - 0.5
    sc = torch.from_numpy(np.exp2(u)).to(torch.bfloat16)
    bi = torch.from_numpy(-sc.to(torch.float64).numpy() * (7.5 + v)).to(torch.bfloat16)
    as_bits = lambda t: t.view(torch.int16).numpy().view(np.uint16).copy()  # noqa: E731
    return as_bits(sc), as_bits(bi)


def uniform_ints(seed: int, stream: int, start: int, count: int, n: int) -> np.ndarray:
    """Integers uniform over [0, n) (multiply-shift on the top 32 bits)."""
    r = words(seed, stream, start, count) >> np.uint64(32)
    return ((r * np.uint64(n)) >> np.uint64(32)).astype(np.int64)


# ------------------------------------------------------------------ canonical tensors

def nvfp4_rows(seed: int, layer: int, codes_t: int, scales_t: int, K: int, rows) -> tuple:
    """Canonical NVFP4 rows (codes [len][K/2], scales [len][K/16]) of a generated matrix."""
    rows = np.asarray(rows, dtype=np.int64)
    c = np.stack([uniform_bytes(seed, stream_id(layer, codes_t), int(n) * (K // 2), K // 2) for n in rows]) \
        if rows.size else np.zeros((0, K // 2), np.uint8)
    s = np.stack([scale_codes(seed, stream_id(layer, scales_t), int(n) * (K // 16), K // 16) for n in rows]) \
        if rows.size else np.zeros((0, K // 16), np.uint8)
    return c, s


def nvfp4_matrix(seed: int, layer: int, codes_t: int, scales_t: int, N: int, K: int) -> tuple:
    c = uniform_bytes(seed, stream_id(layer, codes_t), 0, N * K // 2).reshape(N, K // 2)
    s = scale_codes(seed, stream_id(layer, scales_t), 0, N * K // 16).reshape(N, K // 16)
    return c, s


def fp8_rows(seed: int, layer: int, t: int, K: int, rows) -> np.ndarray:
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size == 0:
        return np.zeros((0, K), np.uint8)
    return np.stack([fp8_normal_codes(seed, stream_id(layer, t), int(n) * K, K) for n in rows])


def fp8_matrix(seed: int, layer: int, t: int, N: int, K: int) -> np.ndarray:
    return fp8_normal_codes(seed, stream_id(layer, t), 0, N * K).reshape(N, K)


def planted_pending(seed: int, t_ref: np.ndarray, vocab: int, prefix=None) -> tuple:
    """Anchor + 7 drafts per lane with a planted matching prefix of length p in 0..7.

    For lane l: p ~ U{0..7} (or ``prefix[l]``); drafts[j] = t_ref[8l + j] for j < p; if p < 7,
    drafts[p] = (t_ref[8l + p] + 1 + r) mod vocab with r uniform in [0, vocab - 1) (so it differs);
    later drafts are uniform over the vocabulary; pending[8l] is a uniform anchor token."""
    t_ref = np.asarray(t_ref, dtype=np.int64)
    lanes = t_ref.size // 8
    s = stream_id(0, T_PENDING)
    r = uniform_ints(seed, s, 0, 32 * lanes, vocab)
    ps = uniform_ints(seed, s + 1, 0, lanes, 8)
    pending = np.zeros(8 * lanes, np.int32)
    planted = np.zeros(lanes, np.int32)
    for l in range(lanes):
        p = int(prefix[l]) if prefix is not None else int(ps[l])
        planted[l] = p
        pending[8 * l] = r[32 * l]
        for j in range(7):
            if j < p:
                d = t_ref[8 * l + j]
            elif j == p:
                d = (t_ref[8 * l + j] + 1 + (r[32 * l + 1 + j] % max(vocab - 1, 1))) % vocab
            else:
                d = r[32 * l + 8 + j]
            pending[8 * l + j + 1] = d
    return pending, planted


# ------------------------------------------------------------------ device fill (synth.cu)

_HERE = os.path.dirname(os.path.abspath(__file__))
_CU = os.path.join(_HERE, "synth.cu")
_SO = os.path.join(_HERE, "libvpsynth.so")
_lock = threading.Lock()
_dev = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_CU):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a", "-Xcompiler", "-fPIC", "-shared",
           _CU, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _devlib():
    global _dev
    with _lock:
        if _dev is None:
            build()
            L = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            u64 = ctypes.c_uint64
            L.vps_fill_bytes.restype = ctypes.c_int
            L.vps_fill_bytes.argtypes = [P, u64, u64, u64, u64, P]
            L.vps_fill_threshold_codes.restype = ctypes.c_int
            L.vps_fill_threshold_codes.argtypes = [P, u64, u64, u64, u64, P, ctypes.c_int, P, P]
            _dev = L
    return _dev


def _cuda_stream_handle():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def gpu_uniform_bytes(t, seed: int, stream: int, start: int = 0) -> None:
    """Fills the uint8 CUDA tensor ``t`` with uniform_bytes(seed, stream, start, t.numel())."""
    rc = _devlib().vps_fill_bytes(ctypes.c_void_p(t.data_ptr()), t.numel(), seed & _M64, stream, start,
                                  _cuda_stream_handle())
    if rc != 0:
        raise RuntimeError(f"vps_fill_bytes failed ({rc})")


def _gpu_threshold_codes(t, seed, stream, start, table):
    import torch
    thr, codes = table
    thr_d = torch.from_numpy(thr.astype(np.uint64).view(np.int64)).to(t.device)
    codes_d = torch.from_numpy(codes.astype(np.uint8)).to(t.device)
    rc = _devlib().vps_fill_threshold_codes(ctypes.c_void_p(t.data_ptr()), t.numel(), seed & _M64, stream,
                                            start, ctypes.c_void_p(thr_d.data_ptr()), int(thr.size),
                                            ctypes.c_void_p(codes_d.data_ptr()), _cuda_stream_handle())
    if rc != 0:
        raise RuntimeError(f"vps_fill_threshold_codes failed ({rc})")
    torch.cuda.current_stream().synchronize()  # keep the small tables alive until the fill ran


def gpu_scale_codes(t, seed: int, stream: int, start: int = 0) -> None:
    _gpu_threshold_codes(t, seed, stream, start, scale_thresholds())


def gpu_fp8_normal_codes(t, seed: int, stream: int, start: int = 0) -> None:
    _gpu_threshold_codes(t, seed, stream, start, fp8_normal_thresholds())

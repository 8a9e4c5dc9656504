"""fp64 CPU oracle for the speculative-verify weight stream (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  The product library never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one thread per output row); this module only
builds it with gcc and marshals numpy arrays through ctypes.  Every function cites, in the C source,
the passage of the pages it follows:

* "lithos-metal: per-layer megakernels for Qwen3.8-27B on an M5 Max" -- "What one token costs the
  bus" (byte table), "Formats, and what runs where" (NVFP4 = E2M1 code x E4M3 block scale per 16 x
  FP32 tensor-scale multiplier; scale codes top out at 448; BF16 activations, wide accumulation),
  "The megakernel is per layer, not per step" (greedy acceptance, 1..8 tokens per round).
* "144 tok/s needs 502 GB/s" (Splash) -- "The engine hard-codes the model" (geometry).
* "Beating Splash on an M5 Max" -- "The bugs a second reviewer found" (one argmax tie rule).
* "144 tok/s needs 502 GB/s" -- "The engine hard-codes the model" (the affine 4-bit "Q4" format:
  per group of 64 inputs, 32 bytes of codes, a bf16 scale and a bf16 bias; ``linear_q4``) and "Exact,
  up to top-32" (speculative sampling over the top_k <= 32 target candidates; ``sample_accept``).
* "lithos-metal ..." -- "The megakernel is per layer, not per step" (the attention core over a BF16
  KV cache with online-softmax partitions and a sigmoid gate; ``attention_verify``; the GDN commit
  re-scan) and "Beating Splash ..." -- "What actually moved the needle" (double-buffered GDN state,
  re-scan of the committed rows; ``gdn_scan``, with the published gated delta rule).
* "Speculative decoding" (mlx-dspark) -- "Lookup (no drafter)", "Lookup drafts" (the continuation of
  an earlier match of the current text is a free draft; ``lookup_drafts``); the embedding gather
  (``embed_nvfp4``) and the history append (``commit_append``) of a decode loop.

Parity status: every function here is pinned by a ``-m "not gpu"`` test against page values,
closed forms, library routines or brute force, except the 64-layer surrogate chain, whose
end-to-end fp64 result is only pinned through its parts and a small independent re-composition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

NVFP4 = 0
FP8 = 1
PTRS_PER_LAYER = 9
SCALES_PER_LAYER = 6


def build(force: bool = False) -> str:
    """Compiles oracle.c into liboracle.so with gcc (portable flags, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-D_DEFAULT_SOURCE", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class Geom(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("inter", ctypes.c_int),
                ("vocab", ctypes.c_int), ("period", ctypes.c_int), ("gdn_in", ctypes.c_int),
                ("gdn_z", ctypes.c_int), ("attn_q", ctypes.c_int), ("attn_kv", ctypes.c_int),
                ("attn_z", ctypes.c_int), ("eps", ctypes.c_double)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            L.orc_e2m1.restype = ctypes.c_double
            L.orc_e2m1.argtypes = [ctypes.c_int]
            L.orc_e4m3.restype = ctypes.c_double
            L.orc_e4m3.argtypes = [ctypes.c_int]
            L.orc_tables.argtypes = [P, P]
            L.orc_bf16_value.restype = ctypes.c_double
            L.orc_bf16_value.argtypes = [ctypes.c_uint16]
            L.orc_bf16_values.argtypes = [P, P, ctypes.c_int64]
            L.orc_bf16_round1.restype = ctypes.c_uint16
            L.orc_bf16_round1.argtypes = [ctypes.c_double]
            L.orc_bf16_round.argtypes = [P, P, ctypes.c_int64]
            L.orc_linear.restype = ctypes.c_int
            L.orc_linear.argtypes = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                     ctypes.c_double, P, ctypes.c_int64, P, P, ctypes.c_int]
            L.orc_linear_q4.restype = ctypes.c_int
            L.orc_linear_q4.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, ctypes.c_int64,
                                        P, P, ctypes.c_int]
            L.orc_q4_bytes.restype = ctypes.c_int64
            L.orc_q4_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
            L.orc_target_dist.restype = ctypes.c_int
            L.orc_target_dist.argtypes = [P, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_double, P, P, P]
            L.orc_sample_accept.restype = ctypes.c_int
            L.orc_sample_accept.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                            ctypes.c_double, P, P, P, P, P, P, P]
            L.orc_attention_verify.restype = ctypes.c_int
            L.orc_attention_verify.argtypes = [P, P, P, P, P, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, P, P]
            L.orc_gdn_scan.restype = ctypes.c_int
            L.orc_gdn_scan.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, P]
            L.orc_embed_nvfp4.argtypes = [P, P, ctypes.c_double, P, ctypes.c_int, ctypes.c_int, P]
            L.orc_lookup_drafts.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
            L.orc_commit_append.restype = ctypes.c_int
            L.orc_commit_append.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_silu_mul.argtypes = [P, P, ctypes.c_int64, P]
            L.orc_rmsnorm.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_double, P]
            L.orc_argmax.restype = ctypes.c_int64
            L.orc_argmax.argtypes = [P, ctypes.c_int64]
            L.orc_accept.argtypes = [P, P, ctypes.c_int, P, P]
            L.orc_accept_rows.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_lookup_drafts_rows.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
            L.orc_commit_append_rows.restype = ctypes.c_int
            L.orc_commit_append_rows.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
            L.orc_verify_pass.restype = ctypes.c_int
            L.orc_verify_pass.argtypes = [ctypes.POINTER(Geom), P, P, P, P, ctypes.c_double, P,
                                          ctypes.c_int, P, P, P, P, P, P, P, ctypes.c_int]
            L.orc_pass_bytes.argtypes = [ctypes.POINTER(Geom), P]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return os.cpu_count() or 1


def e2m1_table() -> np.ndarray:
    a = np.zeros(16, np.float64)
    b = np.zeros(256, np.float64)
    lib().orc_tables(_p(a), _p(b))
    return a


def e4m3_table() -> np.ndarray:
    a = np.zeros(16, np.float64)
    b = np.zeros(256, np.float64)
    lib().orc_tables(_p(a), _p(b))
    return b


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float64)
    lib().orc_bf16_values(_p(bits), _p(out), bits.size)
    return out


def bf16_round(v: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns, round to nearest even, rounding once."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_round(_p(v), _p(out), v.size)
    return out


def linear(fmt: int, x_bf16: np.ndarray, codes: np.ndarray, scales: np.ndarray | None, ts: float,
           N: int, rows: np.ndarray | None = None, with_abs: bool = True, nthreads: int | None = None):
    """y[m][i] = sum_k x[m][k] w[rows[i]][k] (fp64) and a = sum_k |x w| (tolerance scale).

    x_bf16: uint16 [M][K]; codes: NVFP4 uint8 [N][K/2] or FP8 uint8 [N][K]; scales: NVFP4 uint8
    [N][K/16].  rows: optional int32 subset of output rows (codes/scales still hold all N rows, or
    exactly the listed rows when ``rows`` indexes into a row-sampled array)."""
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x_bf16.shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint8) if scales is not None else None
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        n_rows = rows.size
    else:
        n_rows = N
    y = np.zeros((M, n_rows), np.float64)
    a = np.zeros((M, n_rows), np.float64) if with_abs else None
    rc = lib().orc_linear(fmt, _p(x_bf16), M, K, N, _p(codes), _p(sc) if sc is not None else None,
                          float(ts), _p(rows) if rows is not None else None, n_rows, _p(y),
                          _p(a) if a is not None else None, nthreads or default_threads())
    if rc != 0:
        raise ValueError("orc_linear rejected its arguments")
    return (y, a) if with_abs else y


def linear_q4(x_bf16: np.ndarray, codes: np.ndarray, scales: np.ndarray, biases: np.ndarray, N: int,
              rows: np.ndarray | None = None, with_abs: bool = True, nthreads: int | None = None):
    """Affine INT4 linear: y[m][i] = sum_k x[m][k] (scale * q + bias)[rows[i]][k] (fp64), and
    a = sum_k |x| (|scale * q| + |bias|) (tolerance scale).  codes uint8 [N][K/2] (low nibble first),
    scales / biases bf16 bit patterns (uint16) [N][K/64]."""
    x_bf16 = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x_bf16.shape
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(scales, dtype=np.uint16)
    bi = np.ascontiguousarray(biases, dtype=np.uint16)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        n_rows = rows.size
    else:
        n_rows = N
    y = np.zeros((M, n_rows), np.float64)
    a = np.zeros((M, n_rows), np.float64) if with_abs else None
    rc = lib().orc_linear_q4(_p(x_bf16), M, K, N, _p(codes), _p(sc), _p(bi), _p(rows) if rows is not None else None,
                             n_rows, _p(y), _p(a) if a is not None else None, nthreads or default_threads())
    if rc != 0:
        raise ValueError("orc_linear_q4 rejected its arguments")
    return (y, a) if with_abs else y


def q4_bytes(N: int, K: int) -> int:
    return int(lib().orc_q4_bytes(N, K))


def target_dist(logits_row: np.ndarray, temperature: float, top_k: int, top_p: float):
    """(tokens, probs, margin): one row's sampling distribution -- top_k candidates (larger logit
    first, lower index among equals), temperature, top_p truncation, renormalised."""
    v = np.ascontiguousarray(logits_row, dtype=np.float64).reshape(-1)
    tok = np.zeros(32, np.int32)
    prob = np.zeros(32, np.float64)
    mg = np.zeros(1, np.float64)
    n = lib().orc_target_dist(_p(v), v.size, float(temperature), int(top_k), float(top_p), _p(tok), _p(prob), _p(mg))
    if n <= 0:
        raise ValueError("orc_target_dist rejected its arguments")
    return tok[:n].copy(), prob[:n].copy(), float(mg[0])


def sample_accept(logits: np.ndarray, temperature: float, top_k: int, top_p: float, pending: np.ndarray,
                  draft_tokens: np.ndarray | None, draft_probs: np.ndarray | None, uniforms: np.ndarray):
    """Speculative sampling per lane (see orc_sample_accept): returns (n_commit [L], committed [L][8],
    margin [L])."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    M, V = lg.shape
    pend = np.ascontiguousarray(pending, dtype=np.int32)
    dt = np.ascontiguousarray(draft_tokens, dtype=np.int32) if draft_tokens is not None else None
    dp = np.ascontiguousarray(draft_probs, dtype=np.float64) if draft_probs is not None else None
    u = np.ascontiguousarray(uniforms, dtype=np.float64)
    L = M // 8
    nc = np.zeros(L, np.int32)
    cm = np.zeros((L, 8), np.int32)
    mg = np.zeros(L, np.float64)
    rc = lib().orc_sample_accept(_p(lg), M, V, float(temperature), int(top_k), float(top_p), _p(pend),
                                 _p(dt) if dt is not None else None, _p(dp) if dp is not None else None, _p(u),
                                 _p(nc), _p(cm), _p(mg))
    if rc != 0:
        raise ValueError("orc_sample_accept rejected its arguments")
    return nc, cm, mg


def attention_verify(q, k_new, v_new, k_cache, v_cache, ctx, gate=None, with_abs=True):
    """Causal attention of the verify rows over each lane's cache plus the rows' own appended keys
    (see orc_attention_verify); bf16 bit patterns in, fp64 [M][Hq][D] out (and the tolerance scale)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    M, Hq, D = q.shape
    kc = np.ascontiguousarray(k_cache, dtype=np.uint16)
    L, Hkv, cap, _ = kc.shape
    args = [np.ascontiguousarray(x, dtype=np.uint16) for x in (k_new, v_new, v_cache)]
    ctx = np.ascontiguousarray(ctx, dtype=np.int32)
    g = np.ascontiguousarray(gate, dtype=np.uint16) if gate is not None else None
    out = np.zeros((M, Hq, D), np.float64)
    a = np.zeros((M, Hq, D), np.float64) if with_abs else None
    rc = lib().orc_attention_verify(_p(q), _p(args[0]), _p(args[1]), _p(kc), _p(args[2]), _p(ctx), cap,
                                    _p(g) if g is not None else None, M, Hq, Hkv, D, _p(out),
                                    _p(a) if a is not None else None)
    if rc != 0:
        raise ValueError("orc_attention_verify rejected its arguments")
    return (out, a) if with_abs else out


def gdn_scan(state_in, q, k, v, alpha, beta, rows, want_out=True):
    """Gated delta rule scan of each lane's first rows[l] verify rows from state_in [L][H][dv][dk]
    (see orc_gdn_scan); returns (state_out fp64, out fp64 [M][H][dv] or None)."""
    st = np.ascontiguousarray(state_in, dtype=np.float64)
    L, H, dv, dk = st.shape
    q = np.ascontiguousarray(q, dtype=np.uint16)
    M = q.shape[0]
    kk = np.ascontiguousarray(k, dtype=np.uint16)
    vv = np.ascontiguousarray(v, dtype=np.uint16)
    a = np.ascontiguousarray(alpha, dtype=np.float64)
    b = np.ascontiguousarray(beta, dtype=np.float64)
    rw = np.ascontiguousarray(rows, dtype=np.int32)
    so = np.zeros_like(st)
    out = np.zeros((M, H, dv), np.float64) if want_out else None
    rc = lib().orc_gdn_scan(_p(st), _p(so), _p(q), _p(kk), _p(vv), _p(a), _p(b), _p(rw), M, H, dk, dv,
                            _p(out) if out is not None else None)
    if rc != 0:
        raise ValueError("orc_gdn_scan rejected its arguments")
    return so, out


def embed_nvfp4(codes: np.ndarray, scales: np.ndarray, ts: float, tokens: np.ndarray) -> np.ndarray:
    """Rows of a canonical NVFP4 table as bf16 bit patterns [M][K] (one rounding)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    K = codes.shape[1] * 2
    out = np.zeros((tokens.size, K), np.uint16)
    lib().orc_embed_nvfp4(_p(codes), _p(scales), float(ts), _p(tokens), tokens.size, K, _p(out))
    return out


def lookup_drafts(hist: np.ndarray, hist_len: np.ndarray, max_match: int = 8, rows: int = 8) -> np.ndarray:
    """Anchor + rows - 1 lookup drafts per lane (int32 [rows L]) from histories [L][cap]."""
    hist = np.ascontiguousarray(hist, dtype=np.int32)
    L, cap = hist.shape
    hl = np.ascontiguousarray(hist_len, dtype=np.int32)
    out = np.zeros(rows * L, np.int32)
    if rows == 8:
        lib().orc_lookup_drafts(_p(hist), _p(hl), L, cap, int(max_match), _p(out))
    else:
        lib().orc_lookup_drafts_rows(_p(hist), _p(hl), L, cap, int(max_match), int(rows), _p(out))
    return out


def commit_append(hist: np.ndarray, hist_len: np.ndarray, n_commit: np.ndarray, committed: np.ndarray) -> int:
    """Appends each lane's committed tokens (committed [L][rows]) in place; returns 0, or -1 if a lane's
    history is full."""
    assert hist.dtype == np.int32 and hist.flags.c_contiguous and hist_len.dtype == np.int32
    L, cap = hist.shape
    nc = np.ascontiguousarray(n_commit, dtype=np.int32)
    cm = np.ascontiguousarray(committed, dtype=np.int32)
    rows = cm.size // L
    if rows == 8:
        return int(lib().orc_commit_append(_p(hist), _p(hist_len), L, cap, _p(nc), _p(cm)))
    return int(lib().orc_commit_append_rows(_p(hist), _p(hist_len), L, cap, int(rows), _p(nc), _p(cm)))


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    out = np.empty_like(g)
    lib().orc_silu_mul(_p(g), _p(u), g.size, _p(out))
    return out


def rmsnorm(h_bf16: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    h = np.ascontiguousarray(h_bf16, dtype=np.uint16)
    M, D = h.shape
    out = np.empty_like(h)
    lib().orc_rmsnorm(_p(h), M, D, float(eps), _p(out))
    return out


def argmax(v: np.ndarray) -> int:
    v = np.ascontiguousarray(v, dtype=np.float64).reshape(-1)
    return int(lib().orc_argmax(_p(v), v.size))


def accept(t: np.ndarray, pending: np.ndarray, rows: int = 8):
    """Greedy acceptance per lane of `rows` verify rows (anchor + rows - 1 drafts): n_commit [lanes],
    committed [lanes][rows]."""
    t = np.ascontiguousarray(t, dtype=np.int32)
    pending = np.ascontiguousarray(pending, dtype=np.int32)
    lanes = t.size // rows
    nc = np.zeros(lanes, np.int32)
    cm = np.zeros((lanes, rows), np.int32)
    if rows == 8:
        lib().orc_accept(_p(t), _p(pending), lanes, _p(nc), _p(cm))
    else:
        lib().orc_accept_rows(_p(t), _p(pending), lanes, int(rows), _p(nc), _p(cm))
    return nc, cm


def geom(n_layers=64, hidden=5120, inter=17408, vocab=248320, period=4, gdn_in=16384, gdn_z=6144,
         attn_q=12288, attn_kv=2048, attn_z=6144, eps=1e-6) -> Geom:
    return Geom(n_layers, hidden, inter, vocab, period, gdn_in, gdn_z, attn_q, attn_kv, attn_z, eps)


def pass_bytes(g: Geom) -> np.ndarray:
    out = np.zeros(6, np.int64)
    lib().orc_pass_bytes(ctypes.byref(g), _p(out))
    return out


def verify_pass(g: Geom, layers: list, head: tuple, x0_bf16: np.ndarray, pending: np.ndarray,
                want_trace: bool = False, want_logits: bool = False, nthreads: int | None = None):
    """Runs the surrogate pass.  ``layers[l]`` is a dict with keys in, kv (None on GDN layers), out,
    gate_c, gate_s, up_c, up_s, down_c, down_s (canonical uint8 arrays) and s_in, s_kv, s_out,
    ts_gate, ts_up, ts_down (floats).  ``head`` = (codes, scales, ts)."""
    L = g.n_layers
    keep = []
    ptrs = (ctypes.c_void_p * (L * PTRS_PER_LAYER))()
    scs = np.zeros(L * SCALES_PER_LAYER, np.float64)
    names = ["in", "kv", "out", "gate_c", "gate_s", "up_c", "up_s", "down_c", "down_s"]
    snames = ["s_in", "s_kv", "s_out", "ts_gate", "ts_up", "ts_down"]
    for l, d in enumerate(layers):
        for j, nm in enumerate(names):
            a = d.get(nm)
            if a is None:
                ptrs[l * PTRS_PER_LAYER + j] = None
            else:
                a = np.ascontiguousarray(a, dtype=np.uint8)
                keep.append(a)
                ptrs[l * PTRS_PER_LAYER + j] = a.ctypes.data
        for j, nm in enumerate(snames):
            scs[l * SCALES_PER_LAYER + j] = float(d.get(nm, 1.0))
    hc = np.ascontiguousarray(head[0], dtype=np.uint8)
    hs = np.ascontiguousarray(head[1], dtype=np.uint8)
    x0 = np.ascontiguousarray(x0_bf16, dtype=np.uint16)
    M = x0.shape[0]
    pend = np.ascontiguousarray(pending, dtype=np.int32)
    am = np.zeros(M, np.int32)
    nc = np.zeros(M // 8, np.int32)
    cm = np.zeros((M // 8, 8), np.int32)
    trace = np.zeros((2 * L, M, g.hidden), np.uint16) if want_trace else None
    logits = np.zeros((M, g.vocab), np.float64) if want_logits else None
    final_r = np.zeros((M, g.hidden), np.uint16)
    rc = lib().orc_verify_pass(ctypes.byref(g), ctypes.cast(ptrs, ctypes.c_void_p), _p(scs), _p(hc),
                               _p(hs), float(head[2]), _p(x0), M, _p(pend), _p(am), _p(nc), _p(cm),
                               _p(trace) if trace is not None else None,
                               _p(logits) if logits is not None else None, _p(final_r),
                               nthreads or default_threads())
    if rc != 0:
        raise ValueError("orc_verify_pass rejected its arguments")
    return {"argmax": am, "n_commit": nc, "committed": cm, "trace": trace, "logits": logits,
            "final_r": final_r}

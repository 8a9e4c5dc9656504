"""ctypes binding of libverify (include/verify.h): argument marshalling only.

Every function keeps its C name.  Pointer arguments accept a torch tensor (its data_ptr), a plain
integer address, or None (NULL).  Workspace sizes are taken from the tensor when not given.  The
stream defaults to torch's current CUDA stream.  A non-VP_OK status raises VerifyError.  There is no
fallback: if libverify.so has not been built, importing fails with an explicit message.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# VP_LIBVERIFY may name another build of the same library (the phase-traced libverify_trace.so).
LIB_PATH = os.environ.get("VP_LIBVERIFY") or os.path.join(_PKG, "libverify.so")

VP_OK, VP_ERR_INVALID_ARG, VP_ERR_SHAPE, VP_ERR_ALIGNMENT, VP_ERR_WORKSPACE, VP_ERR_CUDA, VP_ERR_TIMEOUT, \
    VP_ERR_UNSUPPORTED = range(8)
VP_OP_NVFP4, VP_OP_FP8, VP_OP_HEAD, VP_OP_ARGMAX, VP_OP_Q4, VP_OP_SAMPLE, VP_OP_ATTN = range(7)
VP_LAYER_GDN, VP_LAYER_ATTN = 0, 1

# Every symbol include/verify.h declares.
EXPORTS = [
    "vp_status_string", "vp_get_last_cuda_error", "vp_workspace_init", "vp_read_status", "vp_packed_bytes_nvfp4",
    "vp_packed_bytes_fp8", "vp_pack_nvfp4", "vp_pack_fp8", "vp_workspace_bytes", "vp_linear_nvfp4",
    "vp_linear_fp8", "vp_head_argmax_accept", "vp_argmax_accept", "vp_model_create", "vp_model_destroy",
    "vp_pass_workspace_bytes", "vp_verify_pass", "vp_verify_blocks", "vp_pass_launch_count",
    "vp_linear_nvfp4_noalloc", "vp_noalloc_read_status", "vp_trace_read", "vp_packed_bytes_q4", "vp_pack_q4", "vp_linear_q4",
    "vp_sample_accept", "vp_attention_verify", "vp_gdn_scan", "vp_embed_nvfp4", "vp_lookup_drafts",
    "vp_commit_append", "vp_decode_steps", "vp_pass_sampled_workspace_bytes", "vp_verify_pass_sampled",
    "vp_argmax_accept_rows", "vp_verify_pass_rows", "vp_lookup_drafts_rows", "vp_commit_append_rows",
    "vp_decode_steps_rows",
    "vp_model_set_cores", "vp_pass_cores_workspace_bytes", "vp_verify_pass_cores", "vp_pass_cores_launch_count", "vp_commit_cores",
]


class VerifyError(RuntimeError):
    def __init__(self, name: str, status: int):
        self.status = status
        msg = f"{name} failed: {status_string(status)}"
        if status == VP_ERR_CUDA:
            msg += f" (cuda error {_L.vp_get_last_cuda_error()})"
        super().__init__(msg)


class vp_layer_desc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int),
                ("w_in", ctypes.c_void_p), ("s_in", ctypes.c_float), ("n_in", ctypes.c_int),
                ("w_kv", ctypes.c_void_p), ("s_kv", ctypes.c_float), ("n_kv", ctypes.c_int),
                ("w_out", ctypes.c_void_p), ("s_out", ctypes.c_float), ("k_out", ctypes.c_int),
                ("w_gate", ctypes.c_void_p), ("ts_gate", ctypes.c_float),
                ("w_up", ctypes.c_void_p), ("ts_up", ctypes.c_float),
                ("w_down", ctypes.c_void_p), ("ts_down", ctypes.c_float)]


class vp_core_desc(ctypes.Structure):
    _fields_ = [("w_a", ctypes.c_void_p), ("w_b", ctypes.c_void_p), ("conv_taps", ctypes.c_void_p),
                ("a_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p),
                ("state_a", ctypes.c_void_p), ("state_b", ctypes.c_void_p), ("window_a", ctypes.c_void_p),
                ("conv_hist", ctypes.c_void_p), ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p)]


class vp_core_geom(ctypes.Structure):
    _fields_ = [("n_qk", ctypes.c_int), ("n_v", ctypes.c_int), ("d", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("D", ctypes.c_int), ("cap", ctypes.c_int)]


class vp_head_desc(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("ts", ctypes.c_float), ("vocab", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libverify.so is not built ({LIB_PATH}); run weight_streaming_gb300.build.build() "
                          "(nvcc, sm_103a) first -- there is no fallback implementation")
    L = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "vp_status_string": (ctypes.c_char_p, [I]),
        "vp_get_last_cuda_error": (I, []),
        "vp_workspace_init": (I, [P, S, P]),
        "vp_read_status": (I, [P, ctypes.POINTER(I), P]),
        "vp_packed_bytes_nvfp4": (S, [I, I]),
        "vp_packed_bytes_fp8": (S, [I, I]),
        "vp_pack_nvfp4": (I, [P, P, I, I, P, S, P]),
        "vp_pack_fp8": (I, [P, I, I, P, S, P]),
        "vp_workspace_bytes": (S, [I, I, I, I]),
        "vp_linear_nvfp4": (I, [P, F, P, P, I, I, I, P, S, P]),
        "vp_linear_fp8": (I, [P, F, P, P, I, I, I, P, S, P]),
        "vp_head_argmax_accept": (I, [P, F, P, I, I, I, P, P, P, P, P, P, S, P]),
        "vp_argmax_accept": (I, [P, I, I, P, P, P, P, P, S, P]),
        "vp_argmax_accept_rows": (I, [P, I, I, I, P, P, P, P, P, S, P]),
        "vp_verify_pass_rows": (I, [P, P, I, I, P, P, P, P, P, P, P, S, P]),
        "vp_lookup_drafts_rows": (I, [P, P, I, I, I, I, P, P, P]),
        "vp_commit_append_rows": (I, [P, P, I, I, I, P, P, P, P]),
        "vp_decode_steps_rows": (I, [P, I, I, P, P, F, I, I, P, P, I, I, I, P, P, P, P, P, P, S, P, P]),
        "vp_model_create": (I, [I, I, F, ctypes.POINTER(vp_layer_desc), I, ctypes.POINTER(vp_head_desc),
                                ctypes.POINTER(P)]),
        "vp_model_destroy": (None, [P]),
        "vp_pass_workspace_bytes": (S, [P, I]),
        "vp_verify_pass": (I, [P, P, I, P, P, P, P, P, P, P, S, P]),
        "vp_verify_blocks": (I, [P, P, I, I, I, P, P, S, P]),
        "vp_pass_launch_count": (I, [P]),
        "vp_linear_nvfp4_noalloc": (I, [P, F, P, P, I, I, I, P]),
        "vp_noalloc_read_status": (I, [ctypes.POINTER(I), P]),
        "vp_trace_read": (I, [I, P, S, ctypes.POINTER(ctypes.c_uint)]),
        "vp_packed_bytes_q4": (S, [I, I]),
        "vp_pack_q4": (I, [P, P, P, I, I, P, S, P]),
        "vp_linear_q4": (I, [P, P, P, I, I, I, P, S, P]),
        "vp_sample_accept": (I, [P, I, I, F, I, F, P, P, P, P, P, P, P, S, P]),
        "vp_attention_verify": (I, [P, P, P, P, P, P, I, P, P, I, I, I, I, P, S, P]),
        "vp_gdn_scan": (I, [P, P, P, P, P, P, P, P, I, I, I, I, P, P]),
        "vp_embed_nvfp4": (I, [P, P, F, P, I, I, I, P, P, P]),
        "vp_lookup_drafts": (I, [P, P, I, I, I, P, P, P]),
        "vp_commit_append": (I, [P, P, I, I, P, P, P, P]),
        "vp_decode_steps": (I, [P, I, P, P, F, I, I, P, P, I, I, I, P, P, P, P, P, P, S, P, P]),
        "vp_pass_sampled_workspace_bytes": (S, [P, I]),
        "vp_verify_pass_sampled": (I, [P, P, I, P, F, I, F, P, P, P, P, P, P, P, P, S, P]),
        "vp_model_set_cores": (I, [P, ctypes.POINTER(vp_core_geom), ctypes.POINTER(vp_core_desc), I]),
        "vp_pass_cores_workspace_bytes": (S, [P, I]),
        "vp_verify_pass_cores": (I, [P, P, I, P, I, P, P, P, P, P, P, P, S, P]),
        "vp_commit_cores": (I, [P, I, P, I, P, S, P]),
        "vp_pass_cores_launch_count": (I, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


_L = _load()


def lib():
    return _L


def status_string(s: int) -> str:
    return _L.vp_status_string(int(s)).decode()


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, st):
    if st != VP_OK:
        raise VerifyError(name, st)


def vp_packed_bytes_nvfp4(N: int, K: int) -> int:
    return _L.vp_packed_bytes_nvfp4(N, K)


def vp_packed_bytes_fp8(N: int, K: int) -> int:
    return _L.vp_packed_bytes_fp8(N, K)


def vp_packed_bytes_q4(N: int, K: int) -> int:
    return _L.vp_packed_bytes_q4(N, K)


def vp_workspace_bytes(op: int, M: int, N: int, K: int) -> int:
    return _L.vp_workspace_bytes(op, M, N, K)


def vp_pack_nvfp4(codes, scales, N: int, K: int, packed, stream=None, packed_bytes=None):
    pb = packed_bytes if packed_bytes is not None else _nbytes(packed)
    _check("vp_pack_nvfp4", _L.vp_pack_nvfp4(_ptr(codes), _ptr(scales), N, K, _ptr(packed), pb, _stream(stream)))


def vp_pack_fp8(w, N: int, K: int, packed, stream=None, packed_bytes=None):
    pb = packed_bytes if packed_bytes is not None else _nbytes(packed)
    _check("vp_pack_fp8", _L.vp_pack_fp8(_ptr(w), N, K, _ptr(packed), pb, _stream(stream)))


def vp_pack_q4(codes, scales, biases, N: int, K: int, packed, stream=None, packed_bytes=None):
    pb = packed_bytes if packed_bytes is not None else _nbytes(packed)
    _check("vp_pack_q4", _L.vp_pack_q4(_ptr(codes), _ptr(scales), _ptr(biases), N, K, _ptr(packed), pb,
                                       _stream(stream)))


def vp_linear_q4(w_packed, x, y, M: int, N: int, K: int, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_linear_q4", _L.vp_linear_q4(_ptr(w_packed), _ptr(x), _ptr(y), M, N, K, _ptr(ws), wb, _stream(stream)))


def vp_linear_nvfp4(w_packed, tensor_scale: float, x, y, M: int, N: int, K: int, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_linear_nvfp4", _L.vp_linear_nvfp4(_ptr(w_packed), tensor_scale, _ptr(x), _ptr(y), M, N, K, _ptr(ws),
                                                 wb, _stream(stream)))


def vp_linear_nvfp4_noalloc(w_packed, tensor_scale: float, x, y, M: int, N: int, K: int, stream=None):
    """vp_linear_nvfp4 on the library's own fixed scratch (no workspace argument, nothing allocated);
    calls must not overlap in time (see include/verify.h)."""
    _check("vp_linear_nvfp4_noalloc", _L.vp_linear_nvfp4_noalloc(_ptr(w_packed), tensor_scale, _ptr(x), _ptr(y), M,
                                                                 N, K, _stream(stream)))


def vp_noalloc_read_status(stream=None) -> int:
    """Status word of the last vp_linear_nvfp4_noalloc call on this device (synchronises the stream)."""
    out = ctypes.c_int(-1)
    _check("vp_noalloc_read_status", _L.vp_noalloc_read_status(ctypes.byref(out), _stream(stream)))
    return out.value


def vp_linear_fp8(w_packed, scale: float, x, y, M: int, N: int, K: int, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_linear_fp8", _L.vp_linear_fp8(_ptr(w_packed), scale, _ptr(x), _ptr(y), M, N, K, _ptr(ws), wb,
                                             _stream(stream)))


def vp_head_argmax_accept(w_packed, tensor_scale: float, x, M: int, V: int, K: int, pending, argmax, n_commit,
                          committed, logits, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_head_argmax_accept",
           _L.vp_head_argmax_accept(_ptr(w_packed), tensor_scale, _ptr(x), M, V, K, _ptr(pending), _ptr(argmax),
                                    _ptr(n_commit), _ptr(committed), _ptr(logits), _ptr(ws), wb, _stream(stream)))


def vp_argmax_accept(logits, M: int, V: int, pending, argmax, n_commit, committed, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_argmax_accept", _L.vp_argmax_accept(_ptr(logits), M, V, _ptr(pending), _ptr(argmax), _ptr(n_commit),
                                                   _ptr(committed), _ptr(ws), wb, _stream(stream)))


def vp_argmax_accept_rows(logits, M: int, V: int, rows: int, pending, argmax, n_commit, committed, ws, stream=None,
                          ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_argmax_accept_rows", _L.vp_argmax_accept_rows(_ptr(logits), M, V, rows, _ptr(pending), _ptr(argmax),
                                                             _ptr(n_commit), _ptr(committed), _ptr(ws), wb,
                                                             _stream(stream)))


def vp_sample_accept(logits, M: int, V: int, temperature: float, top_k: int, top_p: float, pending, draft_tokens,
                     draft_probs, uniforms, n_commit, committed, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_sample_accept",
           _L.vp_sample_accept(_ptr(logits), M, V, temperature, top_k, top_p, _ptr(pending), _ptr(draft_tokens),
                               _ptr(draft_probs), _ptr(uniforms), _ptr(n_commit), _ptr(committed), _ptr(ws), wb,
                               _stream(stream)))


def vp_attention_verify(q, k_new, v_new, k_cache, v_cache, ctx, cap: int, gate, out, M: int, Hq: int, Hkv: int,
                        D: int, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_attention_verify",
           _L.vp_attention_verify(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(ctx), cap,
                                  _ptr(gate), _ptr(out), M, Hq, Hkv, D, _ptr(ws), wb, _stream(stream)))


def vp_gdn_scan(state_in, state_out, q, k, v, alpha, beta, rows, M: int, H: int, dk: int, dv: int, out,
                stream=None):
    _check("vp_gdn_scan", _L.vp_gdn_scan(_ptr(state_in), _ptr(state_out), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                         _ptr(beta), _ptr(rows), M, H, dk, dv, _ptr(out), _stream(stream)))


def vp_embed_nvfp4(codes, scales, ts: float, tokens, M: int, V: int, K: int, x, status=None, stream=None):
    _check("vp_embed_nvfp4", _L.vp_embed_nvfp4(_ptr(codes), _ptr(scales), ts, _ptr(tokens), M, V, K, _ptr(x),
                                               _ptr(status), _stream(stream)))


def vp_lookup_drafts(hist, hist_len, lanes: int, cap: int, max_match: int, pending, status=None, stream=None):
    _check("vp_lookup_drafts", _L.vp_lookup_drafts(_ptr(hist), _ptr(hist_len), lanes, cap, max_match, _ptr(pending),
                                                   _ptr(status), _stream(stream)))


def vp_lookup_drafts_rows(hist, hist_len, lanes: int, rows: int, cap: int, max_match: int, pending, status=None,
                          stream=None):
    _check("vp_lookup_drafts_rows", _L.vp_lookup_drafts_rows(_ptr(hist), _ptr(hist_len), lanes, rows, cap, max_match,
                                                             _ptr(pending), _ptr(status), _stream(stream)))


def vp_commit_append_rows(hist, hist_len, lanes: int, rows: int, cap: int, n_commit, committed, status=None,
                          stream=None):
    _check("vp_commit_append_rows", _L.vp_commit_append_rows(_ptr(hist), _ptr(hist_len), lanes, rows, cap,
                                                             _ptr(n_commit), _ptr(committed), _ptr(status),
                                                             _stream(stream)))


def vp_commit_append(hist, hist_len, lanes: int, cap: int, n_commit, committed, status=None, stream=None):
    _check("vp_commit_append", _L.vp_commit_append(_ptr(hist), _ptr(hist_len), lanes, cap, _ptr(n_commit),
                                                   _ptr(committed), _ptr(status), _stream(stream)))


def vp_decode_steps(model: "vp_model", steps: int, emb_codes, emb_scales, emb_ts: float, vocab: int, hidden: int,
                    hist, hist_len, cap: int, lanes: int, max_match: int, pending, x0, argmax, n_commit, committed,
                    ws, status=None, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_decode_steps",
           _L.vp_decode_steps(model.handle, steps, _ptr(emb_codes), _ptr(emb_scales), emb_ts, vocab, hidden,
                              _ptr(hist), _ptr(hist_len), cap, lanes, max_match, _ptr(pending), _ptr(x0),
                              _ptr(argmax), _ptr(n_commit), _ptr(committed), _ptr(ws), wb, _ptr(status),
                              _stream(stream)))


def vp_decode_steps_rows(model: "vp_model", steps: int, rows: int, emb_codes, emb_scales, emb_ts: float, vocab: int,
                         hidden: int, hist, hist_len, cap: int, lanes: int, max_match: int, pending, x0, argmax,
                         n_commit, committed, ws, status=None, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_decode_steps_rows",
           _L.vp_decode_steps_rows(model.handle, steps, rows, _ptr(emb_codes), _ptr(emb_scales), emb_ts, vocab,
                                   hidden, _ptr(hist), _ptr(hist_len), cap, lanes, max_match, _ptr(pending),
                                   _ptr(x0), _ptr(argmax), _ptr(n_commit), _ptr(committed), _ptr(ws), wb,
                                   _ptr(status), _stream(stream)))


def vp_workspace_init(ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_workspace_init", _L.vp_workspace_init(_ptr(ws), wb, _stream(stream)))


def vp_read_status(ws, stream=None) -> int:
    out = ctypes.c_int(-1)
    _check("vp_read_status", _L.vp_read_status(_ptr(ws), ctypes.byref(out), _stream(stream)))
    return out.value


class vp_model:
    """Owns a vp_model handle (vp_model_create / vp_model_destroy).  ``layers`` is a list of
    vp_layer_desc; the device weights they point to must stay alive while the model is used."""

    def __init__(self, hidden: int, inter: int, rms_eps: float, layers, head: vp_head_desc):
        arr = (vp_layer_desc * len(layers))(*layers)
        self._layers = arr
        self._head = head
        h = ctypes.c_void_p()
        _check("vp_model_create", _L.vp_model_create(hidden, inter, rms_eps, arr, len(layers), ctypes.byref(head),
                                                     ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            _L.vp_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()


def vp_pass_workspace_bytes(model: vp_model, M: int) -> int:
    return _L.vp_pass_workspace_bytes(model.handle, M)


def vp_pass_launch_count(model: vp_model) -> int:
    return _L.vp_pass_launch_count(model.handle)


def vp_verify_pass(model: vp_model, x0, M: int, pending, argmax, n_commit, committed, trace, logits, ws, stream=None,
                   ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_verify_pass", _L.vp_verify_pass(model.handle, _ptr(x0), M, _ptr(pending), _ptr(argmax),
                                               _ptr(n_commit), _ptr(committed), _ptr(trace), _ptr(logits), _ptr(ws),
                                               wb, _stream(stream)))


def vp_verify_pass_rows(model: vp_model, x0, M: int, rows: int, pending, argmax, n_commit, committed, trace, logits,
                        ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_verify_pass_rows", _L.vp_verify_pass_rows(model.handle, _ptr(x0), M, rows, _ptr(pending),
                                                         _ptr(argmax), _ptr(n_commit), _ptr(committed), _ptr(trace),
                                                         _ptr(logits), _ptr(ws), wb, _stream(stream)))


def vp_pass_sampled_workspace_bytes(model: vp_model, M: int) -> int:
    return _L.vp_pass_sampled_workspace_bytes(model.handle, M)


def vp_verify_pass_sampled(model: vp_model, x0, M: int, pending, temperature: float, top_k: int, top_p: float,
                           draft_tokens, draft_probs, uniforms, argmax, n_commit, committed, logits, ws, stream=None,
                           ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_verify_pass_sampled",
           _L.vp_verify_pass_sampled(model.handle, _ptr(x0), M, _ptr(pending), temperature, top_k, top_p,
                                     _ptr(draft_tokens), _ptr(draft_probs), _ptr(uniforms), _ptr(argmax),
                                     _ptr(n_commit), _ptr(committed), _ptr(logits), _ptr(ws), wb, _stream(stream)))


def vp_model_set_cores(model: vp_model, geom: vp_core_geom, cores: list):
    arr = (vp_core_desc * len(cores))(*cores)
    _check("vp_model_set_cores", _L.vp_model_set_cores(model.handle, ctypes.byref(geom), arr, len(cores)))


def vp_pass_cores_workspace_bytes(model: vp_model, M: int) -> int:
    return _L.vp_pass_cores_workspace_bytes(model.handle, M)


def vp_pass_cores_launch_count(model: vp_model) -> int:
    return _L.vp_pass_cores_launch_count(model.handle)


def vp_verify_pass_cores(model: vp_model, x0, M: int, ctx, parity: int, pending, argmax, n_commit, committed, trace,
                         logits, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_verify_pass_cores",
           _L.vp_verify_pass_cores(model.handle, _ptr(x0), M, _ptr(ctx), parity, _ptr(pending), _ptr(argmax),
                                   _ptr(n_commit), _ptr(committed), _ptr(trace), _ptr(logits), _ptr(ws), wb,
                                   _stream(stream)))


def vp_commit_cores(model: vp_model, M: int, n_commit, parity: int, ws, stream=None, ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_commit_cores", _L.vp_commit_cores(model.handle, M, _ptr(n_commit), parity, _ptr(ws), wb,
                                                 _stream(stream)))


def vp_verify_blocks(model: vp_model, h, M: int, block_begin: int, block_end: int, trace, ws, stream=None,
                     ws_bytes=None):
    wb = ws_bytes if ws_bytes is not None else _nbytes(ws)
    _check("vp_verify_blocks", _L.vp_verify_blocks(model.handle, _ptr(h), M, block_begin, block_end, _ptr(trace),
                                                   _ptr(ws), wb, _stream(stream)))


def vp_trace_read(M: int, dst) -> int:
    """Copies the executor's phase timeline into the numpy array `dst` (uint64, up to
    [2][160][256][36]) and returns the number of multi-phase launches completed; raises VerifyError
    (VP_ERR_UNSUPPORTED) unless this is the phase-traced build."""
    n = ctypes.c_uint(0)
    _check("vp_trace_read", _L.vp_trace_read(M, dst.ctypes.data, dst.nbytes, ctypes.byref(n)))
    return n.value

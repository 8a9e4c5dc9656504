"""Host-side checks of the C ABI: the library loads, exports every declared symbol, and rejects bad
arguments before touching the GPU (so these run without one)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def V():
    from weight_streaming_gb300 import build
    build()
    from weight_streaming_gb300 import _lib
    return _lib


def declared_functions():
    src = open(os.path.join(ROOT, "include", "verify.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(vp_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(V):
    decl = declared_functions()
    assert len(decl) >= 18
    lib = ctypes.CDLL(V.LIB_PATH)
    for name in decl:
        assert hasattr(lib, name), name
    assert sorted(V.EXPORTS) == decl


def test_status_strings(V):
    assert V.status_string(0) == "VP_OK"
    assert V.status_string(6) == "VP_ERR_TIMEOUT"
    assert V.status_string(99) == "VP_ERR_UNKNOWN"


def test_packed_and_workspace_sizes(V):
    assert V.vp_packed_bytes_nvfp4(17408, 5120) == 17408 * 5120 * 9 // 16
    assert V.vp_packed_bytes_fp8(16384, 5120) == 16384 * 5120
    assert V.vp_packed_bytes_nvfp4(17, 256) == 0 and V.vp_packed_bytes_nvfp4(16, 128) == 0
    assert V.vp_packed_bytes_fp8(16, 128) == 16 * 128 and V.vp_packed_bytes_fp8(16, 64) == 0
    assert V.vp_workspace_bytes(V.VP_OP_NVFP4, 8, 5120, 17408) > 0
    assert V.vp_workspace_bytes(V.VP_OP_NVFP4, 33, 5120, 17408) == 0
    assert V.vp_workspace_bytes(V.VP_OP_NVFP4, 0, 5120, 17408) == 0
    assert V.vp_workspace_bytes(V.VP_OP_HEAD, 12, 1024, 1024) == 0  # head needs M % 8 == 0
    assert V.vp_workspace_bytes(V.VP_OP_ARGMAX, 8, 248320, 0) > 0
    assert V.vp_workspace_bytes(7, 8, 64, 64) == 0


FAKE = 0x10000000  # an aligned address that is never dereferenced: every call below fails validation first


def test_linear_validation_without_gpu(V):
    L = V.lib()
    ws = V.vp_workspace_bytes(V.VP_OP_NVFP4, 8, 256, 1024)
    ok = (FAKE, 1.0, FAKE, FAKE, 8, 256, 1024, FAKE, ws, None)
    for fn in (L.vp_linear_nvfp4, L.vp_linear_fp8):
        assert fn(None, *ok[1:]) == V.VP_ERR_INVALID_ARG
        assert fn(*ok[:2], None, *ok[3:]) == V.VP_ERR_INVALID_ARG
        assert fn(*ok[:7], None, *ok[8:]) == V.VP_ERR_INVALID_ARG
        for M, N, K in ((0, 256, 1024), (33, 256, 1024), (8, 250, 1024), (8, 256, 1000), (8, 0, 1024),
                        (8, 256, 65536 + 256)):
            assert fn(FAKE, 1.0, FAKE, FAKE, M, N, K, FAKE, 1 << 30, None) == V.VP_ERR_SHAPE
        assert fn(FAKE + 8, *ok[1:]) == V.VP_ERR_ALIGNMENT
        assert fn(*ok[:2], FAKE + 2, *ok[3:]) == V.VP_ERR_ALIGNMENT
        assert fn(*ok[:7], FAKE + 16, *ok[8:]) == V.VP_ERR_ALIGNMENT
        assert fn(*ok[:8], ws - 1, None) == V.VP_ERR_WORKSPACE


def test_q4_sizes_and_validation_without_gpu(V):
    assert V.vp_packed_bytes_q4(17408, 5120) == 17408 * 5120 * 9 // 16 == 50_135_040
    assert V.vp_packed_bytes_q4(16, 128) == 0 and V.vp_packed_bytes_q4(24, 256) == 0
    assert V.vp_workspace_bytes(V.VP_OP_Q4, 8, 17408, 5120) > 0
    assert V.vp_workspace_bytes(V.VP_OP_Q4, 33, 17408, 5120) == 0
    L = V.lib()
    ws = V.vp_workspace_bytes(V.VP_OP_Q4, 8, 256, 1024)
    ok = (FAKE, FAKE, FAKE, 8, 256, 1024, FAKE, ws, None)
    assert L.vp_linear_q4(None, *ok[1:]) == V.VP_ERR_INVALID_ARG
    assert L.vp_linear_q4(*ok[:6], None, *ok[7:]) == V.VP_ERR_INVALID_ARG
    for M, N, K in ((0, 256, 1024), (33, 256, 1024), (8, 250, 1024), (8, 256, 1000), (8, 256, 65536 + 256)):
        assert L.vp_linear_q4(FAKE, FAKE, FAKE, M, N, K, FAKE, 1 << 30, None) == V.VP_ERR_SHAPE
    assert L.vp_linear_q4(FAKE + 8, *ok[1:]) == V.VP_ERR_ALIGNMENT
    assert L.vp_linear_q4(FAKE, FAKE + 2, *ok[2:]) == V.VP_ERR_ALIGNMENT
    assert L.vp_linear_q4(*ok[:7], ws - 1, None) == V.VP_ERR_WORKSPACE
    pb = V.vp_packed_bytes_q4(256, 1024)
    assert L.vp_pack_q4(None, FAKE, FAKE, 256, 1024, FAKE, pb, None) == V.VP_ERR_INVALID_ARG
    assert L.vp_pack_q4(FAKE, FAKE, None, 256, 1024, FAKE, pb, None) == V.VP_ERR_INVALID_ARG
    assert L.vp_pack_q4(FAKE, FAKE, FAKE, 256, 1000, FAKE, pb, None) == V.VP_ERR_SHAPE
    assert L.vp_pack_q4(FAKE, FAKE, FAKE, 256, 1024, FAKE, pb - 1, None) == V.VP_ERR_INVALID_ARG
    assert L.vp_pack_q4(FAKE, FAKE + 1, FAKE, 256, 1024, FAKE, pb, None) == V.VP_ERR_ALIGNMENT
    assert L.vp_pack_q4(FAKE, FAKE, FAKE, 256, 1024, FAKE + 8, pb, None) == V.VP_ERR_ALIGNMENT


def test_sample_accept_validation_without_gpu(V):
    L = V.lib()
    assert V.vp_workspace_bytes(V.VP_OP_SAMPLE, 8, 248320, 0) > 0
    ws = V.vp_workspace_bytes(V.VP_OP_SAMPLE, 8, 1000, 0)
    assert ws > 0 and V.vp_workspace_bytes(V.VP_OP_SAMPLE, 12, 1000, 0) == 0
    assert V.vp_workspace_bytes(V.VP_OP_SAMPLE, 8, (1 << 20) + 1, 0) == 0
    F = FAKE
    ok = [F, 8, 1000, 1.0, 20, 0.9, F, F, F, F, F, F, F, ws, None]

    def call(**kw):
        a = list(ok)
        names = ["logits", "M", "V", "T", "k", "p", "pending", "dt", "dp", "u", "nc", "cm", "ws", "wsb", "s"]
        for key, val in kw.items():
            a[names.index(key)] = val
        return L.vp_sample_accept(*a)
    assert call(logits=None) == V.VP_ERR_INVALID_ARG
    assert call(dt=None) == V.VP_ERR_INVALID_ARG  # draft tokens without probabilities
    assert call(T=0.0) == V.VP_ERR_INVALID_ARG and call(T=float("inf")) == V.VP_ERR_INVALID_ARG
    assert call(p=0.0) == V.VP_ERR_INVALID_ARG and call(p=1.5) == V.VP_ERR_INVALID_ARG
    assert call(M=12) == V.VP_ERR_SHAPE and call(k=33) == V.VP_ERR_SHAPE and call(k=0) == V.VP_ERR_SHAPE
    assert call(V=10, k=11) == V.VP_ERR_SHAPE
    assert call(logits=F + 2) == V.VP_ERR_ALIGNMENT and call(ws=F + 16) == V.VP_ERR_ALIGNMENT
    assert call(wsb=ws - 1) == V.VP_ERR_WORKSPACE


def test_attention_validation_without_gpu(V):
    L = V.lib()
    ws = V.vp_workspace_bytes(V.VP_OP_ATTN, 8, 4, 4096)
    assert ws > 0 and V.vp_workspace_bytes(V.VP_OP_ATTN, 9, 4, 4096) == 0 and V.vp_workspace_bytes(V.VP_OP_ATTN, 8, 4, 7) == 0
    F = FAKE
    ok = [F, F, F, F, F, F, 4096, F, F, 8, 24, 4, 256, F, ws, None]
    names = ["q", "kn", "vn", "kc", "vc", "ctx", "cap", "gate", "out", "M", "Hq", "Hkv", "D", "ws", "wsb", "s"]

    def call(**kw):
        a = list(ok)
        for key, val in kw.items():
            a[names.index(key)] = val
        return L.vp_attention_verify(*a)
    assert call(q=None) == V.VP_ERR_INVALID_ARG and call(ctx=None) == V.VP_ERR_INVALID_ARG
    assert call(D=128) == V.VP_ERR_SHAPE and call(Hq=25) == V.VP_ERR_SHAPE and call(Hq=40, Hkv=4) == V.VP_ERR_SHAPE
    assert call(M=12) == V.VP_ERR_SHAPE and call(cap=7) == V.VP_ERR_SHAPE
    assert call(kc=F + 8) == V.VP_ERR_ALIGNMENT and call(ctx=F + 2) == V.VP_ERR_ALIGNMENT
    assert call(wsb=ws - 1) == V.VP_ERR_WORKSPACE


def test_gdn_validation_without_gpu(V):
    L = V.lib()
    F = FAKE
    ok = [F, F, F, F, F, F, F, F, 8, 48, 128, 128, F, None]
    names = ["si", "so", "q", "k", "v", "a", "b", "rows", "M", "H", "dk", "dv", "out", "s"]

    def call(**kw):
        a = list(ok)
        for key, val in kw.items():
            a[names.index(key)] = val
        return L.vp_gdn_scan(*a)
    assert call(si=None) == V.VP_ERR_INVALID_ARG and call(rows=None) == V.VP_ERR_INVALID_ARG
    assert call(M=12) == V.VP_ERR_SHAPE and call(dk=64) == V.VP_ERR_SHAPE and call(H=0) == V.VP_ERR_SHAPE
    assert call(si=F + 2) == V.VP_ERR_ALIGNMENT and call(a=F + 2) == V.VP_ERR_ALIGNMENT


def test_loop_validation_without_gpu(V):
    L = V.lib()
    F = FAKE
    assert L.vp_embed_nvfp4(None, F, 1.0, F, 8, 100, 256, F, None, None) == V.VP_ERR_INVALID_ARG
    assert L.vp_embed_nvfp4(F, F, 1.0, F, 8, 100, 250, F, None, None) == V.VP_ERR_SHAPE
    assert L.vp_embed_nvfp4(F, F, 1.0, F + 2, 8, 100, 256, F, None, None) == V.VP_ERR_ALIGNMENT
    assert L.vp_lookup_drafts(F, F, 5, 100, 8, F, None, None) == V.VP_ERR_SHAPE
    assert L.vp_lookup_drafts(F, F, 1, 100, 0, F, None, None) == V.VP_ERR_SHAPE
    assert L.vp_lookup_drafts(F, None, 1, 100, 8, F, None, None) == V.VP_ERR_INVALID_ARG
    assert L.vp_commit_append(F, F, 0, 100, F, F, None, None) == V.VP_ERR_SHAPE
    assert L.vp_commit_append(F, F, 1, 100, F, F + 2, None, None) == V.VP_ERR_ALIGNMENT
    assert L.vp_decode_steps(None, 1, F, F, 1.0, 100, 256, F, F, 100, 1, 8, F, F, F, F, F, F, 256, None,
                             None) == V.VP_ERR_INVALID_ARG


def test_decode_steps_checks_everything_before_launching(V):
    """vp_decode_steps rejects a bad argument of any of its four steps before its first launch (every
    call below either fails a check or has steps == 0, so nothing is enqueued)."""
    L = V.lib()
    F = FAKE
    m = V.vp_model(256, 512, 1e-6, [_layer(V)], V.vp_head_desc(FAKE, 1.0, 2048))
    need = V.vp_pass_workspace_bytes(m, 8)

    def call(steps=1, vocab=2048, hidden=256, cap=100, lanes=1, mm=8, x0=F, ws=F, ws_bytes=need, hist=F):
        return L.vp_decode_steps(m.handle, steps, F, F, 1.0, vocab, hidden, hist, F, cap, lanes, mm, F, x0, F, F, F, ws,
                                 ws_bytes, None, None)
    assert call(steps=0) == V.VP_OK  # the checks alone
    assert call(steps=-1) == V.VP_ERR_SHAPE and call(lanes=5) == V.VP_ERR_SHAPE
    assert call(cap=0) == V.VP_ERR_SHAPE and call(cap=1 << 24) == V.VP_ERR_SHAPE
    assert call(mm=0) == V.VP_ERR_SHAPE and call(mm=128) == V.VP_ERR_SHAPE
    assert call(vocab=0) == V.VP_ERR_SHAPE and call(hidden=250) == V.VP_ERR_SHAPE
    # the embedding's row width must be the model's: a wider or narrower x0 row is refused
    assert call(hidden=512) == V.VP_ERR_SHAPE and call(hidden=128) == V.VP_ERR_SHAPE
    assert call(steps=0, hidden=512) == V.VP_ERR_SHAPE
    assert call(x0=F + 8) == V.VP_ERR_ALIGNMENT and call(hist=F + 2) == V.VP_ERR_ALIGNMENT
    assert call(ws=F + 128) == V.VP_ERR_ALIGNMENT
    assert call(ws_bytes=need - 1) == V.VP_ERR_WORKSPACE
    m.close()


def test_head_and_argmax_validation_without_gpu(V):
    L = V.lib()
    ws = V.vp_workspace_bytes(V.VP_OP_HEAD, 8, 1024, 512)
    args = [FAKE, 1.0, FAKE, 8, 1024, 512, FAKE, FAKE, FAKE, FAKE, None, FAKE, ws, None]
    a = list(args)
    a[3] = 12
    assert L.vp_head_argmax_accept(*a) == V.VP_ERR_SHAPE
    a = list(args)
    a[6] = None
    assert L.vp_head_argmax_accept(*a) == V.VP_ERR_INVALID_ARG
    a = list(args)
    a[12] = ws - 256
    assert L.vp_head_argmax_accept(*a) == V.VP_ERR_WORKSPACE
    assert L.vp_argmax_accept(FAKE, 9, 100, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == V.VP_ERR_SHAPE
    assert L.vp_argmax_accept(FAKE, 8, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == V.VP_ERR_SHAPE
    assert L.vp_argmax_accept(FAKE + 2, 8, 100, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None) == V.VP_ERR_ALIGNMENT


def _layer(V, kind=0, n_in=512, k_out=256, n_kv=0):
    d = V.vp_layer_desc()
    d.kind = kind
    d.w_in, d.s_in, d.n_in = FAKE, 1.0, n_in
    d.w_kv, d.s_kv, d.n_kv = (FAKE, 1.0, n_kv) if kind == 1 else (None, 1.0, 0)
    d.w_out, d.s_out, d.k_out = FAKE, 1.0, k_out
    d.w_gate, d.ts_gate = FAKE, 1.0
    d.w_up, d.ts_up = FAKE, 1.0
    d.w_down, d.ts_down = FAKE, 1.0
    return d


def test_model_create_validation_without_gpu(V):
    head = V.vp_head_desc(FAKE, 1.0, 2048)
    m = V.vp_model(256, 512, 1e-6, [_layer(V), _layer(V, 1, 384, 256, 128)], head)
    assert V.vp_pass_launch_count(m) == 1  # 9 phases: one executor launch
    assert V.vp_pass_workspace_bytes(m, 8) > 0
    assert V.vp_pass_workspace_bytes(m, 1) > 0 and V.vp_pass_workspace_bytes(m, 12) > 0  # block runs take any M
    assert V.vp_pass_workspace_bytes(m, 0) == 0 and V.vp_pass_workspace_bytes(m, 33) == 0
    # the sampled pass: whole lanes only, and more workspace than the greedy pass (its logits)
    assert V.vp_pass_sampled_workspace_bytes(m, 8) > V.vp_pass_workspace_bytes(m, 8) + 8 * 2048 * 4
    assert V.vp_pass_sampled_workspace_bytes(m, 12) == 0
    ps = V.vp_pass_sampled_workspace_bytes(m, 8)
    bad = lambda **kw: L.vp_verify_pass_sampled(  # noqa: E731
        m.handle, FAKE, 8, FAKE, kw.get("T", 1.0), kw.get("k", 20), kw.get("p", 0.9), kw.get("dt", None),
        kw.get("dp", None), FAKE, FAKE, FAKE, FAKE, None, 1 << 20, kw.get("wb", ps), None)
    L = V.lib()
    assert bad(T=0.0) == V.VP_ERR_INVALID_ARG and bad(p=1.5) == V.VP_ERR_INVALID_ARG
    assert bad(dt=FAKE) == V.VP_ERR_INVALID_ARG  # draft tokens without their probabilities
    assert bad(k=0) == V.VP_ERR_SHAPE and bad(k=33) == V.VP_ERR_SHAPE
    assert bad(wb=ps - 1) == V.VP_ERR_WORKSPACE
    L = V.lib()
    ws_fake = 1 << 20  # never dereferenced: the row count is checked first
    # the pass itself needs whole lanes of 8 rows
    assert L.vp_verify_pass(m.handle, FAKE, 12, FAKE, FAKE, FAKE, FAKE, None, None, ws_fake,
                            V.vp_pass_workspace_bytes(m, 12), None) == V.VP_ERR_SHAPE
    m.close()
    with pytest.raises(V.VerifyError):
        V.vp_model(256, 512, 1e-6, [_layer(V, k_out=1024)], head)  # k_out > n_in
    with pytest.raises(V.VerifyError):
        V.vp_model(250, 512, 1e-6, [_layer(V)], head)
    with pytest.raises(V.VerifyError):
        V.vp_model(256, 512, 1e-6, [_layer(V, kind=1, n_kv=0)], head)
    m64 = V.vp_model(256, 512, 1e-6, [_layer(V, 1 if l % 4 == 3 else 0, 384 if l % 4 == 3 else 512, 256,
                                             128 if l % 4 == 3 else 0) for l in range(64)], head)
    assert V.vp_pass_launch_count(m64) == 2  # 257 phases, at most 160 per launch
    m64.close()
    bad = _layer(V)
    bad.w_up = FAKE + 4
    with pytest.raises(V.VerifyError):
        V.vp_model(256, 512, 1e-6, [bad], head)


def _core(V, gdn=True, **kw):
    c = V.vp_core_desc()
    names = ("w_a", "w_b", "conv_taps", "a_log", "dt_bias", "norm_w", "state_a", "state_b", "window_a", "conv_hist") \
        if gdn else ("q_norm", "k_norm", "k_cache", "v_cache")
    for n in names:
        setattr(c, n, kw.get(n, FAKE))
    return c


def test_cores_validation_without_gpu(V):
    """vp_model_set_cores checks the widths against the core geometry, the pointers and their
    alignment; the cores pass and its commit check parity, rows and workspace before launching."""
    L = V.lib()
    head = V.vp_head_desc(FAKE, 1.0, 2048)
    # layer 0 Gated DeltaNet (n_qk = n_v = 1, d = 128), layer 1 attention (Hq = Hkv = 1, D = 256)
    layers = [_layer(V, 0, 512, 128), _layer(V, 1, 512, 256, 512)]
    m = V.vp_model(256, 512, 1e-6, layers, head)
    geom = V.vp_core_geom(1, 1, 128, 1, 1, 256, 64)
    assert V.vp_pass_cores_workspace_bytes(m, 8) == 0  # no cores yet
    assert L.vp_verify_pass_cores(m.handle, FAKE, 8, FAKE, 0, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 30,
                                  None) == V.VP_ERR_INVALID_ARG
    arr = lambda cs: (V.vp_core_desc * 2)(*cs)  # noqa: E731
    set_cores = lambda g, cs, n=2: L.vp_model_set_cores(m.handle, ctypes.byref(g), arr(cs), n)  # noqa: E731
    good = [_core(V), _core(V, gdn=False)]
    assert set_cores(geom, good, 1) == V.VP_ERR_INVALID_ARG                       # one descriptor per layer
    assert set_cores(V.vp_core_geom(1, 2, 128, 1, 1, 256, 64), good) == V.VP_ERR_SHAPE  # GDN widths
    assert set_cores(V.vp_core_geom(1, 1, 64, 1, 1, 256, 64), good) == V.VP_ERR_SHAPE   # d != 128
    assert set_cores(V.vp_core_geom(1, 1, 128, 2, 1, 256, 64), good) == V.VP_ERR_SHAPE  # attention widths
    assert set_cores(geom, [_core(V, w_b=None), good[1]]) == V.VP_ERR_INVALID_ARG
    assert set_cores(geom, [_core(V, w_a=FAKE + 2), good[1]]) == V.VP_ERR_ALIGNMENT    # A / B need 16 bytes
    assert set_cores(geom, [good[0], _core(V, gdn=False, k_cache=FAKE + 8)]) == V.VP_ERR_ALIGNMENT
    assert set_cores(geom, good) == V.VP_OK
    wb = V.vp_pass_cores_workspace_bytes(m, 8)
    assert wb > V.vp_pass_workspace_bytes(m, 8)
    assert V.vp_pass_cores_workspace_bytes(m, 12) == 0 and V.vp_pass_cores_workspace_bytes(m, 40) == 0
    # launches: 3 executor programs ([in 0], then 4 phases after each core), 1 GDN core, 4 attention
    assert V.vp_pass_cores_launch_count(m) == 3 + 1 + 4
    pc = lambda **kw: L.vp_verify_pass_cores(  # noqa: E731
        m.handle, FAKE, kw.get("M", 8), FAKE, kw.get("parity", 0), FAKE, FAKE, FAKE, FAKE, None, None, FAKE,
        kw.get("wb", wb), None)
    assert pc(parity=2) == V.VP_ERR_INVALID_ARG and pc(parity=-1) == V.VP_ERR_INVALID_ARG
    assert pc(wb=wb - 1) == V.VP_ERR_WORKSPACE
    assert pc(M=12, wb=1 << 30) == V.VP_ERR_SHAPE
    cc = lambda **kw: L.vp_commit_cores(m.handle, kw.get("M", 8), kw.get("nc", FAKE), kw.get("parity", 0),  # noqa: E731
                                         kw.get("ws", FAKE), kw.get("wb", wb), None)
    assert cc(parity=2) == V.VP_ERR_INVALID_ARG and cc(nc=None) == V.VP_ERR_INVALID_ARG
    assert cc(M=12) == V.VP_ERR_SHAPE and cc(M=0) == V.VP_ERR_SHAPE
    assert cc(ws=FAKE + 16) == V.VP_ERR_ALIGNMENT and cc(nc=FAKE + 2) == V.VP_ERR_ALIGNMENT
    assert cc(wb=wb - 1) == V.VP_ERR_WORKSPACE
    m.close()
    m2 = V.vp_model(256, 512, 1e-6, layers, head)  # a model without cores has nothing to commit
    assert L.vp_commit_cores(m2.handle, 8, FAKE, 0, FAKE, 1 << 30, None) == V.VP_ERR_INVALID_ARG
    m2.close()


def test_phase_trace_only_in_traced_build(V):
    """The phase timeline is recorded only by the VP_PHASE_TRACE build; the product library says so
    without touching a device."""
    import numpy as np
    buf = np.zeros(16, np.uint64)
    with pytest.raises(V.VerifyError) as e:
        V.vp_trace_read(8, buf)
    assert e.value.status == V.VP_ERR_UNSUPPORTED
    with pytest.raises(V.VerifyError) as e:
        V.vp_trace_read(0, buf)
    assert e.value.status == V.VP_ERR_SHAPE


def test_wide_verify_validation_without_gpu(V):
    """The R-rows entry points refuse rows outside 1..32, M not a multiple of rows, more than 128 rows
    in all, or more than 32 rows that do not split into runs of 32 rows of whole lanes, before any
    launch."""
    L = V.lib()
    F = FAKE
    arg = lambda M, Vv, rows, lg=F: L.vp_argmax_accept_rows(lg, M, Vv, rows, F, F, F, F, F, 1 << 20, None)
    assert arg(32, 100, 0) == V.VP_ERR_SHAPE and arg(32, 100, 33) == V.VP_ERR_SHAPE
    assert arg(24, 100, 16) == V.VP_ERR_SHAPE and arg(8, 100, 16) == V.VP_ERR_SHAPE
    assert arg(48, 100, 16) == V.VP_ERR_SHAPE and arg(96, 100, 12) == V.VP_ERR_SHAPE  # runs of 32: M % 32, 32 % R
    assert arg(160, 100, 32) == V.VP_ERR_SHAPE
    assert arg(32, 0, 16) == V.VP_ERR_SHAPE and arg(32, 100, 16, lg=F + 2) == V.VP_ERR_ALIGNMENT
    assert L.vp_argmax_accept_rows(None, 32, 100, 16, F, F, F, F, F, 1 << 20, None) == V.VP_ERR_INVALID_ARG
    assert L.vp_lookup_drafts_rows(F, F, 5, 32, 100, 8, F, None, None) == V.VP_ERR_SHAPE   # 160 rows
    assert L.vp_lookup_drafts_rows(F, F, 33, 1, 100, 8, F, None, None) == V.VP_ERR_SHAPE   # 33 lanes
    assert L.vp_lookup_drafts_rows(F, F, 1, 0, 100, 8, F, None, None) == V.VP_ERR_SHAPE
    assert L.vp_lookup_drafts_rows(F, F, 1, 32, 100, 8, F + 2, None, None) == V.VP_ERR_ALIGNMENT
    assert L.vp_commit_append_rows(F, F, 9, 16, 100, F, F, None, None) == V.VP_ERR_SHAPE   # 144 rows
    assert L.vp_commit_append_rows(F, F, 33, 1, 100, F, F, None, None) == V.VP_ERR_SHAPE   # 33 lanes
    assert L.vp_commit_append_rows(F, F, 1, 33, 100, F, F, None, None) == V.VP_ERR_SHAPE
    assert L.vp_commit_append_rows(F, None, 1, 16, 100, F, F, None, None) == V.VP_ERR_INVALID_ARG

    m = V.vp_model(256, 512, 1e-6, [_layer(V)], V.vp_head_desc(FAKE, 1.0, 2048))
    need = V.vp_pass_workspace_bytes(m, 32)
    assert all(V.vp_pass_workspace_bytes(m, M) == need for M in (64, 96, 128))  # passes of 32 rows share it
    assert V.vp_pass_workspace_bytes(m, 48) == 0 and V.vp_pass_workspace_bytes(m, 160) == 0

    def vp(M=32, rows=16, x0=F, ws=F, wb=need):
        return L.vp_verify_pass_rows(m.handle, x0, M, rows, F, F, F, F, None, None, ws, wb, None)
    assert vp(rows=0) == V.VP_ERR_SHAPE and vp(rows=33) == V.VP_ERR_SHAPE and vp(M=24) == V.VP_ERR_SHAPE
    assert vp(M=8, rows=16) == V.VP_ERR_SHAPE and vp(M=40, rows=8) == V.VP_ERR_SHAPE
    assert vp(M=96, rows=12) == V.VP_ERR_SHAPE and vp(M=160, rows=32) == V.VP_ERR_SHAPE
    assert L.vp_verify_pass_rows(m.handle, F, 64, 16, F, F, F, F, F, None, F, need, None) == V.VP_ERR_SHAPE  # trace
    assert vp(x0=F + 8) == V.VP_ERR_ALIGNMENT and vp(ws=F + 128) == V.VP_ERR_ALIGNMENT
    assert vp(wb=need - 1) == V.VP_ERR_WORKSPACE
    assert L.vp_verify_pass_rows(m.handle, None, 32, 16, F, F, F, F, None, None, F, need, None) == V.VP_ERR_INVALID_ARG

    def ds(steps=0, rows=16, lanes=2, hidden=256):
        return L.vp_decode_steps_rows(m.handle, steps, rows, F, F, 1.0, 2048, hidden, F, F, 100, lanes, 8, F, F, F, F,
                                      F, F, need, None, None)
    assert ds() == V.VP_OK  # the checks alone
    assert ds(rows=32, lanes=2) == V.VP_OK and ds(rows=16, lanes=8) == V.VP_OK  # 64, 128 rows
    assert ds(lanes=3) == V.VP_ERR_SHAPE and ds(rows=0) == V.VP_ERR_SHAPE and ds(rows=12, lanes=8) == V.VP_ERR_SHAPE
    assert ds(rows=32, lanes=5) == V.VP_ERR_SHAPE
    assert ds(hidden=512) == V.VP_ERR_SHAPE
    m.close()

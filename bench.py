"""Benchmark of the verify-pass weight stream on GB300.

One step = one full verify pass (64 layers + vocabulary head with argmax and greedy acceptance,
17,555,292,160 weight bytes at the Qwen3.8-27B shapes) over M = 8 rows (one lane), captured once into
a CUDA graph and replayed; weights and inputs are resident in HBM and far larger than L2, so every
replay streams the weights from DRAM.  The JSON line reports verify-pass GB/s (weight bytes / pass
time), ms per pass, the same at M = 16/24/32, the dominant kernel's roofline, an end-to-end figure
through the C ABI with host buffers, and the fp64 oracle on the host cores as the CPU baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: the library runs the pass on one GPU (replicas only): under torchrun every rank runs its
own replica on its own GPU; value = total bytes streamed by all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-pass HBM GB/s (% of GB300 roofline) and ms/pass at M=8 and M=32"
UNIT = "GB/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-components", action="store_true", help="skip the one-MLP-layer and head+accept figures")
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--kernel", default=None, choices=["gate", "down", "gdn_in", "head", "q4_gate", "q4_down", "q4_head", "sample", "attn",
                             "gdn", "decode", "mlp", "head_accept", "pass"],
                    help="time one GEMM shape alone (for profiling) instead of the pass")
    ap.add_argument("--M", type=int, default=8)
    ap.add_argument("--ctx", type=int, default=None,
                    help="context length per lane: --kernel attn (default 32768), --kernel pass --cores (4096)")
    ap.add_argument("--cores", action="store_true", help="--kernel pass: the pass with the real mixer cores")
    return ap.parse_args()


def aggregate(bytes_per_rank: float, times_s: list) -> tuple:
    """Whole-job GB/s over ranks that each stream `bytes_per_rank`: total bytes / slowest time."""
    t = max(times_s)
    return bytes_per_rank * len(times_s) / t / 1e9, t


def dist_setup(n):
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1
    import torch
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    world = int(os.environ["WORLD_SIZE"])
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
    dist.init_process_group("nccl")
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Every rank's value of x (all-gather; CPU tensors under gloo, device tensors under NCCL)."""
    if world <= 1:
        return [x]
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    out = [torch.zeros_like(t) for _ in range(world)]
    dist.all_gather(out, t)
    return [float(o.item()) for o in out]


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.Q}", "--format=csv,noheader",
                                       "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p:
            time.sleep(0.2)
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
                self.out, _ = self.p.communicate()

    def summary(self):
        rows = []
        for r in csv.reader(io.StringIO(self.out or "")):
            if len(r) < 9:
                continue
            try:
                rows.append({"sm": float(r[1].split()[0]), "max": float(r[2].split()[0]),
                             "hw": r[5].strip(), "hwt": r[6].strip(), "swt": r[7].strip(), "pcap": r[8].strip()})
            except (ValueError, IndexError):
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        import statistics
        reasons = set()
        for r in rows:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


# The sources the pass's kernel and its phase program are built from (not the Q4 instantiation's
# launch unit or the sampling kernel, which the pass does not run).
PASS_SOURCES = ["api.cu", "exec.cuh", "exec_launch.h", "exec_nt12.cu", "exec_nt34.cu", "internal.h", "ptx.cuh",
                "trace.cuh"]


def kernel_source_hash() -> str:
    """sha256 over the CUDA sources of the pass's executor (a profile taken on other sources is stale)."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "weight_streaming_gb300", "csrc")
    for f in PASS_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def profiled_traffic(pass_bytes: int):
    """DRAM bytes (read + write) per pass of the executor from the committed ncu capture
    (profiles/pass_m8_traffic.json), or None when that capture was taken on other kernel sources."""
    try:
        d = json.load(open(os.path.join(ROOT, "profiles", "pass_m8_traffic.json")))
    except (OSError, ValueError):
        return None
    if d.get("source_sha256") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_pass")


# ------------------------------------------------------------------ CPU baseline (the oracle)

def oracle_sample(geom, seed: int, M: int, target_s: float = 12.0):
    """Times the fp64 oracle (as it stands, all host cores) on whole MLP blocks of layers 0, 1, ...
    (RMSNorm, gate, up, SiLU*up, down) at M rows until about target_s seconds of work, and returns
    (weight bytes processed, seconds, threads, description)."""
    import numpy as np

    import oracle
    import synth
    H, I = geom.hidden, geom.inter
    x = synth.normal_bf16(seed, synth.stream_id(0, synth.T_X0), (M, H))
    nbytes, secs, l = 0, 0.0, 0
    threads = oracle.default_threads()
    while (l == 0 or secs < target_s) and l < geom.n_layers:
        gc, gs = synth.nvfp4_matrix(seed, l, synth.T_GATE_C, synth.T_GATE_S, I, H)
        uc, us = synth.nvfp4_matrix(seed, l, synth.T_UP_C, synth.T_UP_S, I, H)
        dc, ds = synth.nvfp4_matrix(seed, l, synth.T_DOWN_C, synth.T_DOWN_S, H, I)
        t0 = time.perf_counter()
        r = oracle.rmsnorm(x, geom.eps)
        g = oracle.linear(oracle.NVFP4, r, gc, gs, 1.0, I, with_abs=False, nthreads=threads)
        u = oracle.linear(oracle.NVFP4, r, uc, us, 1.0, I, with_abs=False, nthreads=threads)
        a = oracle.bf16_round(oracle.silu_mul(g, u))
        y = oracle.linear(oracle.NVFP4, a, dc, ds, 1.0, H, with_abs=False, nthreads=threads)
        x = oracle.bf16_round(oracle.bf16_value(x) + y)
        secs += time.perf_counter() - t0
        nbytes += 3 * I * H * 9 // 16
        l += 1
    desc = f"fp64 oracle, MLP blocks of layers 0..{l - 1} ({l} x 150.4 MB NVFP4) at M={M}, all host cores"
    return nbytes, secs, threads, desc


def run_reference(args):
    """The oracle arm: the same metric (weight GB/s of the verify pass) for the fp64 CPU oracle."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from weight_streaming_gb300.geometry import Geometry  # shapes only: no libverify.so in this process
    geom = Geometry(n_layers=args.layers)
    for _ in range(args.warmup):
        oracle_sample(geom, 0, 8, target_s=0.0)
    tot_b, tot_s, thr, desc = 0, 0.0, 1, ""
    for _ in range(args.steps):
        b, s, thr, desc = oracle_sample(geom, 0, 8, target_s=0.0)
        tot_b += b
        tot_s += s
    v = tot_b / tot_s / 1e9
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "verify-pass weight stream, M=8 (bounded sample: one MLP block per step)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": desc},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the GPU arm

def graph_time(fn, steps: int, warmup: int) -> float:
    """Seconds per call of fn (a sequence of library launches on the current stream), captured once
    in a CUDA graph and replayed, so that the host's launch path is not timed; CUDA events on the
    capturing stream."""
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the library's one-time set-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / steps


def run_sample(args):
    """vp_sample_accept alone over fp32 logits [M][248320] (top_k 20, top_p 0.95, temperature 0.7,
    draft distributions of 16 candidates); prints one JSON line with the time per call and the logit
    bytes read per second."""
    import torch

    from weight_streaming_gb300 import _lib as V
    M, Vv = args.M, 248320
    g = torch.Generator(device="cuda").manual_seed(0)
    logits = torch.randn((M, Vv), device="cuda", generator=g)
    pending = torch.randint(0, Vv, (M,), device="cuda", dtype=torch.int32, generator=g)
    dt = torch.randint(0, Vv, (M, 16), device="cuda", dtype=torch.int32, generator=g)
    dp = torch.full((M, 16), 1.0 / 16, device="cuda")
    u = torch.rand((M, 2), device="cuda", generator=g)
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    ws = torch.zeros(V.vp_workspace_bytes(V.VP_OP_SAMPLE, M, Vv, 0), dtype=torch.uint8, device="cuda")

    def call():
        V.vp_sample_accept(logits, M, Vv, 0.7, 20, 0.95, pending, dt, dp, u, nc, cm, ws)
    t = graph_time(call, args.steps, args.warmup)
    nbytes = M * Vv * 4
    print(json.dumps({"kernel": "sample", "M": M, "V": Vv, "us_per_call": t * 1e6, "launches_per_call": 1,
                      "logit_gbps": nbytes / t / 1e9, "bytes_per_call": nbytes}), flush=True)


def run_attn(args):
    """vp_attention_verify alone: the pages' attention heads (24 q / 4 kv, head dim 256), every lane
    at the context --ctx, rotating over 4 cache copies when they fit (so the cache streams from
    DRAM); prints one JSON line with the time per call and the cache bytes read per second."""
    import torch

    from weight_streaming_gb300 import _lib as V
    M, Hq, Hkv, D = args.M, 24, 4, 256
    L, ctx = M // 8, args.ctx
    cap = ctx + 8
    cache_bytes = L * Hkv * cap * D * 2 * 2
    copies = 4 if 4 * cache_bytes < (16 << 30) else 1
    g = torch.Generator(device="cuda").manual_seed(0)
    rnd = lambda *sh: torch.randn(sh, device="cuda", generator=g).to(torch.bfloat16)  # noqa: E731
    caches = [(rnd(L, Hkv, cap, D), rnd(L, Hkv, cap, D)) for _ in range(copies)]
    q, kn, vn, gate = rnd(M, Hq, D), rnd(M, Hkv, D), rnd(M, Hkv, D), rnd(M, Hq, D)
    ctx_d = torch.full((L,), ctx, dtype=torch.int32, device="cuda")
    out = torch.empty((M, Hq, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(V.vp_workspace_bytes(V.VP_OP_ATTN, M, Hkv, cap), dtype=torch.uint8, device="cuda")

    def calls():  # one call per cache copy
        for kc, vc in caches:
            V.vp_attention_verify(q, kn, vn, kc, vc, ctx_d, cap, gate, out, M, Hq, Hkv, D, ws)
    t = graph_time(calls, args.steps, args.warmup) / copies
    nbytes = L * Hkv * (ctx + 8) * D * 2 * 2  # keys and values read once
    peak = (measured_peaks() or {}).get("hbm_gbs")
    print(json.dumps({"kernel": "attn", "M": M, "ctx": ctx, "heads": [Hq, Hkv, D], "us_per_call": t * 1e6,
                      "launches_per_call": 3, "timing": "CUDA graph of one call per cache copy, replayed", "kv_gbps": nbytes / t / 1e9, "bytes_per_call": nbytes, "copies": copies,
                      "frac_of_measured_copy": (nbytes / t / 1e9 / peak) if peak else None}), flush=True)


def run_gdn(args):
    """vp_gdn_scan for the 48 Gated DeltaNet layers of one pass (48 heads of 128 x 128 fp32 state per
    layer and lane, parity A -> B, 8 verify rows), one launch per layer; prints one JSON line with
    the time per layer and the state bytes read + written per second."""
    import torch

    from weight_streaming_gb300 import _lib as V
    M, H, d, layers = args.M, 48, 128, 48
    L = M // 8
    g = torch.Generator(device="cuda").manual_seed(0)
    sa = torch.randn((layers, L, H, d, d), device="cuda", generator=g) * 0.1
    sb = torch.empty_like(sa)
    q = torch.randn((M, H, d), device="cuda", generator=g).to(torch.bfloat16)
    k = (torch.randn((M, H, d), device="cuda", generator=g) / d ** 0.5).to(torch.bfloat16)
    v = torch.randn((M, H, d), device="cuda", generator=g).to(torch.bfloat16)
    a = torch.full((M, H), 0.95, device="cuda")
    b = torch.full((M, H), 0.5, device="cuda")
    rows = torch.full((L,), 8, dtype=torch.int32, device="cuda")
    out = torch.empty((M, H, d), device="cuda")

    def step():
        for layer in range(layers):
            V.vp_gdn_scan(sa[layer], sb[layer], q, k, v, a, b, rows, M, H, d, d, out)
    t = graph_time(step, args.steps, args.warmup) / layers
    nbytes = L * H * d * d * 4 * 2
    peak = (measured_peaks() or {}).get("hbm_gbs")
    print(json.dumps({"kernel": "gdn", "M": M, "heads": H, "us_per_layer": t * 1e6, "state_gbps": nbytes / t / 1e9,
                      "bytes_per_layer": nbytes, "us_per_pass_48_layers": t * 1e6 * layers,
                      "frac_of_measured_copy": (nbytes / t / 1e9 / peak) if peak else None}), flush=True)


def run_decode(args):
    """The device-resident decode loop (vp_decode_steps: embedding gather, the 64-layer verify pass,
    history append, lookup drafts) on the full synthetic model, --M rows (M / 8 lanes). Times R rounds
    captured in one CUDA graph and replayed, the same rounds enqueued one at a time with a host
    synchronisation and a read of n_commit after each (a host-driven loop), and the pass alone; prints
    one JSON line with the time per round of each and the tokens committed per round."""
    import numpy as np
    import torch

    import synth
    from weight_streaming_gb300 import _lib as V
    from weight_streaming_gb300.model import Geometry, SyntheticModel

    geom = Geometry(n_layers=args.layers)
    M, R, T0, cap, mm, ts = args.M, 8, 512, 8192, 8, 1.0
    L = M // 8
    sm = SyntheticModel(geom, seed=0)
    ec = torch.empty((geom.vocab, geom.hidden // 2), dtype=torch.uint8, device="cuda")
    es = torch.empty((geom.vocab, geom.hidden // 16), dtype=torch.uint8, device="cuda")
    synth.gpu_uniform_bytes(ec, 0, synth.stream_id(synth.HEAD_LAYER + 1, synth.T_HEAD_C))
    synth.gpu_scale_codes(es, 0, synth.stream_id(synth.HEAD_LAYER + 1, synth.T_HEAD_S))
    rng = np.random.default_rng(5)
    hist0 = np.zeros((L, cap), np.int32)
    for l in range(L):  # a text over a small alphabet with a copied span, so that lookup finds matches
        base = rng.integers(0, 2000, T0)
        base[T0 // 2:] = base[:T0 // 2]
        hist0[l, :T0] = base
    hl0 = np.full(L, T0, np.int32)
    ws = sm.workspace(M)
    x0 = torch.empty((M, geom.hidden), dtype=torch.bfloat16, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(L, dtype=torch.int32, device="cuda")
    cm = torch.empty((L, 8), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pend = torch.empty(M, dtype=torch.int32, device="cuda")

    def state():
        return torch.from_numpy(hist0).cuda(), torch.from_numpy(hl0).cuda()

    def rounds(h, hl, n, s):
        V.vp_decode_steps(sm.model, n, ec, es, ts, geom.vocab, geom.hidden, h, hl, cap, L, mm, pend, x0, am, nc,
                          cm, ws, st, stream=s)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        # R rounds in one graph, replayed
        h, hl = state()
        V.vp_lookup_drafts(h, hl, L, cap, mm, pend, st, stream=s)
        rounds(h, hl, 1, s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rounds(h, hl, R, s)
        for _ in range(args.warmup):
            g.replay()
        s.synchronize()
        before = int(hl.sum().item())
        e0, e1 = ev(), ev()
        e0.record(s)
        for _ in range(args.steps):
            g.replay()
        e1.record(s)
        s.synchronize()
        t_graph = e0.elapsed_time(e1) / 1e3 / (args.steps * R)
        tok_graph = (int(hl.sum().item()) - before) / (args.steps * R * L)
        # the same rounds, one call per round, the host waiting for each round's n_commit
        h, hl = state()
        V.vp_lookup_drafts(h, hl, L, cap, mm, pend, st, stream=s)
        nch = torch.empty(L, dtype=torch.int32).pin_memory()
        for _ in range(args.warmup):
            rounds(h, hl, 1, s)
            nch.copy_(nc, non_blocking=True)
            s.synchronize()
        e0, e1 = ev(), ev()
        e0.record(s)
        for _ in range(args.steps * R):
            rounds(h, hl, 1, s)
            nch.copy_(nc, non_blocking=True)
            s.synchronize()
        e1.record(s)
        s.synchronize()
        t_host = e0.elapsed_time(e1) / 1e3 / (args.steps * R)
    assert int(st.item()) == 0 and V.vp_read_status(ws) == V.VP_OK
    t_pass = graph_time(lambda: sm.run(x0, pend, am, nc, cm, ws), args.steps, args.warmup)
    launches = sm.launch_count() + 3
    print(json.dumps({"kernel": "decode", "M": M, "lanes": L, "layers": args.layers, "rounds_per_graph": R,
                      "ms_per_round_graph": t_graph * 1e3, "ms_per_round_host_sync": t_host * 1e3,
                      "ms_per_pass_alone": t_pass * 1e3, "loop_overhead_us_graph": (t_graph - t_pass) * 1e6,
                      "loop_overhead_us_host_sync": (t_host - t_pass) * 1e6,
                      "tokens_committed_per_lane_round": tok_graph, "launches_per_round": launches,
                      "history_tokens_at_start": T0, "max_match": mm}), flush=True)


def measure_mlp_layer(M_list, steps: int, warmup: int, copies: int = 4) -> dict:
    """One MLP layer of the pass (RMSNorm, gate + up with SiLU(gate) * up, down with the residual) through
    vp_verify_blocks, as the pass runs it, rotating over `copies` layers' weights (> L2, so every call
    streams from DRAM); per M: microseconds per layer and weight GB/s (150,405,120 B per layer)."""
    import torch

    import synth
    from weight_streaming_gb300 import _lib as V
    from weight_streaming_gb300.geometry import Geometry
    from weight_streaming_gb300.model import SyntheticModel
    geom = Geometry(n_layers=copies)
    sm = SyntheticModel(geom, seed=0)
    H, I = geom.hidden, geom.inter
    nbytes = 3 * I * H * 9 // 16
    out = {}
    for M in M_list:
        h = torch.from_numpy(synth.normal_bf16(M, synth.stream_id(0, synth.T_X0), (M, H)).view("int16"))
        h = h.cuda().view(torch.bfloat16)
        ws = torch.zeros(V.vp_pass_workspace_bytes(sm.model, M), dtype=torch.uint8, device="cuda")

        def calls():  # the MLP block (2l + 1) of every copy
            for l in range(copies):
                V.vp_verify_blocks(sm.model, h, M, 2 * l + 1, 2 * l + 2, None, ws)
        t = graph_time(calls, steps, warmup) / copies
        assert V.vp_read_status(ws) == V.VP_OK
        out[f"M{M}"] = {"us_per_layer": t * 1e6, "gbps": nbytes / t / 1e9}
    del sm
    torch.cuda.empty_cache()
    return {"workload": f"one MLP layer (gate, up [5120->17408], down [17408->5120] NVFP4) as the pass runs it, "
                        f"{copies} rotating copies", "bytes_per_layer": nbytes, **out}


def measure_head_accept(lanes_list, steps: int, warmup: int) -> dict:
    """The NVFP4 vocabulary head [5120 -> 248320] fused with argmax and greedy acceptance
    (vp_head_argmax_accept) at M = 8 lanes, planted draft prefixes of 0..7; per lane count: microseconds
    per call and weight GB/s (715,161,600 B; larger than L2, so every call streams from DRAM)."""
    import torch

    import synth
    from weight_streaming_gb300 import _lib as V
    from weight_streaming_gb300.model import pack_nvfp4
    V_, K = 248320, 5120
    c = torch.empty((V_, K // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty((V_, K // 16), dtype=torch.uint8, device="cuda")
    synth.gpu_uniform_bytes(c, 0, synth.stream_id(synth.HEAD_LAYER, synth.T_HEAD_C))
    synth.gpu_scale_codes(sc, 0, synth.stream_id(synth.HEAD_LAYER, synth.T_HEAD_S))
    w = pack_nvfp4(c, sc)
    del c, sc
    nbytes = V_ * K * 9 // 16
    out = {}
    for L in lanes_list:
        M = 8 * L
        x = torch.from_numpy(synth.normal_bf16(M, synth.stream_id(0, synth.T_X0), (M, K)).view("int16"))
        x = x.cuda().view(torch.bfloat16)
        t_ref = synth.uniform_ints(M, synth.stream_id(0, synth.T_PENDING) + 7, 0, M, V_)
        pending, planted = synth.planted_pending(M, t_ref, V_)
        pend = torch.from_numpy(pending).cuda()
        am = torch.empty(M, dtype=torch.int32, device="cuda")
        nc = torch.empty(L, dtype=torch.int32, device="cuda")
        cm = torch.empty((L, 8), dtype=torch.int32, device="cuda")
        ws = torch.zeros(V.vp_workspace_bytes(V.VP_OP_HEAD, M, V_, K), dtype=torch.uint8, device="cuda")

        def call():
            V.vp_head_argmax_accept(w, 1.0, x, M, V_, K, pend, am, nc, cm, None, ws)
        t = graph_time(call, steps, warmup)
        n = nc.cpu().numpy()
        assert (n >= 1).all() and (n <= 8).all() and V.vp_read_status(ws) == V.VP_OK
        out[f"L{L}"] = {"M": M, "us_per_call": t * 1e6, "gbps": nbytes / t / 1e9,
                        "planted_prefixes": [int(p) for p in planted]}
    del w
    torch.cuda.empty_cache()
    return {"workload": "NVFP4 head [5120->248320] + argmax (lowest index) + greedy accept", "bytes": nbytes, **out}


def measure_cores_pass(sm, M_list, ctx: int, steps: int, warmup: int) -> dict:
    """The verify pass with the real mixer cores (vp_verify_pass_cores) at each M, every lane at
    context ctx: CUDA-graph replays, CUDA events; alone, and followed by the commit of the rows it
    accepted (vp_commit_cores).  Every replay reads parity buffer A and the same window and cache
    rows and rewrites the same outputs, so replays repeat the same work.  Weight GB/s counts the projection weights only; the cores' own reads (the
    key / value cache rows, the delta-rule states) are reported beside it."""
    import numpy as np
    import torch

    import synth
    from weight_streaming_gb300 import _lib as V
    geom = sm.geom
    out = {}
    for M in M_list:
        lanes = M // 8
        x0 = torch.from_numpy(synth.normal_bf16(M, synth.stream_id(0, synth.T_X0), (M, geom.hidden)).view(np.int16))
        x0 = x0.cuda().view(torch.bfloat16)
        t = synth.uniform_ints(M, synth.stream_id(0, synth.T_PENDING) + 7, 0, M, geom.vocab)
        pend = torch.from_numpy(synth.planted_pending(M, t, geom.vocab)[0]).cuda()
        ctx_d = torch.full((lanes,), ctx, dtype=torch.int32, device="cuda")
        am = torch.empty(M, dtype=torch.int32, device="cuda")
        nc = torch.empty(lanes, dtype=torch.int32, device="cuda")
        cm = torch.empty((lanes, 8), dtype=torch.int32, device="cuda")
        ws = sm.cores_workspace(M)
        tp = graph_time(lambda: sm.run_cores(x0, ctx_d, pend, am, nc, cm, ws), steps, warmup)
        assert V.vp_read_status(ws) == V.VP_OK

        def step():  # the pass, then the commit of the rows it accepted (parity 0 both times)
            sm.run_cores(x0, ctx_d, pend, am, nc, cm, ws)
            sm.commit_cores(M, nc, 0, ws)
        tpc = graph_time(step, steps, warmup)
        assert V.vp_read_status(ws) == V.VP_OK
        nb = geom.pass_bytes()
        n_gdn = sum(not geom.is_attn(l) for l in range(geom.n_layers))
        state = n_gdn * lanes * geom.n_v * geom.d * geom.d * 4 * 2  # read state_a, write state_b
        out[f"M{M}"] = {"ms_per_pass": tp * 1e3, "ms_per_pass_and_commit": tpc * 1e3, "weight_gbps": nb / tp / 1e9,
                        "kv_cache_bytes": lanes * geom.kv_bytes(ctx), "state_bytes": state,
                        "all_bytes_gbps": (nb + lanes * geom.kv_bytes(ctx) + state) / tp / 1e9,
                        "launches_per_pass": V.vp_pass_cores_launch_count(sm.model)}
        del ws
    return out


def run_pass_only(args):
    """The verify pass alone (--layers layers, --M rows), CUDA-graph replays with nothing else on the
    device: a small case for profiling; prints one JSON line with the time per pass and weight GB/s."""
    import numpy as np
    import torch

    import synth
    from weight_streaming_gb300 import _lib as V
    from weight_streaming_gb300.geometry import Geometry
    from weight_streaming_gb300.model import SyntheticModel
    geom = Geometry(n_layers=args.layers)
    sm = SyntheticModel(geom, seed=0)
    M, H = args.M, geom.hidden
    x0 = torch.from_numpy(synth.normal_bf16(0, synth.stream_id(0, synth.T_X0), (M, H)).view(np.int16))
    x0 = x0.cuda().view(torch.bfloat16)
    t = synth.uniform_ints(0, synth.stream_id(0, synth.T_PENDING) + 7, 0, M, geom.vocab)
    pend = torch.from_numpy(synth.planted_pending(0, t, geom.vocab)[0]).cuda()
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
    cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
    if args.cores:
        sm.attach_cores(max(1, M // 8), args.ctx + 8)
        r = measure_cores_pass(sm, [M], args.ctx, args.steps, args.warmup)[f"M{M}"]
        print(json.dumps({"kernel": "pass_cores", "layers": args.layers, "M": M, "ctx": args.ctx, **r}), flush=True)
        return
    ws = sm.workspace(M)
    tp = graph_time(lambda: sm.run(x0, pend, am, nc, cm, ws), args.steps, args.warmup)
    assert V.vp_read_status(ws) == V.VP_OK
    nbytes = geom.pass_bytes()
    print(json.dumps({"kernel": "pass", "layers": args.layers, "M": M, "ms_per_pass": tp * 1e3,
                      "gbps": nbytes / tp / 1e9, "bytes_per_pass": nbytes,
                      "launches_per_pass": sm.launch_count()}), flush=True)


def run_kernel(args):
    """One GEMM of the pass alone through the C ABI, rotating over 4 weight copies (> L2) so every
    launch streams from DRAM; prints one JSON line with the average launch time and GB/s."""
    import torch
    if args.kernel == "gdn":
        run_gdn(args)
        return
    if args.kernel == "decode":
        run_decode(args)
        return
    if args.kernel == "sample":
        run_sample(args)
        return
    if args.kernel == "attn":
        run_attn(args)
        return
    if args.kernel == "pass":
        run_pass_only(args)
        return
    if args.kernel == "mlp":
        print(json.dumps({"kernel": "mlp", **measure_mlp_layer([1, 8, 16, 24, 32], args.steps, args.warmup)}), flush=True)
        return
    if args.kernel == "head_accept":
        print(json.dumps({"kernel": "head_accept", **measure_head_accept([1, 4], args.steps, args.warmup)}), flush=True)
        return

    import synth
    from weight_streaming_gb300 import _lib as V
    from weight_streaming_gb300.model import pack_fp8, pack_nvfp4
    shapes = {"gate": ("nvfp4", 17408, 5120), "down": ("nvfp4", 5120, 17408), "gdn_in": ("fp8", 16384, 5120),
              "head": ("nvfp4", 248320, 5120), "q4_gate": ("q4", 17408, 5120), "q4_down": ("q4", 5120, 17408),
              "q4_head": ("q4", 248320, 5120)}
    fmt, N, K = shapes[args.kernel]
    M = args.M
    copies = 1 if args.kernel in ("head", "q4_head") else 4
    ws_list = []
    for c in range(copies):
        if fmt == "nvfp4":
            cc = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
            sc = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
            synth.gpu_uniform_bytes(cc, 0, synth.stream_id(c, synth.T_GATE_C))
            synth.gpu_scale_codes(sc, 0, synth.stream_id(c, synth.T_GATE_S))
            ws_list.append(pack_nvfp4(cc, sc))
        elif fmt == "q4":
            cc = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
            synth.gpu_uniform_bytes(cc, 0, synth.stream_id(c, synth.T_GATE_C))
            sb = synth.q4_scales_biases(0, synth.stream_id(c, synth.T_GATE_S), 0, N * K // 64)
            sc16, bi16 = (torch.from_numpy(a.view("int16")).cuda() for a in sb)
            packed = torch.empty(V.vp_packed_bytes_q4(N, K), dtype=torch.uint8, device="cuda")
            V.vp_pack_q4(cc, sc16, bi16, N, K, packed)
            ws_list.append(packed)
        else:
            w = torch.empty((N, K), dtype=torch.uint8, device="cuda")
            synth.gpu_fp8_normal_codes(w, 0, synth.stream_id(c, synth.T_IN))
            ws_list.append(pack_fp8(w))
    x = torch.randn((M, K), device="cuda").to(torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    op = {"nvfp4": V.VP_OP_NVFP4, "fp8": V.VP_OP_FP8, "q4": V.VP_OP_Q4}[fmt]
    ws = torch.zeros(V.vp_workspace_bytes(op, M, N, K), dtype=torch.uint8, device="cuda")
    if fmt == "q4":
        def fn(w, scale, x_, y_, M_, N_, K_, ws_):
            V.vp_linear_q4(w, x_, y_, M_, N_, K_, ws_)
    else:
        fn = V.vp_linear_nvfp4 if fmt == "nvfp4" else V.vp_linear_fp8
    torch.cuda.synchronize()

    def calls():  # one launch per weight copy
        for w in ws_list:
            fn(w, 1.0, x, y, M, N, K, ws)
    t = graph_time(calls, args.steps, args.warmup) / copies
    nbytes = N * K * 9 // 16 if fmt in ("nvfp4", "q4") else N * K
    peak = (measured_peaks() or {}).get("hbm_gbs")
    print(json.dumps({"kernel": args.kernel, "fmt": fmt, "M": M, "N": N, "K": K, "us_per_launch": t * 1e6,
                      "gbps": nbytes / t / 1e9, "bytes_per_launch": nbytes,
                      "frac_of_measured_copy": (nbytes / t / 1e9 / peak) if peak else None}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.kernel:
        if args.ctx is None:
            args.ctx = 4096 if args.kernel == "pass" else 32768
        run_kernel(args)
        return
    import numpy as np
    import torch

    import synth
    from weight_streaming_gb300 import _lib as V
    from weight_streaming_gb300.model import Geometry, SyntheticModel

    rank, world = dist_setup(args.gpus)
    dev = torch.cuda.current_device()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    geom = Geometry(n_layers=args.layers)
    pass_bytes = geom.pass_bytes()
    sm = SyntheticModel(geom, seed=0)
    H = geom.hidden

    def make_io(M, seed):
        x0 = torch.from_numpy(synth.normal_bf16(seed, synth.stream_id(0, synth.T_X0), (M, H)).view(np.int16))
        x0 = x0.cuda().view(torch.bfloat16)
        t = synth.uniform_ints(seed, synth.stream_id(0, synth.T_PENDING) + 7, 0, M, geom.vocab)
        pending, _ = synth.planted_pending(seed, t, geom.vocab)
        pend = torch.from_numpy(pending).cuda()
        am = torch.empty(M, dtype=torch.int32, device="cuda")
        nc = torch.empty(M // 8, dtype=torch.int32, device="cuda")
        cm = torch.empty((M // 8, 8), dtype=torch.int32, device="cuda")
        ws = sm.workspace(M)
        return x0, pend, am, nc, cm, ws

    def graph_for(M, seed):
        io_ = make_io(M, seed)
        x0, pend, am, nc, cm, ws = io_
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for _ in range(2):
                sm.run(x0, pend, am, nc, cm, ws, stream=s)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                sm.run(x0, pend, am, nc, cm, ws, stream=s)
        torch.cuda.synchronize()
        assert V.vp_read_status(ws) == V.VP_OK
        return g, s, io_

    def time_graph(g, s, steps, warmup):
        with torch.cuda.stream(s):
            for _ in range(warmup):
                g.replay()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(s)
        with torch.cuda.stream(s):
            for _ in range(steps):
                g.replay()
        e1.record(s)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / 1e3

    # ---- headline: M = 8
    g8, s8, io8 = graph_for(8, 0)
    with Clocks(dev) as clk:
        t8 = time_graph(g8, s8, args.steps, args.warmup)
    times = max_over_ranks(t8, world)
    value, tmax = aggregate(pass_bytes * args.steps, times)
    ms8 = 1e3 * tmax / args.steps

    # ---- the other widths (1 graph each)
    also = {}
    for M in (16, 24, 32):
        g, s, _ = graph_for(M, M)
        t = time_graph(g, s, max(3, args.steps // 2), 3)
        steps_m = max(3, args.steps // 2)
        gbs = pass_bytes * steps_m / t / 1e9
        also[f"M{M}"] = {"gbps": gbs, "ms_per_pass": 1e3 * t / steps_m, "passes_per_s": steps_m / t,
                         "implied_tok_s": (M // 8) * 4.8 / (t / steps_m)}
        del g
    also["M8"] = {"gbps": value / world, "ms_per_pass": ms8, "passes_per_s": 1e3 / ms8,
                  "implied_tok_s": 4.8 / (ms8 / 1e3)}
    # run-to-run spread of the headline: the same graph timed in three more runs of K steps
    runs = [ms8] + [1e3 * time_graph(g8, s8, args.steps, 3) / args.steps for _ in range(3)]
    srt = sorted(runs)
    also["M8_runs_ms_per_pass"] = {"runs": runs, "min": srt[0], "median": 0.5 * (srt[1] + srt[2]), "max": srt[-1]}
    # the pass with sampled acceptance at M = 8 (top_k 20, top_p 0.95, temperature 0.7, point-mass drafts)
    x0s, pends, ams, ncs, cms, _ = io8
    wss = torch.zeros(V.vp_pass_sampled_workspace_bytes(sm.model, 8), dtype=torch.uint8, device="cuda")
    us = torch.rand((8, 2), device="cuda", generator=torch.Generator(device="cuda").manual_seed(0))
    t_s = graph_time(lambda: V.vp_verify_pass_sampled(sm.model, x0s, 8, pends, 0.7, 20, 0.95, None, None, us, ams,
                                                      ncs, cms, None, wss), max(3, args.steps // 2), 3)
    also["M8_sampled"] = {"ms_per_pass": t_s * 1e3, "gbps": pass_bytes / t_s / 1e9,
                          "what": "vp_verify_pass_sampled: the pass, its logits written, then sampled acceptance"}
    del wss
    # the per-component workloads: one MLP layer at M = 1 .. 32, and the head with acceptance at 1 / 4 lanes
    if not args.no_components:
        also["config_mlp_layer"] = measure_mlp_layer([1, 8, 16, 24, 32], max(5, args.steps), 3)
        also["config_head_accept"] = measure_head_accept([1, 4], max(5, args.steps), 3)
        # the pass with the real mixer cores in place of the stand-in slice, every lane at context 4096
        sm.attach_cores(4, 4096 + 8)
        also["pass_with_cores_ctx4096"] = measure_cores_pass(sm, [8, 32], 4096, max(5, args.steps // 2), 3)

    # ---- dominant kernel: the pass is two launches of one persistent kernel (exec_kernel<1, 0> at M = 8,
    # 4 phases per layer + the head); its algorithmic bytes are the pass's weight bytes, its duration
    # the event-timed graph replay above (the 80 KB x0 copy in the graph is negligible).
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    achieved = pass_bytes / (tmax / args.steps) / 1e9
    traffic = profiled_traffic(pass_bytes)

    # ---- copy roofline re-measured in this run (torch copy, read + write bytes)
    a = torch.empty(1 << 30, dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    b.copy_(a)
    best = 1e9
    for _ in range(5):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        b.copy_(a)
        c1.record()
        torch.cuda.synchronize()
        best = min(best, c0.elapsed_time(c1) / 1e3)
    copy_gbs = 2 * a.numel() * 2 / best / 1e9
    del a, b
    nominal = None
    try:
        out = subprocess.run(["nvidia-smi", f"--id={dev}", "--query-gpu=clocks.max.memory", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=10).stdout
        mem_mhz = float(out.split()[0])
        nominal = 2 * mem_mhz * 1e6 * 7936 / 8 / 1e9  # double data rate x bus width (bits)
    except Exception:
        pass

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    x0d, pend, am, nc, cm, ws = io8
    x0h = x0d.cpu().pin_memory()
    pendh = pend.cpu().pin_memory()
    amh = torch.empty_like(am, device="cpu").pin_memory()
    nch = torch.empty_like(nc, device="cpu").pin_memory()
    cmh = torch.empty_like(cm, device="cpu").pin_memory()
    se = torch.cuda.Stream()
    with torch.cuda.stream(se):
        for it in range(args.warmup + args.steps):
            if it == args.warmup:
                se.synchronize()
                ee0 = torch.cuda.Event(enable_timing=True)
                ee0.record(se)
                w0 = time.perf_counter()
            x0d.copy_(x0h, non_blocking=True)
            pend.copy_(pendh, non_blocking=True)
            sm.run(x0d, pend, am, nc, cm, ws, stream=se)
            amh.copy_(am, non_blocking=True)
            nch.copy_(nc, non_blocking=True)
            cmh.copy_(cm, non_blocking=True)
        ee1 = torch.cuda.Event(enable_timing=True)
        ee1.record(se)
        se.synchronize()
        wall = time.perf_counter() - w0
    t_e2e = max(ee0.elapsed_time(ee1) / 1e3, 0.0)
    t_e2e = max(t_e2e, wall)
    e2e_times = max_over_ranks(t_e2e, world)
    e2e_val, _ = aggregate(pass_bytes * args.steps, e2e_times)
    h2d = x0h.numel() * 2 + pendh.numel() * 4
    d2h = amh.numel() * 4 + nch.numel() * 4 + cmh.numel() * 4
    assert int(nch.min()) >= 1 and int(nch.max()) <= 8

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world >= 1:
        b, s, thr, desc = oracle_sample(geom, 0, 8)
        cpu = {"value": b / s / 1e9, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": desc}
    frac = achieved / peak
    n_attn = sum(1 for l in range(geom.n_layers) if geom.is_attn(l))
    n_gdn = geom.n_layers - n_attn
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms8, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 mma (nvfp4/fp8 weights exact in f16), f32 accumulate", "data": "synthetic",
        "config": {"workload": f"full verify pass: {geom.n_layers} layers ({n_gdn} GDN + {n_attn} attention FP8 "
                               "projections, NVFP4 MLP) + NVFP4 head + argmax + greedy accept, Qwen3.8-27B shapes, "
                               "M=8 (1 lane)",
                   "bytes_per_pass": pass_bytes, "M": 8, "graph": "one CUDA graph per pass",
                   "l2": "no flush needed: 17.6 GB of weights per pass >> 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": frac,
                     "traffic": traffic,
                     "kernel": f"exec_kernel<1, 0>: the whole pass, {sm.launch_count()} launches "
                               f"({pass_bytes / 1e9:.2f} GB of weights per pass)",
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks else "fallback (of fallback)"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": sm.launch_count() * args.steps,
        "clocks": clk.summary(),
        "also": {**also, "pass_pct_of_measured_copy": 100 * (value / world) / peak,
                 "copy_gbs_this_run": copy_gbs, "pass_pct_of_this_run_copy": 100 * (value / world) / copy_gbs,
                 "nominal_hbm_gbs": nominal},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

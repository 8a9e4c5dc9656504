"""Cost breakdown of the executor's unit loop: the SM's compute rate for one NVFP4 unit (16 rows x
512 K) at 1-4 n-tiles of 8 tokens, with parts of the computation taken out (csrc/unit_bench.cu: the
measurement build libverify_unitbench.so).  Units and activations sit in shared memory, so no memory
traffic is timed; rates are weight bytes per second over all SMs (TB/s-equivalent).

  variant 0  full unit (code and scale loads, conversion and block scaling, activation loads, MMAs)
  variant 1  no MMA
  variant 2  no conversion (code words straight into the MMAs)
  variant 3  conversion only (no activation loads, no MMA)
  variant 4  the gate+up unit: two row blocks' chunks share each activation load

  python -m weight_streaming_gb300.unit_bench [--reps 2000] [--nt 4 --variant 0]   (one configuration)

--ring: the executor's ring streaming from device memory instead (vp_ring_bench): every warp of
152 CTAs streams its own contiguous range of a 12 GB buffer through S slots of B bytes, first with
nothing but one shared-memory load per slot (the ring's own rate, for several slot shapes), then
with the NVFP4 unit at 1-4 n-tiles on each 4608-byte slot (the executor's streaming step with no
phase boundaries).  Rates are bytes read from device memory per second.

  python -m weight_streaming_gb300.unit_bench --ring
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

VARIANTS = ("full", "no MMA", "no conversion", "conversion only", "pairs")


def main(argv=None) -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=2000)
    ap.add_argument("--nt", type=int, default=None, help="one n-tile count (with --variant): a launch to profile")
    ap.add_argument("--variant", type=int, default=0)
    ap.add_argument("--ring", action="store_true", help="the ring streaming from device memory")
    args = ap.parse_args(argv)

    from .build import build
    lib = ctypes.CDLL(build(variant="unitbench"))
    lib.vp_unit_bench.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                  ctypes.c_void_p]
    lib.vp_unit_bench.restype = ctypes.c_int
    import torch

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import synth
    from . import _lib as V

    # two packed units: row block 0 of a 16 x 1024 NVFP4 matrix (chunks 0-1 and 2-3)
    N, K = 16, 1024
    codes = synth.uniform_bytes(0, 1, 0, N * K // 2).reshape(N, K // 2)
    scales = synth.scale_codes(0, 2, 0, N * K // 16).reshape(N, K // 16)
    packed = torch.empty(V.vp_packed_bytes_nvfp4(N, K), dtype=torch.uint8, device="cuda")
    V.vp_pack_nvfp4(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), N, K, packed)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    out = torch.empty((G, 512), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    if args.ring:
        ring(lib, G, out, s)
        return
    if args.nt is not None:  # one configuration, two launches (the second is the one to profile)
        for _ in range(2):
            st = lib.vp_unit_bench(args.nt, args.variant, packed.data_ptr(), args.reps, out.data_ptr(), G, s.cuda_stream)
            assert st == 0, f"vp_unit_bench: cuda error {st}"
        torch.cuda.synchronize()
        print(f"n-tiles {args.nt}, variant {args.variant} ({VARIANTS[args.variant]}): done")
        return
    print(f"unit loop, {G} CTAs x 16 warps, {args.reps} x 4 chunks of 2304 B per warp (TB/s-equivalent)")
    print(f"{'n-tiles':>8s} " + " ".join(f"{v:>16s}" for v in VARIANTS))
    for nt in (1, 2, 3, 4):
        row = []
        for var in range(len(VARIANTS)):
            st = lib.vp_unit_bench(nt, var, packed.data_ptr(), args.reps, out.data_ptr(), G, s.cuda_stream)
            assert st == 0, f"vp_unit_bench: cuda error {st}"
            torch.cuda.synchronize()
            best = None
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                st = lib.vp_unit_bench(nt, var, packed.data_ptr(), args.reps, out.data_ptr(), G, s.cuda_stream)
                e1.record(s)
                torch.cuda.synchronize()
                assert st == 0
                t = e0.elapsed_time(e1) / 1e3
                best = t if best is None else min(best, t)
            nbytes = G * 16 * args.reps * 4 * 2304
            row.append(nbytes / best / 1e12)
        print(f"{nt:8d} " + " ".join(f"{r:16.2f}" for r in row), flush=True)
    assert np.isfinite(out.cpu().numpy()).any()


def ring(lib, G, out, s) -> None:
    import torch

    lib.vp_ring_bench.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                  ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.vp_ring_bench.restype = ctypes.c_int
    nbytes = 12 << 30
    # every byte 0x11: E2M1 codes 0.5, E4M3 scales 2^-6 * 1.125 (finite values; the timing does not
    # depend on them)
    src = torch.full((nbytes,), 0x11, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def rate(nt, W, S, B):
        best = None
        for rep in range(4):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            st = lib.vp_ring_bench(nt, W, S, B, src.data_ptr(), nbytes, G, err.data_ptr(), out.data_ptr(), s.cuda_stream)
            e1.record(s)
            torch.cuda.synchronize()
            assert st == 0, f"vp_ring_bench: cuda error {st}"
            assert err.item() == 0, "a ring wait ran out"
            t = e0.elapsed_time(e1) / 1e3
            if rep > 0:
                best = t if best is None else min(best, t)
        return (nbytes // (G * W * B)) * G * W * B / best / 1e9

    print(f"ring alone ({G} CTAs; GB/s read)")
    print(f"{'warps':>6s} {'slots':>6s} {'bytes':>6s} {'per SM':>8s} {'GB/s':>8s}")
    for W, S, B in ((16, 1, 4608), (16, 2, 4608), (16, 4, 2304), (16, 3, 3072), (16, 6, 1536), (16, 3, 4608),
                    (8, 4, 4608), (8, 3, 9216)):
        print(f"{W:6d} {S:6d} {B:6d} {W * S * B:8d} {rate(0, W, S, B):8.0f}", flush=True)
    print(f"ring + NVFP4 unit (16 warps, slots of 4608 B; GB/s read)")
    print(f"{'n-tiles':>8s} {'1 slot':>8s} {'2 slots':>8s}")
    for nt in (1, 2, 3, 4):
        print(f"{nt:8d} {rate(nt, 16, 1, 4608):8.0f} {rate(nt, 16, 2, 4608):8.0f}", flush=True)


if __name__ == "__main__":
    main()

"""Child process of test_wait_timeout_gpu.py (run with VP_LIBVERIFY naming the wait-test build of the
library, whose bounded waits give up after milliseconds).

A small verify pass runs once normally; then the workspace's test hook makes CTA 0 leave its first
grid-barrier arrival out, so that every other CTA's barrier wait runs out: the call must return,
the workspace's status word must read VP_ERR_TIMEOUT, and, after vp_workspace_init, the next pass
must return exactly the first pass's results.  Prints one line per check."""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import dev_bf16, dev_i32, workspace  # noqa: E402
from passutil import DeviceModel, make_layers  # noqa: E402
from weight_streaming_gb300 import _lib as V  # noqa: E402

SKIP_WORD = 32 // 4  # int32 index of the hook word (byte offset 32 from the status word)


def main():
    assert "waittest" in V.LIB_PATH, V.LIB_PATH
    G = oracle.geom(n_layers=4, hidden=256, inter=512, vocab=2064, period=4, gdn_in=512, gdn_z=384, attn_q=384,
                    attn_kv=128, attn_z=256)
    layers, head = make_layers(G, seed=23)
    dm = DeviceModel(V, G, layers, head)
    M = 8
    x0 = dev_bf16(synth.normal_bf16(9, synth.stream_id(0, synth.T_X0), (M, G.hidden)))
    pend = dev_i32(np.zeros(M, np.int32))
    ws = workspace(V.vp_pass_workspace_bytes(dm.model, M))

    def run():
        am = torch.full((M,), -7, dtype=torch.int32, device="cuda")
        nc = torch.empty(1, dtype=torch.int32, device="cuda")
        cm = torch.empty((1, 8), dtype=torch.int32, device="cuda")
        lg = torch.empty((M, G.vocab), dtype=torch.float32, device="cuda")
        V.vp_verify_pass(dm.model, x0, M, pend, am, nc, cm, None, lg, ws)
        torch.cuda.synchronize()
        return am.cpu(), lg.cpu()

    am0, lg0 = run()
    print("normal status", V.vp_read_status(ws), flush=True)
    ws.view(torch.int32)[SKIP_WORD] = 1  # CTA 0 skips its first arrival
    torch.cuda.synchronize()
    run()
    print("skipped-arrival status", V.vp_read_status(ws), flush=True)
    V.vp_workspace_init(ws)
    torch.cuda.synchronize()
    am1, lg1 = run()
    print("after-init status", V.vp_read_status(ws), flush=True)
    print("after-init equal", int(torch.equal(am0, am1) and torch.equal(lg0, lg1)), flush=True)


if __name__ == "__main__":
    main()

"""Run one libdn kernel on a small case for profiling (a few launches, inputs > L2).

    python -m deltanet_recurrent_state_gb300.profile_case verify  [--layers 8] [--launches 3] [--T 16] [--per-layer]
    python -m deltanet_recurrent_state_gb300.profile_case accept  [--requests 128]
    python -m deltanet_recurrent_state_gb300.profile_case commit  [--layers 48]
    python -m deltanet_recurrent_state_gb300.profile_case prefill [--tokens 4096] [--sequences 1] [--engine mma|tc]
    python -m deltanet_recurrent_state_gb300.profile_case context [--tokens 268000] [--requests 64]
    python -m deltanet_recurrent_state_gb300.profile_case deltas  [--layers 8]

Shapes are those of the single-user workload (48 heads, 128 x 128 fp16 state,
T = 16) with fewer layers, sized so the footprint stays a few hundred MB but
above the 129 MB L2, so DRAM counters mean something.
"""

import argparse
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from deltanet_recurrent_state_gb300 import binding as dn  # noqa: E402
from deltanet_recurrent_state_gb300 import inputs  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["verify", "accept", "commit", "prefill", "context", "deltas"])
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--requests", type=int, default=128)
    ap.add_argument("--tokens", type=int, default=4096)
    ap.add_argument("--sequences", type=int, default=1)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--engine", choices=["mma", "tc"], default="mma", help="prefill engine")
    ap.add_argument("--T", type=int, default=16, help="verify block width (accept: positions per request)")
    ap.add_argument("--per-layer", action="store_true",
                    help="verify: each pass is one launch per layer (N = 1) instead of one over all layers")
    a = ap.parse_args()
    dev = torch.device("cuda:0")
    H, d, T, V = 48, 128, a.T, 151936
    if a.kernel in ("verify", "commit"):
        x = inputs.recurrence_inputs(a.layers, T, H, d, d, seed=1, device=dev)
        out, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
        acc = torch.full((1,), T - 1, dtype=torch.int32, device=dev)
        for _ in range(a.warmup + a.launches):
            if a.kernel == "verify" and a.per_layer:
                for l in range(a.layers):
                    dn.dn_verify_block(x["q"][l:l + 1], x["k"][l:l + 1], x["v"][l:l + 1], x["beta"][l:l + 1],
                                       x["g"][l:l + 1], x["state"][l:l + 1], out[l:l + 1], ckpt[l:l + 1])
            elif a.kernel == "verify":
                dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], out, ckpt)
            else:
                dn.dn_commit(ckpt, acc, x["state"])
    elif a.kernel == "accept":
        B, T4 = a.requests, a.T
        logits, target = inputs.logits_inputs(B, T4, V, dtype="f16", std=2.0, seed=2, device=dev)
        draft = inputs.draft_ids(target, inputs.accepted_lengths(B, T4, "uniform", seed=3), V)
        ws = dn.accept_workspace(B, T4, V, dev)
        for _ in range(a.warmup + a.launches):
            dn.dn_accept_greedy(logits, draft, workspace=ws)
    elif a.kernel == "deltas":
        x = inputs.recurrence_inputs(a.layers, T, H, d, d, seed=1, device=dev)
        out = torch.empty_like(x["v"])
        delta = torch.empty(x["v"].shape, dtype=torch.float32, device=dev)
        acc = torch.full((1,), 15, dtype=torch.int32, device=dev)
        for _ in range(a.warmup + a.launches):
            dn.dn_verify_block_deltas(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], out, delta)
            dn.dn_commit_deltas(x["k"], x["g"], delta, acc, x["state"])
    elif a.kernel == "context":
        ctx, lens = inputs.context_inputs(a.requests, a.tokens, 500, V, quote=True, seed=5)
        ctx, lens = ctx.to(dev), lens.to(dev)
        for _ in range(a.warmup + a.launches):
            dn.dn_context_drafts(ctx, lens, 4, 1, 8)
    else:
        x = inputs.recurrence_inputs(a.sequences, a.tokens, H, d, d, seed=4, device=dev)
        for _ in range(a.warmup + a.launches):
            dn.dn_prefill_checkpoint(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], engine=a.engine)
    torch.cuda.synchronize()
    print("profile_case %s done" % a.kernel)


if __name__ == "__main__":
    main()

"""Benchmark of the DeltaNet verify -> accept -> commit step on one or more GB300s.

One step is one pass of the decode hot path over one batch of seeded synthetic
input, all 48 layers of a request folded into one launch per operation:

    dn_verify_block (48 layers x 48 heads x 128x128 fp16 state, T = 16)
    dn_accept_greedy (16 positions x 151,936-entry fp16 logits rows)
    dn_commit (the checkpoint at the accepted position becomes the state)

The metric counts verified token-layers (B x T x layers) per second. Inputs are
larger than L2 and three buffer sets rotate, so no step reads what the previous
two steps touched. Extra rows time the batch-64 step and the 25,000-token prefill.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs the same per-GPU workload on its own requests
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DeltaNet verify tokens/s (B×T×layers) on 1 GB300; achieved HBM GB/s vs peak"
UNIT = "token-layers/s"
HEADLINE = "single_user_l48_h48_d128_t16_f16"
FALLBACK_HBM_GBS = 6800.0
ROTATE = 3


# ----------------------------------------------------------------------------- byte counts

def verify_bytes(N, T, H, dk, dv, esz):
    """Algorithmic HBM bytes of one dn_verify_block launch: read state, q, k, v, beta, g;
    write out and T checkpoints."""
    per_head = (dv * dk * esz + T * (2 * dk + 2 * dv) * esz + T * 8 + T * dv * dk * esz)
    return N * H * per_head


def accept_bytes(B, T, V, lsz):
    return B * T * V * lsz + B * T * 8 + B * 4


def commit_bytes(L, acc, H, dk, dv, esz):
    """2 x one state set (read checkpoint, write state) per (layer, request) with a >= 1."""
    return 2 * L * int((acc >= 1).sum()) * H * dv * dk * esz


def verify_deltas_bytes(N, T, H, dk, dv, esz):
    """dn_verify_block_deltas: read state, q, k, v, beta, g; write out and delta (fp32)."""
    return N * H * (dv * dk * esz + T * (2 * dk + 2 * dv) * esz + T * 8 + T * dv * 4)


def commit_deltas_bytes(L, acc, H, dk, dv, esz):
    """dn_commit_deltas: per (layer, request) with a >= 1 read and write the state, read
    a keys, gates and deltas."""
    total = 0
    for a in acc.tolist():
        if a >= 1:
            total += L * H * (2 * dv * dk * esz + a * (dk * esz + 4 + dv * 4))
    return total


def prefill_bytes(N, P, H, dk, dv, esz, chunk=64):
    per_head = (P * (2 * dk + 2 * dv) * esz + P * 8 + 2 * dv * dk * esz +
                (P // chunk) * dv * dk * esz)
    return N * H * per_head


# ----------------------------------------------------------------------------- ranks

def max_over_ranks(value, dist, device):
    """The largest `value` over all ranks (the job's duration is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base, rank, buffer_set):
    """Seed of a rank's buffer set: every rank verifies its own requests."""
    return base + 1000 * rank + 17 * buffer_set


# ----------------------------------------------------------------------------- environment

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_hash(files=None):
    """Hash of the kernel sources (all of csrc, or the named files) the counters were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "deltanet_recurrent_state_gb300", "csrc")
    names = sorted(files) if files else sorted(os.listdir(csrc))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_counters.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    k = d.get("kernels", {}).get(kernel)
    if k is None or k.get("sources_sha256_16") != kernel_sources_hash(k.get("sources")):
        return None
    return k.get("dram_bytes_per_launch_full")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples (200 ms) while the GPU works."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0, t1, gpu_index):
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
                rows.append(dict(ts=ts, idx=int(f[1]), sm=float(f[2]), smax=float(f[3]),
                                 hw=f[6], hwt=f[7], swt=f[8], pcap=f[9]))
            except Exception:
                continue
        idxs = sorted(set(r["idx"] for r in rows))
        if gpu_index not in idxs and len(idxs) == 1:
            gpu_index = idxs[0]
        rows = [r for r in rows if r["idx"] == gpu_index]
        win = [r for r in rows if t0 - 0.25 <= r["ts"] <= t1 + 0.25]
        where = "timed region"
        if not win:
            win = [r for r in rows if r["sm"] > 0.5 * r["smax"]] or rows
            where = "whole benchmark (timed region shorter than one sample)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in win):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in win),
                "sm_max_mhz": max(r["smax"] for r in win), "reasons": reasons,
                "samples": len(win), "window": where}


# ----------------------------------------------------------------------------- workloads

def make_step_sets(w, device, rank, count):
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    from deltanet_recurrent_state_gb300 import inputs

    N, B, T = w["L"] * w["B"], w["B"], w["T"]
    sets = []
    for r in range(count):
        seed = rank_seed(w["seed"], rank, r)
        x = inputs.recurrence_inputs(N, T, w["H"], w["dk"], w["dv"], io=w["io"], state=w["state"],
                                     seed=seed, device=device)
        logits, target = inputs.logits_inputs(B, T, w["V"], dtype=w["logit_dtype"],
                                              std=w["logit_std"], seed=seed + 1, device=device)
        acc = inputs.accepted_lengths(B, T, w["accept"], seed=seed + 2, value=w.get("accept_value"))
        draft = inputs.draft_ids(target, acc, w["V"], seed=seed + 3)
        x.update(logits=logits, draft=draft, acc_plan=acc)
        x["out"] = torch.empty((N, T, w["H"], w["dv"]), dtype=x["q"].dtype, device=device)
        x["ckpt"] = torch.empty((N, T, w["H"], w["dv"], w["dk"]), dtype=x["state"].dtype,
                                device=device)
        x["tgt"] = torch.empty((B, T), dtype=torch.int32, device=device)
        x["acc"] = torch.empty((B,), dtype=torch.int32, device=device)
        x["ws"] = dn.accept_workspace(B, T, w["V"], device)
        sets.append(x)
    return sets


def side_stream(device):
    """A high-priority second stream: accept runs on it beside verify."""
    import torch
    lo, hi = torch.cuda.Stream.priority_range()
    return torch.cuda.Stream(device=device, priority=hi)


def run_step(x, stream, evs=None, side=None):
    """One step: verify, accept, commit. With `side`, accept (which reads only the logits and
    the draft ids) runs on the side stream concurrently with verify, and commit waits for
    both; with `evs` (the per-kernel breakdown) the three run one after another with events
    between them."""
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    if side is not None and not evs:
        fork = torch.cuda.Event()
        fork.record(stream)
        side.wait_event(fork)
        dn.dn_accept_greedy(x["logits"], x["draft"], x["tgt"], x["acc"], x["ws"], stream=side)
        join = torch.cuda.Event()
        join.record(side)
        dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], x["out"], x["ckpt"],
                           stream=stream)
        stream.wait_event(join)
        dn.dn_commit(x["ckpt"], x["acc"], x["state"], stream=stream)
        return
    if evs:
        evs[0].record(stream)
    dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], x["out"], x["ckpt"],
                       stream=stream)
    if evs:
        evs[1].record(stream)
    dn.dn_accept_greedy(x["logits"], x["draft"], x["tgt"], x["acc"], x["ws"], stream=stream)
    if evs:
        evs[2].record(stream)
    dn.dn_commit(x["ckpt"], x["acc"], x["state"], stream=stream)
    if evs:
        evs[3].record(stream)


def timed_steps(sets, steps, warmup, stream, dist, per_kernel=True, graphs=True, by_set=None):
    """Warm up, then time exactly `steps` steps between barriers; returns (seconds,
    per-kernel mean ms [verify, accept, commit], wall-clock bounds). With a list `by_set`,
    it also receives (set index, [verify, accept, commit] ms) of every eager step. Accept runs on a second
    stream beside verify (run_step). With `graphs`, each buffer set's step (the three calls)
    is captured once in a CUDA graph and a timed step is one replay, as a serving loop
    launches a fixed step; the per-kernel durations then come from a separate eager pass with
    the three launches one after another and events recorded between them."""
    import torch
    side = side_stream(stream.device)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            run_step(sets[i % len(sets)], stream, side=side)
    torch.cuda.synchronize()
    if graphs:
        gs = []
        for x in sets:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                run_step(x, stream, side=side)
            gs.append(gr)
        with torch.cuda.stream(stream):
            for i in range(warmup):
                gs[i % len(gs)].replay()

        def step(i):
            gs[i % len(gs)].replay()
    else:
        def step(i):
            run_step(sets[i % len(sets)], stream, side=side)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            step(i)
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist is not None:
        dist.barrier()
    secs = start.elapsed_time(end) / 1e3
    per = None
    if per_kernel:
        n = min(steps, 500)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(n):
                run_step(sets[i % len(sets)], stream, evs[i])
        torch.cuda.synchronize()
        per = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(3)]
        if by_set is not None:
            by_set.extend((i % len(sets), [e[j].elapsed_time(e[j + 1]) for j in range(3)]) for i, e in enumerate(evs))
    return secs, per, (t_wall0, t_wall1)


def e2e_group_bounds(L, groups):
    """State-set boundaries [0, ..., L] of the end-to-end step's layer groups: `groups` is
    a count of equal groups or a list of group sizes."""
    if isinstance(groups, int):
        if groups < 1 or L % groups != 0:
            raise ValueError("%d layers do not split into %d equal groups" % (L, groups))
        sizes = [L // groups] * groups
    else:
        sizes = [int(x) for x in groups]
    if not sizes or min(sizes) < 1 or sum(sizes) != L:
        raise ValueError("group sizes %s do not cover %d layers" % (sizes, L))
    return [sum(sizes[:i]) for i in range(len(sizes) + 1)]


def e2e_growing_groups(L):
    """Group sizes of the pipelined end-to-end step: L/12, L/6, L/3 and the rest (4, 8, 16, 20
    for 48 layers), or one group when L is too small to split."""
    if L < 12:
        return [L]
    sizes = [L // 12, L // 6, L // 3]
    return sizes + [L - sum(sizes)]


def e2e_steps(w, sets, steps, warmup, stream, device, graphs=True, groups=1):
    """The same step through the public API with host inputs: every step copies its
    inputs from pinned host memory and reads its results back (the target ids and the
    accepted length, which a serving loop needs to emit tokens; the outputs o feed the
    next sub-layer on the device), and the host waits for them before the next step.
    A step's inputs sit in one pinned buffer and its results in one device region (the
    tensors the calls take are views of them).
    `groups` is a count of equal groups or a list of group sizes (state sets per group). With
    one group the inputs go over in a single copy before the three calls. With more the step
    is pipelined over the layers: the state sets split into contiguous groups, each
    group's q, k, v, beta and g are one contiguous piece of the
    pinned buffer and go over in their own copy on a copy stream, and the group's verify
    (dn_verify_block on that slice of the state sets) starts on the compute stream as soon
    as its copy has landed, so the host link carries the later groups while the earlier
    ones verify. The logits and draft ids go last; accept and commit follow as before.
    With `graphs`, each buffer set's step (the copies, the calls and the device-to-host
    copy, all issued through the public binding) is captured once in a CUDA graph, and a
    step is one replay; otherwise every call is issued from Python each step. Returns
    (seconds, h2d bytes per step, d2h bytes per step)."""
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    bounds = e2e_group_bounds(sets[0]["q"].shape[0], groups)
    groups = len(bounds) - 1
    group_keys = ("q", "k", "v", "beta", "g")
    tail_keys = ("logits", "draft")
    out_keys = ("tgt", "acc")  # what the serving loop needs back; o stays on the device

    def entries_in(x):
        e = [("%s%d" % (k, gi), x[k][bounds[gi]:bounds[gi + 1]]) for gi in range(groups) for k in group_keys]
        return e + [(k, x[k]) for k in tail_keys]

    def packed(entries, pinned):
        """One byte buffer holding the tensors of `entries` in order (256-byte aligned),
        views of it with their shapes and dtypes, and each entry's byte offset."""
        offs, total = {}, 0
        for name, t in entries:
            offs[name] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(total, dtype=torch.uint8, pin_memory=pinned) if pinned else \
            torch.empty(total, dtype=torch.uint8, device=device)
        views = {name: buf[offs[name]:offs[name] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for name, t in entries}
        return buf, views, offs, total

    host, dev_in, dev_out, host_out, segs = [], [], [], [], None
    for x in sets:
        ent = entries_in(x)
        hb, hv, offs, total = packed(ent, True)
        db, dv_, _, _ = packed(ent, False)
        for name, t in ent:
            hv[name].copy_(t.cpu())
            dv_[name].copy_(t)
        outs = [(k, x[k]) for k in out_keys]
        ob, ov, _, _ = packed(outs, False)
        hob, _, _, _ = packed(outs, True)
        host.append(hb)
        dev_in.append((db, dv_))
        dev_out.append((ob, ov))
        host_out.append(hob)
        # byte ranges copied one by one: each group's inputs, then the logits and drafts
        starts = [offs["q%d" % gi] for gi in range(groups)] + [offs["logits"]]
        segs = [(starts[i], starts[i + 1]) for i in range(groups)] + [(offs["logits"], total)]
    h2d = host[0].numel()
    d2h = host_out[0].numel()
    copy_stream = torch.cuda.Stream(device=device)
    side = side_stream(device)
    events = [[torch.cuda.Event() for _ in range(groups + 1)] for _ in sets]
    joins = [torch.cuda.Event() for _ in sets]

    def body(j):
        x = dict(sets[j])
        dvw = dev_in[j][1]
        x.update(dev_out[j][1])
        if groups == 1:
            dev_in[j][0].copy_(host[j], non_blocking=True)  # one pinned copy (the host link's full rate)
            side.wait_stream(stream)
        else:
            copy_stream.wait_stream(stream)
            with torch.cuda.stream(copy_stream):
                for i, (a0, a1) in enumerate(segs):
                    dev_in[j][0][a0:a1].copy_(host[j][a0:a1], non_blocking=True)
                    events[j][i].record(copy_stream)
            side.wait_event(events[j][groups])  # the logits and drafts have landed
        # accept beside the verify calls (it reads only the logits and drafts)
        dn.dn_accept_greedy(dvw["logits"], dvw["draft"], x["tgt"], x["acc"], x["ws"], stream=side)
        joins[j].record(side)
        for gi in range(groups):
            if groups > 1:
                stream.wait_event(events[j][gi])
            sl = slice(bounds[gi], bounds[gi + 1])
            dn.dn_verify_block(dvw["q%d" % gi], dvw["k%d" % gi], dvw["v%d" % gi], dvw["beta%d" % gi],
                               dvw["g%d" % gi], x["state"][sl], x["out"][sl], x["ckpt"][sl], stream=stream)
        stream.wait_event(joins[j])
        dn.dn_commit(x["ckpt"], x["acc"], x["state"], stream=stream)
        host_out[j].copy_(dev_out[j][0], non_blocking=True)

    def eager(i):
        with torch.cuda.stream(stream):
            body(i % len(sets))
        stream.synchronize()

    for i in range(warmup):
        eager(i)
    torch.cuda.synchronize()
    step = eager
    if graphs:
        gs = []
        for j in range(len(sets)):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                body(j)
            gs.append(gr)

        def step(i):
            with torch.cuda.stream(stream):
                gs[i % len(sets)].replay()
            stream.synchronize()

        for i in range(warmup):
            step(i)
        torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    return time.perf_counter() - t0, h2d, d2h


def prefill_row(device, stream, reps=2):
    """The 25,000-token prefill of 48 layers, two ways: 48 per-layer launches (one
    sequence each, two layer buffers rotating) and one launch over 48 independent
    sequences (N = 48, the throughput view)."""
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    from deltanet_recurrent_state_gb300 import inputs
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS
    w = WORKLOADS["prefill_p25000_l48_h48_d128_c64_f16"]
    P, H, d, L = w["P"], w["H"], w["dk"], w["L"]

    def bufs(N, seed):
        x = inputs.recurrence_inputs(N, P, H, d, d, seed=seed, device=device)
        x["out"] = torch.empty((N, P, H, d), dtype=torch.float16, device=device)
        x["ckpt"] = torch.empty((N, P // 64, H, d, d), dtype=torch.float16, device=device)
        x["s_out"] = torch.empty((N, H, d, d), dtype=torch.float16, device=device)
        return x

    def launch(x):
        dn.dn_prefill_checkpoint(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], x["out"],
                                 x["ckpt"], x["s_out"], stream=stream)

    def timed(fn, count):
        with torch.cuda.stream(stream):
            for i in range(2):
                fn(i)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            with torch.cuda.stream(stream):
                for i in range(count):
                    fn(i)
            e.record(stream)
            torch.cuda.synchronize()
            t = s.elapsed_time(e) / 1e3
            best = t if best is None else min(best, t)
        return best

    layer = [bufs(1, w["seed"] + r) for r in range(2)]
    t_layers = timed(lambda i: launch(layer[i % 2]), L)
    del layer
    folded = bufs(L, w["seed"] + 7)
    t_fold = timed(lambda i: launch(folded), 1)
    del folded
    nbytes = prefill_bytes(1, P, H, d, d, 2) * L
    return {"workload": "prefill_p25000_l48_h48_d128_c64_f16",
            "per_layer_launches": {"launches": L, "ms_all_layers": t_layers * 1e3,
                                   "token_layers_per_s": P * L / t_layers,
                                   "achieved_gbs": nbytes / t_layers / 1e9},
            "folded_one_launch": {"sequences": L, "ms": t_fold * 1e3,
                                  "token_layers_per_s": P * L / t_fold,
                                  "achieved_gbs": nbytes / t_fold / 1e9},
            "algorithmic_bytes": nbytes}


def add_prefill_fractions(row, hbm):
    """Both prefill launch forms as fractions of the measured copy peak and of 8 TB/s."""
    for form in ("per_layer_launches", "folded_one_launch"):
        r = row[form]
        r["frac"] = r["achieved_gbs"] / hbm
        r["frac_of_nominal_8tbs"] = r["achieved_gbs"] / 8000.0
    return row


def deltas_row(sets, device, stream, steps=200, warmup=5):
    """The single-user step with recompute on commit: verify without checkpoints (delta_t
    per row instead), greedy accept, commit rebuilding the accepted state from delta."""
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS
    w = WORKLOADS[HEADLINE]
    N, B, T, H, dk, dv = w["L"] * w["B"], w["B"], w["T"], w["H"], w["dk"], w["dv"]
    for x in sets:
        x["delta"] = torch.empty((N, T, H, dv), dtype=torch.float32, device=device)

    side = side_stream(device)

    def step(x, evs=None):
        if not evs:  # accept beside verify, commit after both (as run_step)
            fork = torch.cuda.Event()
            fork.record(stream)
            side.wait_event(fork)
            dn.dn_accept_greedy(x["logits"], x["draft"], x["tgt"], x["acc"], x["ws"], stream=side)
            join = torch.cuda.Event()
            join.record(side)
            dn.dn_verify_block_deltas(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], x["out"],
                                      x["delta"], stream=stream)
            stream.wait_event(join)
            dn.dn_commit_deltas(x["k"], x["g"], x["delta"], x["acc"], x["state"], stream=stream)
            return
        if evs:
            evs[0].record(stream)
        dn.dn_verify_block_deltas(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], x["out"],
                                  x["delta"], stream=stream)
        if evs:
            evs[1].record(stream)
        dn.dn_accept_greedy(x["logits"], x["draft"], x["tgt"], x["acc"], x["ws"], stream=stream)
        if evs:
            evs[2].record(stream)
        dn.dn_commit_deltas(x["k"], x["g"], x["delta"], x["acc"], x["state"], stream=stream)
        if evs:
            evs[3].record(stream)

    with torch.cuda.stream(stream):
        for i in range(warmup):
            step(sets[i % len(sets)])
    torch.cuda.synchronize()
    # the timed steps are CUDA graph replays (one per buffer set), as for the main step
    gs = []
    for x in sets:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(x)
        gs.append(gr)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            gs[i % len(gs)].replay()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            gs[i % len(gs)].replay()
    s1.record(stream)
    torch.cuda.synchronize()
    secs = s0.elapsed_time(s1) / 1e3
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            step(sets[i % len(sets)], evs[i])
    torch.cuda.synchronize()
    per = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(3)]
    del gs
    vb = verify_deltas_bytes(N, T, H, dk, dv, 2)
    cb = commit_deltas_bytes(w["L"], sets[0]["acc_plan"], H, dk, dv, 2)
    for x in sets:
        del x["delta"]
    return {"workload": HEADLINE + " (recompute on commit)", "ms_per_step": secs / steps * 1e3,
            "token_layers_per_s": B * T * w["L"] * steps / secs,
            "verify_deltas_ms": per[0], "verify_deltas_gbs": vb / (per[0] / 1e3) / 1e9,
            "accept_ms": per[1], "commit_deltas_ms": per[2],
            "commit_deltas_gbs": cb / (per[2] / 1e3) / 1e9,
            "state_pages_per_request_layer": "1 (+ fp32 deltas: T x H x dv x 4 B) instead of T + 1",
            "algorithmic_bytes_per_step": vb + cb + accept_bytes(B, T, w["V"], 2)}


def verify_per_layer_row(sets, device, stream, reps=50, warmup=5):
    """The single-user verify as a model runs it, one layer at a time: 48 launches of
    dn_verify_block over one state set each (B = 1, 48 heads, T = 16; layer l + 1's q/k/v
    come out of layer l), captured in one CUDA graph per buffer set and timed per replay,
    beside the same 48 layers folded into one launch."""
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS
    w = WORKLOADS[HEADLINE]
    L, T, H, dk, dv = w["L"], w["T"], w["H"], w["dk"], w["dv"]

    def layers(x):
        for l in range(L):
            sl = {k: x[k][l:l + 1] for k in ("q", "k", "v", "beta", "g", "state", "out", "ckpt")}
            dn.dn_verify_block(sl["q"], sl["k"], sl["v"], sl["beta"], sl["g"], sl["state"], sl["out"],
                               sl["ckpt"], stream=stream)

    def folded(x):
        dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], x["out"], x["ckpt"],
                           stream=stream)

    res = {"workload": HEADLINE + " verify, one launch per layer", "layers": L}
    for name, body in (("per_layer", layers), ("folded", folded)):
        with torch.cuda.stream(stream):
            for i in range(warmup):
                body(sets[i % len(sets)])
        torch.cuda.synchronize()
        gs = []
        for x in sets:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                body(x)
            gs.append(gr)
        with torch.cuda.stream(stream):
            for i in range(warmup):
                gs[i % len(gs)].replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for i in range(reps):
                gs[i % len(gs)].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        vb = verify_bytes(L, T, H, dk, dv, 2)
        res[name] = {"ms_per_48_layers": ms, "us_per_layer": ms / L * 1e3,
                     "gbs": vb / (ms / 1e3) / 1e9, "token_layers_per_s": T * L / (ms / 1e3)}
        del gs
    hbm, _ = peaks()
    for name in ("per_layer", "folded"):
        res[name]["frac"] = res[name]["gbs"] / hbm
    res["bytes_per_layer_launch"] = verify_bytes(1, T, H, dk, dv, 2)
    # 32-row CTAs, or 16-row ones when a launch has fewer 32-row CTAs than two per SM
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    res["ctas_per_layer_launch"] = H * dv // 32 if H * dv // 32 >= 2 * sms else H * dv // 16
    return res


def commit_alone_row(sets, device, stream, reps=20, warmup=3):
    """dn_commit of the single-user step (48 state sets, T = 16) timed by itself, in two
    conditions: after an L2 flush (a 512 MB read), and right after the step's verify (its
    checkpoint stores leave up to an L2's worth of dirty lines, written back while commit
    runs). The first is the copy's own rate; the second is what it costs inside the step."""
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS
    w = WORKLOADS[HEADLINE]
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    flush.fill_(1.0)
    sink = torch.empty((), dtype=torch.float32, device=device)
    with torch.cuda.stream(stream):
        for x in sets:  # targets and accepted lengths of every set
            dn.dn_accept_greedy(x["logits"], x["draft"], x["tgt"], x["acc"], x["ws"], stream=stream)
    torch.cuda.synchronize()
    res = {"workload": HEADLINE + " commit"}
    for cond in ("after_l2_flush", "after_verify"):
        times, nbytes = [], []
        for i in range(warmup + reps):
            x = sets[i % len(sets)]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                if cond == "after_l2_flush":
                    torch.sum(flush, dim=0, out=sink)
                else:
                    dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], x["out"],
                                       x["ckpt"], stream=stream)
                e0.record(stream)
                dn.dn_commit(x["ckpt"], x["acc"], x["state"], stream=stream)
                e1.record(stream)
            torch.cuda.synchronize()
            if i >= warmup:
                times.append(e0.elapsed_time(e1))
                nbytes.append(commit_bytes(w["L"], x["acc_plan"], w["H"], w["dk"], w["dv"], 2))
        ms = statistics.median(times)
        gbs = statistics.mean(nbytes) / (ms / 1e3) / 1e9
        res[cond] = {"us": ms * 1e3, "gbs": gbs}
    hbm, _ = peaks()
    for cond in ("after_l2_flush", "after_verify"):
        res[cond]["frac"] = res[cond]["gbs"] / hbm
    del flush
    return res


def decode_row(device, stream, steps=1000, warmup=10, nsets=8):
    """The single-user decode loop: 1000 consecutive verify (T = 8) -> accept -> commit steps
    timed as one loop, each step committing into the state the next step of its buffer set
    reads. Accepted lengths are geometric with mean 4, clamped at T (one draw per buffer set;
    8 rotating sets, ~0.7 GB each, so no step finds its inputs in L2)."""
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS
    w = WORKLOADS["decode_loop_l48_h48_d128_t8_f16"]
    sets = make_step_sets(w, device, 0, nsets)
    by_set = []
    secs, per, _ = timed_steps(sets, steps, warmup, stream, None, by_set=by_set)
    N, B, T = w["L"] * w["B"], w["B"], w["T"]
    vb = verify_bytes(N, T, w["H"], w["dk"], w["dv"], 2)
    plans = [int(x["acc_plan"][0]) for x in sets]
    cbs = [commit_bytes(w["L"], x["acc_plan"], w["H"], w["dk"], w["dv"], 2) for x in sets]
    cb = statistics.mean(cbs)
    # the steps whose request accepted at least one token (the others launch commit but copy nothing)
    copying = [(cbs[i], ms[2]) for i, ms in by_set if cbs[i] > 0]
    res = {"workload": "decode_loop_l48_h48_d128_t8_f16", "steps": steps,
           "ms_per_step": secs / steps * 1e3, "loop_ms": secs * 1e3,
           "token_layers_per_s": B * T * w["L"] * steps / secs,
           "accepted_per_set": plans, "accepted_mean": statistics.mean(plans),
           "verify_ms": per[0], "verify_gbs": vb / (per[0] / 1e3) / 1e9,
           "accept_ms": per[1], "commit_ms": per[2],
           "commit_gbs": cb / (per[2] / 1e3) / 1e9 if per[2] > 0 else None}
    if copying:
        ms_copy = statistics.mean(t for _, t in copying)
        res["commit_copying_steps"] = {"steps": len(copying), "ms": ms_copy,
                                       "gbs": statistics.mean(b for b, _ in copying) / (ms_copy / 1e3) / 1e9}
    del sets
    return res


def batch_row(device, stream, steps=10, warmup=3):
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS
    w = WORKLOADS["batch64_l48_h48_d128_t4_f16"]
    sets = make_step_sets(w, device, 0, 2)
    secs, per, _ = timed_steps(sets, steps, warmup, stream, None)
    N, B, T = w["L"] * w["B"], w["B"], w["T"]
    vb = verify_bytes(N, T, w["H"], w["dk"], w["dv"], 2)
    cb = commit_bytes(w["L"], sets[0]["acc_plan"], w["H"], w["dk"], w["dv"], 2)
    res = {"workload": "batch64_l48_h48_d128_t4_f16", "ms_per_step": secs / steps * 1e3,
           "token_layers_per_s": B * T * w["L"] * steps / secs,
           "verify_ms": per[0], "verify_gbs": vb / (per[0] / 1e3) / 1e9,
           "accept_ms": per[1], "commit_ms": per[2],
           "commit_gbs": cb / (per[2] / 1e3) / 1e9 if per[2] > 0 else None}
    del sets
    return res


def context_bytes(lengths, K):
    """Algorithmic bytes of one dn_context_drafts launch: every context token read once,
    plus the length read and the drafts, count and match length written per request."""
    return 4 * int(sum(int(x) for x in lengths)) + len(lengths) * 4 * (1 + K + 2)


def context_row(device, stream, launches=200, warmup=5):
    """Drafting from the request's own context, once per verify step: the single-user
    document-reproduction case (25,000-token prompt + 1,000 quoted tokens) and 64 requests
    at a 268,000-token context (4 rotating sets, 274 MB, larger than L2)."""
    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    from deltanet_recurrent_state_gb300 import inputs
    out = {}
    for name, N, prompt, gen, nsets in [("single_user_p25000_g1000", 1, 25000, 1000, 3),
                                        ("batch64_p268000_g500", 64, 268000, 500, 4)]:
        sets = []
        for i in range(nsets):
            ctx, lens = inputs.context_inputs(N, prompt, gen, 151936, quote=True, seed=1100 + i)
            sets.append((ctx.to(device), lens.to(device),
                         torch.empty((N, 8), dtype=torch.int32, device=device),
                         torch.empty((N,), dtype=torch.int32, device=device),
                         torch.empty((N,), dtype=torch.int32, device=device)))
        with torch.cuda.stream(stream):
            for i in range(warmup):
                c = sets[i % nsets]
                dn.dn_context_drafts(c[0], c[1], 4, 1, 8, c[2], c[3], c[4], stream=stream)
        # the lookups are captured in one CUDA graph (as a serving loop would launch them,
        # ahead of the GPU) so that host launch overhead does not sit between them
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(launches):
                c = sets[i % nsets]
                dn.dn_context_drafts(c[0], c[1], 4, 1, 8, c[2], c[3], c[4], stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            graph.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / launches
        nbytes = context_bytes(sets[0][1].tolist(), 8)
        found = int(sets[(launches - 1) % nsets][3].min())
        out[name] = {"us_per_lookup": ms * 1e3, "gbs": nbytes / (ms / 1e3) / 1e9,
                     "bytes": nbytes, "drafts_found_min": found, "n_max": 4, "K": 8}
        del sets, graph
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_inputs(w, heads, seed):
    """One layer of workload w restricted to `heads` heads, as float64 arrays."""
    from deltanet_recurrent_state_gb300 import inputs
    B, T = w["B"], w["T"]
    x = inputs.recurrence_inputs(B, T, heads, w["dk"], w["dv"], io=w["io"], state=w["state"],
                                 seed=seed, device="cpu")
    logits, target = inputs.logits_inputs(B, T, w["V"], dtype=w["logit_dtype"], std=w["logit_std"],
                                          seed=seed + 1)
    acc = inputs.accepted_lengths(B, T, w["accept"], seed=seed + 2, value=w.get("accept_value"))
    d = {k: x[k].double().numpy() for k in ("q", "k", "v", "beta", "g", "state")}
    d["logits"] = logits.double().numpy()
    d["draft"] = inputs.draft_ids(target, acc, w["V"], seed=seed + 3).numpy()
    d["heads"] = heads
    return d


def oracle_step(w, d):
    """The oracle's verify + accept + commit on the sample `d`; returns (seconds,
    token-layers), counting a layer restricted to h of H heads as h/H of a layer."""
    import oracle
    t0 = time.perf_counter()
    _, ckpt = oracle.verify_block(d["q"], d["k"], d["v"], d["beta"], d["g"], d["state"],
                                  store=w["state"], io=w["io"])
    _, a = oracle.accept_greedy(d["logits"], d["draft"])
    oracle.commit(d["state"], ckpt, a)
    return time.perf_counter() - t0, w["B"] * w["T"] * d["heads"] / w["H"]


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def reference_arm(args, rank, world, budget_s=120.0):
    """The CPU oracle, as it stands, on the same workload, metric and unit. Each step is
    one layer of the verify step (verify + commit on a sample of heads, greedy accept over
    the full vocabulary), with the head sample sized so the whole run stays near
    `budget_s` seconds."""
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS
    if rank != 0:
        return
    w = WORKLOADS[HEADLINE]
    d = oracle_inputs(w, w["H"], w["seed"])
    t1, _ = oracle_step(w, d)
    heads = int(max(1, min(w["H"], w["H"] * budget_s / ((args.steps + args.warmup) * t1))))
    if heads < w["H"]:
        d = oracle_inputs(w, heads, w["seed"])
    for _ in range(args.warmup):
        oracle_step(w, d)
    total_s, total_u = 0.0, 0.0
    for _ in range(args.steps):
        s, u = oracle_step(w, d)
        total_s += s
        total_u += u
    v = total_u / total_s
    sample = ("per step: 1 of %d layers, %d of %d heads, T=%d verify + commit, greedy accept of "
              "%d rows over V=%d" % (w["L"], heads, w["H"], w["T"], w["T"], w["V"]))
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": HEADLINE, "layers": w["L"], "B": w["B"], "T": w["T"], "H": w["H"],
                   "dk": w["dk"], "dv": w["dv"], "V": w["V"], "step_sample": sample},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-rows", action="store_true", help="skip the batch and prefill rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import torch
    from deltanet_recurrent_state_gb300 import binding as dn
    from deltanet_recurrent_state_gb300.workloads import WORKLOADS

    dn.load_library()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=device)
        dist = tdist

    w = WORKLOADS[HEADLINE]
    N, B, T, H, dk, dv = w["L"] * w["B"], w["B"], w["T"], w["H"], w["dk"], w["dv"]
    sets = make_step_sets(w, device, rank, ROTATE)
    stream = torch.cuda.Stream(device)
    clocks = ClockSampler()
    time.sleep(0.3)

    secs, per, (tw0, tw1) = timed_steps(sets, args.steps, args.warmup, stream, dist)
    secs = max_over_ranks(secs, dist, device)
    units_per_rank = B * T * w["L"] * args.steps
    value = units_per_rank * world / secs

    e2e_k = max(3, min(args.steps, 200))
    # layer groups of the pipelined step, growing (48 layers: 4, 8, 16, 20): the first group's
    # copy is short so the verify starts early, and each later copy lands about when the
    # verify of the groups before it ends (copies move a layer in ~3.4 us, verify takes ~4.3 us)
    e2e_groups = e2e_growing_groups(w["L"])
    e2e_s, h2d, d2h = e2e_steps(w, sets, e2e_k, 3, stream, device, groups=e2e_groups)
    e2e_value = B * T * w["L"] * e2e_k / e2e_s
    e2e_eager_s, _, _ = e2e_steps(w, sets, e2e_k, 3, stream, device, graphs=False, groups=e2e_groups)
    e2e_serial_s, _, _ = e2e_steps(w, sets, e2e_k, 3, stream, device, groups=1)

    rows = {}
    if not args.no_rows and rank == 0:
        rows["verify_per_layer"] = verify_per_layer_row(sets, device, stream)
        rows["commit_alone"] = commit_alone_row(sets, device, stream)
        rows["recompute_on_commit_step"] = deltas_row(sets, device, stream)
        rows["decode_loop"] = decode_row(device, stream)
        rows["batch64_step"] = batch_row(device, stream)
        rows["prefill"] = prefill_row(device, stream)
        rows["context_drafts"] = context_row(device, stream)
    clocks.stop()
    gpu_index = local
    cvd = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if cvd and cvd.split(",")[local].strip().isdigit():
        gpu_index = int(cvd.split(",")[local])
    clock_info = clocks.summary(tw0, tw1, gpu_index)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    hbm, peak_kind = peaks()
    if "prefill" in rows:
        add_prefill_fractions(rows["prefill"], hbm)
    vb = verify_bytes(N, T, H, dk, dv, 2)
    ab = accept_bytes(B, T, w["V"], 2)
    cb = commit_bytes(w["L"], sets[0]["acc_plan"], H, dk, dv, 2)
    v_ms, a_ms, c_ms = per
    achieved = vb / (v_ms / 1e3) / 1e9
    traffic = ncu_traffic("verify_block_kernel")

    cpu = None
    if not args.no_cpu and world == 1:
        d = oracle_inputs(w, H, w["seed"] + 500)
        s_tot, u_tot, n = 0.0, 0.0, 0
        while s_tot < 10.0 or n < 2:
            s, u = oracle_step(w, d)
            s_tot, u_tot, n = s_tot + s, u_tot + u, n + 1
        cpu = {"value": u_tot / s_tot, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": "%d repetitions of 1 of 48 layers (48 heads, T=16 verify + commit, "
                         "greedy accept over V=151936), %.1f s" % (n, s_tot)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded; planted argmax, 15 of 16 accepted)",
        "config": {"workload": HEADLINE, "layers": w["L"], "B": B, "T": T, "H": H, "dk": dk,
                   "dv": dv, "V": w["V"], "accepted": int(sets[0]["acc_plan"][0]),
                   "l2": "inputs larger than L2 (%.2f GB per step), %d rotating buffer sets"
                         % ((vb + ab + cb) / 1e9, ROTATE),
                   "parallelism": "replicas" if world == 1 else "dp%d (independent requests)" % world,
                   "launch": "one CUDA graph replay per step: verify, accept beside it on a second "
                             "stream (it reads only logits and drafts), then commit; per-kernel "
                             "durations from an eager pass with the three launches one after "
                             "another and events between them"},
        "roofline": {"bound": "hbm", "kernel": "dn_verify_block", "achieved": achieved,
                     "peak": hbm, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / hbm,
                     "frac_of_nominal_8tbs": achieved / 8000.0, "traffic": traffic,
                     "algorithmic_bytes_per_launch": vb, "ms_per_launch": v_ms},
        "kernels": {
            "dn_verify_block": {"ms": v_ms, "gbs": achieved, "bytes": vb, "frac": achieved / hbm},
            "dn_accept_greedy": {"ms": a_ms, "gbs": ab / (a_ms / 1e3) / 1e9, "bytes": ab,
                                 "frac": ab / (a_ms / 1e3) / 1e9 / hbm},
            "dn_commit": {"ms": c_ms, "gbs": cb / (c_ms / 1e3) / 1e9, "bytes": cb,
                          "frac": cb / (c_ms / 1e3) / 1e9 / hbm},
        },
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_k,
                "how": "one CUDA graph replay per step: the inputs of layer groups of %s layers go "
                       "over in one copy each on a copy stream, each group's verify starts when its "
                       "copy has landed, then the logits and drafts, whose accept runs beside the "
                       "verify on a second stream, commit and the device-to-host read of the target "
                       "ids and accepted length; the host waits for each step's results"
                       % "/".join(str(x) for x in e2e_groups),
                "eager_value": B * T * w["L"] * e2e_k / e2e_eager_s,
                "serial_value": B * T * w["L"] * e2e_k / e2e_serial_s,
                "serial_how": "the same step with all inputs in one copy before the three calls"},
        "gpu_launches": 3 * args.steps,
        "clocks": clock_info,
        "cpu_baseline": cpu,
        "rows": rows,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

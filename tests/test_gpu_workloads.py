"""Full-size workloads on the GPU, in the launch configuration bench.py times.

The CUDA path runs the whole workload; the float64 oracle recomputes a seeded
sample of independent (state set, head) units from the same inputs, and the
integer results (target ids, accepted lengths) are compared in full.
"""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs
from deltanet_recurrent_state_gb300.workloads import WORKLOADS
from tests.parity import TOL, assert_close, np64

pytestmark = pytest.mark.gpu
KEYS = ("q", "k", "v", "beta", "g")


def _units(N, H, count, seed):
    gen = torch.Generator().manual_seed(seed)
    pick = torch.randperm(N * H, generator=gen)[:count].tolist()
    return [(p // H, p % H) for p in pick]


def _gather(x, units):
    """Inputs of the chosen (n, h) units as an oracle batch with N = len(units), H = 1."""
    out = {}
    for k in KEYS:
        out[k] = np.stack([np64(x[k][n, :, h]) for n, h in units])[:, :, None]
    if x.get("state") is not None:
        out["state"] = np.stack([np64(x["state"][n, h]) for n, h in units])[:, None]
    return out


def _verify_step_workload(name, cuda, sample):
    w = WORKLOADS[name]
    N, B = w["L"] * w["B"], w["B"]
    x = inputs.recurrence_inputs(N, w["T"], w["H"], w["dk"], w["dv"], io=w["io"], state=w["state"],
                                 seed=w["seed"], device=cuda)
    logits, target = inputs.logits_inputs(B, w["T"], w["V"], dtype=w["logit_dtype"],
                                          std=w["logit_std"], seed=w["seed"] + 1, device=cuda)
    a = inputs.accepted_lengths(B, w["T"], w["accept"], seed=w["seed"] + 2,
                                value=w.get("accept_value"))
    draft = inputs.draft_ids(target, a, w["V"], seed=w["seed"] + 3)
    out, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    tgt, acc = dn.dn_accept_greedy(logits, draft)
    state = x["state"].clone()
    dn.dn_commit(ckpt, acc, state)
    torch.cuda.synchronize()

    tgt_ref, acc_ref = oracle.accept_greedy(np64(logits), draft.cpu().numpy())
    np.testing.assert_array_equal(tgt.cpu().numpy(), tgt_ref)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    np.testing.assert_array_equal(acc_ref, a.numpy())

    units = _units(N, w["H"], sample, w["seed"] + 4)
    u = _gather(x, units)
    o_ref, c_ref = oracle.verify_block(u["q"], u["k"], u["v"], u["beta"], u["g"], u["state"],
                                       store=w["state"], io=w["io"])
    o_gpu = torch.stack([out[n, :, h] for n, h in units])[:, :, None]
    c_gpu = torch.stack([ckpt[n, :, h] for n, h in units])[:, :, None]
    assert_close("out", o_gpu, o_ref, TOL[w["io"]])
    assert_close("ckpt", c_gpu, c_ref, TOL[w["state"]])
    for i, (n, h) in enumerate(units):
        an = int(acc_ref[n % B])
        want = u["state"][i, 0] if an == 0 else c_ref[i, an - 1, 0]
        assert_close("committed state", state[n, h], want, TOL[w["state"]])


def test_tiny_workload_end_to_end(cuda):
    # 1 layer, 1 request, 4 heads, dk = dv = 64, T = 8, fp32 state, V = 512 fp32 logits,
    # a ~ U{0..T}: verify -> accept -> commit, every unit against the oracle (the sample is
    # all N * H = 4 units), ids and the accepted length bit-exact
    w = WORKLOADS["tiny_h4_d64_t8_f32"]
    _verify_step_workload("tiny_h4_d64_t8_f32", cuda, sample=w["L"] * w["B"] * w["H"])


def test_single_user_t16_full_size(cuda):
    _verify_step_workload("single_user_l48_h48_d128_t16_f16", cuda, sample=12)


def test_batch64_t4_full_size(cuda):
    _verify_step_workload("batch64_l48_h48_d128_t4_f16", cuda, sample=12)


def test_decode_loop_1000_steps(cuda):
    """1000 verify -> accept -> commit steps feeding the committed state forward.

    The inputs of step i are pool entry i % 4 (q, k, v, beta, g and logits), with
    per-step drafts planting a geometric accepted length. The oracle runs the whole
    chain on its own for a sample of units, from its own committed state.
    """
    w = WORKLOADS["decode_loop_l48_h48_d128_t8_f16"]
    N, B, T, H, d, V = w["L"] * w["B"], w["B"], w["T"], w["H"], w["dk"], w["V"]
    steps, R = w["steps"], 4
    pool = [inputs.recurrence_inputs(N, T, H, d, d, seed=w["seed"] + 10 * r, device=cuda,
                                     with_state=(r == 0)) for r in range(R)]
    s0 = pool[0]["state"].clone()
    lg = [inputs.logits_inputs(B, T, V, dtype="f16", std=2.0, seed=w["seed"] + 10 * r + 1,
                               device=cuda) for r in range(R)]
    a_plan = inputs.accepted_lengths(steps, T, "geometric", seed=w["seed"] + 5)
    drafts = [inputs.draft_ids(lg[i % R][1], a_plan[i:i + 1], V, seed=w["seed"] + 100 + i)
              for i in range(steps)]

    state = s0.clone()
    ws = dn.accept_workspace(B, T, V, cuda)
    acc_hist = torch.empty((steps,), dtype=torch.int32, device=cuda)
    out = ckpt = None
    for i in range(steps):
        x = pool[i % R]
        out, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], state, out, ckpt)
        _, acc = dn.dn_accept_greedy(lg[i % R][0], drafts[i], workspace=ws,
                                     accepted_len=acc_hist[i:i + 1])
        dn.dn_commit(ckpt, acc, state)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc_hist.cpu().numpy(), a_plan.numpy())
    print("decode loop: mean accepted length %.3f" % a_plan.double().mean().item())

    units = _units(N, H, 4, w["seed"] + 6)
    us = [_gather(pool[r], units) for r in range(R)]
    logits64 = [np64(lg[r][0]) for r in range(R)]
    S = np.stack([np64(s0[n, h]) for n, h in units])[:, None]
    for i in range(steps):
        u = us[i % R]
        _, c_ref = oracle.verify_block(u["q"], u["k"], u["v"], u["beta"], u["g"], S,
                                       store="f16", io="f16")
        _, a_ref = oracle.accept_greedy(logits64[i % R], drafts[i].cpu().numpy())
        assert int(a_ref[0]) == int(a_plan[i])
        S = oracle.commit(S, c_ref, a_ref)
    got = torch.stack([state[n, h] for n, h in units])[:, None]
    assert_close("state after 1000 steps", got, S, TOL["f16"])


def test_prefill_25000_tokens_one_layer(cuda):
    """One layer of the 25,000-token prompt: sampled heads against the oracle over all
    tokens, and the restore-at-24,960 run equal to the full run bit for bit."""
    w = WORKLOADS["prefill_p25000_l48_h48_d128_c64_f16"]
    P, H, d = w["P"], w["H"], w["dk"]
    x = inputs.recurrence_inputs(1, P, H, d, d, seed=w["seed"], device=cuda)
    args = [x[k] for k in KEYS]
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*args, x["state"])
    torch.cuda.synchronize()
    assert ckpt.shape[1] == 390
    start = 64 * 390  # 24,960
    tail = [a[:, start:].contiguous() for a in args]
    o2, ck2, s2 = dn.dn_prefill_checkpoint(*tail, ckpt[:, 389].contiguous())
    torch.cuda.synchronize()
    assert ck2.shape[1] == 0
    assert torch.equal(s2, s_out) and torch.equal(o2, out[:, start:])

    heads = [3, 40]
    u = {k: np64(x[k][:, :, heads]) for k in KEYS}
    o_ref, c_ref, s_ref = oracle.prefill_checkpoint(u["q"], u["k"], u["v"], u["beta"], u["g"],
                                                    np64(x["state"][:, heads]), chunk=64,
                                                    store="f16", io="f16")
    assert_close("out", out[:, :, heads], o_ref, TOL["f16"])
    assert_close("ckpt", ckpt[:, :, heads], c_ref, TOL["f16"])
    assert_close("state_out", s_out[:, heads], s_ref, TOL["f16"])


def test_prefill_25000_tokens_all_layers(cuda):
    """All 48 layers of the 25,000-token prompt in one launch (the launch bench.py times).
    The oracle checks four seeded heads of every layer over the last two chunks and the
    40-token tail, restarted from the GPU's own checkpoint at token 24,832, and every head
    of four layers over the first two chunks from the initial state. (The oracle's explicit
    dv x dk matrix form costs ~4 MFLOP per token and head, so the full 25,000 tokens of all
    2,304 units are out of reach; the one-layer test above covers two heads end to end.)"""
    w = WORKLOADS["prefill_p25000_l48_h48_d128_c64_f16"]
    L, P, H, d = w["L"], w["P"], w["H"], w["dk"]
    x = inputs.recurrence_inputs(L, P, H, d, d, seed=w["seed"], device=cuda)
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"])
    torch.cuda.synchronize()
    assert ckpt.shape == (L, 390, H, d, d) and dn.dn_prefill_wait_timeouts() == 0

    start = 64 * 388  # 24,832: two full chunks and the 40-token tail remain
    gen = torch.Generator().manual_seed(w["seed"] + 1)
    units = [(n, int(h)) for n in range(L) for h in torch.randperm(H, generator=gen)[:4]]
    u = {k: np.stack([np64(x[k][n, start:, h]) for n, h in units])[:, :, None] for k in KEYS}
    s0 = np.stack([np64(ckpt[n, 387, h]) for n, h in units])[:, None]
    o_ref, c_ref, s_ref = oracle.prefill_checkpoint(u["q"], u["k"], u["v"], u["beta"], u["g"], s0,
                                                    chunk=64, store="f16", io="f16")
    assert_close("tail out (every layer)", torch.stack([out[n, start:, h] for n, h in units])[:, :, None],
                 o_ref, TOL["f16"])
    assert_close("checkpoints 24,896 and 24,960", torch.stack([ckpt[n, 388:, h] for n, h in units])[:, :, None],
                 c_ref, TOL["f16"])
    assert_close("state_out", torch.stack([s_out[n, h] for n, h in units])[:, None], s_ref, TOL["f16"])

    layers, head_len = [0, 17, 31, 47], 128
    u = {k: np64(x[k][layers, :head_len]) for k in KEYS}
    o_ref, c_ref, _ = oracle.prefill_checkpoint(u["q"], u["k"], u["v"], u["beta"], u["g"],
                                                np64(x["state"][layers]), chunk=64, store="f16", io="f16")
    assert_close("first two chunks out (4 layers, all heads)", out[layers, :head_len], o_ref, TOL["f16"])
    assert_close("first two checkpoints", ckpt[layers, :head_len // 64], c_ref, TOL["f16"])

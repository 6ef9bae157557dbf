"""dn_commit on the GPU (bit-exact copy semantics) and the verify -> accept -> commit chain."""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs
from tests.parity import TOL, assert_close, np64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt", [torch.float16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
def test_commit_every_accepted_length(dt, d, cuda):
    L, B, H, T = 2, 7, 3, 6
    N = L * B
    gen = torch.Generator().manual_seed(d)
    ckpt = torch.randn((N, T, H, d, d), generator=gen).to(dt)
    state = torch.randn((N, H, d, d), generator=gen).to(dt)
    a = torch.tensor([0, 1, 2, 3, 5, 6, 4], dtype=torch.int32)
    ref = oracle.commit(np64(state), np64(ckpt), a.numpy())
    s = state.to(cuda)
    dn.dn_commit(ckpt.to(cuda), a.to(cuda), s)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(np64(s), ref)


def test_out_of_range_lengths_leave_state(cuda):
    N, B, H, T, d = 4, 4, 2, 3, 64
    ckpt = torch.randn((N, T, H, d, d), device=cuda).half()
    state = torch.randn((N, H, d, d), device=cuda).half()
    before = state.clone()
    dn.dn_commit(ckpt, torch.tensor([-1, 4, 100, 0], dtype=torch.int32, device=cuda), state)
    torch.cuda.synchronize()
    assert torch.equal(state, before)


@pytest.mark.parametrize("dt", ["f16", "f32"])
def test_verify_accept_commit_chain_matches_oracle(dt, cuda):
    L, B, H, T, d, V = 3, 4, 5, 8, 64, 3000
    N = L * B
    x = inputs.recurrence_inputs(N, T, H, d, d, io=dt, state=dt, seed=33, device="cpu")
    logits, target = inputs.logits_inputs(B, T, V, dtype=dt, std=2.0, seed=34)
    a = inputs.accepted_lengths(B, T, "uniform", seed=35)
    draft = inputs.draft_ids(target, a, V, seed=36)
    g = {k: v.to(cuda) for k, v in x.items()}
    out, ckpt = dn.dn_verify_block(g["q"], g["k"], g["v"], g["beta"], g["g"], g["state"])
    tgt, acc = dn.dn_accept_greedy(logits.to(cuda), draft.to(cuda))
    state = g["state"].clone()
    dn.dn_commit(ckpt, acc, state)
    torch.cuda.synchronize()

    o_ref, c_ref = oracle.verify_block(np64(x["q"]), np64(x["k"]), np64(x["v"]), np64(x["beta"]),
                                       np64(x["g"]), np64(x["state"]), store=dt, io=dt)
    tgt_ref, acc_ref = oracle.accept_greedy(np64(logits), draft.numpy())
    s_ref = oracle.commit(np64(x["state"]), c_ref, acc_ref)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    np.testing.assert_array_equal(acc_ref, a.numpy())
    assert_close("committed state", state, s_ref, TOL[dt])
    # the committed state equals running only the first a tokens
    for n in range(N):
        an = int(acc_ref[n % B])
        if an == 0:
            assert torch.equal(state[n], g["state"][n])
            continue
        sl = {k: g[k][n:n + 1, :an].contiguous() for k in ("q", "k", "v", "beta", "g")}
        _, cp = dn.dn_verify_block(sl["q"], sl["k"], sl["v"], sl["beta"], sl["g"],
                                   g["state"][n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(cp[0, an - 1], state[n])


def test_more_sets_than_a_grid_y_dimension(cuda):
    # 70,000 state sets: the set count lives on grid.x, not on the 65,535-wide grid.y
    N, B, H, T, d = 70000, 7, 1, 2, 64
    gen = torch.Generator(device=cuda).manual_seed(4)
    ckpt = torch.randn((N, T, H, d, d), generator=gen, device=cuda).half()
    state = torch.randn((N, H, d, d), generator=gen, device=cuda).half()
    a = torch.tensor([0, 1, 2, 1, 2, 0, 1], dtype=torch.int32)
    before = state.clone()
    dn.dn_commit(ckpt, a.to(cuda), state)
    torch.cuda.synchronize()
    pick = list(range(0, 9)) + list(range(65530, 65545)) + list(range(N - 9, N))
    # the oracle maps set i of its batch to request i % B': give it one request per picked set
    a_pick = np.array([int(a[n % B]) for n in pick], dtype=np.int32)
    ref = oracle.commit(np64(before[pick]), np64(ckpt[pick]), a_pick)
    np.testing.assert_array_equal(np64(state[pick]), ref)
    # every set: changed exactly where its request accepted a token
    changed = (state != before).flatten(1).any(1).cpu()
    want = torch.tensor([int(a[n % B]) > 0 for n in range(N)])
    assert torch.equal(changed, want)

"""Recompute-on-commit (dn_verify_block_deltas + dn_commit_deltas) on the GPU: the same
outputs, bit for bit, as the checkpoint path; committed states equal to its states up to
one fp16 unit in the last place (the closed-form commit sums in another order), and the
oracle."""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs
from tests.parity import TOL, assert_close, np64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("T", [1, 7, 8, 9, 16])
def test_deltas_path_equals_checkpoint_path(dk, dv, T, cuda):
    L, B, H = 2, T + 1, 3          # request b accepts b tokens: every length 0..T
    N = L * B
    x = inputs.recurrence_inputs(N, T, H, dk, dv, seed=700 + T + dk + dv, device=cuda)
    acc = torch.arange(B, dtype=torch.int32, device=cuda)
    out_c, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    s_c = x["state"].clone()
    dn.dn_commit(ckpt, acc, s_c)
    out_d, delta = dn.dn_verify_block_deltas(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    s_d = x["state"].clone()
    dn.dn_commit_deltas(x["k"], x["g"], delta, acc, s_d)
    torch.cuda.synchronize()
    assert torch.equal(out_d, out_c)
    _assert_within_one_ulp(s_d, s_c)


def _assert_within_one_ulp(got, want):
    # one fp16 unit in the last place is at most |x| 2^-10 (normal) or 2^-24 (subnormal)
    g32, w32 = got.float(), want.float()
    ulp = torch.maximum(g32.abs(), w32.abs()) * 2.0 ** -10 + 2.0 ** -24
    assert ((g32 - w32).abs() <= ulp).all()
    assert (got == want).float().mean().item() > 0.99


@pytest.mark.parametrize("a", [0, 1, 5, 16])
def test_beta0_g1_deltas_commit_keeps_the_state(a, cuda):
    # beta = 0, g = 1: every delta is zero and every decay one, so the committed state is the
    # initial state bit for bit whatever the accepted length
    N, T, H, d = 3, 16, 4, 128
    x = inputs.recurrence_inputs(N, T, H, d, d, seed=19, device=cuda)
    x["beta"].zero_()
    x["g"].fill_(1.0)
    _, delta = dn.dn_verify_block_deltas(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    s_d = x["state"].clone()
    acc = torch.full((1,), a, dtype=torch.int32, device=cuda)
    dn.dn_commit_deltas(x["k"], x["g"], delta, acc, s_d)
    torch.cuda.synchronize()
    assert torch.equal(delta, torch.zeros_like(delta))
    assert torch.equal(s_d, x["state"])


@pytest.mark.parametrize("a_all", [1, 8, 9, 16])
def test_deltas_commit_full_size_against_checkpoint_path(a_all, cuda):
    # the single-user launch shape (48 layers x 48 heads x 128 x 128), every set at one length
    L, H, T, d = 48, 48, 16, 128
    x = inputs.recurrence_inputs(L, T, H, d, d, seed=790 + a_all, device=cuda)
    acc = torch.full((1,), a_all, dtype=torch.int32, device=cuda)
    _, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    s_c = x["state"].clone()
    dn.dn_commit(ckpt, acc, s_c)
    del ckpt
    _, delta = dn.dn_verify_block_deltas(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    s_d = x["state"].clone()
    dn.dn_commit_deltas(x["k"], x["g"], delta, acc, s_d)
    torch.cuda.synchronize()
    _assert_within_one_ulp(s_d, s_c)


def test_deltas_commit_matches_oracle(cuda):
    N, T, H, d = 3, 16, 4, 128
    x = inputs.recurrence_inputs(N, T, H, d, d, seed=777, device="cpu")
    g = {k: v.to(cuda) for k, v in x.items()}
    acc = torch.tensor([5, 16, 0], dtype=torch.int32)
    _, delta = dn.dn_verify_block_deltas(g["q"], g["k"], g["v"], g["beta"], g["g"], g["state"])
    s = g["state"].clone()
    dn.dn_commit_deltas(g["k"], g["g"], delta, acc.to(cuda), s)
    torch.cuda.synchronize()
    _, c_ref = oracle.verify_block(np64(x["q"]), np64(x["k"]), np64(x["v"]), np64(x["beta"]),
                                   np64(x["g"]), np64(x["state"]), store="f16", io="f16")
    ref = oracle.commit(np64(x["state"]), c_ref, acc.numpy())
    assert_close("committed state", s, ref, TOL["f16"])


def test_deltas_reject_fp32(cuda):
    x = inputs.recurrence_inputs(1, 4, 2, 64, 64, io="f32", state="f32", seed=1, device=cuda)
    with pytest.raises(dn.DnError) as e:
        dn.dn_verify_block_deltas(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    assert e.value.status == dn.DN_ERR_UNSUPPORTED

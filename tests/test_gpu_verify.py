"""dn_verify_block on the GPU vs the float64 oracle, element by element.

Sizes span several CTAs (dv / 32 row blocks per head, many heads and state
sets), every block width 1..16, both head dims and both dtype pairs.
"""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs
from tests.parity import TOL, assert_close, np64

pytestmark = pytest.mark.gpu


def _run_case(N, T, H, dk, dv, dt, seed, cuda):
    x = inputs.recurrence_inputs(N, T, H, dk, dv, io=dt, state=dt, seed=seed, device="cpu")
    g = {k: v.to(cuda) for k, v in x.items()}
    out, ckpt = dn.dn_verify_block(g["q"], g["k"], g["v"], g["beta"], g["g"], g["state"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle.verify_block(np64(x["q"]), np64(x["k"]), np64(x["v"]), np64(x["beta"]),
                                       np64(x["g"]), np64(x["state"]), store=dt, io=dt)
    assert_close("out", out, o_ref, TOL[dt])
    assert_close("ckpt", ckpt, c_ref, TOL[dt])
    return out, ckpt


def test_tiny_fp32_workload(cuda):
    # 1 layer, 1 request, 4 heads, dk = dv = 64, T = 8, fp32 state
    _run_case(1, 8, 4, 64, 64, "f32", 1000, cuda)


@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 15, 16])
def test_fp16_d128_every_width(T, cuda):
    _run_case(3, T, 5, 128, 128, "f16", 10 + T, cuda)


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("dt", ["f16", "f32"])
def test_mixed_head_dims(dk, dv, dt, cuda):
    _run_case(2, 7, 3, dk, dv, dt, 20 + dk + dv, cuda)


def test_deterministic_bitwise(cuda):
    x = inputs.recurrence_inputs(4, 16, 6, 128, 128, seed=5, device=cuda)
    a = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    b = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_block_equals_chained_single_token_calls(cuda):
    # fp32: one T-wide call and T one-token calls agree within fp32 rounding
    x = inputs.recurrence_inputs(2, 6, 3, 64, 64, io="f32", state="f32", seed=6, device=cuda)
    out, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    s = x["state"]
    for t in range(6):
        sl = lambda k: x[k][:, t:t + 1].contiguous()
        o1, c1 = dn.dn_verify_block(sl("q"), sl("k"), sl("v"), sl("beta"), sl("g"), s)
        torch.testing.assert_close(o1[:, 0], out[:, t], rtol=0, atol=1e-5)
        torch.testing.assert_close(c1[:, 0], ckpt[:, t], rtol=0, atol=1e-5)
        s = c1[:, 0].contiguous()


def test_beta0_g1_leaves_state_unchanged_on_gpu(cuda):
    x = inputs.recurrence_inputs(2, 4, 3, 128, 128, seed=7, device=cuda)
    x["beta"].zero_()
    x["g"].fill_(1.0)
    _, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    torch.cuda.synchronize()
    for t in range(4):
        assert torch.equal(ckpt[:, t], x["state"])


@pytest.mark.parametrize("dt", ["f16", "f32"])
def test_unit_key_write_identity_on_gpu(dt, cuda):
    # beta = 1, g = 1: S_t k_t = (1 - |k_t|^2) S_{t-1} k_t + |k_t|^2 v_t, so S_t k_t = v_t for a
    # unit key (the delta rule writes v_t under k_t). Checked from the stored checkpoints in
    # float64, independent of the oracle; the residual is the checkpoints' own rounding.
    N, T, H, d = 2, 8, 3, 128
    x = inputs.recurrence_inputs(N, T, H, d, d, io=dt, state=dt, seed=17, device=cuda)
    x["beta"].fill_(1.0)
    x["g"].fill_(1.0)
    _, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    torch.cuda.synchronize()
    k, v = np64(x["k"]), np64(x["v"])
    prev = np64(x["state"])
    for t in range(T):
        st = np64(ckpt[:, t])
        kt, vt = k[:, t], v[:, t]                      # [N, H, d]
        kk = (kt * kt).sum(-1, keepdims=True)
        want = (1.0 - kk) * np.einsum("nhij,nhj->nhi", prev, kt) + kk * vt
        got = np.einsum("nhij,nhj->nhi", st, kt)
        assert_close("S_t k_t", got, want, TOL[dt])
        prev = st


def test_outputs_do_not_spill_past_their_buffers(cuda):
    # canaries after out and ckpt stay untouched
    N, T, H, d = 2, 5, 3, 64
    x = inputs.recurrence_inputs(N, T, H, d, d, seed=8, device=cuda)
    out_buf = torch.full((N * T * H * d + 64,), 7.0, dtype=torch.float16, device=cuda)
    ck_buf = torch.full((N * T * H * d * d + 64,), 7.0, dtype=torch.float16, device=cuda)
    out = out_buf[:N * T * H * d].view(N, T, H, d)
    ckpt = ck_buf[:N * T * H * d * d].view(N, T, H, d, d)
    dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"], out, ckpt)
    torch.cuda.synchronize()
    assert (out_buf[-64:] == 7.0).all() and (ck_buf[-64:] == 7.0).all()


@pytest.mark.parametrize("T", [4, 16])
def test_one_layer_launch_matches_folded_launch_and_oracle(T, cuda):
    # One layer of one request (48 heads) is a small grid, which the library runs with
    # 16-row CTAs; 48 layers folded into one launch run with 32-row CTAs. Both follow the
    # same arithmetic per state row, so each layer's results are bit-identical, and a
    # sample of heads matches the oracle.
    L, H, d = 6, 48, 128
    x = inputs.recurrence_inputs(L, T, H, d, d, seed=40 + T, device=cuda)
    out, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    for l in range(L):
        sl = {k: x[k][l:l + 1] for k in ("q", "k", "v", "beta", "g", "state")}
        o1, c1 = dn.dn_verify_block(sl["q"], sl["k"], sl["v"], sl["beta"], sl["g"], sl["state"])
        torch.cuda.synchronize()
        assert torch.equal(o1[0], out[l]) and torch.equal(c1[0], ckpt[l]), l
    heads = [0, 17, 47]
    u = {k: np64(x[k][0:1, :, heads]) for k in ("q", "k", "v", "beta", "g")}
    o_ref, c_ref = oracle.verify_block(u["q"], u["k"], u["v"], u["beta"], u["g"],
                                       np64(x["state"][0:1, heads]), store="f16", io="f16")
    assert_close("out", out[0:1, :, heads], o_ref, TOL["f16"])
    assert_close("ckpt", ckpt[0:1, :, heads], c_ref, TOL["f16"])


@pytest.mark.parametrize("T", [1, 4, 8])
def test_short_blocks_in_large_launches_match_one_layer_launches(T, cuda):
    # Blocks of up to 8 tokens over many state sets run with the 8-token tile capacity, as
    # 64-row CTAs up to 4 tokens and 32-row CTAs above; one set at a time runs as 16-row CTAs.
    # The arithmetic per state row is the same, so the results are bit-identical, and a
    # sample matches the oracle.
    N, H, d = 8, 16, 128
    x = inputs.recurrence_inputs(N, T, H, d, d, seed=60 + T, device=cuda)
    out, ckpt = dn.dn_verify_block(x["q"], x["k"], x["v"], x["beta"], x["g"], x["state"])
    for n in (0, 5, 7):
        sl = {k: x[k][n:n + 1] for k in ("q", "k", "v", "beta", "g", "state")}
        o1, c1 = dn.dn_verify_block(sl["q"], sl["k"], sl["v"], sl["beta"], sl["g"], sl["state"])
        torch.cuda.synchronize()
        assert torch.equal(o1[0], out[n]) and torch.equal(c1[0], ckpt[n]), n
    heads = [1, 9, 15]
    u = {k: np64(x[k][2:4, :, heads]) for k in ("q", "k", "v", "beta", "g")}
    o_ref, c_ref = oracle.verify_block(u["q"], u["k"], u["v"], u["beta"], u["g"],
                                       np64(x["state"][2:4][:, heads]), store="f16", io="f16")
    assert_close("out", out[2:4][:, :, heads], o_ref, TOL["f16"])
    assert_close("ckpt", ckpt[2:4][:, :, heads], c_ref, TOL["f16"])

"""dn_prefill_checkpoint on the GPU vs the oracle, with the chunk-boundary edge cases."""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs
from tests.parity import TOL, assert_close, np64

pytestmark = pytest.mark.gpu

KEYS = ("q", "k", "v", "beta", "g")


def _case(N, P, H, d, dt, seed, with_state, cuda):
    x = inputs.recurrence_inputs(N, P, H, d, d, io=dt, state=dt, seed=seed, device="cpu")
    s_in = x["state"].to(cuda) if with_state else None
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*[x[k].to(cuda) for k in KEYS], s_in,
                                                state_dtype=x["state"].dtype)
    torch.cuda.synchronize()
    ref = oracle.prefill_checkpoint(*[np64(x[k]) for k in KEYS],
                                    np64(x["state"]) if with_state else None,
                                    chunk=64, store=dt, io=dt)
    assert_close("out", out, ref[0], TOL[dt])
    assert ckpt.shape[1] == P // 64
    assert_close("ckpt", ckpt, ref[1], TOL[dt])
    assert_close("state_out", s_out, ref[2], TOL[dt])
    return x, out, ckpt, s_out


@pytest.mark.parametrize("P", [0, 1, 17, 63, 64, 65, 130, 200])
def test_fp32_d64_edges(P, cuda):
    _case(2, P, 3, 64, "f32", 100 + P, True, cuda)


@pytest.mark.parametrize("P", [1, 64, 129])
@pytest.mark.parametrize("with_state", [True, False])
def test_fp16_d128(P, with_state, cuda):
    _case(1, P, 4, 128, "f16", 200 + P, with_state, cuda)


@pytest.mark.parametrize("P", [0, 1, 15, 16, 17, 63, 65, 200])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_fp16_chunkwise_edges(P, dk, dv, cuda):
    # the fp16 path (chunkwise tensor-core form): every sub-chunk / chunk boundary case
    x = inputs.recurrence_inputs(2, P, 3, dk, dv, io="f16", state="f16", seed=400 + P + dk + 2 * dv,
                                 device="cpu")
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*[x[k].to(cuda) for k in KEYS], x["state"].to(cuda))
    torch.cuda.synchronize()
    ref = oracle.prefill_checkpoint(*[np64(x[k]) for k in KEYS], np64(x["state"]), chunk=64,
                                    store="f16", io="f16")
    assert_close("out", out, ref[0], TOL["f16"])
    assert_close("ckpt", ckpt, ref[1], TOL["f16"])
    assert_close("state_out", s_out, ref[2], TOL["f16"])


@pytest.mark.parametrize("engine", ["mma", "tc"])
def test_beta0_g1_prefill_keeps_the_state(engine, cuda):
    # beta = 0, g = 1: nothing is written, so every checkpoint and the final state are the initial
    # state bit for bit, and each output is S0 q_t
    N, P, H, d = 2, 200, 3, 128
    x = inputs.recurrence_inputs(N, P, H, d, d, seed=18, device=cuda)
    x["beta"].zero_()
    x["g"].fill_(1.0)
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"], engine=engine)
    torch.cuda.synchronize()
    assert torch.equal(s_out, x["state"])
    for c in range(P // 64):
        assert torch.equal(ckpt[:, c], x["state"])
    want = np.einsum("nhij,nphj->nphi", np64(x["state"]), np64(x["q"]))
    assert_close("out = S0 q", out, want, TOL["f16"])


def test_restore_from_checkpoint_is_bit_identical(cuda):
    N, P, H, d = 1, 300, 4, 128
    x = inputs.recurrence_inputs(N, P, H, d, d, seed=301, device=cuda)
    args = [x[k] for k in KEYS]
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*args, x["state"])
    for c in range(P // 64):
        start = 64 * (c + 1)
        tail = [a[:, start:].contiguous() for a in args]
        o2, ck2, s2 = dn.dn_prefill_checkpoint(*tail, ckpt[:, c].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(s2, s_out), c
        assert torch.equal(o2, out[:, start:]), c
        assert torch.equal(ck2, ckpt[:, c + 1:]), c


def test_state_out_may_alias_state_in(cuda):
    x = inputs.recurrence_inputs(2, 100, 3, 64, 64, seed=302, device=cuda)
    args = [x[k] for k in KEYS]
    _, _, s_ref = dn.dn_prefill_checkpoint(*args, x["state"])
    s = x["state"].clone()
    dn.dn_prefill_checkpoint(*args, s, state_out=s)
    torch.cuda.synchronize()
    assert torch.equal(s, s_ref)


def test_prefill_equals_verify_blocks_chained(cuda):
    # fp32: 64 prompt tokens through prefill == four 16-token verify blocks chained
    x = inputs.recurrence_inputs(1, 64, 2, 64, 64, io="f32", state="f32", seed=303, device=cuda)
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"])
    s = x["state"]
    for b in range(4):
        sl = {k: x[k][:, 16 * b:16 * (b + 1)].contiguous() for k in KEYS}
        o, c = dn.dn_verify_block(sl["q"], sl["k"], sl["v"], sl["beta"], sl["g"], s)
        torch.testing.assert_close(o, out[:, 16 * b:16 * (b + 1)], rtol=0, atol=1e-5)
        s = c[:, -1].contiguous()
    torch.testing.assert_close(s, s_out, rtol=0, atol=1e-5)
    torch.testing.assert_close(s, ckpt[:, 0], rtol=0, atol=1e-5)


def test_no_input_wait_ran_out(cuda):
    # the bounded input waits of the fp16 prefill never gave up in this process
    x = inputs.recurrence_inputs(2, 300, 4, 128, 128, seed=500, device=cuda)
    dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"])
    torch.cuda.synchronize()
    assert dn.dn_prefill_wait_timeouts() == 0


def test_whole_and_half_row_ctas_agree(cuda):
    # N*H >= the SM count runs one CTA per (sequence, head); a single sequence runs two
    # CTAs per head (half the rows each). Same arithmetic per row: bit-identical results.
    N, P, H, d = 4, 130, 48, 128
    assert N * H >= torch.cuda.get_device_properties(0).multi_processor_count
    x = inputs.recurrence_inputs(N, P, H, d, d, seed=600, device=cuda)
    o_all, c_all, s_all = dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"])
    for n in range(N):
        xs = [x[k][n:n + 1].contiguous() for k in KEYS]
        o1, c1, s1 = dn.dn_prefill_checkpoint(*xs, x["state"][n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(o1, o_all[n:n + 1]) and torch.equal(c1, c_all[n:n + 1])
        assert torch.equal(s1, s_all[n:n + 1])
    heads = [0, 47]
    u = {k: np64(x[k][:1, :, heads]) for k in KEYS}
    ref = oracle.prefill_checkpoint(u["q"], u["k"], u["v"], u["beta"], u["g"],
                                    np64(x["state"][:1, heads]), chunk=64, store="f16", io="f16")
    assert_close("out", o_all[:1, :, heads], ref[0], TOL["f16"])
    assert_close("ckpt", c_all[:1, :, heads], ref[1], TOL["f16"])
    assert_close("state_out", s_all[:1, heads], ref[2], TOL["f16"])


@pytest.mark.parametrize("extra", [10, 100])
def test_folded_launch_tail_agrees_with_single_sequences(extra, cuda):
    # N*H = SMs + extra pairs: a folded launch (one full-height CTA a pair) whose last wave is
    # partial. Each sequence must equal its own single-sequence launch (half-height CTAs) bit
    # for bit, and its last pair the oracle.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, P, H, d = (sms + extra) // 2, 130, 2, 128
    x = inputs.recurrence_inputs(N, P, H, d, d, seed=640 + extra, device=cuda)
    o_all, c_all, s_all = dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"])
    torch.cuda.synchronize()
    assert dn.dn_prefill_wait_timeouts() == 0
    for n in range(N):
        xs = [x[k][n:n + 1].contiguous() for k in KEYS]
        o1, c1, s1 = dn.dn_prefill_checkpoint(*xs, x["state"][n:n + 1].contiguous())
        assert torch.equal(o1, o_all[n:n + 1]) and torch.equal(c1, c_all[n:n + 1]), n
        assert torch.equal(s1, s_all[n:n + 1]), n
    last = N - 1
    u = {k: np64(x[k][last:]) for k in KEYS}
    ref = oracle.prefill_checkpoint(u["q"], u["k"], u["v"], u["beta"], u["g"], np64(x["state"][last:]),
                                    chunk=64, store="f16", io="f16")
    assert_close("out", o_all[last:], ref[0], TOL["f16"])
    assert_close("ckpt", c_all[last:], ref[1], TOL["f16"])
    assert_close("state_out", s_all[last:], ref[2], TOL["f16"])


def test_binding_rejects_wrong_shapes_and_dtypes(cuda):
    # The C ABI takes raw pointers and cannot see sizes: the binding stops a mis-sized or
    # mis-typed tensor with ValueError (not an assert that python -O would strip).
    x = inputs.recurrence_inputs(1, 70, 2, 64, 64, seed=5, device=cuda)
    base = [x[k] for k in KEYS]
    with pytest.raises(ValueError):
        dn.dn_prefill_checkpoint(*base[:3], x["beta"][:, :-1].contiguous(), x["g"], x["state"])
    with pytest.raises(ValueError):
        dn.dn_prefill_checkpoint(*base[:3], x["beta"].half(), x["g"], x["state"])
    with pytest.raises(ValueError):
        dn.dn_prefill_checkpoint(*base, x["state"], out=torch.empty(1, 69, 2, 64, dtype=x["q"].dtype, device=cuda))


# ---------------------------------------------------------------------------- tcgen05 engine

@pytest.mark.parametrize("P", [0, 1, 15, 63, 64, 65, 129, 200])
def test_tc_engine_against_oracle(P, cuda):
    x = inputs.recurrence_inputs(2, P, 3, 128, 128, io="f16", state="f16", seed=700 + P, device="cpu")
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*[x[k].to(cuda) for k in KEYS], x["state"].to(cuda), engine="tc")
    torch.cuda.synchronize()
    ref = oracle.prefill_checkpoint(*[np64(x[k]) for k in KEYS], np64(x["state"]), chunk=64, store="f16", io="f16")
    assert_close("out", out, ref[0], TOL["f16"])
    assert_close("ckpt", ckpt, ref[1], TOL["f16"])
    assert_close("state_out", s_out, ref[2], TOL["f16"])


def test_tc_engine_no_initial_state_and_restore(cuda):
    N, P, H, d = 1, 300, 4, 128
    x = inputs.recurrence_inputs(N, P, H, d, d, seed=701, device=cuda)
    args = [x[k] for k in KEYS]
    o0, c0, s0 = dn.dn_prefill_checkpoint(*args, None, state_dtype=torch.float16, engine="tc")
    ref = oracle.prefill_checkpoint(*[np64(a) for a in args], None, chunk=64, store="f16", io="f16")
    assert_close("state_out", s0, ref[2], TOL["f16"])
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*args, x["state"], engine="tc")
    for c in range(P // 64):
        start = 64 * (c + 1)
        tail = [a[:, start:].contiguous() for a in args]
        o2, ck2, s2 = dn.dn_prefill_checkpoint(*tail, ckpt[:, c].contiguous(), engine="tc")
        torch.cuda.synchronize()
        assert torch.equal(s2, s_out) and torch.equal(o2, out[:, start:]) and torch.equal(ck2, ckpt[:, c + 1:])


def test_tc_engine_rejects_other_shapes(cuda):
    x = inputs.recurrence_inputs(1, 64, 2, 64, 128, seed=702, device=cuda)
    with pytest.raises(dn.DnError):
        dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"], engine="tc")


def test_tc_engine_full_size_layer_sampled(cuda):
    # one 25,000-token layer (48 heads); sampled heads against the oracle
    x = inputs.recurrence_inputs(1, 25000, 48, 128, 128, seed=703, device=cuda)
    out, ckpt, s_out = dn.dn_prefill_checkpoint(*[x[k] for k in KEYS], x["state"], engine="tc")
    torch.cuda.synchronize()
    assert dn.dn_prefill_wait_timeouts() == 0
    heads = [0, 29, 47]
    u = {k: np64(x[k][:, :, heads]) for k in KEYS}
    ref = oracle.prefill_checkpoint(u["q"], u["k"], u["v"], u["beta"], u["g"], np64(x["state"][:, heads]),
                                    chunk=64, store="f16", io="f16")
    assert_close("out", out[:, :, heads], ref[0], TOL["f16"])
    assert_close("ckpt", ckpt[:, :, heads], ref[1], TOL["f16"])
    assert_close("state_out", s_out[:, heads], ref[2], TOL["f16"])


@pytest.mark.parametrize("budget_us", [10, 2000])
def test_bounded_wait_gives_up_drains_and_reports(budget_us, cuda):
    # the prefill kernels' waits are bounded in time: on a barrier nothing arrives on, the wait
    # runs out after the budget and raises the abort flag; after the arrival the same wait
    # returns; a copy in flight when the CTA aborts is drained and lands; each failure is
    # counted once. No kernel is made to fault or hang.
    assert dn.dn_wait_selftest(budget_us, device=cuda) == (1, 1, 1, 2)


def test_wait_selftest_rejects_bad_arguments(cuda):
    lib = dn.load_library()
    buf = torch.zeros(8, dtype=torch.int32, device=cuda)
    assert lib.dn_wait_selftest(0, buf.data_ptr(), None) == 1          # DN_ERR_INVALID_ARG
    assert lib.dn_wait_selftest(1000001, buf.data_ptr(), None) == 1
    assert lib.dn_wait_selftest(10, None, None) == 1
    assert lib.dn_wait_selftest(10, buf.data_ptr() + 4, None) == 1     # not 16-byte aligned

"""The seeded input generator: determinism, distributions, planted answers (no GPU)."""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import inputs
from deltanet_recurrent_state_gb300.workloads import WORKLOADS


def test_recurrence_inputs_deterministic_and_normalised():
    a = inputs.recurrence_inputs(3, 5, 2, 64, 32, io="f32", state="f32", seed=7)
    b = inputs.recurrence_inputs(3, 5, 2, 64, 32, io="f32", state="f32", seed=7)
    for key in a:
        assert torch.equal(a[key], b[key])
    np.testing.assert_allclose(a["q"].norm(dim=-1).numpy(), 1.0, atol=1e-6)
    np.testing.assert_allclose(a["k"].norm(dim=-1).numpy(), 1.0, atol=1e-6)
    assert (a["beta"] > 0).all() and (a["beta"] < 1).all()
    assert (a["g"] > 0).all() and (a["g"] < 1).all()
    assert a["state"].shape == (3, 2, 32, 64)


def test_recurrence_inputs_fp16_chunked_generation_matches_shapes():
    d = inputs.recurrence_inputs(300, 2, 1, 64, 64, io="f16", state="f16", seed=1)
    assert d["q"].dtype == torch.float16 and d["state"].dtype == torch.float16
    assert d["q"].shape == (300, 2, 1, 64)
    s = d["state"].float()
    assert 0.09 < s.std().item() < 0.11


@pytest.mark.parametrize("kind,T", [("uniform", 8), ("geometric", 8), ("fixed", 16)])
def test_planted_argmax_and_accepted_length_hold(kind, T):
    B, V = 5, 1000
    logits, target = inputs.logits_inputs(B, T, V, dtype="f16", std=2.0, seed=3)
    a = inputs.accepted_lengths(B, T, kind, seed=4, value=15 if kind == "fixed" else None)
    d = inputs.draft_ids(target, a, V, seed=5)
    tgt, acc = oracle.accept_greedy(logits.float().numpy(), d.numpy())
    np.testing.assert_array_equal(tgt, target.numpy())
    np.testing.assert_array_equal(acc, a.numpy())


def test_geometric_lengths_mean():
    a = inputs.accepted_lengths(20000, 8, "geometric", seed=9).double()
    # geometric(p=0.2) on {0,1,...} clamped at 8: mean = sum_{j=1..8} 0.8^j
    want = sum(0.8 ** j for j in range(1, 9))
    assert abs(a.mean().item() - want) < 0.05
    assert a.max().item() <= 8 and a.min().item() >= 0


def test_workload_table_shapes():
    for name, w in WORKLOADS.items():
        assert w["dk"] in (64, 128) and w["dv"] in (64, 128), name
        if "T" in w:
            assert 1 <= w["T"] <= 16


def test_context_inputs_quote_copies_a_prompt_passage():
    ctx, lens = inputs.context_inputs(3, 500, 40, 151936, seed=5)
    assert ctx.shape == (3, 540) and ctx.dtype == torch.int32 and (lens == 540).all()
    assert int(ctx.min()) >= 0 and int(ctx.max()) < 151936
    c = ctx.numpy()
    for r in range(3):
        gen = c[r, 500:].tolist()
        assert any(c[r, s:s + 40].tolist() == gen for s in range(461))
    again, _ = inputs.context_inputs(3, 500, 40, 151936, seed=5)
    assert torch.equal(ctx, again)
    # the quoted passage continues in the prompt: the oracle's drafts are that continuation
    d, n, e = oracle.context_drafts_row(c[0], 4, 1, 8)
    assert n == 4 and c[0, e - 4:e].tolist() == c[0, -4:].tolist()


def test_context_inputs_ragged_lengths_in_range():
    _, lens = inputs.context_inputs(200, 30, 10, 1000, quote=False, ragged=True, seed=6)
    assert int(lens.min()) >= 0 and int(lens.max()) <= 40 and len(set(lens.tolist())) > 10

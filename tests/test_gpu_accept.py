"""dn_accept_greedy on the GPU vs the oracle: target ids and accepted lengths bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs

pytestmark = pytest.mark.gpu


def _check(logits, draft, cuda, ws=None):
    tgt, acc = dn.dn_accept_greedy(logits.to(cuda), draft.to(cuda), workspace=ws)
    torch.cuda.synchronize()
    tgt_ref, acc_ref = oracle.accept_greedy(logits.double().numpy(), draft.numpy())
    np.testing.assert_array_equal(tgt.cpu().numpy(), tgt_ref)
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)
    return tgt_ref, acc_ref


def _drafts_from(tgt_ref, V, gen):
    B, T = tgt_ref.shape
    d = torch.randint(0, V, (B, T), generator=gen, dtype=torch.int32)
    for b in range(B):
        a = int(torch.randint(0, T + 1, (1,), generator=gen))
        d[b, :a] = torch.from_numpy(tgt_ref[b, :a])
    return d


@pytest.mark.parametrize("V", [1, 2, 7, 13, 512, 8191, 8192, 8193, 40000, 151936])
@pytest.mark.parametrize("dt", [torch.float16, torch.float32])
def test_random_rows_with_forced_ties(V, dt, cuda):
    gen = torch.Generator().manual_seed(V)
    B, T = 3, 5
    logits = (torch.randn((B, T, V), generator=gen) * 2).to(dt)
    # plant copies of each row's maximum at random places (ties, both sides of the max)
    if V > 2:
        m = logits.float().max(-1).values
        for b in range(B):
            for t in range(T):
                for i in torch.randint(0, V, (3,), generator=gen):
                    logits[b, t, int(i)] = m[b, t].to(dt)
    tgt_ref, _ = oracle.accept_greedy(logits.double().numpy(), np.zeros((B, T), np.int32))
    _check(logits, _drafts_from(tgt_ref, V, gen), cuda)


@pytest.mark.parametrize("dt", [torch.float16, torch.float32])
def test_signed_zero_and_all_equal_rows(dt, cuda):
    V = 1000
    logits = torch.full((1, 4, V), -1.0, dtype=dt)
    logits[0, 0, :] = 0.0
    logits[0, 0, 0] = -0.0          # -0 ties +0: index 0
    logits[0, 1, 5] = -0.0
    logits[0, 1, 3] = 0.0           # lowest of the tied zeros: 3
    logits[0, 2, :] = 0.25          # all equal: 0
    logits[0, 3, 999] = 3.0         # last entry
    draft = torch.tensor([[0, 3, 0, 999]], dtype=torch.int32)
    tgt, acc = _check(logits, draft, cuda)
    assert list(tgt[0]) == [0, 3, 0, 999] and acc[0] == 4


def test_negative_values_and_extremes_fp16(cuda):
    V = 20000
    gen = torch.Generator().manual_seed(3)
    logits = -(torch.rand((2, 3, V), generator=gen) * 60000 + 1).to(torch.float16)
    logits[1, 2, 12345] = 65504.0
    logits[0, 0, 7] = -0.0
    _check(logits, torch.zeros((2, 3), dtype=torch.int32), cuda)


# B x T up to 16 rows take the one-level reduction (the grid's last CTA finishes every row and
# request), more rows the two-level one; (2, 8) and (17, 1) sit on either side of that line.
@pytest.mark.parametrize("B,T", [(1, 1), (1, 16), (2, 8), (17, 1), (64, 4), (7, 3)])
def test_planted_prefix_lengths(B, T, cuda):
    V = 151936
    logits, target = inputs.logits_inputs(B, T, V, dtype="f16", std=2.0, seed=B * 100 + T)
    a = inputs.accepted_lengths(B, T, "uniform", seed=B + T)
    draft = inputs.draft_ids(target, a, V, seed=9)
    _, acc_ref = _check(logits, draft, cuda)
    np.testing.assert_array_equal(acc_ref, a.numpy())


@pytest.mark.parametrize("B,T", [(5, 4), (4, 4), (1, 17)])
def test_workspace_reused_across_calls(B, T, cuda):
    # the counters reset themselves: the same workspace serves many calls in a row (both the
    # one-level reduction, 16 rows, and the two-level one)
    V = 30000
    ws = dn.accept_workspace(B, T, V, cuda)
    for s in range(6):
        logits, target = inputs.logits_inputs(B, T, V, dtype="f32", std=1.0, seed=50 + s)
        a = inputs.accepted_lengths(B, T, "uniform", seed=60 + s)
        _check(logits, inputs.draft_ids(target, a, V, seed=70 + s), cuda, ws=ws)
    assert int(ws.count_nonzero()) > 0  # keys stay, counters are zero again
    n_keys = B * T * ((V + 8191) // 8192) * 8
    assert int(ws[n_keys:].count_nonzero()) == 0


@pytest.mark.parametrize("dt", [torch.float16, torch.float32])
def test_masked_rows_with_minus_infinity(dt, cuda):
    # vocabulary entries masked to -inf: a row that is -inf throughout gives index 0 in both
    # dtypes, a row with one finite entry gives that entry, and +inf wins like any maximum
    V = 9000  # two chunks, the last one partly filled
    logits = torch.full((2, 4, V), float("-inf"), dtype=dt)
    logits[0, 1, 8500] = -3.0
    logits[0, 2, 17] = float("inf")
    logits[0, 2, 4000] = float("inf")
    logits[0, 3, 8999] = -65504.0
    logits[1] = (torch.randn((4, V), generator=torch.Generator().manual_seed(2)) * 2).to(dt)
    logits[1, :, ::2] = float("-inf")
    draft = torch.tensor([[0, 8500, 17, 8999], [0, 0, 0, 0]], dtype=torch.int32)
    tgt, acc = _check(logits, draft, cuda)
    assert list(tgt[0]) == [0, 8500, 17, 8999] and acc[0] == 4


def test_more_rows_than_a_grid_y_dimension(cuda):
    # 70,000 rows: the row count lives on grid.x, not on the 65,535-wide grid.y
    B, T, V = 35000, 2, 40
    gen = torch.Generator().manual_seed(11)
    logits = torch.randint(-4, 5, (B, T, V), generator=gen).float()  # many ties
    tgt_ref, _ = oracle.accept_greedy(logits.double().numpy(), np.zeros((B, T), np.int32))
    _check(logits, _drafts_from(tgt_ref, V, gen), cuda)

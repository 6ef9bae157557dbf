"""dn_context_drafts on the GPU vs the oracle: bit-exact drafts, counts and match lengths."""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs

pytestmark = pytest.mark.gpu


def _check(ctx, lens, n_max, n_min, K, cuda):
    d, c, m = dn.dn_context_drafts(ctx.to(cuda), lens.to(cuda), n_max, n_min, K)
    torch.cuda.synchronize()
    rd, rc, rm = oracle.context_drafts(ctx.numpy(), lens.numpy(), n_max, n_min, K)
    np.testing.assert_array_equal(c.cpu().numpy(), rc)
    np.testing.assert_array_equal(m.cpu().numpy(), rm)
    np.testing.assert_array_equal(d.cpu().numpy(), rd)
    return rc


# strides span one CTA per request (<= 4096), 3-CTA clusters and the 8-CTA cap
@pytest.mark.parametrize("stride", [1, 2, 37, 4096, 4097, 10000, 40000])
@pytest.mark.parametrize("vocab", [2, 5, 1000])
def test_random_ragged_contexts(stride, vocab, cuda):
    g = torch.Generator().manual_seed(stride * 7 + vocab)
    N = 24
    ctx = torch.randint(0, vocab, (N, stride), generator=g, dtype=torch.int32)
    lens = torch.randint(0, stride + 1, (N,), generator=g, dtype=torch.int32)
    lens[0], lens[-1] = stride, min(stride, 1)
    for n_max, n_min, K in [(4, 1, 8), (16, 1, 16), (3, 3, 1), (1, 1, 5)]:
        _check(ctx, lens, n_max, n_min, K, cuda)


def test_edge_cases(cuda):
    rows = [
        [],                      # empty
        [5],                     # one token: nothing can follow an earlier occurrence
        [5, 5],                  # match at e = 1, one draft
        [7, 7, 7, 7, 7, 7],      # overlapping occurrences: latest is e = L-1
        [1, 2, 3, 4, 5, 6, 7],   # no repeat
        [9, 1, 2, 9, 1, 2],      # whole-pattern match, drafts run to the end
        [0, -3, 0, -3, 2, 0, -3],  # negative ids compare like any other value
    ]
    stride = 8
    ctx = torch.full((len(rows), stride), 123, dtype=torch.int32)
    lens = torch.zeros(len(rows), dtype=torch.int32)
    for r, t in enumerate(rows):
        ctx[r, :len(t)] = torch.tensor(t, dtype=torch.int32)
        lens[r] = len(t)
    for n_max, n_min, K in [(4, 1, 8), (2, 2, 3), (16, 1, 16)]:
        _check(ctx, lens, n_max, n_min, K, cuda)


def test_lengths_out_of_range_are_clamped(cuda):
    ctx = torch.tensor([[1, 2, 1, 2, 3, 1, 2]], dtype=torch.int32)
    d1, c1, m1 = dn.dn_context_drafts(ctx.to(cuda), torch.tensor([99], dtype=torch.int32, device=cuda))
    d2, c2, m2 = dn.dn_context_drafts(ctx.to(cuda), torch.tensor([7], dtype=torch.int32, device=cuda))
    d3, c3, _ = dn.dn_context_drafts(ctx.to(cuda), torch.tensor([-5], dtype=torch.int32, device=cuda))
    torch.cuda.synchronize()
    assert torch.equal(d1, d2) and torch.equal(c1, c2) and torch.equal(m1, m2)
    assert int(c3[0]) == 0 and (d3 == -1).all()
    assert d2[0, :3].tolist() == [3, 1, 2] and int(c2[0]) == 3  # latest "1 2" ending before the end


@pytest.mark.parametrize("N,prompt,gen", [(1, 25000, 1000), (64, 25000, 1000), (2, 268000, 500)])
def test_document_reproduction_workloads(N, prompt, gen, cuda):
    ctx, lens = inputs.context_inputs(N, prompt, gen, 151936, quote=True, seed=800 + N)
    rc = _check(ctx, lens, 4, 1, 8, cuda)
    assert (rc == 8).all()  # the quoted passage continues in the prompt


def test_chat_like_workload_ragged(cuda):
    ctx, lens = inputs.context_inputs(64, 3000, 200, 151936, quote=False, ragged=True, seed=810)
    _check(ctx, lens, 4, 1, 8, cuda)
    _check(ctx, lens, 4, 2, 8, cuda)


def test_row_pitch_larger_than_lengths_and_noncontiguous_guard(cuda):
    ctx, lens = inputs.context_inputs(5, 300, 20, 50, quote=True, seed=820)
    _check(ctx, lens - 7, 3, 1, 4, cuda)
    with pytest.raises(ValueError):
        dn.dn_context_drafts(ctx.to(cuda)[:, ::2], lens.to(cuda))

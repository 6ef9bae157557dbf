"""The allocation-free greedy-accept entry point against the regular one (GPU).

dn_accept_greedy_noalloc serves callers that cannot allocate device memory where
they verify: an engine that has given nearly all GPU memory to its own page pool,
or C code embedded in a host whose allocator it cannot reach. It keeps its scratch
in a fixed array inside libdn.so instead of a caller workspace. These tests call
it through the C ABI and require the same target ids and accepted lengths
(bit-exact, as for every integer result here) as dn_accept_greedy on the same
inputs, on two calls in a row, plus the size limit; and the same results as the
float64 oracle directly, also right after a larger call has left its scratch
full of non-zero keys where the next call keeps its counters. They depend on no
other test, so they pass alone in a fresh process and after the rest of the suite.
"""

import numpy as np
import pytest
import torch

import oracle
from deltanet_recurrent_state_gb300 import binding as dn
from deltanet_recurrent_state_gb300 import inputs

pytestmark = pytest.mark.gpu

_DT = {torch.float16: dn.DN_F16, torch.float32: dn.DN_F32}
SCRATCH_LIMIT = 256 * 1024  # DN_ACCEPT_NOALLOC_SCRATCH_BYTES in include/dn.h


def _noalloc(lib, logits, draft, stream):
    B, T, V = logits.shape
    tgt = torch.full((B, T), -7, dtype=torch.int32, device=logits.device)
    acc = torch.full((B,), -7, dtype=torch.int32, device=logits.device)
    st = lib.dn_accept_greedy_noalloc(B, T, V, _DT[logits.dtype], logits.data_ptr(),
                                      draft.data_ptr(), tgt.data_ptr(), acc.data_ptr(), stream)
    return st, tgt, acc


def _case(B, T, V, dt, seed, cuda):
    logits, target = inputs.logits_inputs(B, T, V, dtype=dt, std=2.0, seed=seed, device=cuda)
    a = inputs.accepted_lengths(B, T, "uniform", seed=seed + 1)
    draft = inputs.draft_ids(target, a, V, seed=seed + 2)
    return logits, draft


def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(cuda):
    lib = dn.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [_case(1, 16, 151936, "f16", 900, cuda), _case(64, 4, 151936, "f16", 910, cuda)]
    for logits, draft in cases:  # two calls in a row, sharing the library's scratch array
        st, tgt, acc = _noalloc(lib, logits, draft, stream)
        assert st == dn.DN_OK, dn.dn_status_string(st)
        ref_tgt, ref_acc = dn.dn_accept_greedy(logits, draft)
        torch.cuda.synchronize()
        assert torch.equal(tgt, ref_tgt)
        assert torch.equal(acc, ref_acc)


def test_noalloc_repeated_calls_fp32_and_ties(cuda):
    lib = dn.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    gen = torch.Generator().manual_seed(5)
    for r in range(2):
        logits = torch.randint(-3, 4, (3, 5, 9001), generator=gen).float().to(cuda)  # many ties
        draft = torch.randint(0, 4, (3, 5), generator=gen, dtype=torch.int32).to(cuda)
        st, tgt, acc = _noalloc(lib, logits, draft, stream)
        assert st == dn.DN_OK
        ref_tgt, ref_acc = dn.dn_accept_greedy(logits, draft)
        torch.cuda.synchronize()
        assert torch.equal(tgt, ref_tgt) and torch.equal(acc, ref_acc), r


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda):
    lib = dn.load_library()
    B, T, V = 1800, 1, 151936
    assert dn.dn_accept_workspace_bytes(B, T, V) > SCRATCH_LIMIT
    assert dn.dn_accept_workspace_bytes(1600, 1, V) <= SCRATCH_LIMIT
    # real buffers of the full size, so nothing could read out of bounds even if the
    # check were missing; the call must refuse before launching anything
    logits = torch.empty((B, T, V), dtype=torch.float16, device=cuda)
    draft = torch.zeros((B, T), dtype=torch.int32, device=cuda)
    st, tgt, acc = _noalloc(lib, logits, draft, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == dn.DN_ERR_INVALID_ARG
    assert (tgt == -7).all() and (acc == -7).all()


def test_noalloc_matches_oracle_after_a_larger_call_left_leftovers(cuda):
    # A call over many rows fills the front of the shared array with its chunk keys (never
    # zero: every key carries the value's order bits). The next, smaller call keeps its
    # counters at an offset inside that region, so it is right only if it clears them first.
    lib = dn.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    V = 151936
    chunks = (V + 8191) // 8192
    big_rows, small = 1500, (1, 16)
    assert dn.dn_accept_workspace_bytes(big_rows, 1, V) <= SCRATCH_LIMIT
    small_counter_offset = small[0] * small[1] * chunks * 8  # keys first, 16-byte aligned
    assert small_counter_offset % 16 == 0 and small_counter_offset < big_rows * chunks * 8
    for B, T in ((big_rows, 1), small, (big_rows, 1), (3, 5)):
        logits, draft = _case(B, T, V, "f16", 920 + B + T, cuda)
        st, tgt, acc = _noalloc(lib, logits, draft, stream)
        assert st == dn.DN_OK, dn.dn_status_string(st)
        torch.cuda.synchronize()
        tgt_ref, acc_ref = oracle.accept_greedy(logits.double().cpu().numpy(), draft.cpu().numpy())
        np.testing.assert_array_equal(tgt.cpu().numpy(), tgt_ref)
        np.testing.assert_array_equal(acc.cpu().numpy(), acc_ref)

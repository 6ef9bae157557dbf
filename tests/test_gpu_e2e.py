"""The pipelined end-to-end step of bench.py (each layer group's inputs copied on a copy stream,
the group's verify started when its copy has landed) computes what the step with one copy
before the three calls computes: after the same steps from the same inputs, the committed
states, the checkpoints and the outputs are bit-identical."""

import pytest
import torch

import bench

pytestmark = pytest.mark.gpu

# a small step: 6 layers x 4 heads x 64 x 64 fp16, T = 8, 5 of 8 drafts accepted
W = {"L": 6, "B": 1, "H": 4, "dk": 64, "dv": 64, "T": 8, "io": "f16", "state": "f16", "V": 5000,
     "logit_dtype": "f16", "logit_std": 2.0, "accept": "fixed", "accept_value": 5, "seed": 77}


@pytest.mark.parametrize("groups", [(1, 2, 3), 3, (5, 1)])
def test_pipelined_step_commits_the_same_states(groups, cuda):
    stream = torch.cuda.Stream(device=cuda)
    single = bench.make_step_sets(W, cuda, 0, 2)
    piped = bench.make_step_sets(W, cuda, 0, 2)
    start = [x["state"].clone() for x in single]
    for x, y in zip(single, piped):
        assert torch.equal(x["state"], y["state"])
    # eager warm-up, graph capture, replayed warm-up and timed steps: the same sequence of
    # steps over the two buffer sets in both runs, each step committing into its set's state
    bench.e2e_steps(W, single, 3, 3, stream, cuda, graphs=True, groups=1)
    bench.e2e_steps(W, piped, 3, 3, stream, cuda, graphs=True, groups=groups)
    torch.cuda.synchronize()
    for x, y in zip(single, piped):
        assert torch.equal(x["state"], y["state"])
        assert torch.equal(x["ckpt"], y["ckpt"])
        assert torch.equal(x["out"], y["out"])
    # the steps did commit (accepted length 5 >= 1), so the comparison is not of untouched states
    assert not any(torch.equal(x["state"], s0) for x, s0 in zip(single, start))


def test_accept_beside_verify_commits_the_same_states(cuda):
    # The timed step runs accept on a second stream beside verify (accept reads only the
    # logits and draft ids) and commit after both; the same steps one after another on one
    # stream give the same targets, accepted lengths, checkpoints and committed states.
    stream = torch.cuda.Stream(device=cuda)
    side = bench.side_stream(cuda)
    serial = bench.make_step_sets(W, cuda, 0, 1)[0]
    beside = bench.make_step_sets(W, cuda, 0, 1)[0]
    with torch.cuda.stream(stream):
        for _ in range(3):
            bench.run_step(serial, stream)
            bench.run_step(beside, stream, side=side)
    torch.cuda.synchronize()
    for key in ("tgt", "acc", "out", "ckpt", "state"):
        assert torch.equal(serial[key], beside[key]), key
    assert int(beside["acc"][0]) == W["accept_value"]

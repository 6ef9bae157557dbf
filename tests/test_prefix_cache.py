"""The host prefix index (dn_prefix_cache_*) against a plain dictionary model (no GPU).

Model: a dict from a token prefix (tuple) whose length is a multiple of the chunk to a
slot, with least-recently-used eviction; lookup returns the longest cached prefix.
"""

import collections
import random

import numpy as np
import pytest

from deltanet_recurrent_state_gb300 import binding
from deltanet_recurrent_state_gb300 import build as dnbuild


@pytest.fixture(scope="module", autouse=True)
def lib():
    dnbuild.build()
    return binding.load_library()


class Model:
    def __init__(self, capacity, chunk):
        self.cap, self.chunk = capacity, chunk
        self.d = collections.OrderedDict()  # prefix -> slot, last = most recent

    def insert(self, tokens, pos, slot):
        key = tuple(tokens[:pos])
        if key in self.d:
            old = self.d.pop(key)
            self.d[key] = slot
            return old if old != slot else -1
        ev = -1
        if len(self.d) >= self.cap:
            _, ev = self.d.popitem(last=False)
        self.d[key] = slot
        return ev

    def lookup(self, tokens):
        for pos in range(len(tokens) - len(tokens) % self.chunk, 0, -self.chunk):
            key = tuple(tokens[:pos])
            if key in self.d:
                self.d.move_to_end(key)
                return pos, self.d[key]
        return 0, -1


def test_longest_prefix_and_exact_match():
    c = binding.PrefixCache(capacity=8, chunk=4)
    doc = list(range(100, 120))
    assert c.insert(doc, 4, 0) == -1
    assert c.insert(doc, 12, 1) == -1
    assert c.lookup(doc) == (12, 1)
    assert c.lookup(doc[:11]) == (4, 0)          # 12 not reachable: only 11 tokens
    other = doc[:8] + [7] + doc[9:]
    assert c.lookup(other) == (4, 0)             # diverges inside the 3rd chunk
    assert c.lookup([1, 2, 3]) == (0, -1)
    assert c.lookup([]) == (0, -1)
    assert len(c) == 2


def test_replace_slot_for_same_prefix():
    c = binding.PrefixCache(capacity=4, chunk=2)
    t = [5, 6, 7, 8]
    assert c.insert(t, 2, 3) == -1
    assert c.insert(t, 2, 9) == 3                # the old slot is handed back
    assert c.insert(t, 2, 9) == -1
    assert c.lookup(t) == (2, 9)


def test_bad_arguments():
    c = binding.PrefixCache(capacity=2, chunk=4)
    for pos in (0, 3, 5):
        with pytest.raises(binding.DnError):
            c.insert(list(range(8)), pos, 0)
    with pytest.raises(binding.DnError):
        c.insert(list(range(8)), 4, -1)
    lib = binding.load_library()
    assert not lib.dn_prefix_cache_create(0, 4)
    assert not lib.dn_prefix_cache_create(64, 0)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_against_model_with_eviction(seed):
    rng = random.Random(seed)
    chunk, cap = 4, 6
    c, m = binding.PrefixCache(capacity=cap, chunk=chunk), Model(cap, chunk)
    # prompts share openings (small alphabet, few templates) so prefixes collide often
    templates = [[rng.randrange(3) for _ in range(24)] for _ in range(4)]
    next_slot = 0
    for _ in range(400):
        base = list(rng.choice(templates))
        cut = rng.randrange(len(base) + 1)
        toks = base[:cut] + [rng.randrange(3) for _ in range(rng.randrange(10))]
        if rng.random() < 0.5 and len(toks) >= chunk:
            pos = chunk * rng.randint(1, len(toks) // chunk)
            assert c.insert(toks, pos, next_slot) == m.insert(toks, pos, next_slot)
            next_slot += 1
        else:
            assert c.lookup(toks) == m.lookup(toks)
        assert len(c) == len(m.d)


def test_exact_compare_survives_many_chunks():
    # many distinct chunks under one parent: every lookup finds its own slot
    c = binding.PrefixCache(capacity=5000, chunk=2)
    for i in range(3000):
        assert c.insert([i, i + 1, 0, 0], 2, i) == -1
    for i in range(0, 3000, 7):
        assert c.lookup([i, i + 1, 9]) == (2, i)


@pytest.mark.gpu
def test_restore_longest_prefix_then_prefill_tail_is_bit_identical(cuda):
    """Serve prompt B from prompt A's cached checkpoints: restore + tail == full prefill of B.

    Layer inputs are a fixed function of the token id (a seeded table), so two prompts with
    the same opening tokens feed the recurrence the same q, k, v, beta, g there.
    """
    import torch

    from deltanet_recurrent_state_gb300 import inputs

    H, d, vocab, C = 4, 128, 50, binding.PREFILL_CHUNK
    tab = inputs.recurrence_inputs(1, vocab, H, d, d, seed=700, device=cuda)
    keys = ("q", "k", "v", "beta", "g")

    def feats(tokens):
        idx = torch.as_tensor(tokens, dtype=torch.long, device=cuda)
        return [tab[k][:, idx].contiguous() for k in keys]

    rng = np.random.default_rng(701)
    prompt_a = rng.integers(0, vocab, 5 * C + 17).tolist()
    prompt_b = prompt_a[:3 * C + 40] + rng.integers(0, vocab, 2 * C + 5).tolist()
    s0 = tab["state"][:1].contiguous()

    cache = binding.PrefixCache(capacity=16)
    pool = torch.empty((16,) + tuple(s0.shape[1:]), dtype=s0.dtype, device=cuda)
    _, ckpt_a, _ = binding.dn_prefill_checkpoint(*feats(prompt_a), s0)
    for c in range(ckpt_a.shape[1]):
        assert cache.insert(prompt_a, C * (c + 1), c) == -1
        pool[c].copy_(ckpt_a[0, c])

    pos, slot = cache.lookup(prompt_b)
    assert (pos, slot) == (3 * C, 2)             # B diverges inside A's 4th chunk
    tail = [f[:, pos:].contiguous() for f in feats(prompt_b)]
    o_tail, ck_tail, s_tail = binding.dn_prefill_checkpoint(*tail, pool[slot:slot + 1].contiguous())
    o_full, ck_full, s_full = binding.dn_prefill_checkpoint(*feats(prompt_b), s0)
    torch.cuda.synchronize()
    assert torch.equal(s_tail, s_full)
    assert torch.equal(o_tail, o_full[:, pos:])
    assert torch.equal(ck_tail, ck_full[:, pos // C:])

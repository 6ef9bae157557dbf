"""Pins of the CPU oracle against what the mathematics fixes (no GPU).

Each pin is chosen so that a plausible slip in the oracle fails it: a dropped
gate, a sign error in the erase term, S k^T instead of v k^T, left- instead of
right-multiplication by (I - beta k k^T), reading S_{t-1} instead of S_t, q and
k swapped, an off-by-one in the commit index, rounding the carry inside a
block, a missing or extra checkpoint, and the wrong argmax tie-break.

The recurrence is the gated delta rule (Yang et al. 2024), the DeltaNet state of
"HyperQwen: 1,000 tok/s on a Single RTX 3090 Through Aggressive Recurrent-State
Speculation" (Technical Insight).
"""

import os
import re
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import wy_chunk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unit(rng, *shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _inputs(rng, N=2, T=5, H=3, dk=6, dv=5):
    return dict(
        q=_unit(rng, N, T, H, dk),
        k=_unit(rng, N, T, H, dk),
        v=rng.standard_normal((N, T, H, dv)),
        beta=1.0 / (1.0 + np.exp(-rng.standard_normal((N, T, H)))),
        g=np.exp(-np.log1p(np.exp(rng.standard_normal((N, T, H))))),
        state_in=0.1 * rng.standard_normal((N, H, dv, dk)),
    )


def _run(inp, store=None, io=None):
    return oracle.verify_block(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                               inp["state_in"], store=store, io=io)


# ----------------------------------------------------------------------------- golden

def _parse_recurrence_golden():
    cases = {}
    name = None
    with open(os.path.join(GOLDEN, "handworked_recurrence.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "case":
                name = parts[1]
                cases[name] = dict(toks=[])
            elif parts[0] == "dims":
                cases[name]["dv"], cases[name]["dk"] = int(parts[1]), int(parts[2])
            elif parts[0] == "S0":
                cases[name]["S0"] = [float(x) for x in parts[1:]]
            elif parts[0] == "tok":
                tok = {}
                for kv in parts[1:]:
                    key, val = kv.split("=")
                    tok[key] = [float(x) for x in val.split(",")]
                cases[name]["toks"].append(tok)
    return cases


@pytest.mark.parametrize("case", ["scalar", "two_by_two"])
@pytest.mark.parametrize("store", [None, "f32", "f16"])
def test_handworked_golden(case, store):
    c = _parse_recurrence_golden()[case]
    dv, dk, toks = c["dv"], c["dk"], c["toks"]
    T = len(toks)
    q = np.array([t["q"] for t in toks]).reshape(1, T, 1, dk)
    k = np.array([t["k"] for t in toks]).reshape(1, T, 1, dk)
    v = np.array([t["v"] for t in toks]).reshape(1, T, 1, dv)
    beta = np.array([t["beta"][0] for t in toks]).reshape(1, T, 1)
    g = np.array([t["g"][0] for t in toks]).reshape(1, T, 1)
    S0 = np.array(c["S0"]).reshape(1, 1, dv, dk)
    o, ckpt = oracle.verify_block(q, k, v, beta, g, S0, store=store, io=store)
    for t, tok in enumerate(toks):
        assert np.array_equal(ckpt[0, t, 0], np.array(tok["S"]).reshape(dv, dk)), (case, t)
        assert np.array_equal(o[0, t, 0], np.array(tok["o"])), (case, t)


# ----------------------------------------------------------------------------- store rounding

def _exact(expr):
    """An exact value written as a signed sum of terms c, c*2^e or 2^e (inf, -inf, -0 allowed).

    Returns a float64. Every term is parsed as an exact rational (a decimal literal
    stands for its nearest float64), so the sum is exact before the one final
    conversion, and every input of the golden file is a float64 value.
    """
    if expr in ("inf", "-inf"):
        return float(expr)
    if expr == "-0":
        return -0.0
    total = Fraction(0)
    for sign, term in re.findall(r"([+-]?)([^+-]+(?:\^-?\d+)?)", expr.replace("^-", "^~")):
        term = term.replace("^~", "^-")
        value = Fraction(1)
        for factor in term.split("*"):
            if factor.startswith("2^"):
                value *= Fraction(2) ** int(factor[2:])
            else:
                value *= Fraction(float(factor)) if "." in factor else Fraction(int(factor))
        total += -value if sign == "-" else value
    x = float(total)
    assert Fraction(x) == total, expr  # every value in the file is a float64
    return x


def _decode(fmt, bits):
    """The value of an IEEE 754 binary16 / binary32 encoding, from the format's definition."""
    ebits, fbits = {"f16": (5, 10), "f32": (8, 23)}[fmt]
    bias = (1 << (ebits - 1)) - 1
    s = bits >> (ebits + fbits)
    e = (bits >> fbits) & ((1 << ebits) - 1)
    f = bits & ((1 << fbits) - 1)
    if e == (1 << ebits) - 1:
        assert f == 0, "no NaN in the golden file"
        mag = float("inf")
    elif e == 0:
        mag = float(Fraction(f, 1 << fbits) * Fraction(2) ** (1 - bias))
    else:
        mag = float((1 + Fraction(f, 1 << fbits)) * Fraction(2) ** (e - bias))
    return -mag if s else mag


def _parse_rounding_golden():
    rows = []
    with open(os.path.join(GOLDEN, "handworked_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, x, want, bits = line.split()
            rows.append((fmt, x, want, int(bits, 16)))
    return rows


def _same_value(a, b):
    return (a == b and np.signbit(a) == np.signbit(b)) or (np.isinf(a) and a == b)


def test_rounding_golden_file_is_self_consistent():
    # each expected value is the value its stated encoding decodes to
    rows = _parse_rounding_golden()
    assert sum(r[0] == "f16" for r in rows) >= 20 and sum(r[0] == "f32" for r in rows) >= 8
    for fmt, _, want, bits in rows:
        assert _same_value(_decode(fmt, bits), _exact(want)), (fmt, want, hex(bits))


def test_round_to_handworked_round_to_nearest_even():
    # oracle.round_to against hand-worked binary16 / binary32 roundings: ties to even,
    # either side of a tie, carries into the next binade, subnormals, overflow, -0
    for fmt, x, want, bits in _parse_rounding_golden():
        with np.errstate(over="ignore"):
            got = float(oracle.round_to(np.array([_exact(x)]), fmt)[0])
        assert _same_value(got, _decode(fmt, bits)), (fmt, x, got, want)


def test_verify_and_prefill_stores_round_to_nearest_even():
    # the stores of verify_block and prefill_checkpoint carry the same rounding: with
    # beta = 0 and g = 1 the state is unchanged and o = S q, so a hand-picked S and q
    # put an exact value on each store. S0 = 1 + 2^-11 + 2^-30 (stored: 1 + 2^-10,
    # not 1 as truncation or double rounding through binary32 would give); q = 1 + 2^-10,
    # so o = S q = 1 + 3*2^-11 + 2^-21 + 2^-30 + 2^-40, just above the tie between
    # 1 + 2^-10 and 1 + 2^-9: stored 1 + 2^-9 (truncation gives 1 + 2^-10).
    s0 = _exact("1+2^-11+2^-30")
    qv = _exact("1+2^-10")
    o_exact = Fraction(s0) * Fraction(qv)
    assert Fraction(_exact("1+3*2^-11")) < o_exact < Fraction(_exact("1+2^-9"))
    one = np.ones((1, 1, 1, 1))
    args = dict(q=qv * one, k=one, v=one, beta=np.zeros((1, 1, 1)), g=np.ones((1, 1, 1)))
    o, ck = oracle.verify_block(args["q"], args["k"], args["v"], args["beta"], args["g"],
                                s0 * np.ones((1, 1, 1, 1)), store="f16", io="f16")
    assert ck[0, 0, 0, 0, 0] == _exact("1+2^-10")
    assert o[0, 0, 0, 0] == _exact("1+2^-9")
    o2, ck2, sf = oracle.prefill_checkpoint(args["q"], args["k"], args["v"], args["beta"], args["g"],
                                            s0 * np.ones((1, 1, 1, 1)), chunk=1, store="f16", io="f16")
    assert ck2[0, 0, 0, 0, 0] == _exact("1+2^-10") and sf[0, 0, 0, 0] == _exact("1+2^-10")
    assert o2[0, 0, 0, 0] == _exact("1+2^-9")


# ----------------------------------------------------------------------------- closed forms

def test_beta0_g1_leaves_state_unchanged():
    rng = np.random.default_rng(1)
    inp = _inputs(rng)
    inp["beta"][:] = 0.0
    inp["g"][:] = 1.0
    o, ckpt = _run(inp)
    S0 = inp["state_in"]
    for t in range(ckpt.shape[1]):
        assert np.array_equal(ckpt[:, t], S0)
        # o_t = S0 q_t, summed element by element
        ref = np.zeros_like(o[:, t])
        for j in range(S0.shape[-1]):
            ref += S0[..., :, j] * inp["q"][:, t, :, None, j]
        np.testing.assert_allclose(o[:, t], ref, rtol=0, atol=1e-14)


def test_beta0_state_decays_by_gate_product():
    rng = np.random.default_rng(2)
    inp = _inputs(rng)
    inp["beta"][:] = 0.0
    _, ckpt = _run(inp)
    gamma = np.cumprod(inp["g"], axis=1)  # [N, T, H]
    for t in range(ckpt.shape[1]):
        np.testing.assert_allclose(ckpt[:, t], gamma[:, t, :, None, None] * inp["state_in"],
                                   rtol=1e-13, atol=1e-15)


def test_beta1_g1_unit_key_writes_value_exactly():
    rng = np.random.default_rng(3)
    inp = _inputs(rng, dk=8, dv=8)
    inp["beta"][:] = 1.0
    inp["g"][:] = 1.0
    _, ckpt = _run(inp)
    T = ckpt.shape[1]
    for t in range(T):
        Sk = np.einsum("nhij,nhj->nhi", ckpt[:, t], inp["k"][:, t])
        np.testing.assert_allclose(Sk, inp["v"][:, t], rtol=0, atol=1e-12)


def test_key_direction_update_general_beta_gate():
    # S_t k_t = g_t (1 - beta_t) S_{t-1} k_t + beta_t v_t  for unit k_t
    rng = np.random.default_rng(4)
    inp = _inputs(rng)
    _, ckpt = _run(inp)
    prev = inp["state_in"]
    for t in range(ckpt.shape[1]):
        k = inp["k"][:, t]
        lhs = np.einsum("nhij,nhj->nhi", ckpt[:, t], k)
        b = inp["beta"][:, t][..., None]
        gg = inp["g"][:, t][..., None]
        rhs = gg * (1 - b) * np.einsum("nhij,nhj->nhi", prev, k) + b * inp["v"][:, t]
        np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
        prev = ckpt[:, t]


def test_directions_orthogonal_to_key_only_decay():
    # x orthogonal to k_t  =>  S_t x = g_t S_{t-1} x   (right-multiplication by the erase)
    rng = np.random.default_rng(5)
    inp = _inputs(rng)
    _, ckpt = _run(inp)
    prev = inp["state_in"]
    for t in range(ckpt.shape[1]):
        k = inp["k"][:, t]
        x = rng.standard_normal(k.shape)
        x = x - np.sum(x * k, axis=-1, keepdims=True) * k
        lhs = np.einsum("nhij,nhj->nhi", ckpt[:, t], x)
        rhs = inp["g"][:, t][..., None] * np.einsum("nhij,nhj->nhi", prev, x)
        np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
        prev = ckpt[:, t]


def test_zero_state_first_token_is_outer_product_v_k():
    # S_0 = 0: S_1[i, j] = beta v_i k_j and o_1 = beta v (k . q)  (reads the updated state)
    rng = np.random.default_rng(6)
    inp = _inputs(rng, T=1, dk=7, dv=4)
    inp["state_in"][:] = 0.0
    o, ckpt = _run(inp)
    b = inp["beta"][:, 0]
    v, k, q = inp["v"][:, 0], inp["k"][:, 0], inp["q"][:, 0]
    for n in range(v.shape[0]):
        for h in range(v.shape[1]):
            for i in range(v.shape[2]):
                for j in range(k.shape[2]):
                    assert abs(ckpt[n, 0, h, i, j] - b[n, h] * v[n, h, i] * k[n, h, j]) < 1e-15
                kq = sum(k[n, h, j] * q[n, h, j] for j in range(k.shape[2]))
                assert abs(o[n, 0, h, i] - b[n, h] * v[n, h, i] * kq) < 1e-14


def test_orthonormal_keys_form_an_exact_associative_memory():
    # g = 1, beta = 1, keys = distinct basis vectors: S_t = S0 (I - sum k k^T) + sum v k^T.
    # Reading with q_t = k_1 returns v_1 at every t (q and k play different roles).
    rng = np.random.default_rng(7)
    N, T, H, dk, dv = 1, 4, 2, 6, 3
    inp = _inputs(rng, N=N, T=T, H=H, dk=dk, dv=dv)
    inp["beta"][:] = 1.0
    inp["g"][:] = 1.0
    perm = [4, 1, 5, 0]
    inp["k"][:] = 0.0
    for t, j in enumerate(perm):
        inp["k"][:, t, :, j] = 1.0
    inp["q"][:] = inp["k"][:, :1]  # q_t = k_1 for all t
    o, ckpt = _run(inp)
    for t in range(T):
        np.testing.assert_allclose(o[:, t], inp["v"][:, 0], rtol=0, atol=1e-14)
        expect = inp["state_in"].copy()
        for s in range(t + 1):
            expect[..., :, perm[s]] = inp["v"][:, s]
        np.testing.assert_allclose(ckpt[:, t], expect, rtol=0, atol=1e-14)


def test_value_permutation_permutes_state_rows():
    rng = np.random.default_rng(8)
    inp = _inputs(rng, dv=6)
    o, ckpt = _run(inp)
    p = rng.permutation(6)
    inp2 = dict(inp)
    inp2["v"] = inp["v"][..., p]
    inp2["state_in"] = inp["state_in"][..., p, :]
    o2, ckpt2 = _run(inp2)
    np.testing.assert_allclose(o2, o[..., p], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ckpt2, ckpt[..., p, :], rtol=0, atol=1e-13)


def test_block_equals_chained_single_tokens():
    rng = np.random.default_rng(9)
    inp = _inputs(rng, T=6)
    o, ckpt = _run(inp)
    S = inp["state_in"]
    for t in range(6):
        one = {key: (val[:, t:t + 1] if key != "state_in" else S) for key, val in inp.items()}
        o1, c1 = _run(one)
        np.testing.assert_array_equal(o1[:, 0], o[:, t])
        np.testing.assert_array_equal(c1[:, 0], ckpt[:, t])
        S = c1[:, 0]


def test_stores_round_only_at_store_not_in_carry():
    # fp16 mode stores round16(S_t) but carries the exact S_t inside the block
    rng = np.random.default_rng(10)
    inp = _inputs(rng, T=4)
    o64, c64 = _run(inp, store=None, io=None)
    o16, c16 = _run(inp, store="f16", io="f16")
    np.testing.assert_array_equal(c16, c64.astype(np.float16).astype(np.float64))
    np.testing.assert_array_equal(o16, o64.astype(np.float16).astype(np.float64))


# ----------------------------------------------------------------------------- commit

@pytest.mark.parametrize("B", [1, 3])
def test_verify_then_commit_equals_prefix_run(B):
    rng = np.random.default_rng(11)
    L, T = 2, 5
    inp = _inputs(rng, N=L * B, T=T)
    _, ckpt = _run(inp, store="f16", io="f16")
    for a0 in range(T + 1):
        a = np.array([(a0 + b) % (T + 1) for b in range(B)], dtype=np.int32)
        S = oracle.commit(inp["state_in"], ckpt, a)
        for n in range(L * B):
            an = int(a[n % B])
            if an == 0:
                np.testing.assert_array_equal(S[n], inp["state_in"][n])
                continue
            pre = {key: (val[n:n + 1, :an] if key != "state_in" else val[n:n + 1])
                   for key, val in inp.items()}
            _, cp = _run(pre, store="f16", io="f16")
            np.testing.assert_array_equal(S[n], cp[0, an - 1])


# ----------------------------------------------------------------------------- prefill

def _prefill_inputs(rng, N=1, P=100, H=2, dk=4, dv=3):
    d = _inputs(rng, N=N, T=P, H=H, dk=dk, dv=dv)
    return d


@pytest.mark.parametrize("P", [1, 7, 8, 9, 17, 24])
def test_prefill_equals_tokenwise_and_checkpoints_at_chunk_ends(P):
    rng = np.random.default_rng(12 + P)
    inp = _prefill_inputs(rng, P=P)
    chunk = 8
    o, ckpt, Sf = oracle.prefill_checkpoint(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                                            inp["state_in"], chunk=chunk, store=None, io=None)
    assert ckpt.shape[1] == P // chunk
    ov, cv = _run(inp)
    np.testing.assert_allclose(o, ov, rtol=0, atol=1e-13)
    for c in range(P // chunk):
        np.testing.assert_allclose(ckpt[:, c], cv[:, chunk * (c + 1) - 1], rtol=0, atol=1e-13)
    np.testing.assert_allclose(Sf, cv[:, P - 1], rtol=0, atol=1e-13)


def test_prefill_zero_initial_state_is_none():
    rng = np.random.default_rng(30)
    inp = _prefill_inputs(rng, P=10)
    a = oracle.prefill_checkpoint(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], None,
                                  chunk=4, store="f16", io="f16")
    b = oracle.prefill_checkpoint(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                                  np.zeros_like(inp["state_in"]), chunk=4, store="f16", io="f16")
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("store", ["f16", "f32"])
def test_prefill_restore_from_checkpoint_equals_full_run(store):
    # a run restored from the last checkpoint and fed only the tail ends where the full run ends
    rng = np.random.default_rng(31)
    P, chunk = 45, 8
    inp = _prefill_inputs(rng, P=P)
    args = (inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"])
    o, ckpt, Sf = oracle.prefill_checkpoint(*args, inp["state_in"], chunk=chunk, store=store, io=store)
    c = P // chunk - 1
    start = chunk * (c + 1)
    tail = [x[:, start:] for x in args]
    o2, _, Sf2 = oracle.prefill_checkpoint(*tail, ckpt[:, c], chunk=chunk, store=store, io=store)
    np.testing.assert_array_equal(Sf2, Sf)
    np.testing.assert_array_equal(o2, o[:, start:])
    # restarting from each checkpoint also reproduces the later checkpoints
    for c0 in range(P // chunk - 1):
        s0 = chunk * (c0 + 1)
        _, ck3, _ = oracle.prefill_checkpoint(*[x[:, s0:] for x in args], ckpt[:, c0],
                                              chunk=chunk, store=store, io=store)
        np.testing.assert_array_equal(ck3, ckpt[:, c0 + 1:])


def test_prefill_carry_rounded_at_chunk_boundaries():
    # fp16 mode: the carry at each chunk end is the fp16 checkpoint (not the exact state)
    rng = np.random.default_rng(32)
    inp = _prefill_inputs(rng, P=16)
    args = (inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"])
    _, ck, _ = oracle.prefill_checkpoint(*args, inp["state_in"], chunk=8, store="f16", io="f16")
    first = oracle.prefill_checkpoint(*[x[:, :8] for x in args], inp["state_in"], chunk=8,
                                      store="f16", io="f16")[1][:, 0]
    assert np.array_equal(first, first.astype(np.float16).astype(np.float64))
    second = oracle.prefill_checkpoint(*[x[:, 8:] for x in args], first, chunk=8,
                                       store="f16", io="f16")[1][:, 0]
    np.testing.assert_array_equal(ck[:, 1], second)


@pytest.mark.parametrize("C", [1, 5, 16, 64])
def test_wy_chunk_algebra_equals_sequential_definition(C):
    # the chunked UT/WY algebra the tensor-core prefill uses equals the definition in float64
    rng = np.random.default_rng(40 + C)
    dk, dv = 16, 12
    inp = _prefill_inputs(rng, N=1, P=C, H=1, dk=dk, dv=dv)
    o_seq, _, S_seq = oracle.prefill_checkpoint(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                                                inp["state_in"], chunk=10 ** 9, store=None, io=None)
    O, S_C = wy_chunk.chunk_forward(inp["state_in"][0, 0], inp["q"][0, :, 0], inp["k"][0, :, 0],
                                    inp["v"][0, :, 0], inp["beta"][0, :, 0], inp["g"][0, :, 0])
    np.testing.assert_allclose(O, o_seq[0, :, 0], rtol=0, atol=1e-10)
    np.testing.assert_allclose(S_C, S_seq[0, 0], rtol=0, atol=1e-10)


# ----------------------------------------------------------------------------- accept

def _parse_accept_golden():
    rows, blocks = [], []
    with open(os.path.join(GOLDEN, "handworked_accept.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            parts = lhs.split()
            if parts[0] == "row":
                rows.append(([float(x) for x in parts[1:]], int(rhs)))
            else:
                kv = dict(p.split("=") for p in parts[1:])
                blocks.append((int(kv["T"]), [int(x) for x in kv["targets"].split(",")],
                               [int(x) for x in kv["drafts"].split(",")], int(rhs)))
    return rows, blocks


def test_accept_handworked_golden():
    rows, blocks = _parse_accept_golden()
    for vals, want in rows:
        assert oracle.argmax_lowest(np.array(vals)) == want, vals
        for dt in (np.float16, np.float32):
            assert oracle.argmax_lowest(np.array(vals, dtype=dt)) == want, (vals, dt)
    for T, targets, drafts, want in blocks:
        V = max(targets + drafts) + 1
        logits = np.zeros((1, T, V))
        for t, tg in enumerate(targets):
            logits[0, t, tg] = 1.0
        tgt, a = oracle.accept_greedy(logits, np.array([drafts]))
        assert list(tgt[0]) == targets
        assert int(a[0]) == want


@pytest.mark.parametrize("V", [1, 2, 3])
def test_argmax_brute_force_property(V):
    # every row over a small value set: the answer holds the maximum and no earlier index ties it
    import itertools
    vals = [-1.0, -0.0, 0.0, 1.0]
    for row in itertools.product(vals, repeat=V):
        r = np.array(row)
        i = oracle.argmax_lowest(r)
        assert all(r[i] >= x for x in r)
        assert all(r[j] < r[i] for j in range(i))


@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_accept_brute_force_all_draft_patterns(T):
    import itertools
    V = 3
    rng = np.random.default_rng(50 + T)
    logits = rng.integers(-2, 3, size=(1, T, V)).astype(np.float64)  # frequent ties
    tgt, _ = oracle.accept_greedy(logits, np.zeros((1, T), dtype=np.int32))
    for draft in itertools.product(range(V), repeat=T):
        _, a = oracle.accept_greedy(logits, np.array([draft]))
        a = int(a[0])
        assert all(draft[t] == tgt[0, t] for t in range(a))
        assert a == T or draft[a] != tgt[0, a]


def test_accept_all_equal_rows_pick_index_zero():
    logits = np.full((2, 3, 17), 0.125)
    tgt, a = oracle.accept_greedy(logits, np.zeros((2, 3), dtype=np.int32))
    assert (tgt == 0).all() and (a == 3).all()


# ----------------------------------------------------------------------------- context drafts

def _parse_context_golden():
    cases = []
    with open(os.path.join(GOLDEN, "handworked_context_drafts.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->", 1)
            parts = lhs.split()
            toks = [int(x) for x in parts[1:] if "=" not in x and x != "-"]
            kv = dict(p.split("=") for p in parts if "=" in p)
            out = dict(p.split("=") for p in rhs.split())
            drafts = [] if out["drafts"] == "-" else [int(x) for x in out["drafts"].split(",")]
            cases.append((toks, int(kv["nmax"]), int(kv["nmin"]), int(kv["K"]), drafts, int(out["n"])))
    return cases


def test_context_drafts_handworked_golden():
    for toks, n_max, n_min, K, want, n in _parse_context_golden():
        d, got_n, _ = oracle.context_drafts_row(toks, n_max, n_min, K)
        assert (d, got_n) == (want, n), toks


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_context_drafts_against_string_rfind(seed):
    # brute force by an independent route: with one character per token, the latest
    # occurrence of the last n tokens that ends before the last token is str.rfind of the
    # pattern in the context without its last token
    rng = np.random.default_rng(900 + seed)
    for _ in range(400):
        L = int(rng.integers(0, 30))
        toks = rng.integers(0, 3 + seed, L).tolist()
        n_max = int(rng.integers(1, 6))
        n_min = int(rng.integers(1, n_max + 1))
        K = int(rng.integers(1, 9))
        s = "".join(chr(97 + t) for t in toks)
        want, want_n = [], 0
        for n in range(n_max, n_min - 1, -1):
            if n > L - 1:
                continue
            j = s[:L - 1].rfind(s[L - n:])
            if j >= 0:
                want, want_n = toks[j + n:j + n + K], n
                break
        d, n, e = oracle.context_drafts_row(toks, n_max, n_min, K)
        assert (d, n) == (want, want_n), (toks, n_max, n_min, K)
        if n:
            assert toks[e - n:e] == toks[L - n:] and len(d) == min(K, L - e)


def test_context_drafts_batch_pads_and_uses_lengths():
    ctx = np.array([[1, 2, 3, 1, 2, 99, 99],
                    [6, 6, 6, 0, 0, 0, 0],
                    [4, 5, 4, 5, 4, 5, 4]])
    d, c, m = oracle.context_drafts(ctx, [5, 3, 7], 3, 1, 4)
    assert d[0].tolist() == [3, 1, 2, -1] and c[0] == 3 and m[0] == 2
    assert d[1].tolist() == [6, -1, -1, -1] and c[1] == 1 and m[1] == 2
    # latest occurrence of 4 5 4 ending before the last token starts at 2: drafts = 5 4
    assert d[2].tolist() == [5, 4, -1, -1] and c[2] == 2 and m[2] == 3

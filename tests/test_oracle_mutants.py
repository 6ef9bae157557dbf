"""Plant plausible mistakes in the oracle (CPU only) and check that the pins catch each.

Every mutant replaces one oracle function for the duration of a test; at least
one of the pin tests must then fail. This shows the pins fix each term of the
gated delta rule and of greedy acceptance, not just the oracle's own output.
"""

import numpy as np
import pytest

import oracle
from oracle import accept as acc_mod
from oracle import recurrence as rec
from tests import test_oracle_pins as pins


def _step_factory(kind):
    def step(S, q, k, v, beta, g):
        S = np.asarray(S, dtype=np.float64)
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        beta, g = np.asarray(beta, dtype=np.float64), np.asarray(g, dtype=np.float64)
        dk = k.shape[-1]
        eye = np.eye(dk)[None]
        kk = k[:, :, None] * k[:, None, :]
        b = beta[:, None, None]
        gg = g[:, None, None]
        erase = eye - b * kk
        write = b * (v[:, :, None] * k[:, None, :])
        if kind == "no_gate":
            S_new = np.matmul(S, erase) + write
        elif kind == "erase_sign":
            S_new = gg * np.matmul(S, eye + b * kk) + write
        elif kind == "erase_without_beta":
            S_new = gg * np.matmul(S, eye - kk) + write
        elif kind == "gate_on_write":
            S_new = gg * (np.matmul(S, erase) + write)
        elif kind == "left_multiply":
            if S.shape[1] != S.shape[2]:
                raise AssertionError("shape mismatch")
            S_new = gg * np.matmul(erase, S) + write
        elif kind == "write_transposed":
            if S.shape[1] != S.shape[2]:
                raise AssertionError("shape mismatch")
            S_new = gg * np.matmul(S, erase) + b * (k[:, :, None] * v[:, None, :])
        elif kind == "output_reads_old_state":
            S_new = gg * np.matmul(S, erase) + write
            return S_new, np.matmul(S, q[:, :, None])[:, :, 0]
        elif kind == "output_uses_key":
            S_new = gg * np.matmul(S, erase) + write
            return S_new, np.matmul(S_new, k[:, :, None])[:, :, 0]
        else:
            raise ValueError(kind)
        return S_new, np.matmul(S_new, q[:, :, None])[:, :, 0]
    return step


RECURRENCE_PINS = [
    lambda: pins.test_handworked_golden("scalar", None),
    lambda: pins.test_handworked_golden("two_by_two", None),
    pins.test_beta0_g1_leaves_state_unchanged,
    pins.test_beta0_state_decays_by_gate_product,
    pins.test_beta1_g1_unit_key_writes_value_exactly,
    pins.test_key_direction_update_general_beta_gate,
    pins.test_directions_orthogonal_to_key_only_decay,
    pins.test_zero_state_first_token_is_outer_product_v_k,
    pins.test_orthonormal_keys_form_an_exact_associative_memory,
    pins.test_value_permutation_permutes_state_rows,
]


def _count_failures(tests):
    failed = 0
    for t in tests:
        try:
            t()
        except (AssertionError, ValueError):
            failed += 1
    return failed


@pytest.mark.parametrize("kind", [
    "no_gate", "erase_sign", "erase_without_beta", "gate_on_write", "left_multiply",
    "write_transposed", "output_reads_old_state", "output_uses_key",
])
def test_recurrence_mutant_is_caught(kind, monkeypatch):
    monkeypatch.setattr(rec, "gated_delta_step", _step_factory(kind))
    assert _count_failures(RECURRENCE_PINS) >= 1, kind


def test_unmutated_recurrence_passes_all_pins():
    assert _count_failures(RECURRENCE_PINS) == 0


def test_block_rounding_carry_mutant_is_caught(monkeypatch):
    real = rec.verify_block

    def rounding_carry(q, k, v, beta, g, state_in, store="f16", io="f16"):
        # wrong: rounds the carried state after every token
        q = np.asarray(q, dtype=np.float64)
        N, T, H, dk = q.shape
        S = np.asarray(state_in, dtype=np.float64)
        os_, cs = [], []
        for t in range(T):
            o, c = real(q[:, t:t + 1], np.asarray(k)[:, t:t + 1], np.asarray(v)[:, t:t + 1],
                        np.asarray(beta)[:, t:t + 1], np.asarray(g)[:, t:t + 1], S, store, io)
            S = c[:, 0]
            os_.append(o)
            cs.append(c)
        return np.concatenate(os_, 1), np.concatenate(cs, 1)

    monkeypatch.setattr(rec, "verify_block", rounding_carry)
    monkeypatch.setattr(oracle, "verify_block", rounding_carry)
    with pytest.raises(AssertionError):
        pins.test_stores_round_only_at_store_not_in_carry()


def test_commit_off_by_one_mutant_is_caught(monkeypatch):
    def commit_wrong(state, ckpt, accepted_len):
        state = np.asarray(state, dtype=np.float64)
        ckpt = np.asarray(ckpt, dtype=np.float64)
        a = np.asarray(accepted_len)
        new = state.copy()
        T = ckpt.shape[1]
        for n in range(state.shape[0]):
            an = int(a[n % a.shape[0]])
            if an > 0:
                new[n] = ckpt[n, min(an, T - 1)]
        return new

    monkeypatch.setattr(oracle, "commit", commit_wrong)
    with pytest.raises(AssertionError):
        pins.test_verify_then_commit_equals_prefix_run(1)


def test_commit_wrong_request_mapping_mutant_is_caught(monkeypatch):
    def commit_wrong(state, ckpt, accepted_len):
        state = np.asarray(state, dtype=np.float64)
        ckpt = np.asarray(ckpt, dtype=np.float64)
        a = np.asarray(accepted_len)
        B = a.shape[0]
        L = state.shape[0] // B
        new = state.copy()
        for n in range(state.shape[0]):
            an = int(a[n // L])  # wrong: sets laid out [B][L]
            if an > 0:
                new[n] = ckpt[n, an - 1]
        return new

    monkeypatch.setattr(oracle, "commit", commit_wrong)
    with pytest.raises(AssertionError):
        pins.test_verify_then_commit_equals_prefix_run(3)


def test_prefill_checkpoint_offset_mutant_is_caught(monkeypatch):
    real = rec.prefill_checkpoint

    def shifted(q, k, v, beta, g, state_in, chunk=64, store="f16", io="f16"):
        o, ck, sf = real(q, k, v, beta, g, state_in, chunk, store, io)
        # wrong: checkpoint taken one token early
        o2, ck2, _ = real(np.asarray(q)[:, :-1], np.asarray(k)[:, :-1], np.asarray(v)[:, :-1],
                          np.asarray(beta)[:, :-1], np.asarray(g)[:, :-1], state_in,
                          chunk - 1 if chunk > 1 else 1, store, io)
        n = min(ck.shape[1], ck2.shape[1])
        ck = ck.copy()
        ck[:, :n] = ck2[:, :n]
        return o, ck, sf

    monkeypatch.setattr(oracle, "prefill_checkpoint", shifted)
    with pytest.raises(AssertionError):
        pins.test_prefill_equals_tokenwise_and_checkpoints_at_chunk_ends(17)


def test_argmax_highest_index_mutant_is_caught(monkeypatch):
    def highest(row):
        row = np.asarray(row, dtype=np.float64)
        return int(np.flatnonzero(row == row.max())[-1])

    monkeypatch.setattr(acc_mod, "argmax_lowest", highest)
    monkeypatch.setattr(oracle, "argmax_lowest", highest)
    with pytest.raises(AssertionError):
        pins.test_accept_handworked_golden()


def test_argmax_signed_zero_mutant_is_caught(monkeypatch):
    def bitwise(row):
        # wrong: orders -0.0 below +0.0
        row = np.asarray(row, dtype=np.float64)
        key = [(x, not np.signbit(x)) for x in row]
        best = max(range(len(key)), key=lambda i: (key[i], -i))
        return best

    monkeypatch.setattr(acc_mod, "argmax_lowest", bitwise)
    monkeypatch.setattr(oracle, "argmax_lowest", bitwise)
    with pytest.raises(AssertionError):
        pins.test_accept_handworked_golden()


def test_accept_counts_matches_not_prefix_mutant_is_caught(monkeypatch):
    def count_matches(logits, draft_ids):
        logits = np.asarray(logits, dtype=np.float64)
        d = np.asarray(draft_ids)
        B, T, _ = logits.shape
        tgt = np.array([[acc_mod.argmax_lowest(logits[b, t]) for t in range(T)] for b in range(B)],
                       dtype=np.int32)
        return tgt, (tgt == d).sum(axis=1).astype(np.int32)

    monkeypatch.setattr(acc_mod, "accept_greedy", count_matches)
    monkeypatch.setattr(oracle, "accept_greedy", count_matches)
    failed = 0
    for T in (2, 3, 4):
        try:
            pins.test_accept_brute_force_all_draft_patterns(T)
        except AssertionError:
            failed += 1
    assert failed >= 1


def _context_mutant(kind):
    from numpy.lib.stride_tricks import sliding_window_view

    def row(context, n_max, n_min, K):
        c = np.asarray(context).astype(np.int64)
        L = c.shape[0]
        order = range(n_min, n_max + 1) if kind == "shortest_first" else range(n_max, n_min - 1, -1)
        for n in order:
            if L - 1 < n:
                continue
            pattern = c[L - n:]
            hay = c if kind == "pattern_matches_itself" else c[:L - 1]
            win = sliding_window_view(hay, n)
            hits = np.flatnonzero((win == pattern).all(axis=1))
            if hits.size:
                j = int(hits[0] if kind == "earliest" else hits[-1])
                e = j + (n + 1 if kind == "skip_one" else (0 if kind == "copy_pattern" else n))
                return c[e:e + K].tolist(), n, e
        return [], 0, -1
    return row


@pytest.mark.parametrize("kind", ["shortest_first", "pattern_matches_itself", "earliest",
                                  "skip_one", "copy_pattern"])
def test_context_drafts_mutant_is_caught(kind, monkeypatch):
    from oracle import context_lookup as ctx_mod
    monkeypatch.setattr(ctx_mod, "context_drafts_row", _context_mutant(kind))
    monkeypatch.setattr(oracle, "context_drafts_row", _context_mutant(kind))
    with pytest.raises(AssertionError):
        pins.test_context_drafts_handworked_golden()


def _round_mutant(kind):
    real = rec.round_to

    def round_to(x, dtype):
        x = np.asarray(x, dtype=np.float64)
        if dtype != "f16":
            return real(x, dtype)
        with np.errstate(over="ignore"):
            if kind == "double_rounding":
                # wrong: rounds to binary32 first, then to binary16
                return x.astype(np.float32).astype(np.float16).astype(np.float64)
            near = x.astype(np.float16).astype(np.float64)
        if kind == "truncate":
            # wrong: rounds toward zero (drops the bits below the last fraction bit)
            over = np.abs(near) > np.abs(x)
            toward0 = np.nextafter(near.astype(np.float16), np.float16(0)).astype(np.float64)
            return np.where(over, toward0, near)
        if kind == "ties_away":
            # wrong: exact ties go away from zero instead of to the even neighbour
            up = np.nextafter(near.astype(np.float16), np.copysign(np.float16(np.inf), x).astype(np.float16))
            up = up.astype(np.float64)
            tie = np.abs(near - x) == np.abs(up - x)
            return np.where(tie & (np.abs(up) > np.abs(near)), up, near)
        raise ValueError(kind)
    return round_to


@pytest.mark.parametrize("kind", ["truncate", "double_rounding", "ties_away"])
def test_round_to_mutant_is_caught(kind, monkeypatch):
    mutant = _round_mutant(kind)
    monkeypatch.setattr(rec, "round_to", mutant)
    monkeypatch.setattr(oracle, "round_to", mutant)
    with pytest.raises(AssertionError):
        pins.test_round_to_handworked_round_to_nearest_even()
    if kind != "ties_away":  # the store-path pin holds no exact tie
        with pytest.raises(AssertionError):
            pins.test_verify_and_prefill_stores_round_to_nearest_even()


def test_unmutated_round_to_passes_its_pins():
    assert _count_failures([pins.test_round_to_handworked_round_to_nearest_even,
                            pins.test_verify_and_prefill_stores_round_to_nearest_even]) == 0

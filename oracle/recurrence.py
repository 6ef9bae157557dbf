"""Oracle for the gated delta-rule recurrence: verify block, commit, prefill.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may import it).

Layouts are the ones the C-ABI uses (row-major, last index fastest):

* q, k      [N, T, H, dk]      (prefill: [N, P, H, dk])
* v, o      [N, T, H, dv]
* beta, g   [N, T, H]
* state     [N, H, dv, dk]     the math state S itself (S[i, j], i over dv, j over dk)
* ckpt      [N, T, H, dv, dk]  (prefill: [N, P // chunk, H, dv, dk])

All arithmetic is float64. ``store`` / ``io`` name the dtype the product stores
states / outputs in ("f16", "f32" or None for none); the oracle rounds to that
dtype exactly where a value is stored and nowhere else.
"""

import numpy as np

_ROUND = {
    None: None,
    "f64": None,
    "f32": np.float32,
    "f16": np.float16,
}


def round_to(x, dtype):
    """Round float64 ``x`` to ``dtype`` ("f16", "f32" or None) and back to float64.

    numpy converts float64 to float16/float32 directly with round-to-nearest-even,
    which is the rounding the product's stores use.
    """
    t = _ROUND[dtype]
    x = np.asarray(x, dtype=np.float64)
    if t is None:
        return x.copy()
    return x.astype(t).astype(np.float64)


def gated_delta_step(S, q, k, v, beta, g):
    """One token of the gated delta rule, for U independent (state set, head) units.

    Definition (gated delta rule, Yang et al. 2024; the DeltaNet state of
    "HyperQwen: 1,000 tok/s on a Single RTX 3090 ...", Technical Insight):

        S_t = g_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
        o_t = S_t q_t

    written out literally: the dk x dk matrix (I - beta k k^T) is formed and
    multiplied on the right of S, and the output reads the updated state.

    S [U, dv, dk], q/k [U, dk], v [U, dv], beta/g [U]  ->  (S_t [U, dv, dk], o_t [U, dv])
    """
    S = np.asarray(S, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    dk = k.shape[-1]
    eye = np.eye(dk)
    # (I - beta k k^T), one dk x dk matrix per unit
    erase = eye[None, :, :] - beta[:, None, None] * (k[:, :, None] * k[:, None, :])
    # beta v k^T, one dv x dk matrix per unit
    write = beta[:, None, None] * (v[:, :, None] * k[:, None, :])
    S_new = g[:, None, None] * np.matmul(S, erase) + write
    o = np.matmul(S_new, q[:, :, None])[:, :, 0]
    return S_new, o


def verify_block(q, k, v, beta, g, state_in, store="f16", io="f16"):
    """Run a verify block of T draft tokens and keep one state checkpoint per position.

    The per-position checkpoints are the "recurrent-state pages" whose number
    grows with the verify width ("HyperQwen: 1,000 tok/s on a Single RTX 3090
    ...", Technical Insight: 1.66 GiB at 15 drafts vs 0.88 GiB at 7); the block is
    at most 16 tokens wide ("HyperQwen on one RTX 3090: a first-time developer's
    guide ...", What actually became faster?).

    S <- state_in; for t = 0..T-1: S, o_t = step(S, ...); ckpt[t] = S (rounded to
    ``store``); o[t] rounded to ``io``. The carried S is not rounded inside the
    block.

    Returns (o [N, T, H, dv], ckpt [N, T, H, dv, dk]) in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    N, T, H, dk = q.shape
    dv = np.asarray(v).shape[-1]
    S = np.asarray(state_in, dtype=np.float64).reshape(N * H, dv, dk).copy()
    o = np.zeros((N, T, H, dv))
    ckpt = np.zeros((N, T, H, dv, dk))
    for t in range(T):
        S, ot = gated_delta_step(
            S,
            q[:, t].reshape(N * H, dk),
            np.asarray(k, dtype=np.float64)[:, t].reshape(N * H, dk),
            np.asarray(v, dtype=np.float64)[:, t].reshape(N * H, dv),
            np.asarray(beta, dtype=np.float64)[:, t].reshape(N * H),
            np.asarray(g, dtype=np.float64)[:, t].reshape(N * H),
        )
        ckpt[:, t] = round_to(S.reshape(N, H, dv, dk), store)
        o[:, t] = round_to(ot.reshape(N, H, dv), io)
    return o, ckpt


def commit(state, ckpt, accepted_len):
    """Commit or roll back each state set to the accepted position.

    Follows the verify step of "Qwen3.8-27B on a Single RTX 3090: ..." (Technical
    Insight, split-KV verify): the accepted prefix is kept and the rejected
    drafts are discarded; for the recurrent state that means the request's state
    becomes the checkpoint after its a-th accepted token, or stays as it was
    when a == 0.

    state [N, H, dv, dk], ckpt [N, T, H, dv, dk], accepted_len [B] with N a
    multiple of B; state set n belongs to request n % B (sets laid out [L][B]).
    Returns the new state (a copy).
    """
    state = np.asarray(state, dtype=np.float64)
    ckpt = np.asarray(ckpt, dtype=np.float64)
    a = np.asarray(accepted_len).astype(np.int64)
    N = state.shape[0]
    B = a.shape[0]
    assert N % B == 0
    T = ckpt.shape[1]
    new = state.copy()
    for n in range(N):
        an = int(a[n % B])
        assert 0 <= an <= T
        if an > 0:
            new[n] = ckpt[n, an - 1]
    return new


def prefill_checkpoint(q, k, v, beta, g, state_in, chunk=64, store="f16", io="f16"):
    """Run a prompt of P tokens through the recurrence and checkpoint every chunk.

    Prefix caching of the recurrent state ("HyperQwen: 1,000 tok/s on a Single RTX
    3090 ...", Technical Insight: the DeltaNet state is checkpointed next to the
    attention context so a later turn resumes instead of recomputing; ~25,000-token
    document in "HyperQwen on one RTX 3090: a first-time developer's guide ...",
    What actually became faster?).

    The token-by-token definition: S <- state_in (zeros if None); for each token
    S, o_t = step(S, ...). After every full chunk the carried state is rounded to
    ``store`` and that value is both the checkpoint and the carry, so a run
    restored from a checkpoint continues exactly as the full run does. The tail
    after the last full chunk writes no checkpoint; S_final is the end state
    rounded to ``store``.

    q/k [N, P, H, dk], v [N, P, H, dv], beta/g [N, P, H], state_in [N, H, dv, dk]
    or None. Returns (o [N, P, H, dv], ckpt [N, P // chunk, H, dv, dk],
    S_final [N, H, dv, dk]) in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    N, P, H, dk = q.shape
    dv = v.shape[-1]
    if state_in is None:
        S = np.zeros((N * H, dv, dk))
    else:
        S = np.asarray(state_in, dtype=np.float64).reshape(N * H, dv, dk).copy()
    o = np.zeros((N, P, H, dv))
    ckpt = np.zeros((N, P // chunk, H, dv, dk))
    for t in range(P):
        S, ot = gated_delta_step(
            S,
            q[:, t].reshape(N * H, dk),
            k[:, t].reshape(N * H, dk),
            v[:, t].reshape(N * H, dv),
            beta[:, t].reshape(N * H),
            g[:, t].reshape(N * H),
        )
        o[:, t] = round_to(ot.reshape(N, H, dv), io)
        if (t + 1) % chunk == 0:
            S = round_to(S, store)
            ckpt[:, (t + 1) // chunk - 1] = S.reshape(N, H, dv, dk)
    S_final = round_to(S, store).reshape(N, H, dv, dk)
    return o, ckpt, S_final

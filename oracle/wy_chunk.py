"""Float64 chunked (WY / UT-transform) form of the gated delta rule.

TEST INFRASTRUCTURE ONLY. This is not the oracle of any entry point: the
prefill oracle is the token-by-token definition in ``recurrence.py``. This
module restates, in float64 and in the plainest matrix form, the algebra that
the chunked prefill kernel relies on, so a test can check that the algebra
equals the definition (to ~1e-10) independently of any CUDA code.

Derivation (gated delta rule, Yang et al. 2024, chunkwise form). Inside one
chunk of C tokens starting from state S0 (dv x dk), write
S_t = g_t S_{t-1} + delta_t k_t^T with delta_t = beta_t (v_t - g_t S_{t-1} k_t).
With G_t = sum_{s<=t} log g_s and gamma_t = exp(G_t):

    S_t = gamma_t S0 + sum_{s<=t} exp(G_t - G_s) delta_s k_s^T
    delta_t = beta_t (v_t - gamma_t S0 k_t - sum_{s<t} exp(G_t - G_s) (k_t . k_s) delta_s)

so, with rows indexed by token,

    A      = strictly-lower( diag(beta) [exp(G_t - G_s) k_t . k_s] )
    Delta  = (I + A)^{-1} diag(beta) (V - diag(gamma) K S0^T)
    O      = diag(gamma) Q S0^T + lower-incl-diag( [exp(G_t - G_s) q_t . k_s] ) Delta
    S_C    = gamma_C S0 + Delta^T diag(exp(G_C - G)) K
"""

import numpy as np


def chunk_forward(S0, q, k, v, beta, g):
    """One chunk for one unit. S0 [dv, dk], q/k [C, dk], v [C, dv], beta/g [C].

    Returns (O [C, dv], S_C [dv, dk]).
    """
    S0 = np.asarray(S0, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    G = np.cumsum(np.log(np.asarray(g, dtype=np.float64)))
    C = k.shape[0]
    decay = np.exp(G[:, None] - G[None, :])  # exp(G_t - G_s); used only where s <= t
    lower_strict = np.tril(np.ones((C, C)), -1)
    lower_incl = np.tril(np.ones((C, C)), 0)
    A = lower_strict * (beta[:, None] * decay * (k @ k.T))
    rhs = beta[:, None] * (v - np.exp(G)[:, None] * (k @ S0.T))
    Delta = np.linalg.solve(np.eye(C) + A, rhs)
    O = np.exp(G)[:, None] * (q @ S0.T) + (lower_incl * decay * (q @ k.T)) @ Delta
    S_C = np.exp(G[-1]) * S0 + Delta.T @ (np.exp(G[-1] - G)[:, None] * k)
    return O, S_C

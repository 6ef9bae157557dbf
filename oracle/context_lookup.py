"""Oracle for drafting from the request's own context (n-gram lookup).

TEST INFRASTRUCTURE ONLY (see the package docstring for who may import it).

The pages describe the mechanism only in words. "HyperQwen: 1,000 tok/s on a Single
RTX 3090 ..." (Technical Insight): in single-user mode the later positions of the
verify block (7 to 14) hold tokens copied out of the prompt and the text generated so
far rather than drafter proposals, since a model that quotes its input repeats it
token for token. "HyperQwen
on one RTX 3090: a first-time developer's guide ..." (What actually became faster?):
when the output starts copying from the input, a lookup proposes further tokens
straight from that context. Neither page says how the place to copy from is found.

Reading used here (the plainest one the pages support): the pattern is the last n
tokens of the context; find its latest earlier occurrence that still has at least one
token after it; the drafts are the (up to K) tokens that follow that occurrence. Try
n from n_max down to n_min and use the first n that has an occurrence. No occurrence
for any n: no drafts.
"""

import numpy as np
from numpy.lib.stride_tricks import sliding_window_view


def context_drafts_row(context, n_max, n_min, K):
    """One request. context: 1-D token ids (prompt then generated tokens).

    Returns (drafts list of length <= K, n used (0 if none), start index e of the drafts
    (-1 if none)).
    """
    c = np.asarray(context).astype(np.int64)
    L = c.shape[0]
    for n in range(n_max, n_min - 1, -1):
        if L - 1 < n:
            continue
        pattern = c[L - n:]
        # windows c[j : j + n] for j = 0 .. L-1-n: every one ends before the last token,
        # so at least one token follows it and the pattern itself is not among them
        win = sliding_window_view(c[:L - 1], n)
        hits = np.flatnonzero((win == pattern).all(axis=1))
        if hits.size:
            e = int(hits[-1]) + n
            return c[e:e + K].tolist(), n, e
    return [], 0, -1


def context_drafts(context, lengths, n_max, n_min, K):
    """context [N, Lmax] int, lengths [N] -> (drafts [N, K] int32 padded with -1,
    count [N] int32, match_len [N] int32). Row r uses context[r, :lengths[r]]."""
    context = np.asarray(context)
    N = context.shape[0]
    drafts = np.full((N, K), -1, dtype=np.int32)
    count = np.zeros((N,), dtype=np.int32)
    match = np.zeros((N,), dtype=np.int32)
    for r in range(N):
        d, n, _ = context_drafts_row(context[r, :int(lengths[r])], n_max, n_min, K)
        drafts[r, :len(d)] = d
        count[r] = len(d)
        match[r] = n
    return drafts, count, match

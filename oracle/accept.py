"""Oracle for greedy acceptance of a verify block.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may import it).

Greedy verification as "Qwen3.8-27B on a Single RTX 3090: ..." describes it
(Technical Insight, split-KV verify: the verifier's logits are compared with
the drafts and the accepted prefix is kept): the target token at each position
is the argmax of that position's logits row, and the accepted length is the
length of the longest prefix on which the drafts equal the targets.
"About 15 of 16" accepted on document reproduction is the figure of "HyperQwen
on one RTX 3090: a first-time developer's guide ...", What actually became
faster?.
"""

import numpy as np


def argmax_lowest(row):
    """Definition: min{ i : row[i] == max_j row[j] } (the lowest index on ties).

    Values compare as float64 numbers, so -0.0 and +0.0 are equal (a tie).
    """
    row = np.asarray(row, dtype=np.float64)
    m = row.max()
    return int(np.flatnonzero(row == m)[0])


def accept_greedy(logits, draft_ids):
    """logits [B, T, V], draft_ids [B, T] -> (target_ids [B, T] int32, accepted_len [B] int32).

    target[b, t] = argmax_lowest(logits[b, t]);
    accepted_len[b] = the first t with draft[b, t] != target[b, t], or T if none.
    """
    logits = np.asarray(logits, dtype=np.float64)
    draft = np.asarray(draft_ids).astype(np.int64)
    B, T, _ = logits.shape
    tgt = np.zeros((B, T), dtype=np.int32)
    acc = np.zeros((B,), dtype=np.int32)
    for b in range(B):
        for t in range(T):
            tgt[b, t] = argmax_lowest(logits[b, t])
        a = T
        for t in range(T):
            if draft[b, t] != tgt[b, t]:
                a = t
                break
        acc[b] = a
    return tgt, acc

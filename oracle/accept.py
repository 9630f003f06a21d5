"""Greedy acceptance of speculative draft trees -- TEST INFRASTRUCTURE
(the oracle of the library's accept step; only tests/ and bench.py's CPU
baseline may use it; it shares no code with the CUDA path).

The step after verification: each request's L_b draft nodes (node 0 the
root, the last token already accepted; parents[i] < i its parent, -1 for
the root; draft_tokens[i] the token node i proposes) carry the target
model's logits, one row per node, predicting the token that follows it.
Reading of the pages (FlashInfer issue #152: trees of Medusa / EAGLE drafts
are verified against the target model's outputs) with greedy decoding:

  * the root is accepted;
  * node i >= 1 is accepted iff its parent is accepted and the argmax of
    the parent's logits row equals draft_tokens[i];
  * argmax takes the first (smallest) index among equal maxima;
  * the accepted path is the root-to-node path of the deepest accepted
    node, the smallest node index among equally deep ones;
  * the bonus token is the argmax of that node's logits row (the token
    the target model emits after the accepted path).

Plain numpy: np.argmax (first occurrence of the maximum) and a loop over
nodes in index order.
"""
from __future__ import annotations

import numpy as np


def accept_greedy(logits, qo_indptr, draft_tokens, parents):
    """logits [total, V] (any real dtype, compared as stored), qo_indptr
    [B+1], draft_tokens [total] int, parents [total] int (local, -1 root).
    Returns (accept_len [B], paths: list of int arrays of local node ids,
    bonus [B], argmax [total])."""
    logits = np.asarray(logits)
    qo_indptr = np.asarray(qo_indptr, dtype=np.int64)
    draft_tokens = np.asarray(draft_tokens, dtype=np.int64)
    parents = np.asarray(parents, dtype=np.int64)
    total = int(qo_indptr[-1])
    am = np.argmax(logits[:total], axis=1) if total else np.zeros(0, np.int64)
    B = len(qo_indptr) - 1
    acc_len = np.zeros(B, np.int64)
    bonus = np.full(B, -1, np.int64)
    paths = []
    for b in range(B):
        o, L = int(qo_indptr[b]), int(qo_indptr[b + 1] - qo_indptr[b])
        if L == 0:
            paths.append(np.zeros(0, np.int64))
            continue
        acc = np.zeros(L, bool)
        depth = np.zeros(L, np.int64)
        for i in range(L):
            p = int(parents[o + i])
            if p < 0:
                acc[i] = True
                depth[i] = 0
            else:
                depth[i] = depth[p] + 1
                acc[i] = acc[p] and int(am[o + p]) == int(draft_tokens[o + i])
        best = 0
        for i in range(L):
            if acc[i] and depth[i] > depth[best]:
                best = i
        path = []
        j = best
        while j >= 0:
            path.append(j)
            j = int(parents[o + j])
        path = np.array(path[::-1], np.int64)
        paths.append(path)
        acc_len[b] = len(path)
        bonus[b] = int(am[o + best])
    return acc_len, paths, bonus, am

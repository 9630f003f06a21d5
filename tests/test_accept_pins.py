"""Pins of the greedy acceptance oracle (oracle/accept.py) against closed
forms and an independent brute force over every root path of the tree."""
import itertools

import numpy as np
import pytest

from oracle.accept import accept_greedy


def _chain(L):
    return np.array([-1] + list(range(L - 1)))


def test_chain_accepts_the_leading_matches():
    """A chain accepts 1 + the number of leading drafts that equal the
    argmax of the node before them, and emits the argmax after the last."""
    rng = np.random.default_rng(1)
    V = 50
    for L in (1, 2, 7):
        for k in range(L):           # first k drafts match, draft k+1 (if any) misses
            logits = rng.standard_normal((L, V))
            am = logits.argmax(axis=1)
            toks = rng.integers(0, V, L)
            for i in range(1, L):
                toks[i] = am[i - 1] if i <= k else (am[i - 1] + 1) % V
            n, paths, bonus, _ = accept_greedy(logits, [0, L], toks, _chain(L))
            assert n[0] == min(k, L - 1) + 1
            assert list(paths[0]) == list(range(n[0]))
            assert bonus[0] == am[n[0] - 1]


def test_argmax_ties_take_the_smallest_index():
    logits = np.zeros((2, 6))
    logits[0, [1, 4]] = 3.0           # tie between tokens 1 and 4
    logits[1, 2] = 1.0
    n, _, bonus, am = accept_greedy(logits, [0, 2], [9, 4], [-1, 0])
    assert am[0] == 1 and n[0] == 1 and bonus[0] == 1
    n, _, bonus, _ = accept_greedy(logits, [0, 2], [9, 1], [-1, 0])
    assert n[0] == 2 and bonus[0] == 2


def test_deepest_branch_wins_and_ties_take_the_smallest_node():
    # root 0 -> {1, 2}; 1 -> 3; 2 -> 4 -> 5
    parents = [-1, 0, 0, 1, 2, 4]
    V = 10
    logits = np.full((6, V), -1.0)
    for node, tok in ((0, 7), (1, 3), (2, 5), (3, 0), (4, 6), (5, 8)):
        logits[node, tok] = 1.0
    # drafts: 1 and 2 both propose 7 (both match the root's argmax)
    toks = [0, 7, 7, 3, 5, 6]
    n, paths, bonus, _ = accept_greedy(logits, [0, 6], toks, parents)
    assert list(paths[0]) == [0, 2, 4, 5] and bonus[0] == 8
    # cut the deep branch at node 5: 3 and 4 are equally deep -> node 3
    toks = [0, 7, 7, 3, 5, 1]
    n, paths, bonus, _ = accept_greedy(logits, [0, 6], toks, parents)
    assert list(paths[0]) == [0, 1, 3] and bonus[0] == 0


def _brute(logits, toks, parents):
    """Every node's root path; the longest whose every edge matches."""
    L = len(parents)
    am = [int(np.argmax(r)) for r in logits]
    best = (1, [0])
    for i in range(L):
        path, j = [], i
        while j >= 0:
            path.append(j)
            j = parents[j]
        path = path[::-1]
        if all(am[path[k - 1]] == toks[path[k]] for k in range(1, len(path))):
            if len(path) > best[0] or (len(path) == best[0] and path[-1] < best[1][-1]):
                best = (len(path), path)
    return best[0], best[1], am[best[1][-1]]


@pytest.mark.parametrize("seed", range(20))
def test_random_trees_match_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    B = 3
    lens = rng.integers(1, 12, B)
    indptr = np.concatenate([[0], np.cumsum(lens)])
    V = int(rng.integers(2, 9))
    logits = rng.integers(-3, 4, (indptr[-1], V)).astype(np.float32)   # many ties
    parents, toks = [], []
    for L in lens:
        par = [-1] + [int(rng.integers(0, i)) for i in range(1, L)]
        parents += par
        toks += [int(rng.integers(0, V)) for _ in range(L)]
    n, paths, bonus, _ = accept_greedy(logits, indptr, toks, parents)
    for b in range(B):
        o = indptr[b]
        L = lens[b]
        bn, bp, bb = _brute(logits[o:o + L], toks[o:o + L], parents[o:o + L])
        assert n[b] == bn and list(paths[b]) == bp and bonus[b] == bb


def test_empty_request():
    n, paths, bonus, _ = accept_greedy(np.zeros((2, 4)), [0, 0, 2], [0, 1], [-1, 0])
    assert n[0] == 0 and bonus[0] == -1 and len(paths[0]) == 0 and n[1] >= 1

"""GPU parity of the greedy acceptance step (verify_accept_greedy) with the
numpy oracle (oracle/accept.py): accepted lengths, paths, bonus tokens and
every row's argmax compared exactly (integer results; both sides compare
the same stored logits, first index among equal maxima)."""
import numpy as np
import pytest
import torch

import synthetic
from oracle.accept import accept_greedy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_gqa_gb300 as m
    return m


def _case(seed, lens, vocab, kind="tree", plant=0.7, ties=False, dtype=torch.bfloat16, pad=0):
    """Random trees (or chains) over `lens` nodes per request; logits N(0,1)
    (integers in [-2, 2] with ties=True); each draft token is the argmax of
    its parent's row with probability `plant` (so paths go deep), else a
    random token."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator().manual_seed(seed)
    total = int(sum(lens))
    if ties:
        lg = torch.randint(-2, 3, (total, vocab + pad), generator=gen).to(dtype)
    else:
        lg = torch.randn((total, vocab + pad), generator=gen).to(dtype)
    host = lg.float().numpy()[:, :vocab]
    am = host.argmax(axis=1)
    indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    parents, toks = [], []
    for b, L in enumerate(lens):
        if L == 0:
            continue
        o = int(indptr[b])
        par = [-1] + ([i - 1 for i in range(1, L)] if kind == "chain"
                      else [int(rng.integers(0, i)) for i in range(1, L)])
        parents += par
        toks.append(int(rng.integers(0, vocab)))
        for i in range(1, L):
            toks.append(int(am[o + par[i]]) if rng.random() < plant else int(rng.integers(0, vocab)))
    return lg, host, indptr, np.array(toks, np.int32), np.array(parents, np.int32)


def _check(va, lg, host, indptr, toks, parents):
    dev = "cuda"
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    acc, path, bonus, am = va.verify_accept_greedy(
        lg.to(dev)[:, :host.shape[1]] if lg.shape[1] == host.shape[1] else lg.to(dev)[:, :host.shape[1]],
        torch.from_numpy(indptr).to(dev), torch.from_numpy(toks).to(dev),
        torch.from_numpy(parents).to(dev), want_argmax=True, status=status)
    torch.cuda.synchronize()
    r_acc, r_paths, r_bonus, r_am = accept_greedy(host, indptr, toks, parents)
    assert int(status.item()) == 0
    assert np.array_equal(am.cpu().numpy(), r_am)
    assert np.array_equal(acc.cpu().numpy(), r_acc)
    assert np.array_equal(bonus.cpu().numpy(), r_bonus)
    p = path.cpu().numpy()
    for b in range(len(indptr) - 1):
        o = int(indptr[b])
        assert np.array_equal(p[o:o + int(r_acc[b])], r_paths[b])
    return r_acc


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("case", [
    dict(lens=[17], vocab=128256),                         # Llama-3 vocabulary, the 17-node tree
    dict(lens=[64] * 8, vocab=128256),                     # the wide tree's 8 x 64 nodes
    dict(lens=[1, 5, 8, 3, 2, 8, 7, 1] * 8, vocab=32016, kind="chain"),  # batched chains
    dict(lens=[9, 0, 4], vocab=1001),                      # odd vocabulary: scalar tails
    dict(lens=[12, 7], vocab=300, ties=True),              # integer logits: many equal maxima
    dict(lens=[5, 6], vocab=4000, pad=24),                 # rows longer than the vocabulary
], ids=["llama3_tree", "wide_tree", "chains", "odd_vocab", "ties", "padded_rows"])
def test_accept_matches_oracle(va, case, dtype):
    case = dict(case)
    lens = case.pop("lens")
    vocab = case.pop("vocab")
    lg, host, indptr, toks, parents = _case(7, lens, vocab, dtype=dtype, **case)
    r_acc = _check(va, lg, host, indptr, toks, parents)
    if len(lens) > 1 and case.get("kind") != "chain":
        assert r_acc.max() >= 3          # the planted matches reach deep


def test_accept_flags_malformed_trees(va):
    lg, host, indptr, toks, parents = _case(3, [5, 4], 64)
    bad = parents.copy()
    bad[5 + 2] = 3            # request 1: node 2's parent is a later node
    dev = "cuda"
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    acc, path, bonus, _ = va.verify_accept_greedy(
        lg.to(dev), torch.from_numpy(indptr).to(dev), torch.from_numpy(toks).to(dev),
        torch.from_numpy(bad).to(dev), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    assert int(acc[1]) == 0 and int(bonus[1]) == -1
    r_acc, _, r_bonus, _ = accept_greedy(host, indptr, toks, parents)
    assert int(acc[0]) == r_acc[0] and int(bonus[0]) == r_bonus[0]   # request 0 untouched

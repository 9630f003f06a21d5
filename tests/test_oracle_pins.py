"""Pins of the fp64 oracle against what the source pages and mathematics fix.

Each test names the identity it checks and where it comes from.  Chosen so
that a plausible slip in the oracle (a transposed mask bit, a wrong GQA head
map, a dropped scale, an off-by-one in the page walk, a wrong merge weight)
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run(wl, rows=None, caches=None):
    return oracle.verify_attn_workload(wl, rows=rows, caches=caches, nthreads=4)


def _gather(wl, kc, vc, b, h):
    """Test-side page walk (numpy indexing) giving request b's K, V of KV
    head h as fp64 [kv_len, d] (decoded, scaled)."""
    n = int(wl.kv_lens[b])
    P = wl.page_size
    pages = wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]]
    pos = np.arange(n)
    kb = kc[pages[pos // P], h, pos % P]
    vb = vc[pages[pos // P], h, pos % P]
    fp8 = wl.kv_dtype == synthetic.FP8
    dec = (lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e4m3fn)
           .double().numpy()) if fp8 else (
        lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.int16)
        .view(torch.bfloat16).double().numpy())
    return dec(kb) * wl.k_scale, dec(vb) * wl.v_scale


def _q(wl, tok, qh):
    return torch.from_numpy(wl.q[tok, qh].copy()).view(torch.int16).view(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- decoding

def test_bf16_decode_matches_torch_for_every_code(oracle_lib):
    codes = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.decode_bf16(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_matches_torch_for_every_code(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_landmarks(oracle_lib):
    # From the format definition (bias 7, 3 mantissa bits, no infinity).
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x3C: 1.5, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for code, val in cases.items():
        assert oracle.decode_e4m3(np.array([code], np.uint8))[0] == val
    assert math.isnan(oracle.decode_e4m3(np.array([0x7F], np.uint8))[0])
    assert math.isnan(oracle.decode_e4m3(np.array([0xFF], np.uint8))[0])


# ---------------------------------------------------------------- golden

def _golden_cases():
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        return json.load(f)["cases"]


def _expr(s):
    return float(eval(s, {"__builtins__": {}}, {"e": math.e, "ln": math.log, "exp": math.exp,
                                                 "inf": math.inf}))


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_worked_examples(oracle_lib, case):
    h_q, h_kv, d, P = case["h_q"], case["h_kv"], case["d"], case["page_size"]
    fp8 = case.get("kv_dtype") == "fp8_e4m3"
    num_pages = case["num_pages"]
    reqs = case["requests"]
    dt = np.uint8 if fp8 else np.uint16
    kc = np.full((num_pages, h_kv, P, d), 0xFF if fp8 else 0xFFFF, dtype=dt)
    vc = kc.copy()

    def bits(vals):
        t = torch.tensor(vals, dtype=torch.float32)
        if fp8:
            return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    kv_indptr, kv_indices, last, qo_indptr, qs, masks = [0], [], [], [0], [], []
    for r, pages in zip(reqs, case["pages"]):
        n = len(r["k"])
        kv_indices += pages
        kv_indptr.append(kv_indptr[-1] + len(pages))
        last.append(n - (len(pages) - 1) * P)
        for j in range(n):
            pg, slot = pages[j // P], j % P
            kc[pg, :, slot, :] = bits([r["k"][j]] * h_kv).reshape(h_kv, d)
            vc[pg, :, slot, :] = bits([r["v"][j]] * h_kv).reshape(h_kv, d)
        qo_indptr.append(qo_indptr[-1] + r["L"])
        qs.append(np.asarray(r["q"], dtype=np.float32).reshape(r["L"], h_q, d))
        masks.append(r["mask"])
    q = torch.from_numpy(np.concatenate(qs)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if any(m is not None for m in masks):
        packed, mask_indptr = synthetic.pack_masks([np.asarray(m, dtype=bool) for m in masks])
    else:
        packed, mask_indptr = None, None
    out, lse = oracle.verify_attn(q, kc, vc, fp8, np.array(kv_indptr), np.array(kv_indices),
                                  np.array(last), np.array(qo_indptr), packed, mask_indptr,
                                  h_q, h_kv, d, P, num_pages, case["sm_scale"],
                                  case.get("k_scale", 1.0), case.get("v_scale", 1.0))
    for ex in case["expect"]:
        row = ex["token"] * h_q + ex["head"]
        want_lse = _expr(ex["lse"])
        if math.isinf(want_lse):
            assert lse[row] == want_lse
        else:
            assert abs(lse[row] - want_lse) < 1e-12
        for e, s in enumerate(ex["out"]):
            assert abs(out[row, e] - _expr(s)) < 1e-12


# ---------------------------------------------------------------- brute force

TINY = [
    dict(batch=3, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [0, 5, 9]),
         qo=("fixed", [3, 1, 5]), mask="causal"),
    dict(batch=2, h_q=4, h_kv=1, d=16, page_size=4, prefix=("fixed", [7, 12]),
         qo=("fixed", [5, 4]), mask="tree"),
    dict(batch=2, h_q=2, h_kv=2, d=8, page_size=1, prefix=("fixed", [3, 0]),
         qo=("fixed", [4, 5]), mask="random"),
    dict(batch=2, h_q=6, h_kv=3, d=8, page_size=16, prefix=("fixed", [20, 1]),
         qo=("fixed", [2, 3]), mask="tree", kv_dtype=synthetic.FP8),
    dict(batch=1, h_q=2, h_kv=1, d=8, page_size=2, prefix=("fixed", [0]),
         qo=("fixed", [4]), mask="none_visible"),
]


@pytest.mark.parametrize("spec", TINY, ids=range(len(TINY)))
def test_matches_scalar_brute_force(oracle_lib, spec):
    wl = synthetic.make_custom(seed=3, **spec)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    bout, blse = brute.verify_attn(wl.q, kc, vc, wl.kv_dtype == synthetic.FP8, wl.kv_indptr,
                                   wl.kv_indices, wl.last_page_len, wl.qo_indptr, wl.mask,
                                   wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                   wl.sm_scale, wl.k_scale, wl.v_scale)
    fin = np.isfinite(blse)
    assert (np.isfinite(lse) == fin).all()
    assert np.all(lse[~fin] == -np.inf)
    np.testing.assert_allclose(lse[fin], blse[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(out, bout, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- identities

def _triu_ninf(n_rows, n_cols, offset):
    """-inf strictly above the (offset-shifted) diagonal, 0 elsewhere."""
    i = np.arange(n_rows)[:, None]
    j = np.arange(n_cols)[None, :]
    return np.where(j > i + offset, -np.inf, 0.0)


def test_triu_ninf_mask_equals_causal(oracle_lib):
    """FlashInfer issue #152: a triu -inf mask (0 elsewhere) equals causal=True."""
    wl = synthetic.make_custom(batch=1, h_q=2, h_kv=1, d=16, page_size=4,
                               prefix=("fixed", [0]), qo=("fixed", [9]), mask="causal", seed=5)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    K, V = _gather(wl, kc, vc, 0, 0)
    for qh in range(wl.h_q):
        Q = np.stack([_q(wl, t, qh) for t in range(9)])
        o2, l2 = oracle.dense_attention(Q, K, V, _triu_ninf(9, 9, 0), wl.sm_scale)
        rows = np.arange(9) * wl.h_q + qh
        np.testing.assert_allclose(out[rows], o2, atol=1e-13, rtol=0)
        np.testing.assert_allclose(lse[rows], l2, atol=1e-13, rtol=0)


def test_minus_5e4_mask_equals_ninf(oracle_lib):
    """FlashInfer issue #152: -5e4 (or -inf) where masked, 0 elsewhere."""
    rng = np.random.default_rng(0)
    Q, K, V = rng.normal(size=(7, 16)), rng.normal(size=(11, 16)), rng.normal(size=(11, 16))
    keep = rng.random((7, 11)) < 0.6
    keep[:, 0] = True
    o1, l1 = oracle.dense_attention(Q, K, V, np.where(keep, 0.0, -np.inf), 0.25)
    o2, l2 = oracle.dense_attention(Q, K, V, np.where(keep, 0.0, -5e4), 0.25)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_allclose(l1, l2, atol=1e-15, rtol=0)


def test_gqa_equals_mha_on_expanded_kv(oracle_lib):
    """vLLM PR #2401: GQA equals MHA with K/V expanded (stride 0) per query head."""
    wl = synthetic.make_custom(batch=2, h_q=6, h_kv=2, d=8, page_size=4,
                               prefix=("fixed", [6, 10]), qo=("fixed", [3, 4]), mask="tree",
                               seed=7)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    G = wl.group
    kx = np.repeat(kc, G, axis=1)   # head h*G + g <- KV head h
    vx = np.repeat(vc, G, axis=1)
    o2, l2 = oracle.verify_attn(wl.q, kx, vx, False, wl.kv_indptr, wl.kv_indices,
                                wl.last_page_len, wl.qo_indptr, wl.mask, wl.mask_indptr,
                                wl.h_q, wl.h_q, wl.d, wl.page_size, wl.num_pages, wl.sm_scale)
    np.testing.assert_array_equal(out, o2)
    np.testing.assert_array_equal(lse, l2)
    # and a wrong head map (h = qh % h_kv) would differ
    kw = np.concatenate([kc] * G, axis=1)
    vw = np.concatenate([vc] * G, axis=1)
    o3, _ = oracle.verify_attn(wl.q, kw, vw, False, wl.kv_indptr, wl.kv_indices,
                               wl.last_page_len, wl.qo_indptr, wl.mask, wl.mask_indptr,
                               wl.h_q, wl.h_q, wl.d, wl.page_size, wl.num_pages, wl.sm_scale)
    assert np.abs(o3 - out).max() > 1e-3


def test_split_partials_merged_by_lse_equal_unsplit(oracle_lib):
    """flashmap verify_attention.py: splits of the key range merged by their
    log-sum-exp give the unsplit result (including empty / fully masked splits)."""
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=8, page_size=4,
                               prefix=("fixed", [13, 22]), qo=("fixed", [4, 6]), mask="tree",
                               seed=11)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    rng = np.random.default_rng(1)
    kvf = wl.kv_dtype == synthetic.FP8
    for b in range(wl.batch):
        n = int(wl.kv_lens[b])
        for t in range(int(wl.qo_lens[b])):
            for qh in range(wl.h_q):
                cuts = sorted(set([0, n] + list(rng.integers(0, n + 1, size=3))))
                outs, lses = [], []
                for lo, hi in zip(cuts[:-1], cuts[1:]):
                    o, l = oracle.attn_range(wl.q, kc, vc, kvf, wl.kv_indptr, wl.kv_indices,
                                             wl.last_page_len, wl.qo_indptr, wl.mask,
                                             wl.mask_indptr, wl.h_q, wl.h_kv, wl.d,
                                             wl.page_size, wl.num_pages, wl.sm_scale,
                                             wl.k_scale, wl.v_scale, b, t, qh, lo, hi)
                    outs.append(o[None]); lses.append([l])
                # an empty split (lse -inf) must carry no mass
                outs.append(np.full((1, wl.d), 123.0)); lses.append([-np.inf])
                mo, ml = oracle.merge_partials(np.stack(outs), np.array(lses))
                row = (int(wl.qo_indptr[b]) + t) * wl.h_q + qh
                np.testing.assert_allclose(mo[0], out[row], atol=1e-12, rtol=0)
                assert abs(ml[0] - lse[row]) < 1e-12


def test_merge_all_empty_gives_zero_and_ninf(oracle_lib):
    mo, ml = oracle.merge_partials(np.ones((3, 2, 4)), np.full((3, 2), -np.inf))
    assert np.all(mo == 0) and np.all(ml == -np.inf)


def test_merge_weights_closed_form(oracle_lib):
    # two parts with lse ln 1 and ln 3: weights 1/4 and 3/4
    outs = np.array([[[4.0, 0.0]], [[0.0, 8.0]]])
    lses = np.array([[0.0], [math.log(3.0)]])
    mo, ml = oracle.merge_partials(outs, lses)
    np.testing.assert_allclose(mo[0], [1.0, 6.0], atol=1e-14)
    assert abs(ml[0] - math.log(4.0)) < 1e-14


def test_single_token_equals_decode(oracle_lib):
    """L = 1 verify is plain single-query decode over every cached key."""
    wl = synthetic.make_custom(batch=3, h_q=4, h_kv=2, d=16, page_size=4,
                               prefix=("fixed", [0, 9, 30]), qo=("fixed", [1, 1, 1]),
                               mask="causal", seed=13)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    for b in range(wl.batch):
        for qh in range(wl.h_q):
            K, V = _gather(wl, kc, vc, b, qh // wl.group)
            tok = int(wl.qo_indptr[b])
            o, l = oracle.dense_attention(_q(wl, tok, qh)[None], K, V,
                                          np.zeros((1, len(K))), wl.sm_scale)
            np.testing.assert_allclose(out[tok * wl.h_q + qh], o[0], atol=1e-13, rtol=0)
            assert abs(lse[tok * wl.h_q + qh] - l[0]) < 1e-13


def test_chain_equals_decodes_at_growing_context(oracle_lib):
    """vLLM PR #1679: a causal chain of L drafts equals L single-query decodes
    with context lengths prefix+1 ... prefix+L."""
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=8, page_size=4,
                               prefix=("fixed", [5, 17]), qo=("fixed", [6, 3]), mask="causal",
                               seed=17)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    for b in range(wl.batch):
        prefix = int(wl.prefix_lens[b])
        for t in range(int(wl.qo_lens[b])):
            tok = int(wl.qo_indptr[b]) + t
            for qh in range(wl.h_q):
                K, V = _gather(wl, kc, vc, b, qh // wl.group)
                n = prefix + t + 1
                o, l = oracle.dense_attention(_q(wl, tok, qh)[None], K[:n], V[:n],
                                              np.zeros((1, n)), wl.sm_scale)
                np.testing.assert_allclose(out[tok * wl.h_q + qh], o[0], atol=1e-13, rtol=0)
                assert abs(lse[tok * wl.h_q + qh] - l[0]) < 1e-13


def test_tree_row_equals_decode_over_root_path(oracle_lib):
    """FlashInfer issue #152: tree node i attends to the prefix and its
    root-to-i path -- the same as one draft sequence decoded as its own request."""
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=8, page_size=4,
                               prefix=("fixed", [9, 4]), qo=("fixed", [7, 6]), mask="tree",
                               seed=19)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    for b in range(wl.batch):
        prefix = int(wl.prefix_lens[b])
        par = wl.parents[b]
        for i in range(int(wl.qo_lens[b])):
            path, j = [], i
            while j >= 0:
                path.append(j)
                j = par[j]
            keys = list(range(prefix)) + [prefix + u for u in sorted(path)]
            tok = int(wl.qo_indptr[b]) + i
            for qh in range(wl.h_q):
                K, V = _gather(wl, kc, vc, b, qh // wl.group)
                o, l = oracle.dense_attention(_q(wl, tok, qh)[None], K[keys], V[keys],
                                              np.zeros((1, len(keys))), wl.sm_scale)
                np.testing.assert_allclose(out[tok * wl.h_q + qh], o[0], atol=1e-13, rtol=0)
                assert abs(lse[tok * wl.h_q + qh] - l[0]) < 1e-13


def test_chain_tree_mask_equals_causal(oracle_lib):
    """A chain tree's ancestor mask is the causal mask."""
    base = dict(batch=2, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [6, 0]),
                qo=("fixed", [5, 7]), seed=23)
    wc = synthetic.make_custom(mask="chain", **base)
    wn = synthetic.make_custom(mask="causal", **base)
    assert np.array_equal(wc.q, wn.q) and np.array_equal(wc.k_tok, wn.k_tok)
    o1, l1 = _run(wc)
    o2, l2 = _run(wn)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------- closed forms

def _const_workload(kv_len, L, d=8, P=4, seed=29):
    return synthetic.make_custom(batch=1, h_q=2, h_kv=1, d=d, page_size=P,
                                 prefix=("fixed", [kv_len - L]), qo=("fixed", [L]),
                                 mask="causal", seed=seed)


def test_identical_keys_give_uniform_weights(oracle_lib):
    wl = _const_workload(kv_len=13, L=4)
    kc, vc = oracle.build_cache(wl)
    pages = wl.kv_indices
    for j in range(13):
        kc[pages[j // 4], 0, j % 4] = kc[pages[0], 0, 0]
    out, lse = _run(wl, caches=(kc, vc))
    K, V = _gather(wl, kc, vc, 0, 0)
    for t in range(4):
        n = 9 + t + 1
        for qh in range(2):
            s = wl.sm_scale * float(_q(wl, t, qh) @ K[0])
            row = t * 2 + qh
            np.testing.assert_allclose(out[row], V[:n].mean(axis=0), atol=1e-13)
            assert abs(lse[row] - (s + math.log(n))) < 1e-12


def test_one_hot_values_give_weight_mass(oracle_lib):
    wl = _const_workload(kv_len=8, L=1, d=8)
    kc, vc = oracle.build_cache(wl)
    one = torch.tensor(1.0, dtype=torch.bfloat16).view(torch.int16).item() & 0xFFFF
    vc[...] = 0
    pages = wl.kv_indices
    for j in range(8):
        vc[pages[j // 4], 0, j % 4, j] = one          # v_j = e_j
    out, lse = _run(wl, caches=(kc, vc))
    K, _ = _gather(wl, kc, vc, 0, 0)
    for qh in range(2):
        s = wl.sm_scale * (K @ _q(wl, 0, qh))
        w = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
        np.testing.assert_allclose(out[qh], w, atol=1e-14)


def test_single_key_returns_its_value(oracle_lib):
    wl = _const_workload(kv_len=1, L=1)
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    K, V = _gather(wl, kc, vc, 0, 0)
    for qh in range(2):
        np.testing.assert_array_equal(out[qh], V[0])
        assert abs(lse[qh] - wl.sm_scale * float(_q(wl, 0, qh) @ K[0])) < 1e-14


# ---------------------------------------------------------------- paging

def test_page_permutation_invariance(oracle_lib):
    base = dict(batch=3, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [9, 0, 14]),
                qo=("fixed", [3, 5, 2]), mask="tree", seed=31)
    w1 = synthetic.make_custom(shuffle_pages=True, **base)
    w2 = synthetic.make_custom(shuffle_pages=False, **base)
    assert not np.array_equal(w1.kv_indices, w2.kv_indices)
    o1, l1 = _run(w1)
    o2, l2 = _run(w2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_append_scatter_is_exact_and_touches_nothing_else(oracle_lib):
    for kvd in (synthetic.BF16, synthetic.FP8):
        wl = synthetic.make_custom(batch=3, h_q=4, h_kv=2, d=8, page_size=4,
                                   prefix=("fixed", [5, 0, 8]), qo=("fixed", [3, 2, 4]),
                                   kv_dtype=kvd, seed=37)
        kc, vc = oracle.build_cache(wl)
        sentinel = synthetic.sentinel_pool(wl)
        written = np.zeros(kc.shape[:3], dtype=bool)
        for b in range(wl.batch):
            pages = wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]]
            for j in range(int(wl.kv_lens[b])):
                tok = int(wl.tok_indptr[b]) + j
                pg, slot = pages[j // 4], j % 4
                assert np.array_equal(kc[pg, :, slot], wl.k_tok[tok])
                assert np.array_equal(vc[pg, :, slot], wl.v_tok[tok])
                written[pg, :, slot] = True
        assert np.array_equal(kc[~written], sentinel[~written])
        assert np.array_equal(vc[~written], sentinel[~written])


def test_append_of_drafts_lands_at_the_last_positions(oracle_lib):
    wl = synthetic.make_custom(batch=2, h_q=2, h_kv=1, d=8, page_size=4,
                               prefix=("fixed", [6, 3]), qo=("fixed", [3, 2]), seed=41)
    kc = synthetic.sentinel_pool(wl)
    vc = synthetic.sentinel_pool(wl)
    kn, vn = wl.new_tokens()
    oracle.paged_kv_append(kn, vn, wl.qo_indptr, wl.kv_indptr, wl.kv_indices, wl.last_page_len,
                           wl.page_size, wl.num_pages, kc, vc)
    for b in range(wl.batch):
        pages = wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]]
        pre = int(wl.prefix_lens[b])
        for i in range(int(wl.qo_lens[b])):
            pos = pre + i
            assert np.array_equal(kc[pages[pos // 4], :, pos % 4], kn[wl.qo_indptr[b] + i])
        for pos in range(pre):
            assert np.all(kc[pages[pos // 4], :, pos % 4] == 0xFFFF)


def test_rejects_bad_page_table(oracle_lib):
    wl = synthetic.make_custom(batch=1, h_q=2, h_kv=1, d=8, page_size=4,
                               prefix=("fixed", [5]), qo=("fixed", [2]), seed=43)
    kc, vc = oracle.build_cache(wl)
    bad = wl.kv_indices.copy()
    bad[0] = wl.num_pages
    with pytest.raises(ValueError):
        oracle.verify_attn(wl.q, kc, vc, False, wl.kv_indptr, bad, wl.last_page_len,
                           wl.qo_indptr, None, None, 2, 1, 8, 4, wl.num_pages, wl.sm_scale)


def test_selected_rows_match_full_run(oracle_lib):
    wl = synthetic.make_workload("tiny_verify")
    kc, vc = oracle.build_cache(wl)
    out, lse = _run(wl, caches=(kc, vc))
    rows = synthetic.sample_rows(wl, 7)
    o2, l2 = _run(wl, rows=rows, caches=(kc, vc))
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(l2, lse[rows])


def test_tiny_verify_workload_shape():
    """The tiny verify case: kv lengths 42 and 75 (37 + 5, 70 + 5), 3 and 5
    pages of 16 in a shuffled 16-page pool, last pages holding 10 and 11."""
    wl = synthetic.make_workload("tiny_verify")
    assert list(wl.kv_lens) == [42, 75]
    assert list(np.diff(wl.kv_indptr)) == [3, 5]
    assert list(wl.last_page_len) == [10, 11]
    assert wl.num_pages == 16 and len(set(wl.kv_indices.tolist())) == 8
    assert wl.sm_scale == 0.125 and wl.mask is None


def test_tree_masks_are_ancestor_sets():
    wl = synthetic.make_custom(batch=2, h_q=2, h_kv=1, d=8, page_size=4,
                               prefix=("fixed", [3, 3]), qo=("fixed", [9, 17]), mask="tree",
                               seed=47)
    bits = np.unpackbits(wl.mask, bitorder="little")
    for b in range(2):
        L = int(wl.qo_lens[b])
        m = bits[wl.mask_indptr[b]:wl.mask_indptr[b] + L * L].reshape(L, L).astype(bool)
        par = wl.parents[b]
        assert par[0] == -1 and all(0 <= par[i] < i for i in range(1, L))
        for i in range(L):
            anc = set()
            j = i
            while j >= 0:
                anc.add(j)
                j = par[j]
            assert set(np.nonzero(m[i])[0].tolist()) == anc
        assert not np.triu(m, 1).any()

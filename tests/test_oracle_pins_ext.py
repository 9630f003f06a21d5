"""Pins of the oracle's extensions against what the pages and mathematics fix:
the fp8-e4m3 quantiser of the quantising append (FlashInfer PR #286's fp8
cache with a per-tensor scale), the bf16 rounding of rotated keys, the rotary
position embedding (FlashInfer PR #286's ROPE_LLAMA; FlashInfer issue #152:
tree drafts need it at their tree positions), the NHD cache layout
(FlashInfer PR #286's kv_layout) and the full-prefix custom-mask layout
(flashmap's L x (prefix + L) mask).  Each test names the identity it checks;
each is chosen so that a plausible slip (a wrong rounding direction, a sign
or pairing error in the rotation, a transposed layout, a mask bit read from
the wrong row) fails it."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic
from oracle import brute


# ---------------------------------------------------------------- e4m3 quantiser

def _e4m3_values():
    codes = np.arange(256, dtype=np.uint8)
    return codes, oracle.decode_e4m3(codes)


def test_e4m3_encode_inverts_decode_on_every_finite_code(oracle_lib):
    codes, vals = _e4m3_values()
    finite = ~np.isnan(vals)
    enc = oracle.encode_e4m3_satfinite(vals[finite].astype(np.float32))
    assert np.array_equal(enc, codes[finite])


def test_e4m3_encode_matches_torch_cast_on_every_bf16_code(oracle_lib):
    """For every bf16 input x and three per-tensor scales, the stored code of
    the correctly rounded binary32 quotient x / scale equals torch's
    float8_e4m3fn cast of the same binary32 quotient, wherever torch does not
    overflow (|q| <= 448; torch turns larger values into NaN, the
    saturating reading clamps them to +-448)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float()
    for scale in (1.0, float(np.float32(0.0123)), 7.5):
        q = (x / np.float32(scale)).numpy()        # IEEE binary32 division
        ok = np.isfinite(q) & (np.abs(q) <= 448.0)
        want = torch.from_numpy(q[ok]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = oracle.encode_e4m3_satfinite(q[ok])
        assert np.array_equal(got, want), scale
        # the quotient rule itself: binary32 division, correctly rounded
        xs = x.numpy()[::97]
        qs = np.array([oracle.div_f32(v, scale) for v in xs], dtype=np.float32)
        with np.errstate(all="ignore"):
            np.testing.assert_array_equal(qs, (xs / np.float32(scale)).astype(np.float32))


def test_e4m3_saturation_nan_and_ties(oracle_lib):
    enc = oracle.encode_e4m3_satfinite
    assert list(enc(np.array([448.0, 449.0, 464.0, 465.0, 1e30, np.inf], np.float32))) == [0x7E] * 6
    assert list(enc(np.array([-448.0, -500.0, -np.inf], np.float32))) == [0xFE] * 3
    assert enc(np.array([np.nan], np.float32))[0] == 0x7F
    # ties go to the even code: 1.0625 between 1.0 (0x38) and 1.125 (0x39),
    # 1.1875 between 1.125 and 1.25 (0x3A); subnormal 1.5 * 2^-9 between codes 1 and 2
    assert list(enc(np.array([1.0625, 1.1875, 1.5 * 2 ** -9, 2.5 * 2 ** -9], np.float32))) == \
        [0x38, 0x3A, 0x02, 0x02]
    # just off a tie goes to the nearer code
    assert enc(np.array([np.nextafter(np.float32(1.0625), np.float32(2))], np.float32))[0] == 0x39


def test_e4m3_encode_is_nearest(oracle_lib):
    """Brute force: for random binary32 values in range, no code is nearer
    than the chosen one."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4000) * np.exp2(rng.integers(-10, 8, 4000))).astype(np.float32)
    x = x[np.abs(x) <= 448]
    codes, vals = _e4m3_values()
    fin = ~np.isnan(vals)
    enc = oracle.encode_e4m3_satfinite(x)
    got = oracle.decode_e4m3(enc)
    best = np.abs(vals[fin][None, :] - x[:, None].astype(np.float64)).min(axis=1)
    np.testing.assert_array_equal(np.abs(got - x), best)


def test_quantising_append_matches_torch_at_the_right_slots(oracle_lib):
    """oracle_paged_kv_append_quant (and the extended append with quantize):
    every new row lands at its slot as torch's e4m3 cast of x / scale, and
    no other byte of the pool changes."""
    wl = synthetic.make_custom(batch=3, h_q=4, h_kv=2, d=16, page_size=4,
                               prefix=("fixed", [5, 0, 9]), qo=("fixed", [3, 4, 2]), seed=61)
    kn, vn = wl.new_tokens()            # bf16 bits
    pool = dict(kv_dtype=synthetic.FP8)
    wf = synthetic.make_custom(batch=3, h_q=4, h_kv=2, d=16, page_size=4,
                               prefix=("fixed", [5, 0, 9]), qo=("fixed", [3, 4, 2]), seed=61,
                               **pool)
    ks, vs = float(np.float32(0.021)), float(np.float32(0.0173))
    for variant in ("quant", "ex"):
        kc = synthetic.sentinel_pool(wf)
        vc = synthetic.sentinel_pool(wf)
        if variant == "quant":
            oracle.paged_kv_append_quant(kn, vn, ks, vs, wl.qo_indptr, wl.kv_indptr,
                                         wl.kv_indices, wl.last_page_len, wl.page_size,
                                         wl.num_pages, kc, vc)
        else:
            oracle.paged_kv_append_ex(kn, vn, wl.qo_indptr, wl.kv_indptr, wl.kv_indices,
                                      wl.last_page_len, wl.page_size, wl.num_pages, kc, vc,
                                      cache_fp8=True, quantize=True, k_scale=ks, v_scale=vs)
        written = np.zeros(kc.shape[:3], dtype=bool)
        for b in range(wl.batch):
            pages = wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]]
            for i in range(int(wl.qo_lens[b])):
                pos = int(wl.prefix_lens[b]) + i
                tok = int(wl.qo_indptr[b]) + i
                for arr, src, sc in ((kc, kn, ks), (vc, vn, vs)):
                    x = torch.from_numpy(src[tok].view(np.int16)).view(torch.bfloat16).float()
                    want = (x / np.float32(sc)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    assert np.array_equal(arr[pages[pos // 4], :, pos % 4], want)
                written[pages[pos // 4], :, pos % 4] = True
        assert np.all(kc[~written] == 0xFF) and np.all(vc[~written] == 0xFF)


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_encode_inverts_decode_and_is_nearest_even(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = oracle.decode_bf16(bits)
    fin = np.isfinite(vals)
    assert np.array_equal(oracle.encode_bf16(vals[fin]), bits[fin])
    # nearest: random doubles against their two bracketing bf16 values
    rng = np.random.default_rng(7)
    x = rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, 3000))
    enc = oracle.encode_bf16(x)
    got = oracle.decode_bf16(enc)
    up = oracle.decode_bf16((enc.astype(np.int32) + 1).astype(np.uint16))
    dn = oracle.decode_bf16((enc.astype(np.int32) - 1).astype(np.uint16))
    err = np.abs(got - x)
    assert np.all(err <= np.abs(up - x)) and np.all(err <= np.abs(dn - x))
    # ties to even: 1 + 2^-8 (between 1 and 1 + 2^-7) -> 1; 1 + 3 * 2^-8 -> 1 + 2^-6
    assert list(oracle.encode_bf16(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)]))) == \
        [0x3F80, 0x3F82, 0xBF80]


# ---------------------------------------------------------------- RoPE

def test_rope_is_the_complex_rotation(oracle_lib):
    """Pair (x_i, x_{i+d/2}) as the complex number x_i + j x_{i+d/2},
    multiplied by exp(j * pos / scale * theta^(-2i/d)) (numpy complex
    arithmetic, a library routine)."""
    rng = np.random.default_rng(3)
    for d, pos, theta, scale in ((8, 5, 10000.0, 1.0), (128, 4113, 500000.0, 1.0),
                                 (64, 32831, 10000.0, 4.0), (2, 1, 10000.0, 1.0)):
        x = rng.standard_normal(d)
        h = d // 2
        z = (x[:h] + 1j * x[h:]) * np.exp(1j * pos / scale * theta ** (-2.0 * np.arange(h) / d))
        want = np.concatenate([z.real, z.imag])
        np.testing.assert_allclose(oracle.rope(x, pos, theta, scale), want, atol=1e-9, rtol=0)
    # d = 2, position 1, theta irrelevant (frequency theta^0 = 1): a 1-radian turn
    np.testing.assert_allclose(oracle.rope([1.0, 0.0], 1, 10000.0), [math.cos(1), math.sin(1)],
                               atol=1e-15)


def test_rope_group_and_relative_position(oracle_lib):
    """R(0) = I, |R(p) x| = |x|, R(a) R(b) = R(a + b), and the score of a
    rotated query and key depends only on their position difference."""
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    th = 10000.0
    np.testing.assert_array_equal(oracle.rope(q, 0, th), q)
    assert abs(np.linalg.norm(oracle.rope(q, 777, th)) - np.linalg.norm(q)) < 1e-12
    np.testing.assert_allclose(oracle.rope(oracle.rope(q, 300, th), 45, th),
                               oracle.rope(q, 345, th), atol=1e-11)
    s0 = oracle.rope(q, 1000, th) @ oracle.rope(k, 990, th)
    for c in (-500, 7, 20000):
        s1 = oracle.rope(q, 1000 + c, th) @ oracle.rope(k, 990 + c, th)
        assert abs(s1 - s0) < 1e-9


def test_rope_append_rounds_the_rotated_key_to_nearest(oracle_lib):
    """The extended append with positions stores, for each new K row, the
    cache-dtype value nearest to the fp64 rotation of the row (bf16), or the
    e4m3 nearest to it over the scale (quantising); V is stored unrotated."""
    for kvd, quant in ((synthetic.BF16, False), (synthetic.FP8, True)):
        wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=16, page_size=4,
                                   prefix=("fixed", [5, 2]), qo=("fixed", [3, 4]), mask="tree",
                                   seed=67, rope_theta=10000.0)
        wb = wl
        kn, vn = wb.new_tokens()          # bf16 bits
        pos = wb.new_positions()
        fp8 = kvd == synthetic.FP8
        wf = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=16, page_size=4,
                                   prefix=("fixed", [5, 2]), qo=("fixed", [3, 4]), mask="tree",
                                   seed=67, rope_theta=10000.0, kv_dtype=kvd)
        kc = synthetic.sentinel_pool(wf)
        vc = synthetic.sentinel_pool(wf)
        ks = vs = float(np.float32(0.01))
        oracle.paged_kv_append_ex(kn, vn, wb.qo_indptr, wb.kv_indptr, wb.kv_indices,
                                  wb.last_page_len, 4, wb.num_pages, kc, vc, cache_fp8=fp8,
                                  quantize=quant, k_scale=ks, v_scale=vs, positions=pos,
                                  rope_theta=10000.0)
        codes = np.arange(256, dtype=np.uint8)
        grid = oracle.decode_e4m3(codes)
        for b in range(wb.batch):
            pages = wb.kv_indices[wb.kv_indptr[b]:wb.kv_indptr[b + 1]]
            for i in range(int(wb.qo_lens[b])):
                p_ = int(wb.prefix_lens[b]) + i
                tok = int(wb.qo_indptr[b]) + i
                for h in range(2):
                    x = oracle.decode_bf16(kn[tok, h])
                    z = oracle.rope(x, int(pos[tok]), 10000.0)
                    got_k = kc[pages[p_ // 4], h, p_ % 4]
                    if fp8:
                        target = z / ks
                        dist = np.abs(grid[None, ~np.isnan(grid)] - target[:, None]).min(axis=1)
                        np.testing.assert_array_equal(
                            np.abs(oracle.decode_e4m3(got_k) - target), dist)
                        want_v = oracle.encode_e4m3_satfinite(
                            np.array([oracle.div_f32(v, vs) for v in oracle.decode_bf16(vn[tok, h])],
                                     np.float32))
                    else:
                        got = oracle.decode_bf16(got_k)
                        ulp = np.exp2(np.floor(np.log2(np.abs(z))) - 7)
                        assert np.all(np.abs(got - z) <= ulp / 2)
                        want_v = vn[tok, h]
                    assert np.array_equal(vc[pages[p_ // 4], h, p_ % 4], want_v)


def _rope_workload(**kw):
    base = dict(batch=2, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [9, 4]),
                qo=("fixed", [7, 6]), mask="tree", seed=19, rope_theta=10000.0)
    base.update(kw)
    return synthetic.make_custom(**base)


def test_rope_tree_positions_are_depths(oracle_lib):
    wl = _rope_workload()
    for b in range(wl.batch):
        pre = int(wl.prefix_lens[b])
        t0 = int(wl.tok_indptr[b])
        assert list(wl.kv_pos[t0:t0 + pre]) == list(range(pre))
        for u, par in enumerate(wl.parents[b]):
            want = pre if par < 0 else int(wl.kv_pos[t0 + pre + par]) + 1
            assert wl.kv_pos[t0 + pre + u] == want
            assert wl.q_pos[int(wl.qo_indptr[b]) + u] == want


def test_rope_tree_row_equals_decode_over_its_rotated_root_path(oracle_lib):
    """FlashInfer issue #152: with rotary positions, tree node i (position
    prefix + depth(i)) attends to the prefix and its root-to-i path, whose
    positions are then contiguous -- the same as that path decoded as one
    ordinary sequence: a new request holding the prefix and the path with
    the same key / value rows, positions 0 .. prefix + depth(i)."""
    wl = _rope_workload()
    kc, vc = oracle.build_cache(wl)
    out, lse = oracle.verify_attn_workload(wl, caches=(kc, vc), nthreads=2)
    for b in range(wl.batch):
        pre = int(wl.prefix_lens[b])
        par = wl.parents[b]
        t0 = int(wl.tok_indptr[b])
        for i in range(int(wl.qo_lens[b])):
            path, j = [], i
            while j >= 0:
                path.append(j)
                j = par[j]
            keys = list(range(pre)) + [pre + u for u in sorted(path)]
            n = len(keys)
            # a one-request chain workload over exactly these tokens
            k_tok = wl.k_tok[t0 + np.array(keys)]
            v_tok = wl.v_tok[t0 + np.array(keys)]
            pages = (n + 3) // 4
            ch = synthetic.Workload(
                name="path", batch=1, h_q=wl.h_q, h_kv=wl.h_kv, d=wl.d, page_size=4,
                kv_dtype=wl.kv_dtype, prefix_lens=np.array([n - 1]), qo_lens=np.array([1]),
                kv_lens=np.array([n]), qo_indptr=np.array([0, 1], np.int32),
                kv_indptr=np.array([0, pages], np.int32),
                kv_indices=np.arange(pages, dtype=np.int32),
                last_page_len=np.array([n - (pages - 1) * 4], np.int32), num_pages=pages,
                tok_indptr=np.array([0, n]), q=wl.q[int(wl.qo_indptr[b]) + i][None],
                k_tok=k_tok, v_tok=v_tok, sm_scale=wl.sm_scale, k_scale=1.0, v_scale=1.0,
                mask_kind="causal", rope_theta=wl.rope_theta,
                q_pos=np.array([n - 1], np.int32), kv_pos=np.arange(n, dtype=np.int32))
            assert int(wl.q_pos[int(wl.qo_indptr[b]) + i]) == n - 1
            o2, l2 = oracle.verify_attn_workload(ch, nthreads=1)
            tok = int(wl.qo_indptr[b]) + i
            rows = slice(tok * wl.h_q, (tok + 1) * wl.h_q)
            np.testing.assert_allclose(out[rows], o2, atol=1e-13, rtol=0)
            np.testing.assert_allclose(lse[rows], l2, atol=1e-13, rtol=0)


def test_rope_at_position_zero_is_no_rope(oracle_lib):
    wl = _rope_workload()
    wl.q_pos = np.zeros_like(wl.q_pos)
    wl.kv_pos = np.zeros_like(wl.kv_pos)
    o1, l1 = oracle.verify_attn_workload(wl, nthreads=2)
    wl.q_pos = wl.kv_pos = None
    wl.rope_theta = None
    o2, l2 = oracle.verify_attn_workload(wl, nthreads=2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------- layouts

def test_nhd_cache_equals_hnd(oracle_lib):
    """The NHD pool is the HND pool with the head and slot axes swapped; the
    attention over it is the same, bit for bit."""
    for kvd in (synthetic.BF16, synthetic.FP8):
        base = dict(batch=3, h_q=8, h_kv=2, d=16, page_size=4, prefix=("fixed", [9, 0, 14]),
                    qo=("fixed", [3, 5, 2]), mask="tree", seed=71, kv_dtype=kvd)
        wh = synthetic.make_custom(**base)
        wn = synthetic.make_custom(kv_layout="nhd", **base)
        kh, vh = oracle.build_cache(wh)
        kn, vn = oracle.build_cache(wn)
        assert kn.shape == (wn.num_pages, 4, 2, 16)
        assert np.array_equal(kn, kh.transpose(0, 2, 1, 3))
        assert np.array_equal(vn, vh.transpose(0, 2, 1, 3))
        o1, l1 = oracle.verify_attn_workload(wh, caches=(kh, vh), nthreads=2)
        o2, l2 = oracle.verify_attn_workload(wn, caches=(kn, vn), nthreads=2)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_full_layout_mask_with_visible_prefix_equals_draft_block(oracle_lib):
    """flashmap's full custom mask (L rows of prefix + L bits) with every
    prefix bit set is the L x L draft-block mask."""
    base = dict(batch=3, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [9, 0, 14]),
                qo=("fixed", [3, 5, 2]), mask="tree", seed=73)
    wq = synthetic.make_custom(**base)
    wf = synthetic.make_custom(mask_layout="full", **base)
    assert wf.mask_indptr[-1] == sum(int(L) * int(n) for L, n in zip(wf.qo_lens, wf.kv_lens))
    o1, l1 = oracle.verify_attn_workload(wq, nthreads=2)
    o2, l2 = oracle.verify_attn_workload(wf, nthreads=2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


EXT_TINY = [
    dict(batch=2, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [6, 3]),
         qo=("fixed", [4, 3]), mask="tree", mask_layout="full", prefix_visible="random", seed=81),
    dict(batch=2, h_q=2, h_kv=1, d=8, page_size=2, prefix=("fixed", [5, 0]),
         qo=("fixed", [3, 4]), mask="random", mask_layout="full", prefix_visible="random",
         kv_layout="nhd", seed=82),
    dict(batch=2, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [7, 2]),
         qo=("fixed", [5, 3]), mask="tree", rope_theta=10000.0, seed=83),
    dict(batch=1, h_q=4, h_kv=1, d=16, page_size=4, prefix=("fixed", [6]),
         qo=("fixed", [4]), mask="causal", rope_theta=500000.0, kv_layout="nhd",
         kv_dtype=synthetic.FP8, seed=84),
    dict(batch=2, h_q=4, h_kv=2, d=8, page_size=4, prefix=("fixed", [3, 5]),
         qo=("fixed", [3, 2]), mask="tree", mask_layout="full", prefix_visible="random",
         rope_theta=10000.0, seed=85),
]


@pytest.mark.parametrize("spec", EXT_TINY, ids=range(len(EXT_TINY)))
def test_extensions_match_scalar_brute_force(oracle_lib, spec):
    """The scalar brute force (its own page walk, mask rule, layout view and
    rotation) on the cache the oracle's append wrote."""
    wl = synthetic.make_custom(**spec)
    kc, vc = oracle.build_cache(wl)
    out, lse = oracle.verify_attn_workload(wl, caches=(kc, vc), nthreads=2)
    bo, bl = brute.verify_attn(wl.q, kc, vc, wl.kv_dtype == synthetic.FP8, wl.kv_indptr,
                               wl.kv_indices, wl.last_page_len, wl.qo_indptr, wl.mask,
                               wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size, wl.sm_scale,
                               wl.k_scale, wl.v_scale, kv_layout=1 if wl.nhd else 0,
                               mask_layout=1 if wl.mask_layout == "full" else 0, q_pos=wl.q_pos,
                               rope_theta=wl.rope_theta or 0.0)
    fin = np.isfinite(bl)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(out, bo, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[fin], bl[fin], atol=1e-12, rtol=0)


# ---------------------------------------------------------------- e4m3 queries

def test_query_quantisation_matches_torch(oracle_lib):
    """oracle_quantize_q_e4m3: amax = max |q|, inv = 448 / amax and qsc = amax
    / 448 in binary32, codes = the e4m3 cast of the binary32 product q * inv
    -- restated with torch's float32 arithmetic and its e4m3 cast."""
    gen = torch.Generator().manual_seed(5)
    for scale in (1.0, 30.0, 1e-3):
        q = (torch.randn((16, 128), generator=gen) * scale).to(torch.bfloat16).float()
        for row in q:
            amax = row.abs().max()
            inv = torch.tensor(448.0, dtype=torch.float32) / amax
            want = (row * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            codes, qsc = oracle.quantize_q_e4m3(row.double().numpy())
            assert np.array_equal(codes, want)
            assert qsc == float(amax / torch.tensor(448.0, dtype=torch.float32))
    codes, qsc = oracle.quantize_q_e4m3(np.zeros(8))
    assert qsc == 1.0 and not codes.any()


def test_e4m3_query_attention_is_attention_over_the_quantised_rows(oracle_lib):
    """verify attention with e4m3 queries = the plain definition over the
    dequantised query rows (codes * scale, built here with torch), per row."""
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=16, page_size=4,
                               prefix=("fixed", [9, 3]), qo=("fixed", [4, 3]), mask="tree",
                               kv_dtype=synthetic.FP8, seed=111)
    kc, vc = oracle.build_cache(wl)
    out, lse = oracle.verify_attn_workload(wl, caches=(kc, vc), q_fp8=True, nthreads=2)
    qd = torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16).float()
    for b in range(wl.batch):
        pre, L = int(wl.prefix_lens[b]), int(wl.qo_lens[b])
        pages = wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]]
        pos = np.arange(pre + L)
        dec = lambda x: torch.from_numpy(np.ascontiguousarray(x)).view(torch.float8_e4m3fn).double().numpy()
        for t in range(L):
            tok = int(wl.qo_indptr[b]) + t
            vis = list(range(pre)) + [pre + u for u in range(L) if wl.mask_dense[b][t, u]]
            for qh in range(wl.h_q):
                h = qh // wl.group
                row = qd[tok, qh]
                amax = row.abs().max()
                inv = torch.tensor(448.0, dtype=torch.float32) / amax
                qsc = float(amax / torch.tensor(448.0, dtype=torch.float32))
                q8 = (row * inv).to(torch.float8_e4m3fn).double() * qsc
                K = dec(kc[pages[pos // 4], h, pos % 4]) * wl.k_scale
                V = dec(vc[pages[pos // 4], h, pos % 4]) * wl.v_scale
                o, l = oracle.dense_attention(q8.numpy()[None], K[vis], V[vis],
                                              np.zeros((1, len(vis))), wl.sm_scale)
                np.testing.assert_allclose(out[tok * wl.h_q + qh], o[0], atol=1e-12, rtol=0)
                assert abs(lse[tok * wl.h_q + qh] - l[0]) < 1e-12


# ---------------------------------------------------------------- value width dv != d

@pytest.mark.parametrize("spec", [
    dict(batch=2, h_q=4, h_kv=2, d=16, dv=8, page_size=4, prefix=("fixed", [9, 3]),
         qo=("fixed", [4, 3]), mask="tree", seed=141),
    dict(batch=2, h_q=2, h_kv=1, d=8, dv=24, page_size=2, prefix=("fixed", [5, 0]),
         qo=("fixed", [3, 4]), mask="causal", kv_dtype=synthetic.FP8, seed=142),
    dict(batch=1, h_q=4, h_kv=2, d=8, dv=16, page_size=4, prefix=("fixed", [6]),
         qo=("fixed", [3]), mask="random", kv_layout="nhd", mask_layout="full",
         prefix_visible="random", seed=143),
], ids=["narrow_values_tree", "wide_values_fp8_chain", "wide_values_nhd_full_mask"])
def test_value_width_matches_scalar_brute_force(oracle_lib, spec):
    """sglang's value head size dv != d: the scalar brute force (which takes
    the value width from the cache it is given) on the cache the oracle's
    append wrote, with key rows of d and value rows of dv elements."""
    wl = synthetic.make_custom(**spec)
    kc, vc = oracle.build_cache(wl)
    assert kc.shape[-1] == wl.d and vc.shape[-1] == wl.dv
    out, lse = oracle.verify_attn_workload(wl, caches=(kc, vc), nthreads=2)
    assert out.shape == (wl.total_qo * wl.h_q, wl.dv)
    bo, bl = brute.verify_attn(wl.q, kc, vc, wl.kv_dtype == synthetic.FP8, wl.kv_indptr,
                               wl.kv_indices, wl.last_page_len, wl.qo_indptr, wl.mask,
                               wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size, wl.sm_scale,
                               wl.k_scale, wl.v_scale, kv_layout=1 if wl.nhd else 0,
                               mask_layout=1 if wl.mask_layout == "full" else 0)
    fin = np.isfinite(bl)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(out, bo, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[fin], bl[fin], atol=1e-12, rtol=0)


def test_value_columns_are_independent(oracle_lib):
    """The weights depend on Q and K alone: with the same keys, values of dv
    columns give exactly the first dv columns (and the same LSE) of the
    result for values widened by extra columns -- so no value row is read
    with the key's width or stride."""
    base = dict(batch=3, h_q=8, h_kv=2, d=32, page_size=4, prefix=("fixed", [13, 0, 7]),
                qo=("fixed", [5, 2, 6]), mask="tree", seed=144)
    narrow = synthetic.make_custom(dv=16, **base)
    wide = synthetic.make_custom(dv=48, **base)
    assert np.array_equal(narrow.q, wide.q) and np.array_equal(narrow.k_tok, wide.k_tok)
    wide.v_tok = wide.v_tok.copy()
    wide.v_tok[..., :16] = narrow.v_tok
    on, ln = oracle.verify_attn_workload(narrow, nthreads=2)
    ow, lw = oracle.verify_attn_workload(wide, nthreads=2)
    np.testing.assert_array_equal(ln, lw)
    np.testing.assert_allclose(on, ow[:, :16], atol=1e-13, rtol=0)
    # and a value width equal to d is the ordinary path
    same = synthetic.make_custom(dv=32, **base)
    plain = synthetic.make_custom(**base)
    o1, l1 = oracle.verify_attn_workload(same, nthreads=2)
    o2, l2 = oracle.verify_attn_workload(plain, nthreads=2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_value_width_append_lands_rows_of_their_width(oracle_lib):
    """The append with dv-wide values: each new V row (dv elements) lands at
    its token's slot of the dv-wide pool, K rows (d elements) at the same
    slot of the d-wide pool, bf16 and quantised to e4m3; nothing else moves."""
    for kvd, quant in ((synthetic.BF16, False), (synthetic.FP8, True)):
        wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=16, dv=8, page_size=4,
                                   prefix=("fixed", [5, 2]), qo=("fixed", [3, 4]), kv_dtype=kvd,
                                   seed=145)
        wb = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=16, dv=8, page_size=4,
                                   prefix=("fixed", [5, 2]), qo=("fixed", [3, 4]), seed=145)
        src = wb if quant else wl
        kn, vn = src.new_tokens()
        kc = synthetic.sentinel_pool(wl)
        vc = synthetic.sentinel_pool(wl, values=True)
        oracle.paged_kv_append_ex(kn, vn, wl.qo_indptr, wl.kv_indptr, wl.kv_indices,
                                  wl.last_page_len, wl.page_size, wl.num_pages, kc, vc,
                                  cache_fp8=kvd == synthetic.FP8, quantize=quant,
                                  k_scale=wl.k_scale, v_scale=wl.v_scale)
        written = np.zeros(kc.shape[:3], bool)
        for b in range(wl.batch):
            L, kv = int(wl.qo_lens[b]), int(wl.kv_lens[b])
            for i in range(L):
                pos = kv - L + i
                page = wl.kv_indices[wl.kv_indptr[b] + pos // wl.page_size]
                slot = pos % wl.page_size
                tok = int(wl.qo_indptr[b]) + i
                for h in range(wl.h_kv):
                    written[page, h, slot] = True
                    if quant:
                        want_k = torch.from_numpy(
                            (torch.from_numpy(kn[tok, h].view(np.int16)).view(torch.bfloat16).float()
                             / np.float32(wl.k_scale)).numpy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                        want_v = torch.from_numpy(
                            (torch.from_numpy(vn[tok, h].view(np.int16)).view(torch.bfloat16).float()
                             / np.float32(wl.v_scale)).numpy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    else:
                        want_k, want_v = kn[tok, h], vn[tok, h]
                    assert np.array_equal(kc[page, h, slot], want_k)
                    assert np.array_equal(vc[page, h, slot], want_v)
        fill = 0xFF if kvd == synthetic.FP8 else 0xFFFF
        assert np.all(kc[~written] == fill) and np.all(vc[~written] == fill)

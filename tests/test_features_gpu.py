"""GPU parity of the interface-breadth features against the fp64 oracle:
the quantising append into an fp8 cache (bit-exact), the NHD cache layout,
flashmap's full-prefix custom-mask layout, and RoPE at the drafts' tree
positions (new keys rotated by the append, queries inside the attention
kernels), on every kernel variant that serves each shape."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import DeviceWorkload, compare, to_dev
from test_fp8_mma_gpu import check as check_e4m3

pytestmark = pytest.mark.gpu

KERNELS = [(1, "mma64"), (2, "mma128"), (3, "tc128"), (4, "tc256")]


@pytest.fixture(scope="module")
def va():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_gqa_gb300 as m
    return m


def _raw(t, fp8):
    return t.view(torch.uint8).cpu().numpy().view(np.uint8 if fp8 else np.uint16)


# ------------------------------------------------------------------ quantising append

@pytest.mark.parametrize("layout", ["hnd", "nhd"])
@pytest.mark.parametrize("case", [
    dict(batch=3, h_q=4, h_kv=2, d=64, page_size=16, prefix=("fixed", [37, 0, 70]),
         qo=("fixed", [5, 3, 1])),
    dict(batch=2, h_q=8, h_kv=8, d=128, page_size=64, prefix=("fixed", [100, 1]),
         qo=("fixed", [30, 64]), value_std=40.0),
], ids=["d64", "d128_saturating"])
def test_quantising_append_is_bit_exact(va, case, layout):
    """bf16 drafts into an fp8-e4m3 cache: stored = e4m3(x / scale), the
    correctly rounded binary32 quotient rounded to nearest even and saturated
    (value_std 40 with a small scale drives some codes past 448), bit for bit
    equal to the oracle's quantiser; no other byte changes."""
    wb = synthetic.make_custom(seed=5, kv_layout=layout, **case)
    wf = synthetic.make_custom(seed=5, kv_layout=layout, kv_dtype=synthetic.FP8, **case)
    kn, vn = wb.new_tokens()
    ks, vs = float(np.float32(wf.k_scale * 0.25)), float(np.float32(wf.v_scale))
    kc = synthetic.sentinel_pool(wf)
    vc = synthetic.sentinel_pool(wf)
    oracle.paged_kv_append_ex(kn, vn, wb.qo_indptr, wb.kv_indptr, wb.kv_indices,
                              wb.last_page_len, wb.page_size, wb.num_pages, kc, vc,
                              cache_fp8=True, quantize=True, k_scale=ks, v_scale=vs,
                              kv_layout=1 if layout == "nhd" else 0)
    assert (kc == 0x7E).any() or case["d"] == 64
    dk = torch.from_numpy(kc.copy()).fill_(0xFF).cuda().view(torch.float8_e4m3fn)
    dv = torch.from_numpy(vc.copy()).fill_(0xFF).cuda().view(torch.float8_e4m3fn)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    va.paged_kv_append(to_dev(kn.view(np.int16), "cuda", torch.bfloat16),
                       to_dev(vn.view(np.int16), "cuda", torch.bfloat16),
                       to_dev(wb.qo_indptr, "cuda"), to_dev(wb.kv_indptr, "cuda"),
                       to_dev(wb.kv_indices, "cuda"), to_dev(wb.last_page_len, "cuda"), dk, dv,
                       k_scale=ks, v_scale=vs, kv_layout=layout, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(_raw(dk, True), kc)
    assert np.array_equal(_raw(dv, True), vc)


def test_quantising_append_then_attention_over_the_fresh_drafts(va):
    """The wide-tree fp8 shape in small: an fp8 prefix, the bf16 drafts
    quantised into the cache by the append, then verify attention (both
    tcgen05 variants) over the cache the append just wrote, against the
    oracle over its own quantised cache."""
    base = dict(batch=2, h_q=32, h_kv=8, d=128, prefix=("fixed", [1000, 300]),
                qo=("fixed", [64, 20]), mask="tree", seed=91)
    wf = synthetic.make_custom(kv_dtype=synthetic.FP8, **base)
    wb = synthetic.make_custom(**base)
    kn, vn = wb.new_tokens()
    # the oracle's pool: every token from the fp8 workload, then the drafts
    # quantised from bf16 over them
    kc, vc = oracle.build_cache(wf)
    oracle.paged_kv_append_quant(kn, vn, wf.k_scale, wf.v_scale, wf.qo_indptr, wf.kv_indptr,
                                 wf.kv_indices, wf.last_page_len, wf.page_size, wf.num_pages,
                                 kc, vc)
    dw = DeviceWorkload(wf)
    va.paged_kv_append(to_dev(kn.view(np.int16), "cuda", torch.bfloat16),
                       to_dev(vn.view(np.int16), "cuda", torch.bfloat16), dw.qo_indptr,
                       dw.kv_indptr, dw.kv_indices, dw.last_page_len, dw.k_cache, dw.v_cache,
                       k_scale=wf.k_scale, v_scale=wf.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(_raw(dw.k_cache, True), kc)
    assert np.array_equal(_raw(dw.v_cache, True), vc)
    for kernel in (3, 4):
        out, lse, plan = dw.run(kernel=kernel)
        torch.cuda.synchronize()
        assert va.verify_attn_device_status(plan) == 0
        compare(wf, out, lse, caches=(kc, vc))


# ------------------------------------------------------------------ NHD layout

@pytest.mark.parametrize("kernel,kname", KERNELS, ids=[k[1] for k in KERNELS])
@pytest.mark.parametrize("kvd", [synthetic.BF16, synthetic.FP8])
def test_nhd_layout_matches_oracle(va, kernel, kname, kvd):
    wl = synthetic.make_custom(batch=3, h_q=16, h_kv=2, d=128, prefix=("fixed", [700, 0, 90]),
                               qo=("fixed", [17, 40, 3]), mask="tree", kv_dtype=kvd,
                               kv_layout="nhd", seed=93)
    dw = DeviceWorkload(wl)
    kc, vc = oracle.build_cache(wl)
    assert np.array_equal(_raw(dw.k_cache, kvd == synthetic.FP8), kc)   # the NHD append, bit-exact
    assert np.array_equal(_raw(dw.v_cache, kvd == synthetic.FP8), vc)
    for splits in (1, 0):
        out, lse, plan = dw.run(kernel=kernel, max_splits=splits)
        torch.cuda.synchronize()
        assert plan.header()["kernel"] == kernel
        assert va.verify_attn_device_status(plan) == 0
        compare(wl, out, lse, caches=(kc, vc))


def test_nhd_layout_d64_page4(va):
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=64, page_size=4, prefix=("fixed", [77, 3]),
                               qo=("fixed", [9, 5]), mask="causal", kv_layout="nhd", seed=94)
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run()
    torch.cuda.synchronize()
    compare(wl, out, lse)


# ------------------------------------------------------------------ full-prefix mask

@pytest.mark.parametrize("kernel,kname", KERNELS, ids=[k[1] for k in KERNELS])
@pytest.mark.parametrize("case", [
    dict(mask="tree", prefix_visible="random"),
    dict(mask="random", prefix_visible="random", kv_dtype=synthetic.FP8),
    dict(mask="tree", prefix_visible="all"),
], ids=["tree_random_prefix", "fp8_random", "tree_visible_prefix"])
def test_full_prefix_mask_matches_oracle(va, kernel, kname, case):
    """flashmap's full custom mask: L rows of (prefix + L) bits, so prefix
    keys can be hidden too (random bits here); every key tile takes its
    visibility from the row's bits."""
    wl = synthetic.make_custom(batch=3, h_q=16, h_kv=2, d=128, prefix=("fixed", [300, 0, 45]),
                               qo=("fixed", [17, 40, 6]), mask_layout="full", seed=95, **case)
    dw = DeviceWorkload(wl)
    for splits in (1, 0):
        out, lse, plan = dw.run(kernel=kernel, max_splits=splits, target_ctas=300)
        torch.cuda.synchronize()
        assert plan.header()["kernel"] == kernel
        assert va.verify_attn_device_status(plan) == 0
        compare(wl, out, lse)


def test_full_prefix_mask_d64(va):
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=64, prefix=("fixed", [60, 200]),
                               qo=("fixed", [12, 33]), mask="random", mask_layout="full",
                               prefix_visible="random", seed=96)
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run()
    torch.cuda.synchronize()
    compare(wl, out, lse)


# ------------------------------------------------------------------ RoPE

@pytest.mark.parametrize("kernel,kname", KERNELS, ids=[k[1] for k in KERNELS])
@pytest.mark.parametrize("case", [
    dict(mask="tree", rope_theta=10000.0),
    dict(mask="tree", rope_theta=500000.0, kv_dtype=synthetic.FP8),
    dict(mask="causal", rope_theta=10000.0, kv_layout="nhd"),
], ids=["tree_bf16", "tree_fp8_llama3_theta", "chain_nhd"])
def test_rope_at_tree_positions_matches_oracle(va, kernel, kname, case):
    """RoPE at the drafts' tree positions (prefix + depth): the append
    rotates every key at its position, the attention kernel rotates each
    query row at its token's position; compared with the oracle, which
    rotates in fp64 (its cache is its own rotated append)."""
    wl = synthetic.make_custom(batch=3, h_q=16, h_kv=2, d=128,
                               prefix=("fixed", [2000, 0, 130]), qo=("fixed", [17, 40, 6]),
                               seed=97, **case)
    dw = DeviceWorkload(wl)
    for splits in (1, 0):
        out, lse, plan = dw.run(kernel=kernel, max_splits=splits, target_ctas=300)
        torch.cuda.synchronize()
        assert plan.header()["kernel"] == kernel
        assert va.verify_attn_device_status(plan) == 0
        compare(wl, out, lse)


def test_rope_d64_and_long_positions(va):
    """Warp-level kernel at head_dim 64, positions past 32K (the angle
    reduction matters there)."""
    wl = synthetic.make_custom(batch=2, h_q=8, h_kv=2, d=64, prefix=("fixed", [33000, 5]),
                               qo=("fixed", [9, 4]), mask="tree", rope_theta=10000.0, seed=98)
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run()
    torch.cuda.synchronize()
    compare(wl, out, lse)


def test_rope_append_rounds_within_one_step(va):
    """The append's rotated keys against the oracle's fp64 rotation rounded
    once: equal, or one step of the cache dtype apart where the fp32 and
    fp64 rotations fall on the two sides of a rounding boundary."""
    for kvd in (synthetic.BF16, synthetic.FP8):
        wl = synthetic.make_custom(batch=2, h_q=8, h_kv=2, d=128, prefix=("fixed", [4000, 31]),
                                   qo=("fixed", [17, 9]), mask="tree", rope_theta=10000.0,
                                   kv_dtype=kvd, seed=99)
        dw = DeviceWorkload(wl)
        torch.cuda.synchronize()
        kc, vc = oracle.build_cache(wl)
        fp8 = kvd == synthetic.FP8
        gk = _raw(dw.k_cache, fp8)
        assert np.array_equal(_raw(dw.v_cache, fp8), vc)      # values are not rotated
        dec = oracle.decode_e4m3 if fp8 else oracle.decode_bf16
        written = kc != (0xFF if fp8 else 0xFFFF)
        a, b = dec(gk[written]), dec(kc[written])
        # one step of the format at the larger of the two: 3 (e4m3) or 7
        # (bf16) fraction bits, subnormal steps below 2^-6 (e4m3) or 2^-126
        # (bf16); plus the fp32 rotation's own absolute error, ~4e-7 times
        # the pair's magnitude (|x| <= ~5 for bf16 rows of N(0, 1) values,
        # <= 448 for e4m3 codes), which decides near-zero results where the
        # two terms of a rotation cancel
        emin = -6.0 if fp8 else -126.0
        e = np.floor(np.log2(np.maximum(np.maximum(np.abs(a), np.abs(b)), 2.0 ** emin)))
        spacing = np.exp2(e - (3 if fp8 else 7))
        slack = 4e-7 * (2 * 448.0 if fp8 else 2 * 6.0)
        bad = np.abs(a - b) > spacing * 1.0001 + slack
        assert not bad.any(), (a[bad][:5], b[bad][:5])
        assert np.mean(gk[written] == kc[written]) > 0.99


def test_rope_plan_needs_positions(va):
    wl = synthetic.make_custom(batch=1, h_q=4, h_kv=2, d=128, prefix=("fixed", [40]),
                               qo=("fixed", [3]), mask="causal", rope_theta=10000.0, seed=100)
    dw = DeviceWorkload(wl)
    plan = dw.plan()
    with pytest.raises(va.VerifyAttnError):
        va.verify_attn_run(dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices,
                           dw.last_page_len, dw.qo_indptr, None, None, plan)
    plain = dw.plan(rope=False)
    with pytest.raises(va.VerifyAttnError):
        va.verify_attn_run(dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices,
                           dw.last_page_len, dw.qo_indptr, None, None, plain,
                           q_position=dw.q_pos)


# ------------------------------------------------------------------ fused append + run

def _fused(va, dw, plan, out=None, lse=None, **kw):
    wl = dw.wl
    return va.verify_attn_append_run(dw.k_new, dw.v_new, dw.q, dw.k_cache, dw.v_cache,
                                     dw.kv_indptr, dw.kv_indices, dw.last_page_len, dw.qo_indptr,
                                     dw.mask, dw.mask_indptr, plan, sm_scale=wl.sm_scale,
                                     k_scale=wl.k_scale, v_scale=wl.v_scale, out=out, lse=lse,
                                     q_position=dw.q_pos, rope_theta=wl.rope_theta or 0.0,
                                     positions=dw.new_pos, kv_layout=wl.kv_layout, **kw)


@pytest.mark.parametrize("early_reads", [False, True], ids=["plain", "early_reads"])
@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER)
def test_append_run_matches_oracle(va, name, early_reads):
    """verify_attn_append_run (the drafts appended and attended in one call,
    the attention reading q and the prefix while the append runs) on a pool
    whose draft slots still hold NaN, for every named workload at full size;
    with early_reads this is the launch configuration the benchmark times
    (and the plan's automatic draft items read the drafts from k_new / v_new):
    every row against the oracle at the strict bound, and the pool equal to
    the oracle's, bit for bit."""
    wl = synthetic.make_workload(name)
    dw = DeviceWorkload(wl, append=False)
    # prefix only: the drafts' slots keep the NaN sentinel until the fused call
    fp8 = wl.kv_dtype == synthetic.FP8
    raw = np.uint8 if fp8 else np.int16
    pre = np.concatenate([np.arange(wl.tok_indptr[b], wl.tok_indptr[b + 1] - wl.qo_lens[b])
                          for b in range(wl.batch)])
    pre_indptr = np.concatenate([[0], np.cumsum(wl.prefix_lens)]).astype(np.int32)
    # appending the prefix alone: a table whose kv_len is the prefix length
    pages = (wl.prefix_lens + wl.page_size - 1) // wl.page_size
    kvp = np.zeros(wl.batch + 1, np.int32)
    idx = []
    for b in range(wl.batch):
        kvp[b + 1] = kvp[b] + pages[b]
        idx.append(wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b] + pages[b]])
    lpl = np.array([int(n) - (int(p) - 1) * wl.page_size if p > 0 else 0
                    for n, p in zip(wl.prefix_lens, pages)], np.int32)
    va.paged_kv_append(to_dev(wl.k_tok[pre].view(raw), "cuda", dw.kvd),
                       to_dev(wl.v_tok[pre].view(raw), "cuda", dw.kvd), to_dev(pre_indptr, "cuda"),
                       to_dev(kvp, "cuda"), to_dev(np.concatenate(idx).astype(np.int32), "cuda"),
                       to_dev(lpl, "cuda"), dw.k_cache, dw.v_cache)
    plan = dw.plan()
    out, lse = _fused(va, dw, plan, early_reads=early_reads)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    kc, vc = oracle.build_cache(wl)
    assert np.array_equal(_raw(dw.k_cache, fp8), kc) and np.array_equal(_raw(dw.v_cache, fp8), vc)
    compare(wl, out, lse, caches=(kc, vc), strict=True)


@pytest.mark.parametrize("case", [
    dict(mask="tree", rope_theta=10000.0),
    dict(mask="causal", kv_layout="nhd"),
    dict(mask="tree", kv_dtype=synthetic.FP8),
], ids=["rope_tree", "nhd_chain", "fp8_tree"])
def test_append_run_features_match_oracle(va, case):
    wl = synthetic.make_custom(batch=3, h_q=32, h_kv=8, d=128, prefix=("fixed", [1500, 0, 300]),
                               qo=("fixed", [17, 40, 6]), seed=101, **case)
    dw = DeviceWorkload(wl)   # drafts already in place: the fused call rewrites the same bits
    plan = dw.plan()
    out, lse = _fused(va, dw, plan)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    compare(wl, out, lse)


@pytest.mark.parametrize("kernel", [3, 4], ids=["tc128", "tc256"])
@pytest.mark.parametrize("case", [
    dict(prefix=("fixed", [37, 700, 0, 2048]), qo=("fixed", [17, 5, 9, 64]), mask="tree"),
    dict(prefix=("fixed", [130, 16, 1000]), qo=("fixed", [3, 1, 8]), mask="causal"),
    dict(prefix=("fixed", [301, 77]), qo=("fixed", [20, 33]), mask="tree", kv_dtype=synthetic.FP8),
    dict(prefix=("fixed", [301, 77]), qo=("fixed", [20, 33]), mask="tree", kv_dtype=synthetic.FP8,
         q_fp8=True),
    dict(prefix=("fixed", [500, 63]), qo=("fixed", [12, 40]), mask="tree", kv_layout="nhd"),
    dict(prefix=("fixed", [500, 63]), qo=("fixed", [12, 40]), mask="random", mask_layout="full",
         prefix_visible="random"),
], ids=["tree_unaligned", "chain", "fp8_tree", "fp8_e4m3_mma", "nhd", "full_mask"])
def test_append_run_draft_items(va, kernel, case):
    """Draft items (plan option draft_items = 1: each split request's drafts
    an item of their own, starting at the prefix length, mid-page) through
    the fused call, which reads them from k_new / v_new and not from the
    pages: first on a pool whose draft slots still hold NaN, then again on
    the appended pool; every row against the oracle and the pool equal to the
    oracle's bit for bit.  Also through verify_attn_run (the drafts read from
    the pages)."""
    case = dict(case)
    q_fp8 = case.pop("q_fp8", False)
    wl = synthetic.make_custom(batch=len(case["prefix"][1]), h_q=16, h_kv=2, d=128, seed=131,
                               **case)
    dw = DeviceWorkload(wl, append=False)
    fp8 = wl.kv_dtype == synthetic.FP8
    raw = np.uint8 if fp8 else np.int16
    # the prefixes only, through a table whose kv_len is the prefix length
    pre = np.concatenate([np.arange(wl.tok_indptr[b], wl.tok_indptr[b + 1] - wl.qo_lens[b])
                          for b in range(wl.batch)]).astype(np.int64)
    pre_indptr = np.concatenate([[0], np.cumsum(wl.prefix_lens)]).astype(np.int32)
    pages = (wl.prefix_lens + wl.page_size - 1) // wl.page_size
    kvp = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    idx = np.concatenate([wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b] + pages[b]]
                          for b in range(wl.batch)]).astype(np.int32)
    lpl = np.array([int(n) - (int(p) - 1) * wl.page_size if p > 0 else 0
                    for n, p in zip(wl.prefix_lens, pages)], np.int32)
    va.paged_kv_append(to_dev(wl.k_tok[pre].view(raw), "cuda", dw.kvd),
                       to_dev(wl.v_tok[pre].view(raw), "cuda", dw.kvd), to_dev(pre_indptr, "cuda"),
                       to_dev(kvp, "cuda"), to_dev(idx, "cuda"), to_dev(lpl, "cuda"), dw.k_cache,
                       dw.v_cache, kv_layout=wl.kv_layout)
    plan = dw.plan(kernel=kernel, draft_items=1, target_ctas=64, min_chunk=128, q_fp8=q_fp8)
    items = plan.items()
    assert any(int(it[4]) == int(wl.prefix_lens[int(it[0])]) and int(it[4]) % 16 for it in items)
    kc, vc = oracle.build_cache(wl)
    cmp = (lambda o, l: check_e4m3(wl, o, l, caches=(kc, vc))) if q_fp8 else \
          (lambda o, l: compare(wl, o, l, caches=(kc, vc)))
    for call in range(2):
        out, lse = _fused(va, dw, plan, early_reads=bool(call))
        torch.cuda.synchronize()
        assert va.verify_attn_device_status(plan) == 0
        assert np.array_equal(_raw(dw.k_cache, fp8), kc) and np.array_equal(_raw(dw.v_cache, fp8), vc)
        cmp(out, lse)
    out, lse, _ = dw.run(plan=plan)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    cmp(out, lse)


def test_append_run_quantises_fresh_drafts(va):
    """The wide fp8 tree in small through the fused call: bf16 drafts are
    quantised into the fp8 cache and attended in the same call."""
    base = dict(batch=2, h_q=32, h_kv=8, d=128, prefix=("fixed", [1000, 300]),
                qo=("fixed", [64, 20]), mask="tree", seed=91)
    wf = synthetic.make_custom(kv_dtype=synthetic.FP8, **base)
    wb = synthetic.make_custom(**base)
    kn, vn = wb.new_tokens()
    kc, vc = oracle.build_cache(wf)
    oracle.paged_kv_append_quant(kn, vn, wf.k_scale, wf.v_scale, wf.qo_indptr, wf.kv_indptr,
                                 wf.kv_indices, wf.last_page_len, wf.page_size, wf.num_pages,
                                 kc, vc)
    dw = DeviceWorkload(wf)
    plan = dw.plan()
    out, lse = va.verify_attn_append_run(
        to_dev(kn.view(np.int16), "cuda", torch.bfloat16),
        to_dev(vn.view(np.int16), "cuda", torch.bfloat16), dw.q, dw.k_cache, dw.v_cache,
        dw.kv_indptr, dw.kv_indices, dw.last_page_len, dw.qo_indptr, dw.mask, dw.mask_indptr,
        plan, sm_scale=wf.sm_scale, k_scale=wf.k_scale, v_scale=wf.v_scale,
        append_k_scale=wf.k_scale, append_v_scale=wf.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(_raw(dw.k_cache, True), kc) and np.array_equal(_raw(dw.v_cache, True), vc)
    compare(wf, out, lse, caches=(kc, vc))


@pytest.mark.parametrize("early_reads", [False, True])
def test_append_run_graph_replays_back_to_back(va, early_reads):
    """The fused call captured in a CUDA graph, replayed many times back to
    back on the same buffers (each replay's append overwrites the drafts the
    previous replay's attention read), then checked: the early reads of q,
    the tables and the prefix must never see a half-written step."""
    wl = synthetic.make_workload("llama3_8b_tree_verify")
    dw = DeviceWorkload(wl)
    plan = dw.plan()
    out = torch.empty_like(dw.q)
    lse = torch.empty(dw.q.shape[:2], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _fused(va, dw, plan, out=out, lse=lse, early_reads=early_reads)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(8):
            _fused(va, dw, plan, out=out, lse=lse, early_reads=early_reads)
    out.zero_()
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    compare(wl, out, lse, strict=True)


@pytest.mark.parametrize("early_reads", [False, True])
def test_layers_sharing_one_workspace(va, early_reads):
    """Four "layers" run back to back in one graph, each with its own q and
    output but one plan and one workspace: a layer's split kernel must not
    overwrite the split partials before the previous layer's merge has read
    them, even when it reads its inputs early."""
    wl = synthetic.make_workload("llama3_8b_tree_verify")
    dw = DeviceWorkload(wl)
    plan = dw.plan()
    assert plan.header()["n_merge"] > 0
    gen = torch.Generator(device="cpu").manual_seed(7)
    qs = [torch.randn(dw.q.shape, generator=gen).to(torch.bfloat16).cuda() for i in range(4)]
    outs = [torch.empty_like(dw.q) for _ in qs]
    lses = [torch.empty(dw.q.shape[:2], dtype=torch.float32, device="cuda") for _ in qs]

    def layers():
        for q, o, l in zip(qs, outs, lses):
            va.verify_attn_run(q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices,
                               dw.last_page_len, dw.qo_indptr, dw.mask, dw.mask_indptr, plan,
                               sm_scale=wl.sm_scale, out=o, lse=l, early_reads=early_reads)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layers()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layers()
    for o in outs:
        o.zero_()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    kc, vc = oracle.build_cache(wl)
    for q, o, l in zip(qs, outs, lses):
        wq = synthetic.make_workload("llama3_8b_tree_verify")
        wq.q = q.cpu().view(torch.int16).numpy().view(np.uint16)
        compare(wq, o, l, caches=(kc, vc), strict=True)


# ------------------------------------------------------------------ value width dv != d

DV_CASES = [
    dict(d=128, dv=64, prefix=("fixed", [700, 0, 90]), qo=("fixed", [17, 40, 3]), mask="tree"),
    dict(d=64, dv=128, prefix=("fixed", [300, 45]), qo=("fixed", [9, 5]), mask="causal"),
    dict(d=128, dv=64, prefix=("fixed", [500, 63]), qo=("fixed", [12, 30]), mask="tree",
         kv_dtype=synthetic.FP8),
    dict(d=64, dv=128, prefix=("fixed", [200, 1000]), qo=("fixed", [6, 20]), mask="random",
         kv_layout="nhd", mask_layout="full", prefix_visible="random"),
]


@pytest.mark.parametrize("kernel", [1, 2], ids=["mma64", "mma128"])
@pytest.mark.parametrize("case", DV_CASES, ids=["d128_dv64_tree", "d64_dv128_chain",
                                                "fp8_d128_dv64", "nhd_full_d64_dv128"])
def test_value_width_matches_oracle(va, kernel, case):
    """sglang's value head size dv != d (plan option head_dim_v): the append
    writes K rows of d and V rows of dv elements (bit-exact against the
    oracle's pools), and the warp-level kernels attend with them, unsplit and
    split (merge over dv-wide partials), against the oracle row by row."""
    wl = synthetic.make_custom(batch=len(case["prefix"][1]), h_q=8, h_kv=2, seed=151, **case)
    dw = DeviceWorkload(wl)
    kc, vc = oracle.build_cache(wl)
    fp8 = wl.kv_dtype == synthetic.FP8
    assert np.array_equal(_raw(dw.k_cache, fp8), kc) and np.array_equal(_raw(dw.v_cache, fp8), vc)
    for splits in (1, 0):
        out, lse, plan = dw.run(kernel=kernel, max_splits=splits, target_ctas=200, min_chunk=64)
        torch.cuda.synchronize()
        hd = plan.header()
        assert hd["kernel"] == kernel and hd["head_dim_v"] == wl.dv
        assert tuple(out.shape) == (wl.total_qo, wl.h_q, wl.dv)
        assert va.verify_attn_device_status(plan) == 0
        compare(wl, out, lse, caches=(kc, vc))


def test_value_width_fused_call_and_quantising_append(va):
    """The fused append + attention call with dv != d, through a plain copy
    and through a quantising append into an fp8 cache."""
    base = dict(batch=2, h_q=8, h_kv=2, d=128, dv=64, prefix=("fixed", [400, 33]),
                qo=("fixed", [17, 6]), mask="tree", seed=152)
    wl = synthetic.make_custom(**base)
    dw = DeviceWorkload(wl)
    plan = dw.plan()
    assert plan.header()["head_dim_v"] == 64 and plan.header()["kernel"] in (1, 2)
    out, lse = _fused(va, dw, plan)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    kc, vc = oracle.build_cache(wl)
    assert np.array_equal(_raw(dw.k_cache, False), kc) and np.array_equal(_raw(dw.v_cache, False), vc)
    compare(wl, out, lse, caches=(kc, vc))
    # quantising: bf16 drafts of the bf16 workload into the fp8 one's cache
    wf = synthetic.make_custom(kv_dtype=synthetic.FP8, **base)
    kn, vn = wl.new_tokens()
    kcf, vcf = oracle.build_cache(wf)
    oracle.paged_kv_append_ex(kn, vn, wf.qo_indptr, wf.kv_indptr, wf.kv_indices,
                              wf.last_page_len, wf.page_size, wf.num_pages, kcf, vcf,
                              cache_fp8=True, quantize=True, k_scale=wf.k_scale,
                              v_scale=wf.v_scale)
    dwf = DeviceWorkload(wf)
    planf = dwf.plan()
    out, lse = va.verify_attn_append_run(
        to_dev(kn.view(np.int16), "cuda", torch.bfloat16),
        to_dev(vn.view(np.int16), "cuda", torch.bfloat16), dwf.q, dwf.k_cache, dwf.v_cache,
        dwf.kv_indptr, dwf.kv_indices, dwf.last_page_len, dwf.qo_indptr, dwf.mask,
        dwf.mask_indptr, planf, sm_scale=wf.sm_scale, k_scale=wf.k_scale, v_scale=wf.v_scale,
        append_k_scale=wf.k_scale, append_v_scale=wf.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(_raw(dwf.k_cache, True), kcf) and np.array_equal(_raw(dwf.v_cache, True), vcf)
    compare(wf, out, lse, caches=(kcf, vcf))

"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Tolerances: max |out - oracle| <= 1e-2 and
max |lse - oracle| <= 1e-3 (bf16 inputs, fp32 accumulation); the paged
append is compared bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import DeviceWorkload, compare, host_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_gqa_gb300 as m
    return m


# ------------------------------------------------------------------ append

APPEND_CASES = [
    dict(batch=3, h_q=4, h_kv=2, d=64, page_size=16, prefix=("fixed", [37, 0, 70]),
         qo=("fixed", [5, 3, 1])),
    dict(batch=2, h_q=8, h_kv=8, d=128, page_size=1, prefix=("fixed", [5, 9]),
         qo=("fixed", [4, 2])),
    dict(batch=2, h_q=4, h_kv=1, d=128, page_size=64, prefix=("fixed", [100, 1]),
         qo=("fixed", [30, 64]), kv_dtype=synthetic.FP8),
    dict(batch=4, h_q=2, h_kv=2, d=64, page_size=256, prefix=("fixed", [0, 255, 256, 3]),
         qo=("fixed", [1, 1, 2, 0]), kv_dtype=synthetic.FP8),
]


@pytest.mark.parametrize("case", APPEND_CASES, ids=range(len(APPEND_CASES)))
def test_append_is_bit_exact(va, case):
    wl = synthetic.make_custom(seed=5, **case)
    dw = DeviceWorkload(wl)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dw.append_drafts(status=status)
    torch.cuda.synchronize()
    kc, vc = oracle.build_cache(wl)
    raw = np.uint8 if wl.kv_dtype == synthetic.FP8 else np.uint16
    gk = dw.k_cache.view(torch.uint8).cpu().numpy().view(raw)
    gv = dw.v_cache.view(torch.uint8).cpu().numpy().view(raw)
    assert np.array_equal(gk.reshape(kc.shape), kc)
    assert np.array_equal(gv.reshape(vc.shape), vc)
    assert int(status.item()) == 0


def test_append_flags_bad_page_and_writes_the_rest(va):
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=64, page_size=16,
                               prefix=("fixed", [20, 20]), qo=("fixed", [3, 3]), seed=9)
    dw = DeviceWorkload(wl, append=False)
    bad = wl.kv_indices.copy()
    bad[wl.kv_indptr[1] + 1] = wl.num_pages + 5  # request 1's drafts (positions 20-22) live on its page 1
    dw.kv_indices = torch.from_numpy(bad).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dw.append_drafts(status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1  # VA_DEV_BAD_PAGE: the tokens of request 1 that map there
    # request 0's drafts landed
    kc = dw.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    kn, _ = wl.new_tokens()
    pages = wl.kv_indices[:wl.kv_indptr[1]]
    for i in range(3):
        pos = 20 + i
        assert np.array_equal(kc[pages[pos // 16], :, pos % 16], kn[i])


# ------------------------------------------------------------------ verify, small

SMALL = [
    ("chain_d64", dict(batch=2, h_q=4, h_kv=2, d=64, prefix=("fixed", [37, 70]),
                       qo=("fixed", [5, 5]), mask="causal")),
    ("tree_d128", dict(batch=3, h_q=8, h_kv=2, d=128, prefix=("fixed", [100, 513, 7]),
                       qo=("fixed", [17, 9, 4]), mask="tree")),
    ("random_mask", dict(batch=2, h_q=4, h_kv=4, d=64, prefix=("fixed", [60, 200]),
                         qo=("fixed", [12, 33]), mask="random")),
    ("decode_L1", dict(batch=5, h_q=32, h_kv=8, d=128, prefix=("fixed", [1, 15, 16, 17, 900]),
                       qo=("fixed", [1, 1, 1, 1, 1]), mask="causal")),
    ("mqa_g16", dict(batch=2, h_q=16, h_kv=1, d=128, prefix=("fixed", [300, 64]),
                     qo=("fixed", [3, 8]), mask="tree")),
    ("prefill_no_prefix", dict(batch=3, h_q=8, h_kv=2, d=128, prefix=("fixed", [0, 0, 0]),
                               qo=("fixed", [300, 17, 64]), mask="causal")),
    ("fp8_tree", dict(batch=2, h_q=8, h_kv=2, d=128, prefix=("fixed", [700, 33]),
                      qo=("fixed", [64, 20]), mask="tree", kv_dtype=synthetic.FP8)),
    ("fp8_d64_chain", dict(batch=2, h_q=4, h_kv=2, d=64, prefix=("fixed", [99, 1000]),
                           qo=("fixed", [3, 8]), mask="causal", kv_dtype=synthetic.FP8)),
    ("page1", dict(batch=2, h_q=4, h_kv=2, d=128, page_size=1, prefix=("fixed", [50, 3]),
                   qo=("fixed", [4, 6]), mask="tree")),
    ("page4", dict(batch=2, h_q=4, h_kv=2, d=64, page_size=4, prefix=("fixed", [77, 0]),
                   qo=("fixed", [9, 5]), mask="causal")),
    ("page256", dict(batch=2, h_q=4, h_kv=2, d=128, page_size=256, prefix=("fixed", [600, 10]),
                     qo=("fixed", [4, 6]), mask="tree")),
    ("empty_request", dict(batch=3, h_q=4, h_kv=2, d=128, prefix=("fixed", [40, 30, 20]),
                           qo=("fixed", [3, 0, 2]), mask="causal")),
    ("fully_masked_rows", dict(batch=2, h_q=4, h_kv=2, d=64, prefix=("fixed", [0, 5]),
                               qo=("fixed", [4, 3]), mask="none_visible")),
    ("full_mask", dict(batch=1, h_q=4, h_kv=2, d=128, prefix=("fixed", [10]),
                       qo=("fixed", [40]), mask="full")),
    ("g3_many_rows", dict(batch=2, h_q=6, h_kv=2, d=128, prefix=("fixed", [129, 1]),
                          qo=("fixed", [50, 45]), mask="tree")),
]


@pytest.mark.parametrize("name,case", SMALL, ids=[s[0] for s in SMALL])
def test_small_cases_match_oracle(va, name, case):
    wl = synthetic.make_custom(seed=11, **case)
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run()
    torch.cuda.synchronize()
    compare(wl, out, lse)
    assert va.verify_attn_device_status(plan) == 0


@pytest.mark.parametrize("opts", [dict(max_splits=1), dict(min_chunk=64, target_ctas=2000),
                                  dict(kernel=1), dict(kernel=2), dict(max_splits=2)])
def test_forced_plans_match_oracle(va, opts):
    wl = synthetic.make_custom(batch=3, h_q=8, h_kv=2, d=128, prefix=("fixed", [1000, 3000, 50]),
                               qo=("fixed", [6, 2, 7]), mask="tree", seed=13)
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run(**opts)
    torch.cuda.synchronize()
    if opts.get("max_splits") == 1:
        assert plan.header()["n_merge"] == 0
    if "target_ctas" in opts:
        assert plan.header()["n_merge"] > 0
    compare(wl, out, lse)


def test_custom_mask_may_open_later_drafts(va):
    """A custom mask is not limited to earlier drafts: rows of the first row
    block must still see every later draft the mask allows (3 row blocks)."""
    wl = synthetic.make_custom(batch=2, h_q=16, h_kv=2, d=128, prefix=("fixed", [70, 3]),
                               qo=("fixed", [40, 33]), mask="random", seed=27)
    assert int((wl.group * wl.qo_lens).max()) > 256
    dw = DeviceWorkload(wl)
    for opts in (dict(), dict(kernel=1), dict(kernel=3), dict(kernel=4)):
        out, lse, plan = dw.run(**opts)
        torch.cuda.synchronize()
        compare(wl, out, lse)


TC_CASES = [
    ("tree_g4", dict(batch=2, h_q=32, h_kv=8, d=128, prefix=("fixed", [700, 64]),
                     qo=("fixed", [17, 40]), mask="tree")),
    ("prefill_g8", dict(batch=3, h_q=16, h_kv=2, d=128, prefix=("fixed", [0, 0, 0]),
                        qo=("fixed", [300, 17, 129]), mask="causal")),
    ("chain_prefix", dict(batch=2, h_q=8, h_kv=1, d=128, prefix=("fixed", [1000, 257]),
                          qo=("fixed", [20, 16]), mask="causal")),
    ("page32", dict(batch=2, h_q=8, h_kv=2, d=128, page_size=32, prefix=("fixed", [333, 31]),
                    qo=("fixed", [40, 33]), mask="tree")),
    ("page256", dict(batch=2, h_q=4, h_kv=2, d=128, page_size=256, prefix=("fixed", [600, 10]),
                     qo=("fixed", [70, 6]), mask="tree")),
    ("g1_mha", dict(batch=1, h_q=2, h_kv=2, d=128, prefix=("fixed", [190]),
                    qo=("fixed", [150]), mask="causal")),
    ("masked_rows", dict(batch=2, h_q=8, h_kv=2, d=128, prefix=("fixed", [0, 5]),
                         qo=("fixed", [40, 37]), mask="none_visible")),
    ("fp8_tree", dict(batch=2, h_q=32, h_kv=8, d=128, prefix=("fixed", [1000, 77]),
                      qo=("fixed", [64, 20]), mask="tree", kv_dtype=synthetic.FP8)),
    ("fp8_chain_page64", dict(batch=3, h_q=16, h_kv=2, d=128, page_size=64,
                              prefix=("fixed", [500, 3, 129]), qo=("fixed", [9, 16, 1]),
                              mask="causal", kv_dtype=synthetic.FP8)),
]


@pytest.mark.parametrize("name,case", TC_CASES, ids=[c[0] for c in TC_CASES])
@pytest.mark.parametrize("splits", [1, 0])
@pytest.mark.parametrize("kernel", [3, 4], ids=["tc128", "tc256"])
def test_tcgen05_kernel_matches_oracle(va, name, case, splits, kernel):
    wl = synthetic.make_custom(seed=29, **case)
    dw = DeviceWorkload(wl)
    opts = dict(kernel=kernel, max_splits=splits)
    if splits == 0:
        opts["target_ctas"] = 600
    out, lse, plan = dw.run(**opts)
    torch.cuda.synchronize()
    assert plan.header()["kernel"] == kernel
    assert va.verify_attn_device_status(plan) == 0
    compare(wl, out, lse)


def test_tcgen05_kernel_rejects_what_it_cannot_serve(va):
    wl = synthetic.make_custom(batch=1, h_q=6, h_kv=2, d=128, prefix=("fixed", [10]),
                               qo=("fixed", [3]), seed=31)
    for kernel in (3, 4):
        with pytest.raises(va.VerifyAttnError):
            va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, None, 6, 2,
                                     128, 16, kernel=kernel, num_sms=152)   # 128 % G != 0


def test_split_and_unsplit_agree(va):
    wl = synthetic.make_workload("llama3_8b_tree_verify")
    dw = DeviceWorkload(wl)
    o1, l1, p1 = dw.run(max_splits=1)
    o2, l2, p2 = dw.run()
    torch.cuda.synchronize()
    assert p1.header()["n_merge"] == 0
    assert p2.header()["n_merge"] > 0
    assert float((o1.float() - o2.float()).abs().max()) <= 1e-2
    assert float((l1 - l2).abs().max()) <= 1e-3
    compare(wl, o1, l1)


def test_page_placement_does_not_change_bits(va):
    base = dict(batch=3, h_q=8, h_kv=2, d=128, prefix=("fixed", [300, 47, 1000]),
                qo=("fixed", [5, 9, 2]), mask="tree", seed=17)
    w1 = synthetic.make_custom(shuffle_pages=True, **base)
    w2 = synthetic.make_custom(shuffle_pages=False, **base)
    d1, d2 = DeviceWorkload(w1), DeviceWorkload(w2)
    o1, l1, _ = d1.run()
    o2, l2, _ = d2.run()
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_chain_mask_equals_causal_on_gpu(va):
    base = dict(batch=2, h_q=8, h_kv=2, d=128, prefix=("fixed", [200, 31]),
                qo=("fixed", [8, 13]), seed=19)
    wc = synthetic.make_custom(mask="chain", **base)
    wn = synthetic.make_custom(mask="causal", **base)
    oc, lc, _ = DeviceWorkload(wc).run()
    on, ln, _ = DeviceWorkload(wn).run()
    torch.cuda.synchronize()
    assert torch.equal(oc.view(torch.int16), on.view(torch.int16))
    assert torch.equal(lc, ln)


def test_partial_then_merge_equals_run(va):
    wl = synthetic.make_workload("llama3_8b_tree_verify")
    dw = DeviceWorkload(wl)
    out1, lse1, plan = dw.run()
    out2 = torch.empty_like(out1)
    lse2 = torch.empty_like(lse1)
    va.verify_attn_partial(dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices,
                           dw.last_page_len, dw.qo_indptr, dw.mask, dw.mask_indptr, plan,
                           sm_scale=wl.sm_scale, out=out2, lse=lse2)
    va.verify_attn_merge(dw.qo_indptr, plan, out2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_lse_may_be_omitted(va):
    wl = synthetic.make_workload("tiny_verify")
    dw = DeviceWorkload(wl)
    out1, lse1, plan = dw.run()
    out2, none = va.verify_attn_run(dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices,
                                    dw.last_page_len, dw.qo_indptr, None, None, plan,
                                    sm_scale=wl.sm_scale, want_lse=False)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_empty_batch_is_a_no_op(va):
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=64, prefix=("fixed", [10, 20]),
                               qo=("fixed", [0, 0]), mask="causal", seed=21)
    dw = DeviceWorkload(wl)
    out = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(0, 4, dtype=torch.float32, device="cuda")
    plan = dw.plan()
    assert plan.launches() == 0
    dw.run(plan=plan, out=out, lse=lse)
    torch.cuda.synchronize()


def test_bad_page_id_is_flagged_not_read(va):
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=128, prefix=("fixed", [100, 100]),
                               qo=("fixed", [3, 3]), mask="causal", seed=23)
    dw = DeviceWorkload(wl)
    bad = wl.kv_indices.copy()
    bad[wl.kv_indptr[1] + 1] = 1 << 30          # request 1, second page
    dw.kv_indices = torch.from_numpy(bad).cuda()
    out, lse, plan = dw.run()
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) & 1
    assert torch.isfinite(out.float()).all()
    # request 0 is unaffected
    rows = np.arange(3 * wl.h_q, dtype=np.int32)
    o, l = host_out(out, lse, wl.d)
    ro, rl = oracle.verify_attn_workload(wl, rows=rows)
    assert np.abs(o[rows] - ro).max() <= 1e-2 and np.abs(l[rows] - rl).max() <= 1e-3


def test_stale_plan_is_flagged(va):
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=64, prefix=("fixed", [40, 40]),
                               qo=("fixed", [3, 3]), mask="causal", seed=25)
    dw = DeviceWorkload(wl)
    plan = dw.plan()
    short = wl.qo_indptr.copy()
    short[2] = short[1] + 1                      # request 1 now has 1 token, the plan says 3
    dw.qo_indptr = torch.from_numpy(short).cuda()
    dw.run(plan=plan)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) & 2


def test_graph_capture_of_append_and_run(va):
    wl = synthetic.make_workload("llama3_8b_tree_verify")
    dw = DeviceWorkload(wl)
    plan = dw.plan()
    out = torch.empty_like(dw.q)
    lse = torch.empty(dw.q.shape[:2], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dw.append_drafts()
        dw.run(plan=plan, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dw.append_drafts()
        dw.run(plan=plan, out=out, lse=lse)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    compare(wl, out, lse, rows=synthetic.sample_rows(wl, 200))


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER)
def test_named_workload_matches_oracle(va, name):
    """Each named workload at full size, in the launch configuration the
    benchmark times (the planner's automatic choice): EVERY (token, query
    head) row of the call against the fp64 oracle at the strict bound
    (|out - oracle| <= 1e-2, |lse - oracle| <= 1e-3), after checking that the
    device page pool written by the append kernel is the oracle's pool, bit
    for bit."""
    wl = synthetic.make_workload(name)
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run()
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    of = out.float()
    assert torch.isfinite(of).all() and torch.isfinite(lse).all()
    raw = np.uint8 if wl.kv_dtype == synthetic.FP8 else np.uint16
    got_k = dw.k_cache.view(torch.uint8).cpu().numpy().view(raw)
    got_v = dw.v_cache.view(torch.uint8).cpu().numpy().view(raw)
    ok, ov = oracle.build_cache(wl)
    assert np.array_equal(got_k, ok) and np.array_equal(got_v, ov)
    compare(wl, out, lse, rows=None, caches=(ok, ov), strict=True)


@pytest.mark.parametrize("num_sms", [1, 3, 7])
@pytest.mark.parametrize("kernel", [3, 4], ids=["tc128", "tc256"])
@pytest.mark.parametrize("case", [
    dict(mask="tree"),
    dict(mask="causal"),
    dict(mask="tree", kv_dtype=synthetic.FP8),
], ids=["tree", "causal", "fp8_tree"])
def test_tcgen05_long_item_chains_match_oracle(va, num_sms, kernel, case):
    """The persistent tcgen05 kernel with few CTAs: each walks a long chain of
    items mixing one and two live Q tiles, split and whole kv ranges, prefix
    and prefill requests; the streaming of Q, keys, S / P and O from one item
    into the next must not leak anything across items."""
    wl = synthetic.make_custom(batch=4, h_q=16, h_kv=2, d=128,
                               prefix=("fixed", [700, 0, 90, 2000]),
                               qo=("fixed", [40, 33, 3, 17]), seed=41, **case)
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run(kernel=kernel, num_sms=num_sms, target_ctas=40)
    torch.cuda.synchronize()
    hd = plan.header()
    assert hd["kernel"] == kernel and hd["n_ctas"] == min(num_sms, hd["n_items"])
    assert hd["n_items"] > 2 * hd["n_ctas"]
    assert va.verify_attn_device_status(plan) == 0
    compare(wl, out, lse)


@pytest.mark.parametrize("kernel", [1, 2, 3, 4], ids=["mma64", "mma128", "tc128", "tc256"])
@pytest.mark.parametrize("case", [
    dict(mask="causal", value_std=3.0),
    dict(mask="tree", value_std=3.0),
    dict(mask="tree", value_std=3.0, kv_dtype=synthetic.FP8),
    dict(mask="causal", value_std=5.0),
], ids=["causal_std3", "tree_std3", "fp8_tree_std3", "causal_std5"])
def test_large_logits_match_oracle(va, kernel, case):
    """Logits with a standard deviation of 9 to 25 (q, k, v drawn with
    standard deviation 3 or 5): a row's running max keeps rising by far more
    than 2^8 from one 32-key chunk to the next, inside a key tile and from
    tile to tile, so every rescale path of the online softmax runs (the
    tcgen05 kernel's in-tile rescale of P already written to tensor memory,
    its rescale of O, a first visible chunk after fully masked ones) and
    must still match the fp64 oracle.  The output bound scales with the
    values: P is rounded to 16 bits (relative error <= 2^-8 for bf16, 2^-11
    for the fp8 variant's f16) before P V while the row sum keeps fp32, so
    |out - oracle| <= 2^-8 max|v| + fp32 rounding; a missing or wrong
    rescale is off by a factor 2^8 or more on some weights instead."""
    wl = synthetic.make_custom(batch=3, h_q=16, h_kv=2, d=128,
                               prefix=("fixed", [700, 300, 1500]),
                               qo=("fixed", [17, 40, 9]), seed=53, **case)
    v = oracle.decode_e4m3(wl.v_tok) * wl.v_scale if wl.kv_dtype == synthetic.FP8 \
        else oracle.decode_bf16(wl.v_tok)
    tol = 2.0 ** -8 * float(np.abs(v).max()) + 1e-3
    dw = DeviceWorkload(wl)
    for splits in (1, 0):
        out, lse, plan = dw.run(kernel=kernel, max_splits=splits)
        torch.cuda.synchronize()
        assert plan.header()["kernel"] == kernel
        assert va.verify_attn_device_status(plan) == 0
        compare(wl, out, lse, out_tol=tol)


@pytest.mark.parametrize("kernel", [2, 3, 4], ids=["mma128", "tc128", "tc256"])
def test_work_list_of_another_plan_is_flagged_not_read(va, kernel):
    """A workspace whose work list was overwritten by a later plan for a
    larger batch, then run with the earlier plan: the kernels must not index
    the call's tables with the foreign requests (they flag the items as a bad
    table instead), and the merge skips them.  Every index a kernel takes
    from the work list is checked against this call's plan before use, so
    the run is safe whatever the list holds."""
    small = synthetic.make_custom(batch=2, h_q=8, h_kv=2, d=128, prefix=("fixed", [300, 200]),
                                  qo=("fixed", [5, 9]), seed=61)
    # later requests longer: the longest-first list starts with requests >= 2
    big = synthetic.make_custom(batch=8, h_q=8, h_kv=2, d=128,
                                prefix=("fixed", [200 * (i + 1) for i in range(8)]),
                                qo=("fixed", [7] * 8), seed=62, with_values=False)
    dw = DeviceWorkload(small)
    opts = dict(kernel=kernel, num_sms=8)
    args_big = (big.kv_indptr, big.qo_indptr, big.last_page_len, big.mask_indptr, big.h_q, big.h_kv,
                big.d, big.page_size)
    args_small = (small.kv_indptr, small.qo_indptr, small.last_page_len, small.mask_indptr,
                  small.h_q, small.h_kv, small.d, small.page_size)
    # one workspace large enough for both plans, so that both upload into it
    need = max(va.verify_attn_plan_host(*args_big, **opts).workspace_bytes,
               va.verify_attn_plan_host(*args_small, **opts).workspace_bytes)
    ws = torch.empty(need, dtype=torch.uint8, device=dw.dev)
    plan_small = va.verify_attn_plan(*args_small, workspace=ws, device=dw.dev, **opts)
    plan_big = va.verify_attn_plan(*args_big, workspace=ws, device=dw.dev, **opts)
    assert plan_small.workspace.data_ptr() == plan_big.workspace.data_ptr() == ws.data_ptr()
    items = plan_big.items()
    assert (items[:plan_small.header()["n_items"], 0] >= small.batch).any()
    dw.run(plan=plan_small)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan_small) & 2

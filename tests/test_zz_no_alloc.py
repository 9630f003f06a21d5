"""The allocation-free entry point, verify_attn_run_static_scratch, for
callers that may not allocate device memory (their framework owns every
allocation, or allocation is forbidden on their hot path).  It must give the
same result as verify_attn_run, call after call, although its scratch is the
library's one static array rather than a caller workspace.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.  Works alone in a fresh process
and after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DeviceWorkload, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_gqa_gb300 as m
    return m


@pytest.mark.parametrize("name", ["llama3_8b_tree_verify", "tiny_verify"])
def test_static_scratch_matches_run_twice_in_a_row(va, name):
    wl = synthetic.make_workload(name)
    dw = DeviceWorkload(wl)
    ref_out, ref_lse, plan = dw.run()            # the existing entry point, caller workspace
    torch.cuda.synchronize()
    # a host-only plan: this caller never allocates a device workspace
    hplan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                     wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                     kv_dtype=wl.kv_dtype)
    if name == "llama3_8b_tree_verify":
        assert hplan.header()["n_merge"] > 0     # the split partials live in the static array
    assert hplan.workspace_bytes <= va.STATIC_SCRATCH_BYTES
    ref_o = ref_out.float().cpu().numpy()
    ref_l = ref_lse.cpu().numpy()
    for call in range(2):
        out = torch.full_like(dw.q, float("nan"))
        lse = torch.full(dw.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        # through the C ABI directly
        L = va.lib()
        rc = L.verify_attn_run_static_scratch(
            va._dp(dw.q), va._dp(dw.k_cache), va._dp(dw.v_cache), va._dp(dw.kv_indptr),
            va._dp(dw.kv_indices), va._dp(dw.last_page_len), va._dp(dw.qo_indptr),
            va._dp(dw.mask), va._dp(dw.mask_indptr), wl.h_q, wl.h_kv, wl.d, wl.page_size,
            ctypes.c_float(wl.sm_scale), ctypes.c_float(wl.k_scale), ctypes.c_float(wl.v_scale),
            va._dp(out), va._dp(lse), wl.num_pages, va._hp(hplan.host),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, va.status_string(rc)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.abs(o - ref_o).max() <= 1e-2
        assert np.abs(l - ref_l).max() <= 1e-3
        compare(wl, out, lse, rows=None if name == "tiny_verify" else synthetic.sample_rows(wl, 64))


def test_static_scratch_wrapper_fp8_two_q_tiles_with_merge(va):
    """The Python wrapper of the same entry point, on an fp8 cache with the
    two-Q-tile tcgen05 kernel and a plan forced to split (so the merge reads
    partials from the static array), twice in a row: equal to
    verify_attn_run with a caller workspace, and to the oracle."""
    wl = synthetic.make_custom(batch=2, h_q=16, h_kv=2, d=128, prefix=("fixed", [900, 130]),
                               qo=("fixed", [40, 20]), mask="tree", kv_dtype=synthetic.FP8,
                               seed=71)
    dw = DeviceWorkload(wl)
    opts = dict(kernel=4, target_ctas=64, min_chunk=128)
    ref_out, ref_lse, _ = dw.run(**opts)
    torch.cuda.synchronize()
    hplan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                     wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                     kv_dtype=wl.kv_dtype, **opts)
    hd = hplan.header()
    assert hd["kernel"] == 4 and hd["n_merge"] > 0
    for call in range(2):
        out = torch.full_like(dw.q, float("nan"))
        lse = torch.full(dw.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        va.verify_attn_run_static_scratch(dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr,
                                          dw.kv_indices, dw.last_page_len, dw.qo_indptr,
                                          dw.mask, dw.mask_indptr, hplan, sm_scale=wl.sm_scale,
                                          k_scale=wl.k_scale, v_scale=wl.v_scale, out=out,
                                          lse=lse)
        torch.cuda.synchronize()
        assert float((out.float() - ref_out.float()).abs().max()) <= 1e-2
        assert float((lse - ref_lse).abs().max()) <= 1e-3
        compare(wl, out, lse)


def test_static_scratch_refuses_plans_beyond_its_size(va):
    # 64 requests x 64 query heads with a long prefix, forced into many splits
    wl = synthetic.make_custom(batch=64, h_q=64, h_kv=8, d=128, prefix=("fixed", [8192] * 64),
                               qo=("fixed", [16] * 64), mask="causal", with_values=False)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, None, 64, 8,
                                    128, 16, min_chunk=64, target_ctas=600, max_splits=64)
    assert plan.workspace_bytes > va.STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(256)
    rc = va.lib().verify_attn_run_static_scratch(
        fake, fake, fake, fake, fake, fake, fake, None, None, 64, 8, 128, 16,
        ctypes.c_float(0.0), ctypes.c_float(1.0), ctypes.c_float(1.0), fake, None, 10,
        va._hp(plan.host), None)
    assert rc == -8


def test_static_scratch_status_reports_device_checks(va):
    """The static array's status word: 0 after a clean call; a page id
    outside the pool (which the kernels skip, zero-fill and flag) raises
    VA_DEV_BAD_PAGE, read once by verify_attn_static_scratch_status and
    cleared by the read."""
    wl = synthetic.make_custom(batch=2, h_q=4, h_kv=2, d=128, prefix=("fixed", [100, 100]),
                               qo=("fixed", [3, 3]), mask="causal", seed=23)
    dw = DeviceWorkload(wl)
    hplan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, None,
                                     wl.h_q, wl.h_kv, wl.d, wl.page_size)
    args = (dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices, dw.last_page_len,
            dw.qo_indptr, None, None, hplan)
    va.verify_attn_run_static_scratch(*args, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert va.verify_attn_static_scratch_status() == 0
    bad = wl.kv_indices.copy()
    bad[wl.kv_indptr[1] + 1] = 1 << 30          # request 1, second page
    out, lse = va.verify_attn_run_static_scratch(
        dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, torch.from_numpy(bad).cuda(),
        dw.last_page_len, dw.qo_indptr, None, None, hplan, sm_scale=wl.sm_scale)
    torch.cuda.synchronize()
    assert va.verify_attn_static_scratch_status() & 1     # VA_DEV_BAD_PAGE
    assert va.verify_attn_static_scratch_status() == 0    # cleared by the read
    assert torch.isfinite(out.float()).all()

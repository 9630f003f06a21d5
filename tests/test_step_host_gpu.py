"""GPU parity of the host-buffer step (verify_attn_step_host): the step's
inputs staged in one pinned host buffer, planned on the host, appended and
attended on the device, out and LSE copied back -- the same bytes as the
device-buffer fused call on the same plan, and every row within the strict
bound of the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import DeviceWorkload, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_gqa_gb300 as m
    return m


def _stage(wl):
    """The step's host arrays, each at a 256-byte offset of one pinned buffer."""
    fp8 = wl.kv_dtype == synthetic.FP8
    raw = np.uint8 if fp8 else np.int16
    kn, vn = wl.new_tokens()
    arrays = dict(q=wl.q.view(np.int16), k_new=kn.view(raw), v_new=vn.view(raw),
                  kv_indptr=wl.kv_indptr, kv_indices=wl.kv_indices,
                  last_page_len=wl.last_page_len, qo_indptr=wl.qo_indptr)
    if wl.mask is not None:
        arrays["mask"], arrays["mask_indptr"] = wl.mask, wl.mask_indptr
    offs, total = {}, 0
    for k, a in arrays.items():
        offs[k] = total
        total += (np.ascontiguousarray(a).nbytes + 255) // 256 * 256
    stage = torch.zeros(max(total, 256), dtype=torch.uint8).pin_memory()
    view = stage.numpy()
    for k, a in arrays.items():
        b = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
        view[offs[k]:offs[k] + b.size] = b
    return stage, offs


@pytest.mark.parametrize("name", ["tiny_verify", "llama3_8b_tree_verify",
                                  "codellama34b_chain_verify", "wide_tree_fp8_verify"])
def test_step_host_matches_fused_call_and_oracle(va, name):
    wl = synthetic.make_workload(name)
    dw = DeviceWorkload(wl)
    stage_h, offs = _stage(wl)
    stage_d = torch.empty_like(stage_h, device="cuda")
    n_out = wl.total_qo * wl.h_q * wl.dv * 2
    lse_off = (n_out + 255) // 256 * 256
    res_d = torch.empty(lse_off + wl.total_qo * wl.h_q * 4, dtype=torch.uint8, device="cuda")
    res_h = torch.zeros_like(res_d, device="cpu").pin_memory()
    out_d = res_d[:n_out].view(torch.bfloat16).view(wl.total_qo, wl.h_q, wl.dv)
    lse_d = res_d[lse_off:].view(torch.float32).view(wl.total_qo, wl.h_q)
    # the device-buffer fused call on its own plan: the reference bytes
    plan = dw.plan()
    ref_out, ref_lse = va.verify_attn_append_run(
        dw.k_new, dw.v_new, dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices,
        dw.last_page_len, dw.qo_indptr, dw.mask, dw.mask_indptr, plan, sm_scale=wl.sm_scale,
        k_scale=wl.k_scale, v_scale=wl.v_scale, early_reads=True)
    torch.cuda.synchronize()
    ws = torch.empty_like(plan.workspace)
    plan_buf = np.zeros(plan.host.nbytes, np.uint8)
    va.verify_attn_step_host(stage_h, stage_d, offs, wl.batch, wl.h_q, wl.h_kv, wl.d,
                             wl.page_size, dw.k_cache, dw.v_cache, out_d, lse_d, res_h, ws,
                             plan_buf, kv_dtype=wl.kv_dtype, num_sms=plan.header()["num_sms"],
                             sm_scale=wl.sm_scale, k_scale=wl.k_scale, v_scale=wl.v_scale,
                             early_reads=True, synchronize=True)
    hv = res_h.numpy()
    out_h = torch.from_numpy(hv[:n_out].view(np.int16).copy()).view(torch.bfloat16)
    lse_h = torch.from_numpy(hv[lse_off:lse_off + wl.total_qo * wl.h_q * 4].view(np.float32).copy())
    assert np.array_equal(out_h.view(torch.int16).numpy().reshape(-1),
                          ref_out.view(torch.int16).cpu().numpy().reshape(-1))
    assert np.array_equal(lse_h.numpy().view(np.uint32), ref_lse.cpu().numpy().reshape(-1).view(np.uint32))
    assert np.array_equal(plan_buf, plan.host)
    assert va.verify_attn_device_status(type(plan)(plan_buf, ws, plan.workspace_bytes, plan.batch,
                                                   plan.num_qo_heads, plan.num_kv_heads,
                                                   plan.head_dim, plan.page_size, plan.kv_dtype,
                                                   plan.has_mask, plan.total_qo)) == 0
    compare(wl, out_h.view(wl.total_qo, wl.h_q, wl.dv), lse_h.view(wl.total_qo, wl.h_q),
            caches=oracle.build_cache(wl), strict=True)


def test_step_host_separate_lse_buffer_and_no_lse(va):
    """out and LSE in separate device buffers (two copies back), and a step
    without LSE."""
    wl = synthetic.make_workload("tiny_verify")
    dw = DeviceWorkload(wl)
    stage_h, offs = _stage(wl)
    stage_d = torch.empty_like(stage_h, device="cuda")
    plan = dw.plan()
    ref_out, ref_lse = dw.run(plan)[:2]
    n_out = wl.total_qo * wl.h_q * wl.dv * 2
    lse_off = (n_out + 255) // 256 * 256
    out_d = torch.empty(wl.total_qo, wl.h_q, wl.dv, dtype=torch.bfloat16, device="cuda")
    lse_d = torch.empty(wl.total_qo, wl.h_q, dtype=torch.float32, device="cuda")
    res_h = torch.zeros(lse_off + wl.total_qo * wl.h_q * 4, dtype=torch.uint8).pin_memory()
    kw = dict(kv_dtype=wl.kv_dtype, num_sms=plan.header()["num_sms"], sm_scale=wl.sm_scale,
              k_scale=wl.k_scale, v_scale=wl.v_scale)
    ws = torch.empty_like(plan.workspace)
    va.verify_attn_step_host(stage_h, stage_d, offs, wl.batch, wl.h_q, wl.h_kv, wl.d,
                             wl.page_size, dw.k_cache, dw.v_cache, out_d, lse_d, res_h, ws,
                             np.zeros(plan.host.nbytes, np.uint8), **kw)
    hv = res_h.numpy()
    assert np.array_equal(hv[:n_out].view(np.int16), ref_out.view(torch.int16).cpu().numpy().reshape(-1))
    assert np.array_equal(hv[lse_off:].view(np.float32), ref_lse.cpu().numpy().reshape(-1))
    res2 = torch.zeros(n_out, dtype=torch.uint8).pin_memory()
    va.verify_attn_step_host(stage_h, stage_d, offs, wl.batch, wl.h_q, wl.h_kv, wl.d,
                             wl.page_size, dw.k_cache, dw.v_cache, out_d, None, res2, ws,
                             np.zeros(plan.host.nbytes, np.uint8), **kw)
    assert np.array_equal(res2.numpy().view(np.int16), ref_out.view(torch.int16).cpu().numpy().reshape(-1))


def test_step_host_quantising_append_and_nhd(va):
    """The step with append options: bf16 drafts quantised into an fp8 NHD
    cache (plan option kv_layout=nhd, e4m3 MMAs off and on), against the
    oracle over its own quantised cache, and the pool bit-equal to it."""
    base = dict(batch=2, h_q=32, h_kv=8, d=128, prefix=("fixed", [700, 260]),
                qo=("fixed", [40, 9]), mask="tree", seed=5, kv_layout="nhd")
    wf = synthetic.make_custom(kv_dtype=synthetic.FP8, **base)
    wb = synthetic.make_custom(**base)
    kn, vn = wb.new_tokens()
    kc, vc = oracle.build_cache(wf)
    oracle.paged_kv_append_ex(kn, vn, wf.qo_indptr, wf.kv_indptr, wf.kv_indices,
                              wf.last_page_len, wf.page_size, wf.num_pages, kc, vc,
                              cache_fp8=True, quantize=True, k_scale=wf.k_scale,
                              v_scale=wf.v_scale, kv_layout=1)
    arrays = dict(q=wf.q.view(np.int16), k_new=kn.view(np.int16), v_new=vn.view(np.int16),
                  kv_indptr=wf.kv_indptr, kv_indices=wf.kv_indices,
                  last_page_len=wf.last_page_len, qo_indptr=wf.qo_indptr, mask=wf.mask,
                  mask_indptr=wf.mask_indptr)
    offs, total = {}, 0
    for k, a in arrays.items():
        offs[k] = total
        total += (np.ascontiguousarray(a).nbytes + 255) // 256 * 256
    stage_h = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for k, a in arrays.items():
        b = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
        stage_h.numpy()[offs[k]:offs[k] + b.size] = b
    stage_d = torch.empty_like(stage_h, device="cuda")
    ao = va.AppendOptions()
    ao.quantize, ao.k_scale, ao.v_scale, ao.kv_layout = 1, wf.k_scale, wf.v_scale, va.LAYOUT_NHD
    n_out = wf.total_qo * wf.h_q * wf.dv * 2
    lse_off = (n_out + 255) // 256 * 256
    for q_fp8 in (False, True):
        dw = DeviceWorkload(wf)   # the pool holds every token, the drafts still as fp8 codes
        res_d = torch.empty(lse_off + wf.total_qo * wf.h_q * 4, dtype=torch.uint8, device="cuda")
        res_h = torch.zeros_like(res_d, device="cpu").pin_memory()
        out_d = res_d[:n_out].view(torch.bfloat16).view(wf.total_qo, wf.h_q, wf.dv)
        lse_d = res_d[lse_off:].view(torch.float32).view(wf.total_qo, wf.h_q)
        plan = dw.plan(q_fp8=q_fp8)
        ws = torch.empty_like(plan.workspace)
        va.verify_attn_step_host(stage_h, stage_d, offs, wf.batch, wf.h_q, wf.h_kv, wf.d,
                                 wf.page_size, dw.k_cache, dw.v_cache, out_d, lse_d, res_h, ws,
                                 np.zeros(plan.host.nbytes, np.uint8), kv_dtype=wf.kv_dtype,
                                 sm_scale=wf.sm_scale, k_scale=wf.k_scale, v_scale=wf.v_scale,
                                 append_options=ao, kv_layout="nhd", q_fp8=q_fp8)
        raw = lambda t: t.view(torch.uint8).cpu().numpy()
        assert np.array_equal(raw(dw.k_cache), kc) and np.array_equal(raw(dw.v_cache), vc)
        hv = res_h.numpy()
        out_h = torch.from_numpy(hv[:n_out].view(np.int16).copy()).view(torch.bfloat16)
        lse_h = torch.from_numpy(hv[lse_off:].view(np.float32).copy())
        if q_fp8:
            from test_fp8_mma_gpu import check as check_e4m3
            check_e4m3(wf, out_h.view(wf.total_qo, wf.h_q, wf.dv), lse_h.view(wf.total_qo, wf.h_q),
                       caches=(kc, vc))
        else:
            compare(wf, out_h.view(wf.total_qo, wf.h_q, wf.dv), lse_h.view(wf.total_qo, wf.h_q),
                    caches=(kc, vc))


def test_prepared_host_step_matches_the_plain_call(va):
    """HostStep (the binding's call with its arguments marshalled once) gives
    the bytes of verify_attn_step_host, also with the cache pair swapped."""
    wl = synthetic.make_workload("llama3_8b_tree_verify")
    dws = [DeviceWorkload(wl), DeviceWorkload(wl)]
    stage_h, offs = _stage(wl)
    stage_d = torch.empty_like(stage_h, device="cuda")
    n_out = wl.total_qo * wl.h_q * wl.dv * 2
    lse_off = (n_out + 255) // 256 * 256
    res_d = torch.empty(lse_off + wl.total_qo * wl.h_q * 4, dtype=torch.uint8, device="cuda")
    out_d = res_d[:n_out].view(torch.bfloat16).view(wl.total_qo, wl.h_q, wl.dv)
    lse_d = res_d[lse_off:].view(torch.float32).view(wl.total_qo, wl.h_q)
    plan = dws[0].plan()
    ws = torch.empty_like(plan.workspace)
    kw = dict(kv_dtype=wl.kv_dtype, num_sms=plan.header()["num_sms"], sm_scale=wl.sm_scale,
              k_scale=wl.k_scale, v_scale=wl.v_scale, early_reads=True)
    ref = torch.zeros_like(res_d, device="cpu").pin_memory()
    va.verify_attn_step_host(stage_h, stage_d, offs, wl.batch, wl.h_q, wl.h_kv, wl.d,
                             wl.page_size, dws[0].k_cache, dws[0].v_cache, out_d, lse_d, ref, ws,
                             np.zeros(plan.host.nbytes, np.uint8), **kw)
    res_h = torch.zeros_like(ref).pin_memory()
    step = va.HostStep(stage_h, stage_d, offs, wl.batch, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                       dws[0].k_cache, dws[0].v_cache, out_d, lse_d, res_h, ws,
                       np.zeros(plan.host.nbytes, np.uint8), **kw)
    for dw in (dws[0], dws[1], dws[0]):
        res_h.zero_()
        step(dw.k_cache, dw.v_cache)
        assert np.array_equal(res_h.numpy(), ref.numpy())

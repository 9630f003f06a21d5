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

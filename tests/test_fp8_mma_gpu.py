"""GPU parity of the e4m3 tensor-core path (plan option q_fp8: both MMAs of
the tcgen05 variants run kind::f8f6f4 on e4m3 operands) against the oracle
with e4m3 queries.

What the two sides share exactly: each query row is quantised the same way
(amax / 448 scale in binary32, round-to-nearest-even satfinite codes), the
cache codes are the same bytes, and Q K^T of e4m3 codes is a sum of exact
products.  So the logits, hence the LSE, keep the fp32 bound of the bf16
path (1e-3).

What the kernel adds: P is fed to the PV MMA as e4m3.  P is taken against a
lazily raised reference (the row's maximum P lies in [1, 2^8]), so a key whose
probability relative to the row maximum is p carries a quantisation error of
at most 2^-4 p (three fraction bits, round to nearest) plus, below e4m3's
normal range, one subnormal step, 2^-10 in the units where the row maximum
is 1.  The kernel settles a tile's reference before it writes any of the
tile's P, so each P is rounded once; the bound below keeps a second
subnormal step as margin (a variant that raised the reference chunk by
chunk rescaled P already written and rounded it once more).  Per element of
the output:

    |out - oracle| <= sum_j e_j |v_j| / sum_j p_j,
    e_j = 2^-4 p_j + min(p_j, 2^-9)

on top of the bf16 path's 1e-2 and the bf16 half-spacing of the output.  The
normaliser sums P before quantisation, so the bound is not relative.  Treating
the roundings as independent and uniform on [-e_j, e_j] gives the expected
RMS error sqrt(sum_j e_j^2 v_j^2 / 3) / sum_j p_j, which the measured RMS
must not exceed twice over."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import DeviceWorkload, LSE_TOL, OUT_TOL, bf16_half_spacing, host_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def va():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_gqa_gb300 as m
    return m


def _keys(wl, cache, b, h):
    """Dequantised (codes only) keys or values of request b, KV head h, in
    key order: [kv_len, d] fp64."""
    n = int(wl.kv_lens[b])
    pos = np.arange(n)
    pages = wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b + 1]][pos // wl.page_size]
    slot = pos % wl.page_size
    codes = cache[pages, slot, h] if wl.nhd else cache[pages, h, slot]
    return _e4m3_table()[codes]


def _e4m3_table():
    """The oracle's decoding of all 256 e4m3 codes (indexed by code)."""
    global _TABLE
    if _TABLE is None:
        _TABLE = oracle.decode_e4m3(np.arange(256, dtype=np.uint8))
    return _TABLE


_TABLE = None


def pv_bounds(wl, kc, vc, rows):
    """Per sampled row: the element-wise worst-case bound and the expected
    variance of the e4m3-P error (the module docstring's formulas), from the
    oracle's own quantised queries and the cache codes."""
    qd = torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16).double().numpy()
    qd = qd.reshape(-1, wl.h_q, wl.d)
    bound = np.zeros((len(rows), wl.d))
    var = np.zeros((len(rows), wl.d))
    tok, qh = np.divmod(np.asarray(rows, np.int64), wl.h_q)
    req = np.searchsorted(wl.qo_indptr, tok, side="right") - 1
    kvh = qh // wl.group
    cache = {}
    for i in np.lexsort((kvh, req)):          # one (request, KV head) at a time
        b, h = int(req[i]), int(kvh[i])
        t = int(tok[i]) - int(wl.qo_indptr[b])
        if (b, h) not in cache:
            cache = {(b, h): (_keys(wl, kc, b, h) * wl.k_scale, _keys(wl, vc, b, h) * wl.v_scale)}
        K, V = cache[(b, h)]
        pre, L = int(wl.prefix_lens[b]), int(wl.qo_lens[b])
        vis = np.ones(pre + L, bool)
        if wl.mask_full is not None:
            vis[:] = wl.mask_full[b][t]
        elif wl.mask_dense is not None:
            vis[pre:] = wl.mask_dense[b][t]
        else:
            vis[pre + t + 1:] = False
        codes, qsc = oracle.quantize_q_e4m3(qd[tok[i], qh[i]])
        q8 = _e4m3_table()[codes] * qsc
        s = (K[vis] @ q8) * wl.sm_scale
        p = np.exp(s - s.max())
        e = 2.0 ** -4 * p + np.minimum(p, 2.0 ** -9)
        Va = np.abs(V[vis])
        bound[i] = (e @ Va) / p.sum()
        var[i] = ((e * e) @ (Va * Va)) / 3.0 / p.sum() ** 2
    return bound, var


def check(wl, out, lse, rows=None, caches=None):
    """Device result (all rows, or the flat rows given) against the oracle
    with e4m3 queries, to the bounds in the module docstring."""
    kc, vc = caches if caches is not None else oracle.build_cache(wl)
    o, l = host_out(out, lse, wl.d)
    ref_o, ref_l = oracle.verify_attn_workload(wl, rows=rows, caches=(kc, vc), q_fp8=True)
    if rows is None:
        rows = np.arange(o.shape[0])
    else:
        o, l = o[rows], l[rows]
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), "-inf LSE rows differ"
    assert np.all(o[~fin] == 0.0)
    err_l = float(np.abs(l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    assert err_l <= LSE_TOL, "max |lse - oracle| = %g" % err_l
    bound, var = pv_bounds(wl, kc, vc, rows[fin])
    diff = np.abs(o[fin] - ref_o[fin])
    excess = diff - (bound + OUT_TOL + bf16_half_spacing(ref_o[fin]))
    assert excess.size == 0 or excess.max() <= 0, \
        "max |out - oracle| = %g beyond its bound by %g" % (diff.max(), excess.max())
    rms, pred = float(np.sqrt(np.mean(diff ** 2))), float(np.sqrt(np.mean(var)))
    print("e4m3 parity %s: max |out err| %.4g (bound up to %.4g), max |lse err| %.3g, "
          "RMS %.4g (expected %.4g)" % (wl.name, diff.max(), bound.max(), err_l, rms, pred))
    assert rms <= 2.0 * pred + 1e-3, "RMS error %g vs expected %g" % (rms, pred)
    return float(diff.max()), err_l, rms, pred


CASES = {
    "tree_ragged": dict(batch=3, h_q=16, h_kv=2, d=128, prefix=("fixed", [700, 0, 90]),
                        qo=("fixed", [17, 40, 3]), mask="tree", seed=121),
    "wide_tree_small": dict(batch=2, h_q=32, h_kv=8, d=128, prefix=("fixed", [1000, 300]),
                            qo=("fixed", [64, 20]), mask="tree", seed=122),
    "chain": dict(batch=4, h_q=64, h_kv=8, d=128, prefix=("fixed", [2000, 513, 31, 0]),
                  qo=("fixed", [8, 1, 5, 3]), mask="causal", seed=123),
    "nhd_full_mask": dict(batch=2, h_q=16, h_kv=2, d=128, prefix=("fixed", [400, 77]),
                          qo=("fixed", [30, 9]), mask="tree", kv_layout="nhd",
                          mask_layout="full", prefix_visible="random", seed=124),
}


@pytest.mark.parametrize("kernel", [3, 4], ids=["tc128", "tc256"])
@pytest.mark.parametrize("name", list(CASES))
def test_e4m3_mma_matches_oracle(va, kernel, name):
    wl = synthetic.make_custom(kv_dtype=synthetic.FP8, **CASES[name])
    dw = DeviceWorkload(wl)
    kc, vc = oracle.build_cache(wl)
    for splits in (1, 0):
        out, lse, plan = dw.run(kernel=kernel, max_splits=splits, target_ctas=300, q_fp8=True)
        torch.cuda.synchronize()
        assert plan.header()["kernel"] == kernel
        assert va.verify_attn_device_status(plan) == 0
        check(wl, out, lse, caches=(kc, vc))


def test_e4m3_mma_full_size_wide_tree(va):
    """The wide fp8 tree at its full size (8 requests, 32K prefix, 64-node
    trees) with the plan the auto rules pick plus q_fp8: sampled rows."""
    wl = synthetic.make_workload("wide_tree_fp8_verify")
    dw = DeviceWorkload(wl)
    out, lse, plan = dw.run(q_fp8=True)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    rows = synthetic.sample_rows(wl, 48)
    check(wl, out, lse, rows=rows)


def test_e4m3_mma_through_the_fused_call(va):
    """verify_attn_append_run with an e4m3 plan: bf16 drafts quantised into
    the cache, then attended with e4m3 queries, in one call."""
    base = CASES["wide_tree_small"]
    wf = synthetic.make_custom(kv_dtype=synthetic.FP8, **base)
    wb = synthetic.make_custom(**base)
    kn, vn = wb.new_tokens()
    kc, vc = oracle.build_cache(wf)
    oracle.paged_kv_append_quant(kn, vn, wf.k_scale, wf.v_scale, wf.qo_indptr, wf.kv_indptr,
                                 wf.kv_indices, wf.last_page_len, wf.page_size, wf.num_pages,
                                 kc, vc)
    dw = DeviceWorkload(wf)
    plan = dw.plan(q_fp8=True)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16))).cuda().view(torch.bfloat16)
    out, lse = va.verify_attn_append_run(
        to(kn), to(vn), dw.q, dw.k_cache, dw.v_cache, dw.kv_indptr, dw.kv_indices,
        dw.last_page_len, dw.qo_indptr, dw.mask, dw.mask_indptr, plan, sm_scale=wf.sm_scale,
        k_scale=wf.k_scale, v_scale=wf.v_scale, append_k_scale=wf.k_scale,
        append_v_scale=wf.v_scale)
    torch.cuda.synchronize()
    assert va.verify_attn_device_status(plan) == 0
    check(wf, out, lse, caches=(kc, vc))


def test_e4m3_mma_zero_and_constant_rows(va):
    """Degenerate query rows: all-zero rows (scale 1, every code 0: uniform
    attention, LSE = log of the visible count) and rows of one repeated
    value (every code 448)."""
    wl = synthetic.make_custom(kv_dtype=synthetic.FP8, **CASES["tree_ragged"])
    q = wl.q.copy().reshape(-1, wl.h_q, wl.d)
    q[0] = 0
    q[1, :, :] = np.uint16(0x3F80)          # bf16 1.0
    q[2, ::2, :] = np.uint16(0xC2F0)        # bf16 -120
    wl.q = q.reshape(wl.q.shape)
    dw = DeviceWorkload(wl)
    for kernel in (3, 4):
        out, lse, plan = dw.run(kernel=kernel, q_fp8=True)
        torch.cuda.synchronize()
        check(wl, out, lse)

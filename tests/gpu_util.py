"""Helpers for the GPU parity tests: put a synthetic workload on the device,
run the CUDA path through the C ABI, and compare with the fp64 oracle."""
import numpy as np
import torch

import oracle
import synthetic

OUT_TOL = 1e-2   # max |out - oracle| (bf16 inputs, fp32 accumulation, bf16 output)
LSE_TOL = 1e-3   # max |lse - oracle|


def to_dev(a, dev, view=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return t.view(view) if view is not None else t


class DeviceWorkload:
    """A workload on the GPU: q, the draft K/V, the index tables, and a page
    pool written by the library's own append kernel (sentinel NaN bytes
    first, then every prefix and draft token, then the drafts again as a
    verify step does)."""

    def __init__(self, wl, dev="cuda", append=True):
        import speculative_decoding_verify_gqa_gb300 as va
        self.wl = wl
        self.dev = torch.device(dev)
        fp8 = wl.kv_dtype == synthetic.FP8
        self.kvd = torch.float8_e4m3fn if fp8 else torch.bfloat16
        raw = np.uint8 if fp8 else np.int16
        self.q = to_dev(wl.q.view(np.int16), dev, torch.bfloat16)
        self.kv_indptr = to_dev(wl.kv_indptr, dev)
        self.kv_indices = to_dev(wl.kv_indices, dev)
        self.last_page_len = to_dev(wl.last_page_len, dev)
        self.qo_indptr = to_dev(wl.qo_indptr, dev)
        self.mask = None if wl.mask is None else to_dev(wl.mask, dev)
        self.mask_indptr = None if wl.mask_indptr is None else to_dev(wl.mask_indptr, dev)
        shape = ((wl.num_pages, wl.page_size, wl.h_kv, wl.d) if wl.nhd
                 else (wl.num_pages, wl.h_kv, wl.page_size, wl.d))
        vshape = shape[:3] + (wl.dv,)
        self.q_pos = None if wl.q_pos is None else to_dev(wl.q_pos, dev)
        self.kv_pos = None if wl.kv_pos is None else to_dev(wl.kv_pos, dev)
        self.new_pos = None if wl.kv_pos is None else to_dev(wl.new_positions(), dev)
        # 0xFF bytes: NaN in bf16 and in fp8-e4m3
        if fp8:
            self.k_cache = torch.full(shape, 0xFF, dtype=torch.uint8, device=dev).view(self.kvd)
            self.v_cache = torch.full(vshape, 0xFF, dtype=torch.uint8, device=dev).view(self.kvd)
        else:
            self.k_cache = torch.full(shape, -1, dtype=torch.int16, device=dev).view(self.kvd)
            self.v_cache = torch.full(vshape, -1, dtype=torch.int16, device=dev).view(self.kvd)
        kn, vn = wl.new_tokens()
        self.k_new = to_dev(kn.view(raw), dev, self.kvd)
        self.v_new = to_dev(vn.view(raw), dev, self.kvd)
        if append:
            k_tok = to_dev(wl.k_tok.view(raw), dev, self.kvd)
            v_tok = to_dev(wl.v_tok.view(raw), dev, self.kvd)
            tok_indptr = to_dev(wl.tok_indptr.astype(np.int32), dev)
            va.paged_kv_append(k_tok, v_tok, tok_indptr, self.kv_indptr, self.kv_indices,
                               self.last_page_len, self.k_cache, self.v_cache,
                               kv_layout=wl.kv_layout, positions=self.kv_pos,
                               rope_theta=wl.rope_theta or 0.0)
            del k_tok, v_tok
            self.append_drafts()

    def append_drafts(self, status=None):
        import speculative_decoding_verify_gqa_gb300 as va
        wl = self.wl
        va.paged_kv_append(self.k_new, self.v_new, self.qo_indptr, self.kv_indptr,
                           self.kv_indices, self.last_page_len, self.k_cache, self.v_cache,
                           status=status, kv_layout=wl.kv_layout, positions=self.new_pos,
                           rope_theta=wl.rope_theta or 0.0)

    def features(self):
        wl = self.wl
        f = dict(kv_layout=wl.kv_layout, mask_layout=wl.mask_layout, rope=wl.q_pos is not None)
        if wl.dv != wl.d:
            f["head_dim_v"] = wl.dv
        return f

    def plan(self, **opts):
        import speculative_decoding_verify_gqa_gb300 as va
        wl = self.wl
        o = self.features()
        o.update(opts)
        return va.verify_attn_plan(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, wl.mask_indptr,
                                   wl.h_q, wl.h_kv, wl.d, wl.page_size, kv_dtype=wl.kv_dtype,
                                   device=self.dev, **o)

    def run(self, plan=None, out=None, lse=None, **opts):
        import speculative_decoding_verify_gqa_gb300 as va
        wl = self.wl
        if plan is None:
            plan = self.plan(**opts)
        out, lse = va.verify_attn_run(self.q, self.k_cache, self.v_cache, self.kv_indptr,
                                      self.kv_indices, self.last_page_len, self.qo_indptr,
                                      self.mask, self.mask_indptr, plan, sm_scale=wl.sm_scale,
                                      k_scale=wl.k_scale, v_scale=wl.v_scale, out=out, lse=lse,
                                      q_position=self.q_pos, rope_theta=wl.rope_theta or 0.0)
        return out, lse, plan


def host_out(out, lse, d):
    o = out.float().cpu().numpy().reshape(-1, d).astype(np.float64)
    l = lse.cpu().numpy().reshape(-1).astype(np.float64)
    return o, l


def bf16_half_spacing(x):
    """Half the spacing of the bf16 grid at |x| (8 significant bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def compare(wl, out, lse, rows=None, caches=None, nthreads=None, strict=False, out_tol=OUT_TOL):
    """Errors of the device result (all rows, or the flat rows given) against
    the oracle.  Asserts -inf agreement, |lse - oracle| <= 1e-3 and
    |out - oracle| <= out_tol (1e-2 unless given) + half the bf16 spacing at
    the oracle value (the output is bf16: where |out| >= 4 that spacing alone
    exceeds 1e-2); strict=True asserts the plain out_tol on every element."""
    o, l = host_out(out, lse, wl.dv)
    ref_o, ref_l = oracle.verify_attn_workload(wl, rows=rows, caches=caches, nthreads=nthreads)
    if rows is not None:
        o, l = o[rows], l[rows]
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), "-inf LSE rows differ"
    assert np.all(l[~fin] == -np.inf)
    assert np.all(o[~fin] == 0.0)
    diff = np.abs(o - ref_o)
    err_o = float(diff.max()) if o.size else 0.0
    err_l = float(np.abs(l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    if strict:
        assert err_o <= out_tol, "max |out - oracle| = %g" % err_o
    else:
        excess = diff - (out_tol + bf16_half_spacing(ref_o))
        assert o.size == 0 or excess.max() <= 0, \
            "max |out - oracle| = %g exceeds %g + bf16 half-spacing" % (err_o, out_tol)
    assert err_l <= LSE_TOL, "max |lse - oracle| = %g" % err_l
    return err_o, err_l

"""Pure-Python scalar brute force of verify attention for tiny inputs --
TEST INFRASTRUCTURE (a second, independent statement of the definition that
pins the C oracle; it shares no code with it).

For each request b, token t and query head qh it walks key positions j of the
request one by one, finds each key through the page table (page
``kv_indices[kv_indptr[b] + j // page_size]``, slot ``j % page_size``),
decides visibility from the rule (prefix always visible; draft column u
visible iff mask bit (t, u) is set, or u <= t without a mask), and evaluates
``lse = log(sum exp(s_j))`` and ``out = sum exp(s_j - lse) v_j`` with
``math.fsum``.  Decoding uses torch's own dtype casts (a library routine),
not the oracle's decoder.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def _decode(bits: np.ndarray, kv_fp8: bool) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits))
    if kv_fp8:
        return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return t.view(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()


def _rotate(x, pos, theta, scale):
    """Rotary embedding of one row, pair (i, i + d/2) as a point in the plane
    turned by pos / scale * theta^(-2i/d) radians counter-clockwise."""
    d = len(x)
    h = d // 2
    y = list(x)
    for i in range(h):
        a = pos / scale * theta ** (-2.0 * i / d)
        y[i] = x[i] * math.cos(a) - x[i + h] * math.sin(a)
        y[i + h] = x[i] * math.sin(a) + x[i + h] * math.cos(a)
    return y


def _round_bf16(x: float) -> float:
    """x rounded to the nearest bf16 value (8 significant bits; ties to even,
    Python's round()), normal range only."""
    if x == 0.0 or not math.isfinite(x):
        return x
    m, e = math.frexp(x)            # x = m * 2^e, 0.5 <= |m| < 1
    return math.ldexp(round(m * 256.0), e - 8)


def verify_attn(q, k_cache, v_cache, kv_fp8, kv_indptr, kv_indices, last_page_len, qo_indptr,
                mask, mask_indptr, h_q, h_kv, d, page_size, sm_scale, k_scale=1.0, v_scale=1.0,
                kv_layout=0, mask_layout=0, q_pos=None, rope_theta=0.0, rope_scale=1.0):
    """kv_layout 1: the cache is [pages, page_size, h_kv, d]; mask_layout 1:
    request b's mask is L rows of kv_len bits (prefix included); q_pos: each
    query row is rotated at its token's position and rounded to bf16 before
    the dot products.  The value rows' width is v_cache's last axis (it may
    differ from d); out rows have that width."""
    qd = _decode(q, False)
    kd = _decode(k_cache, kv_fp8)
    vd = _decode(v_cache, kv_fp8)
    if kv_layout == 1:   # view as [pages, h_kv, P, d] by swapping the middle axes
        kd = kd.transpose(0, 2, 1, 3)
        vd = vd.transpose(0, 2, 1, 3)
    G = h_q // h_kv
    dv = vd.shape[-1]
    total = int(qo_indptr[-1])
    out = np.zeros((total * h_q, dv))
    lse = np.zeros(total * h_q)
    for b in range(len(qo_indptr) - 1):
        npg = int(kv_indptr[b + 1] - kv_indptr[b])
        kv_len = 0 if npg == 0 else (npg - 1) * page_size + int(last_page_len[b])
        L = int(qo_indptr[b + 1] - qo_indptr[b])
        prefix = kv_len - L
        for t in range(L):
            tok = int(qo_indptr[b]) + t
            for qh in range(h_q):
                h = qh // G
                logits, values = [], []
                qrow = [float(qd[tok, qh, e]) for e in range(d)]
                if q_pos is not None:
                    qrow = [_round_bf16(v) for v in
                            _rotate(qrow, float(q_pos[tok]), rope_theta, rope_scale)]
                for j in range(kv_len):
                    if mask is not None and mask_layout == 1:
                        bit = int(mask_indptr[b]) + t * kv_len + j
                        if (int(mask[bit // 8]) >> (bit % 8)) & 1 == 0:
                            continue
                    elif j >= prefix:
                        u = j - prefix
                        if mask is None:
                            vis = u <= t
                        else:
                            bit = int(mask_indptr[b]) + t * L + u
                            vis = (int(mask[bit // 8]) >> (bit % 8)) & 1 == 1
                        if not vis:
                            continue
                    page = int(kv_indices[int(kv_indptr[b]) + j // page_size])
                    slot = j % page_size
                    dot = math.fsum(qrow[e] * float(kd[page, h, slot, e]) * k_scale
                                    for e in range(d))
                    logits.append(sm_scale * dot)
                    values.append([float(vd[page, h, slot, e]) * v_scale for e in range(dv)])
                row = tok * h_q + qh
                if not logits:
                    lse[row] = -math.inf
                    continue
                mx = max(logits)
                l = mx + math.log(math.fsum(math.exp(s - mx) for s in logits))
                lse[row] = l
                w = [math.exp(s - l) for s in logits]
                for e in range(dv):
                    out[row, e] = math.fsum(w[j] * values[j][e] for j in range(len(w)))
    return out, lse

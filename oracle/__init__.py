"""fp64 CPU oracle for paged-KV GQA verify attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arm may import this package.  The product path (the package
``speculative_decoding_verify_gqa_gb300``) never imports it, and this package
never imports the product: the two share nothing but the seeded input
generators in ``synthetic``.

The arithmetic lives in ``verify_attn_oracle.c`` (plain C, double precision,
the definition written out: gather the pages, build the dense mask, softmax,
LSE).  This module compiles it with gcc on first use and wraps it with ctypes.
``brute.py`` holds an independent pure-Python scalar version for tiny inputs.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
what the source pages and the mathematics fix (triu mask == causal, chain tree
== causal, GQA == MHA on expanded K/V, split + LSE merge == unsplit, L = 1 ==
single-query decode, tree row == decode over its root path, closed forms,
hand-worked golden cases, fp8/bf16 decode tables, brute force).  No function
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, no fast-math: IEEE double semantics)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11",
                           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_decode_bf16.restype = dbl
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_e4m3.restype = dbl
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_kv_len.restype = i64
        lib.oracle_kv_len.argtypes = [P, P, i32, i32]
        lib.oracle_dense_attention.restype = None
        lib.oracle_dense_attention.argtypes = [i32, i32, i32, P, i64, P, P, i64, P, dbl, P, P, P]
        lib.oracle_verify_attn.restype = i32
        lib.oracle_verify_attn.argtypes = [P, P, P, i32, P, P, P, P, P, P, i32, i32, i32, i32,
                                           i32, i32, dbl, dbl, dbl, P, i64, P, P, i32]
        lib.oracle_attn_range.restype = i32
        lib.oracle_attn_range.argtypes = [P, P, P, i32, P, P, P, P, P, P, i32, i32, i32, i32,
                                          i32, i32, dbl, dbl, dbl, i32, i64, i32, i64, i64,
                                          P, P]
        lib.oracle_merge_partials.restype = None
        lib.oracle_merge_partials.argtypes = [i32, i32, i32, P, P, P, P]
        lib.oracle_paged_kv_append.restype = i32
        lib.oracle_paged_kv_append.argtypes = [P, P, i32, P, P, P, P, i32, i32, i32, i32, i32,
                                               P, P]
        lib.oracle_encode_e4m3_satfinite.restype = ctypes.c_uint8
        lib.oracle_encode_e4m3_satfinite.argtypes = [ctypes.c_float]
        lib.oracle_div_f32.restype = ctypes.c_float
        lib.oracle_div_f32.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.oracle_paged_kv_append_quant.restype = i32
        lib.oracle_paged_kv_append_quant.argtypes = [P, P, ctypes.c_float, ctypes.c_float, P, P,
                                                     P, P, i32, i32, i32, i32, i32, P, P]
        lib.oracle_encode_bf16.restype = ctypes.c_uint16
        lib.oracle_encode_bf16.argtypes = [dbl]
        lib.oracle_rope_vec.restype = None
        lib.oracle_rope_vec.argtypes = [P, i32, dbl, dbl, dbl]
        lib.oracle_paged_kv_append_ex.restype = i32
        lib.oracle_paged_kv_append_ex.argtypes = [P, P, i32, i32, ctypes.c_float, ctypes.c_float,
                                                  i32, P, dbl, dbl, P, P, P, P, i32, i32, i32,
                                                  i32, i32, P, P]
        lib.oracle_verify_attn_ex.restype = i32
        lib.oracle_verify_attn_ex.argtypes = [P, P, P, i32, i32, P, P, P, P, P, P, i32, P, dbl,
                                              dbl, i32, i32, i32, i32, i32, i32, i32, dbl, dbl,
                                              dbl, P, i64, P, P, i32]
        lib.oracle_quantize_q_e4m3.restype = ctypes.c_float
        lib.oracle_quantize_q_e4m3.argtypes = [P, i32, P]
        lib.oracle_verify_attn_dv.restype = i32
        lib.oracle_verify_attn_dv.argtypes = [P, P, P, i32, i32, P, P, P, P, P, P, i32, P, dbl,
                                              dbl, i32, i32, i32, i32, i32, i32, i32, i32, dbl,
                                              dbl, dbl, P, i64, P, P, i32]
        lib.oracle_paged_kv_append_dv.restype = i32
        lib.oracle_paged_kv_append_dv.argtypes = [P, P, i32, i32, ctypes.c_float, ctypes.c_float,
                                                  i32, P, dbl, dbl, P, P, P, P, i32, i32, i32,
                                                  i32, i32, i32, P, P]
        lib.oracle_dense_attention_dv.restype = None
        lib.oracle_dense_attention_dv.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, i64, P,
                                                  dbl, P, P, P]
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def decode_bf16(bits) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).reshape(-1)
    return np.array([lib.oracle_decode_bf16(int(x)) for x in flat]).reshape(np.shape(bits))


def decode_e4m3(bits) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint8).reshape(-1)
    return np.array([lib.oracle_decode_e4m3(int(x)) for x in flat]).reshape(np.shape(bits))


def dense_attention(Q, K, V, M, scale):
    """softmax(scale * Q K^T + M) V and its natural-log LSE, row by row, in fp64.
    Q [n, d], K [m, d], V [m, dv], M [n, m] additive; out [n, dv]."""
    lib = _load()
    Q = _c(Q, np.float64); K = _c(K, np.float64); V = _c(V, np.float64); M = _c(M, np.float64)
    n, d = Q.shape
    m = K.shape[0]
    dv = V.shape[1]
    out = np.zeros((n, dv)); lse = np.zeros(n)
    s = np.zeros(max(m, 1))
    if dv == d:
        lib.oracle_dense_attention(n, m, d, _p(Q), d, _p(K), _p(V), d, _p(M), float(scale),
                                   _p(out), _p(lse), _p(s))
    else:
        lib.oracle_dense_attention_dv(n, m, d, dv, _p(Q), d, _p(K), d, _p(V), dv, _p(M),
                                      float(scale), _p(out), _p(lse), _p(s))
    return out, lse


def verify_attn(q, k_cache, v_cache, kv_fp8, kv_indptr, kv_indices, last_page_len, qo_indptr,
                mask, mask_indptr, h_q, h_kv, d, page_size, num_pages, sm_scale, k_scale=1.0,
                v_scale=1.0, rows=None, nthreads=None):
    """Verify attention of a batch.  ``rows``: optional flat row ids
    token * h_q + head; returns (out [n, d] fp64, lse [n] fp64)."""
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint8 if kv_fp8 else np.uint16)
    vc = _c(v_cache, np.uint8 if kv_fp8 else np.uint16)
    kv_indptr = _c(kv_indptr, np.int32); kv_indices = _c(kv_indices, np.int32)
    last_page_len = _c(last_page_len, np.int32); qo_indptr = _c(qo_indptr, np.int32)
    mask = _c(mask, np.uint8); mask_indptr = _c(mask_indptr, np.int32)
    batch = len(qo_indptr) - 1
    total_qo = int(qo_indptr[-1])
    sel = _c(rows, np.int32)
    n = total_qo * h_q if sel is None else len(sel)
    out = np.zeros((max(n, 1), d)); lse = np.zeros(max(n, 1))
    rc = lib.oracle_verify_attn(_p(q), _p(kc), _p(vc), int(bool(kv_fp8)), _p(kv_indptr),
                                _p(kv_indices), _p(last_page_len), _p(qo_indptr), _p(mask),
                                _p(mask_indptr), batch, h_q, h_kv, d, page_size, num_pages,
                                float(sm_scale), float(k_scale), float(v_scale), _p(sel),
                                int(n), _p(out), _p(lse),
                                int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_verify_attn rejected its inputs (status %d)" % rc)
    return out[:n], lse[:n]


def verify_attn_ex(q, k_cache, v_cache, kv_fp8, kv_indptr, kv_indices, last_page_len,
                   qo_indptr, mask, mask_indptr, h_q, h_kv, d, page_size, num_pages, sm_scale,
                   k_scale=1.0, v_scale=1.0, kv_layout=0, mask_layout=0, q_pos=None,
                   rope_theta=0.0, rope_scale=1.0, q_fp8=False, rows=None, nthreads=None,
                   dv=None):
    """verify_attn with the cache layout (0 HND, 1 NHD), the mask layout (0:
    L x L draft blocks, 1: L x kv_len rows), optional query positions for
    the rotary embedding of the queries (the cache holds keys as stored) and
    value rows of dv elements (default d); out rows hold dv elements."""
    dv = d if dv is None else int(dv)
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint8 if kv_fp8 else np.uint16)
    vc = _c(v_cache, np.uint8 if kv_fp8 else np.uint16)
    kv_indptr = _c(kv_indptr, np.int32); kv_indices = _c(kv_indices, np.int32)
    last_page_len = _c(last_page_len, np.int32); qo_indptr = _c(qo_indptr, np.int32)
    mask = _c(mask, np.uint8); mask_indptr = _c(mask_indptr, np.int32)
    q_pos = _c(q_pos, np.int32)
    batch = len(qo_indptr) - 1
    total_qo = int(qo_indptr[-1])
    sel = _c(rows, np.int32)
    n = total_qo * h_q if sel is None else len(sel)
    out = np.zeros((max(n, 1), dv)); lse = np.zeros(max(n, 1))
    rc = lib.oracle_verify_attn_dv(_p(q), _p(kc), _p(vc), int(bool(kv_fp8)), int(kv_layout),
                                   _p(kv_indptr), _p(kv_indices), _p(last_page_len),
                                   _p(qo_indptr), _p(mask), _p(mask_indptr), int(mask_layout),
                                   _p(q_pos), float(rope_theta), float(rope_scale), int(bool(q_fp8)),
                                   batch, h_q, h_kv, d, dv, page_size, num_pages, float(sm_scale),
                                   float(k_scale), float(v_scale), _p(sel), int(n), _p(out),
                                   _p(lse), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_verify_attn_dv rejected its inputs (status %d)" % rc)
    return out[:n], lse[:n]


def quantize_q_e4m3(row):
    """The e4m3 codes (uint8) and the binary32 scale of one query row (fp64
    values), as the e4m3 tensor-core path quantises it."""
    lib = _load()
    r = np.ascontiguousarray(row, dtype=np.float64)
    codes = np.zeros(r.shape[0], np.uint8)
    qsc = lib.oracle_quantize_q_e4m3(_p(r), r.shape[0], _p(codes))
    return codes, float(qsc)


def encode_bf16(x) -> np.ndarray:
    """bf16 bits (uint16) of the values nearest to x (ties to even)."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float64).reshape(-1)
    return np.array([lib.oracle_encode_bf16(float(v)) for v in flat],
                    dtype=np.uint16).reshape(np.shape(x))


def rope(x, pos, theta, scale=1.0) -> np.ndarray:
    """LLaMA rotate-half rotary embedding of the last axis of x (fp64) at
    position pos."""
    lib = _load()
    a = np.array(x, dtype=np.float64)
    flat = a.reshape(-1, a.shape[-1])
    for r in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[r])
        lib.oracle_rope_vec(_p(row), row.shape[0], float(pos), float(theta), float(scale))
        flat[r] = row
    return flat.reshape(a.shape)


def paged_kv_append_ex(k_new, v_new, append_indptr, kv_indptr, kv_indices, last_page_len,
                       page_size, num_pages, k_cache, v_cache, cache_fp8, quantize=False,
                       k_scale=1.0, v_scale=1.0, kv_layout=0, positions=None, rope_theta=0.0,
                       rope_scale=1.0):
    """Host scatter with the extended append's options (in place on k_cache /
    v_cache: numpy pools [pages, h_kv, P, d] (HND) or [pages, P, h_kv, d]
    (NHD) of the cache dtype's bits)."""
    lib = _load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    src_dt = np.uint16 if (quantize or not cache_fp8) else np.uint8
    k_new = np.ascontiguousarray(k_new, dtype=src_dt)
    v_new = np.ascontiguousarray(v_new, dtype=src_dt)
    if kv_layout == 1:
        h_kv, d = k_cache.shape[2], k_cache.shape[3]
    else:
        h_kv, d = k_cache.shape[1], k_cache.shape[3]
    dv = v_cache.shape[3]   # value rows may be narrower or wider than key rows
    idx = [_c(a, np.int32) for a in (append_indptr, kv_indptr, kv_indices, last_page_len)]
    pos = _c(positions, np.int32)
    rc = lib.oracle_paged_kv_append_dv(_p(k_new), _p(v_new), int(bool(cache_fp8)),
                                       int(bool(quantize)), float(k_scale), float(v_scale),
                                       int(kv_layout), _p(pos), float(rope_theta),
                                       float(rope_scale), *[_p(a) for a in idx],
                                       len(idx[0]) - 1, h_kv, d, dv, page_size, num_pages,
                                       _p(k_cache), _p(v_cache))
    if rc != 0:
        raise ValueError("oracle_paged_kv_append_dv rejected its inputs (status %d)" % rc)


def attn_range(q, k_cache, v_cache, kv_fp8, kv_indptr, kv_indices, last_page_len, qo_indptr,
               mask, mask_indptr, h_q, h_kv, d, page_size, num_pages, sm_scale, k_scale,
               v_scale, b, t, qh, lo, hi):
    """One row's attention restricted to key positions [lo, hi) of its request."""
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint8 if kv_fp8 else np.uint16)
    vc = _c(v_cache, np.uint8 if kv_fp8 else np.uint16)
    args = [_c(a, np.int32) for a in (kv_indptr, kv_indices, last_page_len, qo_indptr)]
    mask = _c(mask, np.uint8); mask_indptr = _c(mask_indptr, np.int32)
    out = np.zeros(d); lse = np.zeros(1)
    rc = lib.oracle_attn_range(_p(q), _p(kc), _p(vc), int(bool(kv_fp8)), *[_p(a) for a in args],
                               _p(mask), _p(mask_indptr), len(args[3]) - 1, h_q, h_kv, d,
                               page_size, num_pages, float(sm_scale), float(k_scale),
                               float(v_scale), b, t, qh, lo, hi, _p(out), _p(lse))
    if rc != 0:
        raise ValueError("oracle_attn_range rejected its inputs (status %d)" % rc)
    return out, float(lse[0])


def merge_partials(outs, lses):
    """outs [S, n, d], lses [S, n] -> (out [n, d], lse [n])."""
    lib = _load()
    outs = _c(outs, np.float64); lses = _c(lses, np.float64)
    S, n, d = outs.shape
    out = np.zeros((n, d)); lse = np.zeros(n)
    lib.oracle_merge_partials(S, n, d, _p(outs), _p(lses), _p(out), _p(lse))
    return out, lse


def paged_kv_append(k_new, v_new, append_indptr, kv_indptr, kv_indices, last_page_len,
                    page_size, num_pages, k_cache, v_cache):
    """Host scatter (in place on k_cache / v_cache, numpy [pages, h_kv, P, d])."""
    lib = _load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new); v_new = np.ascontiguousarray(v_new)
    h_kv, d = k_cache.shape[1], k_cache.shape[3]
    idx = [_c(a, np.int32) for a in (append_indptr, kv_indptr, kv_indices, last_page_len)]
    rc = lib.oracle_paged_kv_append(_p(k_new), _p(v_new), k_cache.itemsize, *[_p(a) for a in idx],
                                    len(idx[0]) - 1, h_kv, d, page_size, num_pages,
                                    _p(k_cache), _p(v_cache))
    if rc != 0:
        raise ValueError("oracle_paged_kv_append rejected its inputs (status %d)" % rc)


def encode_e4m3_satfinite(x) -> np.ndarray:
    """fp8-e4m3 codes (uint8) of binary32 values: round to nearest even,
    saturating finite overflow and infinities to +-448, NaN -> 0x7F."""
    lib = _load()
    flat = np.asarray(x, dtype=np.float32).reshape(-1)
    return np.array([lib.oracle_encode_e4m3_satfinite(float(v)) for v in flat],
                    dtype=np.uint8).reshape(np.shape(x))


def div_f32(x: float, scale: float) -> float:
    """The correctly rounded binary32 quotient x / scale."""
    return float(_load().oracle_div_f32(float(x), float(scale)))


def paged_kv_append_quant(k_new, v_new, k_scale, v_scale, append_indptr, kv_indptr, kv_indices,
                          last_page_len, page_size, num_pages, k_cache, v_cache):
    """Quantising host scatter: bf16 rows (uint16 bits) into an fp8-e4m3 pool
    (uint8 [pages, h_kv, P, d], in place), stored = e4m3(x / scale)."""
    lib = _load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    h_kv, d = k_cache.shape[1], k_cache.shape[3]
    idx = [_c(a, np.int32) for a in (append_indptr, kv_indptr, kv_indices, last_page_len)]
    rc = lib.oracle_paged_kv_append_quant(_p(k_new), _p(v_new), float(k_scale), float(v_scale),
                                          *[_p(a) for a in idx], len(idx[0]) - 1, h_kv, d,
                                          page_size, num_pages, _p(k_cache), _p(v_cache))
    if rc != 0:
        raise ValueError("oracle_paged_kv_append_quant rejected its inputs (status %d)" % rc)


# ---- convenience over synthetic.Workload (inputs only; no arithmetic here) ----

def build_cache(wl):
    """The workload's page pool, written by the oracle's own host scatter:
    sentinel-filled (NaN bytes), then every token of every request appended
    (in the workload's cache layout; keys rotated at their positions when the
    workload uses rotary positions)."""
    import synthetic
    kc = synthetic.sentinel_pool(wl)
    vc = synthetic.sentinel_pool(wl, values=True)
    if not wl.nhd and wl.kv_pos is None and wl.dv == wl.d:
        paged_kv_append(wl.k_tok, wl.v_tok, wl.tok_append_indptr(), wl.kv_indptr, wl.kv_indices,
                        wl.last_page_len, wl.page_size, wl.num_pages, kc, vc)
        return kc, vc
    paged_kv_append_ex(wl.k_tok, wl.v_tok, wl.tok_append_indptr(), wl.kv_indptr, wl.kv_indices,
                       wl.last_page_len, wl.page_size, wl.num_pages, kc, vc,
                       cache_fp8=wl.kv_dtype == "fp8_e4m3", kv_layout=1 if wl.nhd else 0,
                       positions=wl.kv_pos, rope_theta=wl.rope_theta or 0.0)
    return kc, vc


def verify_attn_workload(wl, rows=None, nthreads=None, caches=None, q_fp8=False):
    kc, vc = caches if caches is not None else build_cache(wl)
    if not wl.nhd and wl.mask_layout == "qlen" and wl.q_pos is None and not q_fp8 and wl.dv == wl.d:
        return verify_attn(wl.q, kc, vc, wl.kv_dtype == "fp8_e4m3", wl.kv_indptr, wl.kv_indices,
                           wl.last_page_len, wl.qo_indptr, wl.mask, wl.mask_indptr, wl.h_q,
                           wl.h_kv, wl.d, wl.page_size, wl.num_pages, wl.sm_scale, wl.k_scale,
                           wl.v_scale, rows=rows, nthreads=nthreads)
    return verify_attn_ex(wl.q, kc, vc, wl.kv_dtype == "fp8_e4m3", wl.kv_indptr, wl.kv_indices,
                          wl.last_page_len, wl.qo_indptr, wl.mask, wl.mask_indptr, wl.h_q,
                          wl.h_kv, wl.d, wl.page_size, wl.num_pages, wl.sm_scale, wl.k_scale,
                          wl.v_scale, kv_layout=1 if wl.nhd else 0,
                          mask_layout=1 if wl.mask_layout == "full" else 0, q_pos=wl.q_pos,
                          rope_theta=wl.rope_theta or 0.0, q_fp8=q_fp8, rows=rows,
                          nthreads=nthreads, dv=wl.dv)

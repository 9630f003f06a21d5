"""Python binding of libverify_attn.so: GQA/MQA verify attention over a paged
KV cache, hand-written CUDA for sm_103a (GB300).

The functions mirror the C ABI (include/verify_attn.h) and only marshal
arguments: torch tensors supply device memory and the current CUDA stream;
every step of the computation runs in the library's kernels.  There is no
CPU or PyTorch fallback: if the shared library is missing, importing the
binding's functions raises.

Typical step::

    plan = verify_attn_plan(kv_indptr_h, qo_indptr_h, last_page_len_h,
                            mask_indptr_h, num_qo_heads, num_kv_heads,
                            head_dim, page_size, kv_dtype="bf16")
    paged_kv_append(k_new, v_new, qo_indptr, kv_indptr, kv_indices,
                    last_page_len, k_cache, v_cache)
    verify_attn_run(q, k_cache, v_cache, kv_indptr, kv_indices,
                    last_page_len, qo_indptr, mask, mask_indptr, plan,
                    out=out, lse=lse)
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

__all__ = [
    "VerifyAttnError", "Plan", "lib", "verify_attn_plan", "verify_attn_run",
    "verify_attn_partial", "verify_attn_merge", "paged_kv_append",
    "verify_attn_device_status", "verify_attn_plan_bounds", "verify_attn_plan_host",
    "verify_attn_workspace_size", "verify_attn_run_static_scratch", "verify_attn_append_run",
    "verify_accept_greedy",
    "status_string", "num_sms", "KV_BF16", "KV_FP8_E4M3", "library_path",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libverify_attn.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1
_DTYPES = {"bf16": KV_BF16, "bfloat16": KV_BF16, "fp8_e4m3": KV_FP8_E4M3,
           "float8_e4m3fn": KV_FP8_E4M3, torch.bfloat16: KV_BF16,
           torch.float8_e4m3fn: KV_FP8_E4M3}

VA_OK = 0
VA_ERR_DEVICE_CHECK = -6
VA_ERR_PLAN_BUFFER_TOO_SMALL = -7

_lib = None


class VerifyAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (fn, status_string(status), status))


class PlanOptions(ctypes.Structure):
    _fields_ = [("max_splits", ctypes.c_int), ("min_chunk", ctypes.c_int),
                ("target_ctas", ctypes.c_int), ("kernel", ctypes.c_int),
                ("mask_layout", ctypes.c_int), ("kv_layout", ctypes.c_int),
                ("rope", ctypes.c_int), ("q_fp8", ctypes.c_int), ("draft_items", ctypes.c_int),
                ("head_dim_v", ctypes.c_int)]


class RunOptions(ctypes.Structure):
    _fields_ = [("q_position", ctypes.c_void_p), ("rope_theta", ctypes.c_float),
                ("rope_scale", ctypes.c_float), ("early_reads", ctypes.c_int),
                ("reserved", ctypes.c_int * 3)]


class AppendOptions(ctypes.Structure):
    _fields_ = [("quantize", ctypes.c_int), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("kv_layout", ctypes.c_int),
                ("positions", ctypes.c_void_p), ("rope_theta", ctypes.c_float),
                ("rope_scale", ctypes.c_float), ("head_dim_v", ctypes.c_int),
                ("reserved", ctypes.c_int * 3)]


class StepOffsets(ctypes.Structure):
    """Byte offsets of a host step's arrays in its staging buffers (-1: absent)."""
    _fields_ = [(n, ctypes.c_int64) for n in ("q", "k_new", "v_new", "kv_indptr", "kv_indices",
                                              "last_page_len", "qo_indptr", "mask", "mask_indptr")]


def step_offsets(**offsets) -> StepOffsets:
    """A StepOffsets from keyword byte offsets; the mask fields default to -1."""
    o = StepOffsets(mask=-1, mask_indptr=-1)
    for k, v in offsets.items():
        setattr(o, k, -1 if v is None else int(v))
    return o


MASK_QLEN, MASK_FULL = 0, 1
LAYOUT_HND, LAYOUT_NHD = 0, 1
_LAYOUTS = {"hnd": LAYOUT_HND, "nhd": LAYOUT_NHD, LAYOUT_HND: LAYOUT_HND, LAYOUT_NHD: LAYOUT_NHD}
_MASK_LAYOUTS = {"qlen": MASK_QLEN, "full": MASK_FULL, MASK_QLEN: MASK_QLEN, MASK_FULL: MASK_FULL}


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise ImportError(
            "libverify_attn.so is not built (expected at %s); run "
            "`python -c 'import __graft_entry__ as g; g.build()'`" % library_path)
    L = ctypes.CDLL(library_path)
    P, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                            ctypes.c_float)
    Psz = ctypes.POINTER(ctypes.c_size_t)
    Pi = ctypes.POINTER(ctypes.c_int)
    sigs = {
        "verify_attn_status_string": (ctypes.c_char_p, [i32]),
        "verify_attn_num_sms": (i32, [Pi]),
        "verify_attn_plan_bounds": (i32, [i32, i64, i32, i32, i32, i32, Psz, Psz]),
        "verify_attn_workspace_size": (i32, [i32, i32, i32, i32, i32, i32, Psz]),
        "verify_attn_plan_host": (i32, [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                        P, P, sz, Psz]),
        "verify_attn_plan": (i32, [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, P, P,
                                   sz, P, sz, P]),
        "verify_attn_run": (i32, [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, f32, f32, f32,
                                  P, P, i32, P, P, sz, P]),
        "verify_attn_partial": (i32, [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, f32, f32,
                                      f32, P, P, i32, P, P, sz, P]),
        "verify_attn_run_ex": (i32, [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, f32, f32,
                                     f32, P, P, i32, P, P, sz, P, P]),
        "verify_attn_partial_ex": (i32, [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32, f32,
                                         f32, f32, P, P, i32, P, P, sz, P, P]),
        "paged_kv_append_ex": (i32, [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                     P, P, P]),
        "verify_attn_append_run": (i32, [P, P, P, P, P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                         f32, f32, f32, P, P, i32, P, P, sz, P, P]),
        "verify_accept_workspace_size": (i32, [i64, i32, i32, Psz]),
        "verify_accept_greedy": (i32, [P, i32, i64, i32, i64, P, i32, P, P, P, P, P, P, P, i32,
                                       P, sz, P]),
        "verify_attn_merge": (i32, [P, i32, i32, i32, P, P, P, P, sz, P]),
        "verify_attn_plan_launches": (i32, [P, Pi]),
        "verify_attn_plan_upload": (i32, [P, P, sz, P]),
        "verify_attn_device_status": (i32, [P, Pi, P]),
        "paged_kv_append": (i32, [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64, P,
                                  P]),
        "verify_attn_run_static_scratch": (i32, [P, P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                 f32, f32, f32, P, P, i32, P, P]),
        "verify_attn_static_scratch_status": (i32, [Pi, P]),
        "verify_attn_step_host": (i32, [P, P, sz, P, i32, i32, i32, i32, i32, i32, i32, P, P, sz,
                                        P, sz, P, P, P, i32, f32, f32, f32, P, P, P, sz, P, i32,
                                        P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().verify_attn_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != VA_OK:
        raise VerifyAttnError(fn, status)


def num_sms() -> int:
    n = ctypes.c_int(0)
    _check("verify_attn_num_sms", lib().verify_attn_num_sms(ctypes.byref(n)))
    return n.value


def _kv_code(kv_dtype) -> int:
    if isinstance(kv_dtype, int):
        return kv_dtype
    return _DTYPES[kv_dtype]


def _host_i32(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _addr(a: np.ndarray) -> int:
    """Host address of a contiguous numpy array (a plain int).  Through a
    ctypes view of the array's buffer when it is writable and not empty (a
    fraction of the cost of numpy's .ctypes), else numpy's own."""
    try:
        return ctypes.addressof(ctypes.c_char.from_buffer(a))
    except (TypeError, ValueError, BufferError):
        return a.ctypes.data


def _hp(a: Optional[np.ndarray]):
    return None if a is None else _addr(a)


# The last host buffer whose address was taken, kept referenced so that its
# address stays valid: a caller that plans into the same buffer every step
# pays the (slow) address lookup once.
_LAST_HOST = [None]   # (array, address), replaced as one object


def _hp_buf(a: np.ndarray) -> int:
    cached = _LAST_HOST[0]
    if cached is None or cached[0] is not a:
        cached = (a, _addr(a))
        _LAST_HOST[0] = cached
    return cached[1]


def _tables(*arrays):
    """Host index arrays (int32) staged in one contiguous buffer: their
    addresses (None for a missing one) and the buffer, which the caller keeps
    alive for the call."""
    parts = [a for a in arrays if a is not None]
    buf = np.concatenate(parts) if parts else np.zeros(1, np.int32)
    base = _addr(buf)
    ptrs, off = [], 0
    for a in arrays:
        if a is None:
            ptrs.append(None)
        else:
            ptrs.append(base + 4 * off)
            off += a.shape[0]
    return ptrs, buf


def _dp(t: Optional[torch.Tensor]):
    """Device address of a contiguous CUDA tensor (a plain int: ctypes
    passes it as the void* argument)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    """The cudaStream_t of `stream`, or of torch's current stream (read
    through torch's raw-stream query when it has one: a fraction of the cost
    of building a Stream object on every call)."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


_OPTIONS_CACHE: dict = {}


def _options(**kw):
    """The PlanOptions struct of these keyword options (built once per
    distinct set and kept: the library only reads it)."""
    key = tuple(sorted(kw.items()))
    o = _OPTIONS_CACHE.get(key)
    if o is None:
        o = _OPTIONS_CACHE[key] = _make_options(**kw)
    return o


def _make_options(max_splits=0, min_chunk=0, target_ctas=0, kernel=0, mask_layout="qlen",
                  kv_layout="hnd", rope=False, q_fp8=False, draft_items=0, head_dim_v=0):
    o = PlanOptions()
    o.max_splits, o.min_chunk, o.target_ctas, o.kernel = (int(max_splits), int(min_chunk),
                                                          int(target_ctas), int(kernel))
    o.mask_layout = _MASK_LAYOUTS[mask_layout]
    o.kv_layout = _LAYOUTS[kv_layout]
    o.rope = int(bool(rope))
    o.q_fp8 = int(bool(q_fp8))
    o.draft_items = int(draft_items)
    o.head_dim_v = int(head_dim_v or 0)
    return o


@dataclass
class Plan:
    """A plan: the host buffer (numpy) and the device workspace (torch) it was
    uploaded to, plus the shapes it was built for."""
    host: np.ndarray
    workspace: Optional[torch.Tensor]
    workspace_bytes: int
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: int
    has_mask: bool
    total_qo: int

    def header(self) -> dict:
        h = self.host[:184].view(np.uint8)
        ints = np.frombuffer(h[:72].tobytes(), dtype=np.int32)
        i64 = np.frombuffer(h[72:96].tobytes(), dtype=np.int64)
        return dict(group=int(ints[10]), kernel=int(ints[11]), block_rows=int(ints[12]),
                    tile_keys=int(ints[13]), n_items=int(ints[14]), n_merge=int(ints[15]),
                    n_units=int(ints[16]), num_sms=int(ints[17]), total_qo=int(i64[0]),
                    part_rows=int(i64[1]), chunk=int(i64[2]),
                    ws_bytes=int(np.frombuffer(h[136:144].tobytes(), dtype=np.uint64)[0]),
                    n_ctas=int(np.frombuffer(h[160:168].tobytes(), dtype=np.int64)[0]),
                    head_dim_v=int(np.frombuffer(h[168:176].tobytes(), dtype=np.int64)[0]),
                    max_nsplit=int(np.frombuffer(h[176:184].tobytes(), dtype=np.int64)[0]))

    def launches(self) -> int:
        n = ctypes.c_int(0)
        _check("verify_attn_plan_launches",
               lib().verify_attn_plan_launches(_hp(self.host), ctypes.byref(n)))
        return n.value

    def items(self) -> np.ndarray:
        """The work list as an [n_items, 8] int32 array (b, h, row0, nrows,
        kv_lo, kv_hi, part_row, next)."""
        hd = self.header()
        raw = self.host[184:184 + 32 * hd["n_items"]].tobytes()
        return np.frombuffer(raw, dtype=np.int32).reshape(-1, 8)

    def merges(self) -> np.ndarray:
        hd = self.header()
        off = 184 + 32 * hd["n_items"]
        raw = self.host[off:off + 32 * hd["n_merge"]].tobytes()
        return np.frombuffer(raw, dtype=np.int32).reshape(-1, 8)


def verify_attn_plan_bounds(batch, total_qo, num_qo_heads, num_kv_heads, head_dim, num_sms=0):
    pb, wb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("verify_attn_plan_bounds",
           lib().verify_attn_plan_bounds(int(batch), int(total_qo), int(num_qo_heads),
                                         int(num_kv_heads), int(head_dim), int(num_sms),
                                         ctypes.byref(pb), ctypes.byref(wb)))
    return pb.value, wb.value


def verify_attn_plan_host(kv_indptr_h, qo_indptr_h, last_page_len_h, mask_indptr_h,
                          num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype="bf16",
                          has_mask=None, num_sms=0, **options) -> Plan:
    """Host-only plan (no CUDA call when num_sms > 0)."""
    kvp, qop, lpl, mip = (_host_i32(kv_indptr_h), _host_i32(qo_indptr_h),
                          _host_i32(last_page_len_h), _host_i32(mask_indptr_h))
    batch = len(qop) - 1
    if has_mask is None:
        has_mask = mip is not None
    total_qo = int(qop[-1]) if batch >= 0 else 0
    if num_sms <= 0:
        num_sms = globals()["num_sms"]()
    pb, _ = verify_attn_plan_bounds(batch, total_qo, num_qo_heads, num_kv_heads, head_dim,
                                    num_sms)
    host = np.zeros(pb, dtype=np.uint8)
    need = ctypes.c_size_t(0)
    opt = _options(**options)
    tp, _keep = _tables(kvp, qop, lpl, mip)
    rc = lib().verify_attn_plan_host(*tp, batch,
                                     int(num_qo_heads), int(num_kv_heads), int(head_dim),
                                     int(page_size), 0, _kv_code(kv_dtype), int(bool(has_mask)),
                                     int(num_sms), ctypes.byref(opt), _hp(host), host.nbytes,
                                     ctypes.byref(need))
    _check("verify_attn_plan_host", rc)
    return Plan(host, None, need.value, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                _kv_code(kv_dtype), bool(has_mask), total_qo)


def verify_attn_workspace_size(batch, num_qo_heads, num_kv_heads, head_dim, max_qo_len,
                               num_sms=0) -> int:
    """Device workspace bytes that serve every plan of a batch of at most
    `batch` requests with at most `max_qo_len` query tokens each."""
    n = ctypes.c_size_t(0)
    _check("verify_attn_workspace_size",
           lib().verify_attn_workspace_size(int(batch), int(num_qo_heads), int(num_kv_heads),
                                            int(head_dim), int(max_qo_len), int(num_sms),
                                            ctypes.byref(n)))
    return n.value


def verify_attn_plan(kv_indptr_h, qo_indptr_h, last_page_len_h, mask_indptr_h, num_qo_heads,
                     num_kv_heads, head_dim, page_size, kv_dtype="bf16", has_mask=None,
                     workspace: Optional[torch.Tensor] = None, device=None, stream=None,
                     num_sms=0, plan_buffer: Optional[np.ndarray] = None, **options) -> Plan:
    """Plan a batch from HOST index arrays and upload the work list to a
    device workspace, planning once: with a workspace given (it must hold the
    plan), one call of the library's verify_attn_plan; without, the host plan
    is made first, a workspace of exactly its size is allocated here with
    torch, and the plan is uploaded.  plan_buffer (uint8, at least
    verify_attn_plan_bounds' plan bytes) may be passed to reuse a host
    buffer."""
    kvp, qop, lpl, mip = (_host_i32(kv_indptr_h), _host_i32(qo_indptr_h),
                          _host_i32(last_page_len_h), _host_i32(mask_indptr_h))
    batch = len(qop) - 1
    if has_mask is None:
        has_mask = mip is not None
    total_qo = int(qop[-1]) if batch >= 0 else 0
    if num_sms <= 0:
        num_sms = globals()["num_sms"]()
    opt = _options(**options)
    if workspace is None:
        # plan on the host, allocate the workspace this plan needs, upload
        plan = verify_attn_plan_host(kvp, qop, lpl, mip, num_qo_heads, num_kv_heads, head_dim,
                                     page_size, kv_dtype, has_mask, num_sms, **options)
        plan.workspace = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8,
                                     device=device or "cuda")
        _check("verify_attn_plan_upload",
               lib().verify_attn_plan_upload(_hp_buf(plan.host), _dp(plan.workspace),
                                             plan.workspace.numel(), _stream(stream)))
        return plan
    # the caller's host buffer first; sized from verify_attn_plan_bounds when
    # there is none or the library reports it too small
    host = plan_buffer
    strm = _stream(stream)
    tp, _keep = _tables(kvp, qop, lpl, mip)
    for attempt in range(2):
        if host is None:
            pb, _ = verify_attn_plan_bounds(batch, total_qo, num_qo_heads, num_kv_heads,
                                            head_dim, num_sms)
            host = np.zeros(pb, dtype=np.uint8)
        rc = lib().verify_attn_plan(*tp, batch,
                                    int(num_qo_heads), int(num_kv_heads), int(head_dim),
                                    int(page_size), 0, _kv_code(kv_dtype), int(bool(has_mask)),
                                    int(num_sms), ctypes.byref(opt), _hp_buf(host), host.nbytes,
                                    _dp(workspace), workspace.numel(), strm)
        if rc != VA_ERR_PLAN_BUFFER_TOO_SMALL or attempt:
            break
        host = None
    _check("verify_attn_plan", rc)
    ws_bytes = int(host[136:144].view(np.uint64)[0])   # the header's workspace size
    return Plan(host, workspace, ws_bytes, batch, num_qo_heads, num_kv_heads, head_dim,
                page_size, _kv_code(kv_dtype), bool(has_mask), total_qo)


def _run_args(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr, mask,
              mask_indptr, plan: Plan, sm_scale, k_scale, v_scale, out, lse, num_pages):
    if q.dtype != torch.bfloat16:
        raise ValueError("q must be bfloat16")
    if out.dtype != torch.bfloat16:
        raise ValueError("out must be bfloat16")
    if lse is not None and lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    if num_pages is None:
        num_pages = k_cache.shape[0]
    return (_dp(q), _dp(k_cache), _dp(v_cache), _dp(kv_indptr), _dp(kv_indices),
            _dp(last_page_len), _dp(qo_indptr), _dp(mask), _dp(mask_indptr),
            plan.num_qo_heads, plan.num_kv_heads, plan.head_dim, plan.page_size,
            float(sm_scale), float(k_scale), float(v_scale), _dp(out), _dp(lse),
            int(num_pages), _hp_buf(plan.host), _dp(plan.workspace), plan.workspace.numel())


def _alloc_out(q, plan, out, lse, want_lse):
    if out is None:
        dv = plan.header()["head_dim_v"]
        out = q.new_empty(q.shape[0], q.shape[1], dv)
    if lse is None and want_lse:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    return out, lse


_EARLY_READS = RunOptions()
_EARLY_READS.early_reads = 1


def _run_options(q_position, rope_theta, rope_scale, early_reads=False):
    if q_position is None and not early_reads:
        return None
    if q_position is None:
        return _EARLY_READS   # shared: the library only reads it
    o = RunOptions()
    if q_position is not None:
        o.q_position = _dp(q_position)
        o.rope_theta = float(rope_theta)
        o.rope_scale = float(rope_scale)
    o.early_reads = int(bool(early_reads))
    return o


def verify_attn_run(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr,
                    mask, mask_indptr, plan: Plan, sm_scale=0.0, k_scale=1.0, v_scale=1.0,
                    out=None, lse=None, want_lse=True, num_pages=None, stream=None,
                    q_position=None, rope_theta=10000.0, rope_scale=1.0, early_reads=False):
    """out = softmax(q k^T * sm_scale * k_scale + mask) v * v_scale, and its LSE.
    q_position (int32 device tensor [total_qo]) rotates the queries by RoPE
    at those positions; the plan must have been made with rope=True.
    early_reads: the caller promises that q, the tables, the mask and the
    positions were complete before the preceding kernel in the stream
    started, and that it writes none of them nor a prefix slot (see
    va_run_options_t)."""
    out, lse = _alloc_out(q, plan, out, lse, want_lse)
    args = _run_args(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr, mask,
                     mask_indptr, plan, sm_scale, k_scale, v_scale, out, lse, num_pages)
    ro = _run_options(q_position, rope_theta, rope_scale, early_reads)
    if ro is None:
        _check("verify_attn_run", lib().verify_attn_run(*args, _stream(stream)))
    else:
        _check("verify_attn_run_ex",
               lib().verify_attn_run_ex(*args, ctypes.byref(ro), _stream(stream)))
    return out, lse


def verify_attn_partial(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr,
                        mask, mask_indptr, plan: Plan, sm_scale=0.0, k_scale=1.0, v_scale=1.0,
                        out=None, lse=None, want_lse=True, num_pages=None, stream=None,
                        q_position=None, rope_theta=10000.0, rope_scale=1.0, early_reads=False):
    out, lse = _alloc_out(q, plan, out, lse, want_lse)
    args = _run_args(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len, qo_indptr, mask,
                     mask_indptr, plan, sm_scale, k_scale, v_scale, out, lse, num_pages)
    ro = _run_options(q_position, rope_theta, rope_scale, early_reads)
    if ro is None:
        _check("verify_attn_partial", lib().verify_attn_partial(*args, _stream(stream)))
    else:
        _check("verify_attn_partial_ex",
               lib().verify_attn_partial_ex(*args, ctypes.byref(ro), _stream(stream)))
    return out, lse


def verify_attn_merge(qo_indptr, plan: Plan, out, lse=None, stream=None):
    _check("verify_attn_merge",
           lib().verify_attn_merge(_dp(qo_indptr), plan.num_qo_heads, plan.num_kv_heads,
                                   plan.head_dim, _dp(out), _dp(lse), _hp_buf(plan.host),
                                   _dp(plan.workspace), plan.workspace.numel(), _stream(stream)))
    return out, lse


def verify_attn_device_status(plan: Plan, stream=None) -> int:
    """OR of VA_DEV_* bits raised by kernels since the plan (synchronises)."""
    bits = ctypes.c_int(0)
    rc = lib().verify_attn_device_status(_dp(plan.workspace), ctypes.byref(bits), _stream(stream))
    if rc not in (VA_OK, VA_ERR_DEVICE_CHECK):
        _check("verify_attn_device_status", rc)
    return bits.value


def paged_kv_append(k_new, v_new, append_indptr, kv_indptr, kv_indices, last_page_len, k_cache,
                    v_cache, total_new=None, num_pages=None, status=None, stream=None,
                    kv_layout="hnd", k_scale=None, v_scale=None, positions=None,
                    rope_theta=10000.0, rope_scale=1.0):
    """Write new tokens' K/V into their pages.  By default a bit-exact copy
    (k_new / v_new in the cache dtype).  With a bf16 k_new / v_new and an fp8
    cache, a quantising append (k_scale / v_scale required).  positions
    (int32 device tensor [total_new]) rotates the new keys by RoPE first.
    kv_layout "nhd" for a [pages, P, h_kv, d] cache.  total_new defaults to
    k_new.shape[0]."""
    fp8_cache = k_cache.element_size() == 1
    quantize = fp8_cache and k_new.dtype == torch.bfloat16
    if not quantize and (k_cache.dtype != k_new.dtype or v_cache.dtype != v_new.dtype):
        raise ValueError("k_new / v_new must be in the cache dtype (or bf16 into an fp8 cache)")
    if quantize and (k_scale is None or v_scale is None or v_new.dtype != torch.bfloat16):
        raise ValueError("a quantising append needs bf16 k_new / v_new and k_scale / v_scale")
    kv_dtype = KV_FP8_E4M3 if fp8_cache else KV_BF16
    batch = append_indptr.shape[0] - 1
    if total_new is None:
        total_new = k_new.shape[0]
    if num_pages is None:
        num_pages = k_cache.shape[0]
    layout = _LAYOUTS[kv_layout]
    if layout == LAYOUT_NHD:
        page_size, h_kv, head_dim = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    else:
        h_kv, page_size, head_dim = k_cache.shape[1], k_cache.shape[2], k_cache.shape[3]
    head_dim_v = v_cache.shape[3]
    common = (_dp(k_new), _dp(v_new), _dp(append_indptr), _dp(kv_indptr), _dp(kv_indices),
              _dp(last_page_len), _dp(k_cache), _dp(v_cache), int(batch), int(h_kv),
              int(head_dim), int(page_size), int(num_pages), kv_dtype, int(total_new))
    if not quantize and positions is None and layout == LAYOUT_HND and head_dim_v == head_dim:
        rc = lib().paged_kv_append(*common, _dp(status), _stream(stream))
        _check("paged_kv_append", rc)
        return
    o = AppendOptions()
    o.quantize = int(quantize)
    o.k_scale = float(k_scale) if quantize else 0.0
    o.v_scale = float(v_scale) if quantize else 0.0
    o.kv_layout = layout
    o.positions = _dp(positions) if positions is not None else None
    o.rope_theta = float(rope_theta) if positions is not None else 0.0
    o.rope_scale = float(rope_scale) if positions is not None else 0.0
    o.head_dim_v = int(head_dim_v)
    rc = lib().paged_kv_append_ex(*common, ctypes.byref(o), _dp(status), _stream(stream))
    _check("paged_kv_append_ex", rc)


def verify_attn_append_run(k_new, v_new, q, k_cache, v_cache, kv_indptr, kv_indices,
                           last_page_len, qo_indptr, mask, mask_indptr, plan: Plan, sm_scale=0.0,
                           k_scale=1.0, v_scale=1.0, out=None, lse=None, want_lse=True,
                           num_pages=None, stream=None, q_position=None, rope_theta=10000.0,
                           rope_scale=1.0, append_k_scale=None, append_v_scale=None,
                           positions=None, kv_layout="hnd", early_reads=False):
    """One verification step: append the drafts' K/V (k_new / v_new, one row
    per query token in qo_indptr order; bf16 into an fp8 cache quantises with
    append_k_scale / append_v_scale; positions rotates the new keys by RoPE),
    then verify attention over the cache just written.  Returns (out, lse).
    early_reads as for verify_attn_run."""
    out, lse = _alloc_out(q, plan, out, lse, want_lse)
    if num_pages is None:
        num_pages = k_cache.shape[0]
    fp8_cache = k_cache.element_size() == 1
    quantize = fp8_cache and k_new.dtype == torch.bfloat16
    layout = _LAYOUTS[kv_layout]
    ao = None
    if quantize or positions is not None or layout != LAYOUT_HND:
        ao = AppendOptions()
        ao.quantize = int(quantize)
        ao.k_scale = float(append_k_scale) if quantize else 0.0
        ao.v_scale = float(append_v_scale) if quantize else 0.0
        ao.kv_layout = layout
        ao.positions = _dp(positions) if positions is not None else None
        ao.rope_theta = float(rope_theta) if positions is not None else 0.0
        ao.rope_scale = float(rope_scale) if positions is not None else 0.0
    ro = _run_options(q_position, rope_theta, rope_scale, early_reads)
    if q.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("q and out must be bfloat16")
    rc = lib().verify_attn_append_run(
        _dp(k_new), _dp(v_new), None if ao is None else ctypes.byref(ao), _dp(q), _dp(k_cache),
        _dp(v_cache), _dp(kv_indptr), _dp(kv_indices), _dp(last_page_len), _dp(qo_indptr),
        _dp(mask), _dp(mask_indptr), plan.num_qo_heads, plan.num_kv_heads, plan.head_dim,
        plan.page_size, float(sm_scale), float(k_scale), float(v_scale), _dp(out), _dp(lse),
        int(num_pages), _hp_buf(plan.host), _dp(plan.workspace), plan.workspace.numel(),
        None if ro is None else ctypes.byref(ro), _stream(stream))
    _check("verify_attn_append_run", rc)
    return out, lse


def _host_ptr(b) -> int:
    """Host address of a CPU torch tensor or a numpy array."""
    if isinstance(b, torch.Tensor):
        if b.is_cuda or not b.is_contiguous():
            raise ValueError("expected a contiguous host tensor")
        return b.data_ptr()
    return _hp_buf(b)


def _nbytes(b) -> int:
    return b.numel() * b.element_size() if isinstance(b, torch.Tensor) else b.nbytes


def verify_attn_step_host(staging_h, staging_d, offsets, batch, num_qo_heads, num_kv_heads,
                          head_dim, page_size, k_cache, v_cache, out, lse, result_h,
                          workspace, plan_buffer, kv_dtype="bf16", num_sms=0, sm_scale=0.0,
                          k_scale=1.0, v_scale=1.0, num_pages=None, append_options=None,
                          early_reads=False, synchronize=True, stream=None, **options):
    """One verification step from host buffers in one library call
    (verify_attn_step_host): the pinned staging buffer `staging_h` (uint8,
    the step's inputs at `offsets`, a StepOffsets or a dict) goes to
    `staging_d` in one copy, the plan is made from its host tables into
    `plan_buffer` (host, uint8) and `workspace`, the drafts are appended and
    attended, and out (then the LSE at round_up(out bytes, 256)) comes back
    into the pinned `result_h`.  With synchronize the call returns once
    result_h is filled."""
    if isinstance(offsets, dict):
        offsets = step_offsets(**offsets)
    if num_pages is None:
        num_pages = k_cache.shape[0]
    ro = _run_options(None, 0.0, 0.0, early_reads)
    rc = lib().verify_attn_step_host(
        _host_ptr(staging_h), _dp(staging_d), _nbytes(staging_h), ctypes.byref(offsets),
        int(batch), int(num_qo_heads), int(num_kv_heads), int(head_dim), int(page_size),
        _kv_code(kv_dtype), int(num_sms), ctypes.byref(_options(**options)),
        _host_ptr(plan_buffer), _nbytes(plan_buffer), _dp(workspace), workspace.numel(),
        None if append_options is None else ctypes.byref(append_options), _dp(k_cache),
        _dp(v_cache), int(num_pages), float(sm_scale), float(k_scale), float(v_scale),
        _dp(out), _dp(lse), _host_ptr(result_h), _nbytes(result_h),
        None if ro is None else ctypes.byref(ro), int(bool(synchronize)), _stream(stream))
    _check("verify_attn_step_host", rc)


class HostStep:
    """verify_attn_step_host with its arguments marshalled once: every
    buffer of a step loop stays put (the staging and result buffers, out /
    lse, the workspace, the plan buffer) and so does the stream (the one
    given, else torch's current stream when the object is made), so each
    call passes the same converted arguments -- only the cache pair may
    change between calls."""

    def __init__(self, staging_h, staging_d, offsets, batch, num_qo_heads, num_kv_heads,
                 head_dim, page_size, k_cache, v_cache, out, lse, result_h, workspace,
                 plan_buffer, kv_dtype="bf16", num_sms=0, sm_scale=0.0, k_scale=1.0,
                 v_scale=1.0, num_pages=None, append_options=None, early_reads=False,
                 synchronize=True, stream=None, **options):
        if isinstance(offsets, dict):
            offsets = step_offsets(**offsets)
        if num_pages is None:
            num_pages = k_cache.shape[0]
        ro = _run_options(None, 0.0, 0.0, early_reads)
        # the objects the arguments point into, kept alive with this call
        self._keep = (staging_h, staging_d, offsets, out, lse, result_h, workspace, plan_buffer,
                      append_options, ro, k_cache, v_cache)
        V, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        self._fn = lib().verify_attn_step_host
        self._args = [
            V(_host_ptr(staging_h)), V(_dp(staging_d)), S(_nbytes(staging_h)), ctypes.byref(offsets),
            I(int(batch)), I(int(num_qo_heads)), I(int(num_kv_heads)), I(int(head_dim)),
            I(int(page_size)), I(_kv_code(kv_dtype)), I(int(num_sms)),
            ctypes.byref(_options(**options)), V(_host_ptr(plan_buffer)), S(_nbytes(plan_buffer)),
            V(_dp(workspace)), S(workspace.numel()),
            None if append_options is None else ctypes.byref(append_options),
            V(_dp(k_cache)), V(_dp(v_cache)), I(int(num_pages)), F(float(sm_scale)),
            F(float(k_scale)), F(float(v_scale)), V(_dp(out)), V(_dp(lse)),
            V(_host_ptr(result_h)), S(_nbytes(result_h)),
            None if ro is None else ctypes.byref(ro), I(int(bool(synchronize))),
            V(_stream(stream))]
        self._caches = {}

    def __call__(self, k_cache=None, v_cache=None):
        """One step; k_cache / v_cache (both or neither) replace the pair the
        call was prepared with."""
        args = self._args
        if k_cache is not None:
            key = (k_cache.data_ptr(), v_cache.data_ptr())
            args = self._caches.get(key)
            if args is None:
                args = list(self._args)
                args[17], args[18] = ctypes.c_void_p(_dp(k_cache)), ctypes.c_void_p(_dp(v_cache))
                self._caches[key] = args
                self._keep = self._keep + (k_cache, v_cache)
        _check("verify_attn_step_host", self._fn(*args))


def verify_accept_greedy(logits, qo_indptr, draft_tokens, parents, workspace=None,
                         want_argmax=False, status=None, stream=None):
    """Greedy acceptance of draft trees (see include/verify_attn.h):
    logits [total, vocab] bf16 or fp32 (device), qo_indptr [B+1],
    draft_tokens / parents [total] int32 (device).  Returns (accept_len [B],
    accepted_nodes [total], bonus_token [B], argmax [total] or None), all
    int32 device tensors; request b's path is accepted_nodes[qo_indptr[b] :
    qo_indptr[b] + accept_len[b]]."""
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be [total, vocab] with unit column stride")
    if logits.dtype == torch.bfloat16:
        code = 0
    elif logits.dtype == torch.float32:
        code = 2
    else:
        raise ValueError("logits must be bfloat16 or float32")
    total, vocab = logits.shape
    batch = qo_indptr.shape[0] - 1
    dev = logits.device
    n = ctypes.c_size_t(0)
    _check("verify_accept_workspace_size",
           lib().verify_accept_workspace_size(int(total), int(vocab), 0, ctypes.byref(n)))
    if workspace is None or workspace.numel() < n.value:
        workspace = torch.empty(max(n.value, 256), dtype=torch.uint8, device=dev)
    acc = torch.empty(batch, dtype=torch.int32, device=dev)
    path = torch.full((max(total, 1),), -1, dtype=torch.int32, device=dev)
    bonus = torch.empty(batch, dtype=torch.int32, device=dev)
    am = torch.empty(max(total, 1), dtype=torch.int32, device=dev) if want_argmax else None
    if not logits.is_cuda:
        raise ValueError("expected a CUDA tensor")
    # rows may be padded (row stride > vocab): the row stride is passed explicitly
    rc = lib().verify_accept_greedy(ctypes.c_void_p(logits.data_ptr()), code, int(total), int(vocab),
                                    int(logits.stride(0)), _dp(qo_indptr), int(batch),
                                    _dp(draft_tokens), _dp(parents), _dp(acc), _dp(path),
                                    _dp(bonus), _dp(am), _dp(status), 0, _dp(workspace),
                                    workspace.numel(), _stream(stream))
    _check("verify_accept_greedy", rc)
    return acc, path[:total], bonus, None if am is None else am[:total]


STATIC_SCRATCH_BYTES = 32 << 20


def verify_attn_static_scratch_status(stream=None) -> int:
    """Device check bits (VA_DEV_*) of the last static-scratch call in this
    context; cleared by the read.  0 when every check passed."""
    bits = ctypes.c_int(0)
    rc = lib().verify_attn_static_scratch_status(ctypes.byref(bits), _stream(stream))
    if rc not in (VA_OK, VA_ERR_DEVICE_CHECK):
        _check("verify_attn_static_scratch_status", rc)
    return bits.value


def verify_attn_run_static_scratch(q, k_cache, v_cache, kv_indptr, kv_indices, last_page_len,
                                   qo_indptr, mask, mask_indptr, plan: Plan, sm_scale=0.0,
                                   k_scale=1.0, v_scale=1.0, out=None, lse=None, want_lse=True,
                                   num_pages=None, stream=None):
    """verify_attn_run for callers that cannot allocate device memory: the
    library's own static scratch array (STATIC_SCRATCH_BYTES) stands in for
    the workspace, so `plan` may come from verify_attn_plan_host (no device
    workspace).  The first call in each CUDA context looks up the array's
    address; calls that overlap on the GPU share the array and race."""
    out, lse = _alloc_out(q, plan, out, lse, want_lse)
    if num_pages is None:
        num_pages = k_cache.shape[0]
    rc = lib().verify_attn_run_static_scratch(
        _dp(q), _dp(k_cache), _dp(v_cache), _dp(kv_indptr), _dp(kv_indices), _dp(last_page_len),
        _dp(qo_indptr), _dp(mask), _dp(mask_indptr), plan.num_qo_heads, plan.num_kv_heads,
        plan.head_dim, plan.page_size, float(sm_scale), float(k_scale), float(v_scale), _dp(out),
        _dp(lse), int(num_pages), _hp_buf(plan.host), _stream(stream))
    _check("verify_attn_run_static_scratch", rc)
    return out, lse

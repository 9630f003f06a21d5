"""Seeded synthetic workloads for paged-KV GQA verify attention.

This module only draws and lays out inputs: request lengths, draft-tree
parents (and the ancestor mask they imply), a shuffled page pool, and the
q / k / v values, in the shapes the source pages describe.  It holds none of
the attention arithmetic; both the fp64 oracle (``oracle/``) and the CUDA
path consume what it returns.

Layouts (all numpy, host memory):

* ``q``        [sum L_b, h_q, d]        bf16 bit patterns (uint16)
* ``k_tok``    [sum kv_len_b, h_kv, d]  every token of every request, prefix
  followed by the L_b draft tokens, in the cache dtype's bit patterns
  (uint16 for bf16, uint8 for fp8-e4m3); ``v_tok`` likewise
* ``tok_indptr`` [B+1]                  offsets of each request in k_tok/v_tok
* page table in FlashInfer's paged-KV convention (FlashInfer PR #286
  "Separate Q and KV dtypes for decode", ``begin_forward`` parameters):
  ``kv_indptr`` [B+1], ``kv_indices`` [kv_indptr[-1]], ``last_page_len`` [B];
  after the drafts are appended, kv_len_b = (pages_b - 1) * page_size +
  last_page_len_b covers the prefix and the drafts
* ``qo_indptr`` [B+1]                   ranges of each request's query tokens
* ``mask`` bit-packed uint8, LSB first; request b's L_b x L_b row-major block
  starts at bit ``mask_indptr[b]`` (None for the causal chain)

Random draws use one CPU ``torch.Generator`` in a fixed order: lengths, tree
parents, page permutation, q, k, v.  Normal values are drawn in fp32 and
rounded to bf16 (round to nearest even).  For fp8-e4m3 caches the per-tensor
scale is amax|x| / 448 over the whole tensor and the stored code is
``(x / scale)`` rounded by torch's float8_e4m3fn cast.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

BF16 = "bf16"
FP8 = "fp8_e4m3"

# The workloads, named by what they are.  Shapes follow the source pages'
# scenarios: the tiny verify case, a Llama-3-8B-shaped tree verify, a
# CodeLLaMA-34B-shaped batched chain verify (64 q / 8 kv heads, d = 128, the
# shape of the vLLM #2401 prefill benchmark), GQA varlen causal prefill of
# 10 x 1024-token prompts, and a wide-tree long-context verify over fp8 KV.
WORKLOADS = {
    "tiny_verify": dict(
        batch=2, h_q=4, h_kv=2, d=64, page_size=16, kv_dtype=BF16,
        prefix=("fixed", [37, 70]), qo=("fixed", [5, 5]), mask="causal",
        pool_pages=16, sm_scale=1.0 / 8.0),
    "llama3_8b_tree_verify": dict(
        batch=1, h_q=32, h_kv=8, d=128, page_size=16, kv_dtype=BF16,
        prefix=("fixed", [4096]), qo=("fixed", [17]), mask="tree"),
    "codellama34b_chain_verify": dict(
        batch=64, h_q=64, h_kv=8, d=128, page_size=16, kv_dtype=BF16,
        prefix=("uniform", (512, 8192)), qo=("uniform", (1, 8)), mask="causal"),
    "gqa_varlen_prefill": dict(
        batch=10, h_q=64, h_kv=8, d=128, page_size=16, kv_dtype=BF16,
        prefix=("fixed", [0] * 10), qo=("fixed", [1024] * 10), mask="causal"),
    "wide_tree_fp8_verify": dict(
        batch=8, h_q=32, h_kv=8, d=128, page_size=16, kv_dtype=FP8,
        prefix=("fixed", [32768] * 8), qo=("fixed", [64] * 8), mask="tree"),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclass
class Workload:
    name: str
    batch: int
    h_q: int
    h_kv: int
    d: int
    page_size: int
    kv_dtype: str
    prefix_lens: np.ndarray          # [B] int64
    qo_lens: np.ndarray              # [B] int64
    kv_lens: np.ndarray              # [B] int64 = prefix + qo
    qo_indptr: np.ndarray            # [B+1] int32
    kv_indptr: np.ndarray            # [B+1] int32 (pages)
    kv_indices: np.ndarray           # [nnz pages] int32
    last_page_len: np.ndarray        # [B] int32
    num_pages: int                   # pool size
    tok_indptr: np.ndarray           # [B+1] int64 offsets into k_tok / v_tok
    q: np.ndarray                    # [sum L, h_q, d] uint16 (bf16 bits)
    k_tok: np.ndarray                # [sum kv_len, h_kv, d] uint16 or uint8
    v_tok: np.ndarray
    sm_scale: float
    k_scale: float
    v_scale: float
    mask_kind: str                   # "causal" (no mask), "tree", "chain", "random", "full", "none_visible"
    parents: Optional[list] = None   # per request list of parent ids (tree/chain)
    mask_dense: Optional[list] = None  # per request bool [L, L] (True = visible)
    mask: Optional[np.ndarray] = None  # bit-packed uint8
    mask_indptr: Optional[np.ndarray] = None  # [B+1] int32 bit offsets
    extra: dict = field(default_factory=dict)
    kv_layout: str = "hnd"           # "hnd" [pages, h_kv, P, d] or "nhd" [pages, P, h_kv, d]
    mask_layout: str = "qlen"        # "qlen": L x L draft blocks; "full": L x kv_len rows
    mask_full: Optional[list] = None  # per request bool [L, kv_len] (mask_layout "full")
    rope_theta: Optional[float] = None  # RoPE base when the workload uses rotary positions
    q_pos: Optional[np.ndarray] = None  # [sum L] int32 position of each query token
    kv_pos: Optional[np.ndarray] = None  # [sum kv_len] int32 position of each key, k_tok order
    dv: int = 0                      # elements of a value row (0: the key's d)

    def __post_init__(self):
        if not self.dv:
            self.dv = self.d

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv

    @property
    def total_qo(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == FP8 else 2

    @property
    def has_mask(self) -> bool:
        return self.mask is not None

    @property
    def nhd(self) -> bool:
        return self.kv_layout == "nhd"

    def new_positions(self):
        """Positions of the draft tokens' keys, in qo_indptr order (what an
        append with RoPE rotates the new keys by)."""
        if self.kv_pos is None:
            return None
        sel = np.concatenate([
            np.arange(self.tok_indptr[b + 1] - self.qo_lens[b], self.tok_indptr[b + 1])
            for b in range(self.batch)]) if self.batch else np.zeros(0, np.int64)
        return self.kv_pos[sel].astype(np.int32)

    def new_tokens(self):
        """The draft tokens' K/V (the last L_b tokens of each request), laid
        out [sum L, h_kv, d] in qo_indptr order: what an append writes."""
        sel = np.concatenate([
            np.arange(self.tok_indptr[b + 1] - self.qo_lens[b], self.tok_indptr[b + 1])
            for b in range(self.batch)]) if self.batch else np.zeros(0, np.int64)
        return self.k_tok[sel], self.v_tok[sel]

    def tok_append_indptr(self) -> np.ndarray:
        """Append offsets that write every token of every request (prefix and
        drafts) in one call: n_b = kv_len_b."""
        return self.tok_indptr.astype(np.int32)


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _fp8_bits(x: torch.Tensor, scale: float) -> np.ndarray:
    return (x / scale).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _draw_lengths(spec, batch, gen):
    kind, val = spec
    if kind == "fixed":
        assert len(val) == batch
        return np.asarray(val, dtype=np.int64)
    lo, hi = val
    return torch.randint(lo, hi + 1, (batch,), generator=gen).numpy().astype(np.int64)


def _draw_tree(n, gen):
    """parent[0] = -1 (the root); parent[i] uniform in [0, i)."""
    parents = [-1]
    for i in range(1, n):
        parents.append(int(torch.randint(0, i, (1,), generator=gen).item()))
    return parents


def ancestor_mask(parents) -> np.ndarray:
    """Dense [L, L] bool: row i sees column j iff j == i or j is an ancestor
    of i (the tree-attention mask of FlashInfer issue #152, "How to implement
    a tree attention")."""
    n = len(parents)
    m = np.zeros((n, n), dtype=bool)
    for i in range(n):
        j = i
        while j >= 0:
            m[i, j] = True
            j = parents[j]
    return m


def pack_masks(dense_list):
    """Bit-pack per-request bool blocks ([L_b, L_b], or [L_b, kv_len_b] for the
    full layout) LSB-first into one uint8 array; returns (bytes, bit offsets
    [B+1])."""
    offs = [0]
    for m in dense_list:
        offs.append(offs[-1] + m.size)
    nbits = offs[-1]
    bits = np.zeros(max(nbits, 1), dtype=np.uint8)
    if nbits:
        bits[:nbits] = np.concatenate([m.reshape(-1) for m in dense_list if m.size]).astype(np.uint8)
    packed = np.packbits(bits, bitorder="little")
    return packed, np.asarray(offs, dtype=np.int32)


def make_workload(name: str, seed: int = 0, **overrides) -> Workload:
    """One of the named workloads (``WORKLOADS``), optionally with fields
    overridden (e.g. a smaller batch for a quick test)."""
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    return make_custom(name=name, seed=seed, **spec)


def make_custom(name="custom", seed=0, batch=2, h_q=4, h_kv=2, d=64, page_size=16,
                kv_dtype=BF16, prefix=("fixed", [37, 70]), qo=("fixed", [5, 5]),
                mask="causal", pool_pages=None, pool_factor=1.25, sm_scale=None,
                shuffle_pages=True, value_std=1.0, with_values=True, kv_layout="hnd",
                mask_layout="qlen", prefix_visible="all", rope_theta=None, dv=None) -> Workload:
    """A workload from explicit parameters.  with_values=False draws only the
    tables (lengths, trees, pages; q / k / v come last in the draw order, so the
    tables are the same either way) and leaves q / k_tok / v_tok empty.

    kv_layout "nhd" lays the page pool out [pages, P, h_kv, d].  mask_layout
    "full" packs each request's mask as L rows of kv_len bits (prefix
    columns included): prefix_visible "all" sets every prefix bit, "random"
    draws them (after every other draw).  rope_theta gives the workload rotary
    positions: a prefix key at index j has position j, draft u has position
    prefix + depth(u) (its tree depth; u itself for chains and masks without
    a tree), and each query token has its draft's position.  dv gives value
    rows of their own width (v_tok [sum kv_len, h_kv, dv]); the default is d."""
    gen = torch.Generator().manual_seed(seed)
    prefix_lens = _draw_lengths(prefix, batch, gen)
    qo_lens = _draw_lengths(qo, batch, gen)
    kv_lens = prefix_lens + qo_lens

    # draft structure
    parents, dense = None, None
    if mask in ("tree", "chain", "random", "full", "none_visible"):
        parents, dense = [], []
        for b in range(batch):
            L = int(qo_lens[b])
            if mask == "tree":
                p = _draw_tree(L, gen)
                parents.append(p)
                dense.append(ancestor_mask(p))
            elif mask == "chain":
                p = [i - 1 for i in range(L)]
                parents.append(p)
                dense.append(ancestor_mask(p))
            elif mask == "random":
                parents.append(None)
                dense.append(torch.rand((L, L), generator=gen).numpy() < 0.5)
            elif mask == "full":
                parents.append(None)
                dense.append(np.ones((L, L), dtype=bool))
            else:  # none_visible: no draft column visible (fully masked rows when prefix is 0)
                parents.append(None)
                dense.append(np.zeros((L, L), dtype=bool))
    elif mask != "causal":
        raise ValueError(mask)

    # page table over a shuffled pool
    pages_per = np.array([(int(n) + page_size - 1) // page_size for n in kv_lens], dtype=np.int64)
    total_pages = int(pages_per.sum())
    if pool_pages is None:
        pool_pages = max(1, int(math.ceil(total_pages * pool_factor)))
    assert pool_pages >= total_pages
    # always drawn, so that the q / k / v draws after it do not depend on
    # whether the pages are shuffled
    perm = torch.randperm(pool_pages, generator=gen).numpy()
    if not shuffle_pages:
        perm = np.arange(pool_pages)
    kv_indices = perm[:total_pages].astype(np.int32)
    kv_indptr = np.zeros(batch + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum(pages_per)
    last_page_len = np.array([n - (p - 1) * page_size if p > 0 else 0
                              for n, p in zip(kv_lens, pages_per)], dtype=np.int32)
    qo_indptr = np.zeros(batch + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    tok_indptr = np.zeros(batch + 1, dtype=np.int64)
    tok_indptr[1:] = np.cumsum(kv_lens)

    total_qo = int(qo_indptr[-1])
    total_tok = int(tok_indptr[-1])
    if not with_values:
        total_qo = total_tok = 0
    qf = torch.randn((total_qo, h_q, d), generator=gen) * value_std
    q = _bf16_bits(qf)
    del qf
    kf = torch.randn((total_tok, h_kv, d), generator=gen) * value_std
    if kv_dtype == FP8:
        k_scale = float(np.float32(float(kf.abs().max()) / 448.0)) if total_tok else 1.0
        k_tok = _fp8_bits(kf, k_scale)
    else:
        k_scale = 1.0
        k_tok = _bf16_bits(kf)
    del kf
    dv = d if dv is None else int(dv)
    vf = torch.randn((total_tok, h_kv, dv), generator=gen) * value_std
    if kv_dtype == FP8:
        v_scale = float(np.float32(float(vf.abs().max()) / 448.0)) if total_tok else 1.0
        v_tok = _fp8_bits(vf, v_scale)
    else:
        v_scale = 1.0
        v_tok = _bf16_bits(vf)
    del vf

    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    sm_scale = float(np.float32(sm_scale))

    packed, mask_indptr = (None, None)
    mask_full = None
    if dense is not None and mask_layout == "full":
        mask_full = []
        for b in range(batch):
            L, pre = int(qo_lens[b]), int(prefix_lens[b])
            m = np.zeros((L, pre + L), dtype=bool)
            if prefix_visible == "random":
                m[:, :pre] = torch.rand((L, pre), generator=gen).numpy() < 0.5
            else:
                m[:, :pre] = True
            m[:, pre:] = dense[b]
            mask_full.append(m)
        packed, mask_indptr = pack_masks(mask_full)
    elif dense is not None:
        packed, mask_indptr = pack_masks(dense)
    elif mask_layout != "qlen":
        raise ValueError("a full-layout mask needs a mask kind other than causal")

    q_pos = kv_pos = None
    if rope_theta is not None:
        kv_pos = np.zeros(int(tok_indptr[-1]), dtype=np.int32)
        q_pos = np.zeros(int(qo_indptr[-1]), dtype=np.int32)
        for b in range(batch):
            L, pre = int(qo_lens[b]), int(prefix_lens[b])
            depth = list(range(L))
            if parents is not None and parents[b] is not None:
                for u in range(L):
                    depth[u] = 0 if parents[b][u] < 0 else depth[parents[b][u]] + 1
            t0 = int(tok_indptr[b])
            kv_pos[t0:t0 + pre] = np.arange(pre)
            kv_pos[t0 + pre:t0 + pre + L] = pre + np.asarray(depth, dtype=np.int64)
            q_pos[int(qo_indptr[b]):int(qo_indptr[b]) + L] = pre + np.asarray(depth, dtype=np.int64)

    return Workload(
        name=name, batch=batch, h_q=h_q, h_kv=h_kv, d=d, page_size=page_size,
        kv_dtype=kv_dtype, prefix_lens=prefix_lens, qo_lens=qo_lens, kv_lens=kv_lens,
        qo_indptr=qo_indptr, kv_indptr=kv_indptr, kv_indices=kv_indices,
        last_page_len=last_page_len, num_pages=int(pool_pages), tok_indptr=tok_indptr,
        q=q, k_tok=k_tok, v_tok=v_tok, sm_scale=sm_scale, k_scale=k_scale,
        v_scale=v_scale, mask_kind=mask, parents=parents, mask_dense=dense,
        mask=packed, mask_indptr=mask_indptr, kv_layout=kv_layout, mask_layout=mask_layout,
        mask_full=mask_full, rope_theta=rope_theta, q_pos=q_pos, kv_pos=kv_pos, dv=dv)


def sentinel_pool(wl: Workload, values: bool = False) -> np.ndarray:
    """An empty page pool [num_pages, h_kv, page_size, d] (values=True: rows
    of the value width dv) filled with 0xFF bytes: NaN in both bf16 and
    fp8-e4m3, so any read of an unwritten slot shows up in the result."""
    dt = np.uint8 if wl.kv_dtype == FP8 else np.uint16
    fill = 0xFF if wl.kv_dtype == FP8 else 0xFFFF
    w = wl.dv if values else wl.d
    if wl.nhd:
        return np.full((wl.num_pages, wl.page_size, wl.h_kv, w), fill, dtype=dt)
    return np.full((wl.num_pages, wl.h_kv, wl.page_size, w), fill, dtype=dt)


def sample_rows(wl: Workload, n: int, seed: int = 1):
    """A seeded sample of (token, q-head) output rows, as flat indices
    token * h_q + head; always includes each request's first and last token."""
    rng = np.random.default_rng(seed)
    total = wl.total_qo * wl.h_q
    must = []
    for b in range(wl.batch):
        if wl.qo_lens[b] == 0:
            continue
        for t in (int(wl.qo_indptr[b]), int(wl.qo_indptr[b + 1]) - 1):
            must.append(t * wl.h_q + int(rng.integers(wl.h_q)))
    extra = rng.choice(total, size=min(n, total), replace=False) if total else np.zeros(0, np.int64)
    rows = np.unique(np.concatenate([np.asarray(must, np.int64), extra.astype(np.int64)]))
    return rows.astype(np.int32)

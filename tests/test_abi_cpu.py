"""C-ABI checks that need no GPU: the library loads, exports every function
include/verify_attn.h declares, and the host planner's work lists cover each
request's rows and keys exactly once; argument validation returns the
documented status codes without touching a device."""
import ctypes
import os
import re

import numpy as np
import pytest

import synthetic

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "verify_attn.h")


@pytest.fixture(scope="module")
def va():
    import __graft_entry__
    from speculative_decoding_verify_gqa_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gqa_gb300 as m
    m.lib()
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for", "sizeof")))


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for must in ("verify_attn_plan", "verify_attn_run", "paged_kv_append",
                 "verify_attn_plan_host", "verify_attn_partial", "verify_attn_merge",
                 "verify_attn_device_status", "verify_attn_status_string",
                 "verify_attn_workspace_size"):
        assert must in names


def test_library_exports_every_declared_symbol(va):
    lib = ctypes.CDLL(va.library_path)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(va):
    assert va.status_string(0) == "ok"
    for code in range(-8, 0):
        assert va.status_string(code) != "unknown status"
    assert va.status_string(-99) == "unknown status"


# ------------------------------------------------------------------ planner

def _tables(seed, batch, G, h_kv, page_size, max_prefix, max_L, masked):
    rng = np.random.default_rng(seed)
    prefix = rng.integers(0, max_prefix + 1, size=batch)
    L = rng.integers(0, max_L + 1, size=batch)
    kv_len = prefix + L
    pages = (kv_len + page_size - 1) // page_size
    kv_indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    last = np.where(pages > 0, kv_len - (pages - 1) * page_size, 0).astype(np.int32)
    qo_indptr = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    mask_indptr = np.concatenate([[0], np.cumsum(L * L)]).astype(np.int32) if masked else None
    return dict(masked=masked, prefix=prefix, L=L, kv_len=kv_len, kv_indptr=kv_indptr, last=last,
                qo_indptr=qo_indptr, mask_indptr=mask_indptr, h_q=G * h_kv, h_kv=h_kv,
                G=G, page_size=page_size)


def _check_cover(va, t, plan):
    hd = plan.header()
    items = plan.items()
    merges = plan.merges()
    assert hd["n_items"] == len(items) and hd["n_merge"] == len(merges)
    BM = hd["block_rows"]
    G = t["G"]
    units = {}
    for i, it in enumerate(items):
        b, h, row0, nrows, lo, hi, part_row, _ = (int(x) for x in it)
        assert 0 <= b < len(t["L"]) and 0 <= h < t["h_kv"]
        assert 0 < nrows <= BM and row0 % BM == 0
        # chunks start on key tiles; a draft item (tcgen05 variants) starts
        # at the request's prefix length and holds at most one key tile
        assert lo < hi
        assert lo % 64 == 0 or (lo == int(t["prefix"][b]) and hd["kernel"] in (3, 4)
                                and hi - lo <= 128)
        units.setdefault((b, h, row0, nrows), []).append((lo, hi, part_row))
    for b in range(len(t["L"])):
        R = G * int(t["L"][b])
        for h in range(t["h_kv"]):
            rows = sorted((k[2], k[3]) for k in units if k[0] == b and k[1] == h)
            pos = 0
            for row0, nrows in rows:
                assert row0 == pos
                pos += nrows
            assert pos == R
    merge_by_unit = {(int(m[0]), int(m[1]), int(m[2]), int(m[3])): m for m in merges}
    used = np.zeros(max(hd["part_rows"], 1), dtype=np.int32)
    for (b, h, row0, nrows), chunks in units.items():
        chunks.sort()
        tmax = (row0 + nrows - 1) // G
        if t.get("masked"):   # a custom mask may open later drafts: whole kv range
            kv_end = int(t["prefix"][b]) + int(t["L"][b])
        else:
            kv_end = int(t["prefix"][b]) + tmax + 1
        pos = 0
        for lo, hi, _ in chunks:
            assert lo == pos
            pos = hi
        assert pos == kv_end
        if len(chunks) == 1:
            assert all(c[2] == -1 for c in chunks) and (b, h, row0, nrows) not in merge_by_unit
        else:
            m = merge_by_unit[(b, h, row0, nrows)]
            assert int(m[5]) == len(chunks)
            for s, (lo, hi, part_row) in enumerate(chunks):
                assert part_row == int(m[4]) + s * nrows
                used[part_row:part_row + nrows] += 1
    assert used.max(initial=0) <= 1
    assert used.sum() == hd["part_rows"]


@pytest.mark.parametrize("case", [
    dict(seed=1, batch=5, G=4, h_kv=2, page_size=16, max_prefix=300, max_L=17, masked=True),
    dict(seed=2, batch=64, G=8, h_kv=8, page_size=16, max_prefix=8192, max_L=8, masked=False),
    dict(seed=3, batch=3, G=8, h_kv=1, page_size=1, max_prefix=50, max_L=40, masked=False),
    dict(seed=4, batch=7, G=1, h_kv=4, page_size=64, max_prefix=2000, max_L=200, masked=True),
    dict(seed=5, batch=1, G=16, h_kv=1, page_size=256, max_prefix=0, max_L=300, masked=False),
    dict(seed=6, batch=4, G=2, h_kv=3, page_size=8, max_prefix=5, max_L=0, masked=False),
])
@pytest.mark.parametrize("num_sms", [152, 7])
def test_plan_covers_rows_and_keys_exactly_once(va, case, num_sms):
    t = _tables(**case)
    for opts in (dict(), dict(max_splits=1), dict(max_splits=3, min_chunk=64),
                 dict(target_ctas=10000)):
        plan = va.verify_attn_plan_host(t["kv_indptr"], t["qo_indptr"], t["last"],
                                        t["mask_indptr"], t["h_q"], t["h_kv"], 128,
                                        t["page_size"], num_sms=num_sms, **opts)
        _check_cover(va, t, plan)
        if opts.get("max_splits") == 1:
            assert plan.header()["n_merge"] == 0
        pb, wb = va.verify_attn_plan_bounds(len(t["L"]), int(t["qo_indptr"][-1]), t["h_q"],
                                            t["h_kv"], 128, num_sms)
        assert plan.workspace_bytes <= wb
        assert 184 + 32 * (plan.header()["n_items"] + plan.header()["n_merge"]) <= pb


def _check_chains(plan):
    """Persistent tcgen05 plans: chain c starts at item c, links run through
    the last field, and the chains visit every item exactly once."""
    hd = plan.header()
    it = plan.items()
    n = len(it)
    assert hd["n_ctas"] == min(n, hd["num_sms"])
    seen = np.zeros(n, dtype=np.int32)
    for c in range(hd["n_ctas"]):
        i = c
        while i >= 0:
            assert 0 <= i < n
            seen[i] += 1
            i = int(it[i, 7])
    assert np.all(seen == 1)


@pytest.mark.parametrize("seed", range(32))
def test_random_plans_cover_rows_and_keys(va, seed):
    """Random batches (group size, KV heads, page size, prefix and draft
    lengths, masks, head_dim, SM count) planned for every variant that can
    serve them, under random split options: every (request, KV head) row is
    covered once, each unit's kv range exactly once in order, partial rows
    once, the persistent variants' chains visit every item once, and the plan
    fits the sizes verify_attn_plan_bounds promises."""
    rng = np.random.default_rng(9000 + seed)
    G = int(rng.choice([1, 2, 4, 8, 16]))
    page_size = int(rng.choice([16, 32, 64]))
    t = _tables(seed=seed, batch=int(rng.integers(1, 40)), G=G, h_kv=int(rng.integers(1, 5)),
                page_size=page_size, max_prefix=int(rng.choice([0, 100, 3000])),
                max_L=int(rng.choice([1, 8, 40, 200])), masked=bool(rng.integers(0, 2)))
    d = int(rng.choice([64, 128]))
    num_sms = int(rng.choice([152, 13, 1]))
    kernels = [0, 1, 2] + ([3, 4] if d == 128 and 128 % G == 0 else [])
    for kernel in kernels:
        opts = dict(kernel=kernel, max_splits=int(rng.choice([0, 1, 2, 5])),
                    min_chunk=int(rng.choice([0, 64, 256])),
                    target_ctas=int(rng.choice([0, 50, 5000])))
        plan = va.verify_attn_plan_host(t["kv_indptr"], t["qo_indptr"], t["last"],
                                        t["mask_indptr"], t["h_q"], t["h_kv"], d, page_size,
                                        num_sms=num_sms, **opts)
        hd = plan.header()
        if kernel:
            assert hd["kernel"] == kernel
        _check_cover(va, t, plan)
        if hd["kernel"] in (3, 4):
            _check_chains(plan)
        else:
            assert hd["n_ctas"] == 0 and np.all(plan.items()[:, 7] == -1)
        pb, wb = va.verify_attn_plan_bounds(len(t["L"]), int(t["qo_indptr"][-1]), t["h_q"],
                                            t["h_kv"], d, num_sms)
        assert plan.workspace_bytes <= wb
        assert 184 + 32 * (hd["n_items"] + hd["n_merge"]) <= pb


@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER)
def test_plans_of_the_named_workloads(va, name):
    wl = synthetic.make_workload(name, with_values=False)
    t = dict(masked=wl.mask is not None, prefix=wl.prefix_lens, L=wl.qo_lens, G=wl.group, h_kv=wl.h_kv)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                    wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                    kv_dtype=wl.kv_dtype, num_sms=152)
    _check_cover(va, t, plan)
    hd = plan.header()
    # kernel variant follows the rows per KV head (G * L) and the cache dtype
    rows = int((wl.group * wl.qo_lens).max())
    if wl.d == 128 and 128 % wl.group == 0 and wl.page_size % 16 == 0:
        assert hd["kernel"] == (4 if rows > 128 else 3)
    else:
        assert hd["kernel"] == (1 if rows <= 64 else 2)


@pytest.mark.parametrize("draft_items", [0, 1, -1])
def test_draft_items(va, draft_items):
    """Draft items: with few split units (the Llama-3-8B tree: 8 KV heads,
    each split many ways) every split unit's drafts -- keys prefix .. kv_len
    -- form one item of their own, merged with the prefix chunks; never for
    the warp-level variants or when turned off."""
    wl = synthetic.make_workload("llama3_8b_tree_verify", with_values=False)
    t = dict(masked=True, prefix=wl.prefix_lens, L=wl.qo_lens, G=wl.group, h_kv=wl.h_kv)
    pre, kv = int(wl.prefix_lens[0]), int(wl.kv_lens[0])
    for kernel in (0, 2):
        plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                        wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                        num_sms=152, kernel=kernel, draft_items=draft_items)
        _check_cover(va, t, plan)
        drafts = [it for it in plan.items() if int(it[4]) == pre]
        if kernel == 0 and draft_items >= 0:
            assert len(drafts) == wl.h_kv
            assert all(int(it[5]) == kv and int(it[6]) >= 0 for it in drafts)
            # the chunk before the drafts ends at the prefix
            assert sum(1 for it in plan.items() if int(it[5]) == pre) == wl.h_kv
        elif kernel == 0:
            assert not drafts   # the 17 drafts join the last prefix chunk
    # many split units (the batched chain): none unless forced
    wl = synthetic.make_workload("codellama34b_chain_verify", with_values=False)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, None, wl.h_q,
                                    wl.h_kv, wl.d, wl.page_size, num_sms=152,
                                    draft_items=draft_items)
    t = dict(masked=False, prefix=wl.prefix_lens, L=wl.qo_lens, G=wl.group, h_kv=wl.h_kv)
    _check_cover(va, t, plan)
    n_drafts = sum(1 for it in plan.items() if int(it[4]) == int(wl.prefix_lens[int(it[0])])
                   and int(it[4]) % 64)
    assert (n_drafts > 0) == (draft_items == 1)
    assert _plan_rc(va, [0, 2], [0, 3], [5], None, draft_items=2) == -1


@pytest.mark.parametrize("name", ["gqa_varlen_prefill", "wide_tree_fp8_verify",
                                  "llama3_8b_tree_verify"])
@pytest.mark.parametrize("kernel", [3, 4])
def test_tcgen05_plans_cover_every_row_once(va, name, kernel):
    """The tcgen05 variants' plans (128- and 256-row blocks) cover each
    (request, KV head, row) with chunks that tile its kv range."""
    wl = synthetic.make_workload(name, with_values=False)
    t = dict(masked=wl.mask is not None, prefix=wl.prefix_lens, L=wl.qo_lens, G=wl.group, h_kv=wl.h_kv)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                    wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                    kv_dtype=wl.kv_dtype, num_sms=152, kernel=kernel)
    hd = plan.header()
    assert hd["kernel"] == kernel and hd["block_rows"] == (128 if kernel == 3 else 256)
    _check_cover(va, t, plan)


@pytest.mark.parametrize("name", ["gqa_varlen_prefill", "wide_tree_fp8_verify",
                                  "codellama34b_chain_verify"])
def test_tcgen05_plans_chain_every_item_once(va, name):
    """The persistent tcgen05 kernel walks one chain of items per CTA: chain c
    starts at item c, links run through the last field, and together the
    chains visit every item exactly once, with near-equal loads."""
    wl = synthetic.make_workload(name, with_values=False)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                    wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                    kv_dtype=wl.kv_dtype, num_sms=152, kernel=4)
    hd = plan.header()
    it = plan.items()
    n = len(it)
    assert hd["n_ctas"] == min(n, 152)
    seen = np.zeros(n, dtype=np.int32)
    loads = []
    for c in range(hd["n_ctas"]):
        i, load = c, 0
        while i >= 0:
            assert 0 <= i < n
            seen[i] += 1
            load += int(it[i, 5] - it[i, 4])
            i = int(it[i, 7])
        loads.append(load)
    assert np.all(seen == 1)
    # longest-processing-time dealing: no chain exceeds the mean by more than
    # the longest item
    longest = int((it[:, 5] - it[:, 4]).max())
    assert max(loads) <= np.mean(loads) + longest + 256


@pytest.mark.parametrize("name", ["codellama34b_chain_verify", "gqa_varlen_prefill", "rand"])
def test_chain_dealing_is_longest_first_onto_the_least_loaded_chain(va, name):
    """The chains of a persistent tcgen05 plan are the longest-first dealing
    of its items: items ordered by cost ((hi - lo) (nrows + 16)) descending,
    then (b, h, kv_lo, row0), each to the chain with the least load (key
    tiles + 1, times 5 for a two-Q-tile item, 3 for one), the lowest chain
    index among equal loads -- dealt here one item at a time from a heap."""
    import heapq
    if name == "rand":
        rng = np.random.default_rng(3)
        batch, G, hkv = 57, 4, 8
        L = rng.integers(1, 120, batch)
        kv = rng.integers(0, 5000, batch) + L
        pages = (kv + 15) // 16
        tabs = (np.concatenate([[0], np.cumsum(pages)]).astype(np.int32),
                np.concatenate([[0], np.cumsum(L)]).astype(np.int32),
                (kv - (pages - 1) * 16).astype(np.int32), None, hkv * G, hkv, 128, 16)
        kvd = "bf16"
    else:
        wl = synthetic.make_workload(name, with_values=False)
        tabs = (wl.kv_indptr, wl.qo_indptr, wl.last_page_len, wl.mask_indptr, wl.h_q, wl.h_kv,
                wl.d, wl.page_size)
        kvd = wl.kv_dtype
    plan = va.verify_attn_plan_host(*tabs, kv_dtype=kvd, num_sms=152)
    hd = plan.header()
    assert hd["kernel"] in (3, 4)
    it = plan.items()
    n, nc, tk = len(it), hd["n_ctas"], hd["tile_keys"]
    assert n > nc
    chain = np.full(n, -1)
    for c in range(nc):
        i = c
        while i >= 0:
            chain[i] = c
            i = int(it[i, 7])
    order = sorted(range(n), key=lambda i: (-(int(it[i, 5]) - int(it[i, 4])) * (int(it[i, 3]) + 16),
                                           int(it[i, 0]), int(it[i, 1]), int(it[i, 4]), int(it[i, 2])))
    heap = [(0, c) for c in range(nc)]
    for i in order:
        load, c = heapq.heappop(heap)
        assert chain[i] == c
        tiles = -(-(int(it[i, 5]) - int(it[i, 4])) // tk) + 1
        heapq.heappush(heap, (load + tiles * (5 if it[i, 3] > 128 else 3), c))
    # and within a chain the items run in the dealing order
    pos = {i: k for k, i in enumerate(order)}
    for c in range(nc):
        i, last = c, -1
        while i >= 0:
            assert pos[i] > last
            last = pos[i]
            i = int(it[i, 7])


@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER)
def test_plan_header_records_the_largest_split(va, name):
    """The merge kernel sizes its load batch from the plan header's largest
    split count: it must equal the largest nsplit of the merge list (0 with
    no merges)."""
    wl = synthetic.make_workload(name, with_values=False)
    for opts in ({}, {"kernel": 3}, {"max_splits": 3}):
        plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                        wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                        kv_dtype=wl.kv_dtype, num_sms=152,
                                        **(opts if wl.d == 128 or "kernel" not in opts else {}))
        m = plan.merges()
        assert plan.header()["max_nsplit"] == (int(m[:, 5].max()) if len(m) else 0)


def _model_chunk(kvp, qop, lpl, has_mask, h_q, h_kv, d, page, fp8, num_sms, kernel):
    """The split size the planner's cost model picks, restated item by item:
    units of row blocks, candidate chunk sizes (1-4 waves of CTA slots, equal
    or full-plus-remainder cuts, and for the tcgen05 variants the n-way cuts
    of the longest unit), each scored by placing every item longest-first on
    the least-loaded slot (a heap), the first clearly (3 %) better kept."""
    import heapq
    cdiv = lambda a, b: -(-a // b)
    tc = kernel in (3, 4)
    G = h_q // h_kv
    bm = 64 if kernel == 1 else (256 if kernel == 4 else 128)
    tk = 128 if tc else 64
    units = []
    for b in range(len(qop) - 1):
        npg, L = int(kvp[b + 1] - kvp[b]), int(qop[b + 1] - qop[b])
        kv = (npg - 1) * page + int(lpl[b]) if npg > 0 else 0
        prefix = kv - L
        for row0 in range(0, G * L, bm):
            nrows = min(bm, G * L - row0)
            units.append((nrows, prefix + L if has_mask else prefix + (row0 + nrows - 1) // G + 1))
    W = sum(k for _, k in units) * h_kv
    slots = num_sms * ((1 if fp8 else 2) if kernel == 3 else (2 if kernel == 1 else 1))
    key_bytes = 2 * d * (1 if fp8 else 2)
    fixed = 64 * 1024 if tc else 48 * 1024
    min_chunk = 2 * tk
    chunk_for = lambda t: max(min_chunk, cdiv(cdiv(W, max(t, 1)), tk) * tk)
    latency = tc and W * key_bytes <= 4 * 64 * 1024 * num_sms
    cand_slots = max(1, 2 * num_sms // 3) if latency else slots
    longest = max(k for _, k in units)
    whole = max(min_chunk, cdiv(longest, tk) * tk)
    cands = []

    def add(c, eq):
        if c >= whole:
            c, eq = whole, True
        if (c, eq) not in cands:
            cands.append((c, eq))
    for cand in range(8):
        add(chunk_for(min((1 + (cand >> 1)) * cand_slots, 4 * num_sms)), cand % 2 == 0)
    unit_heads = max(1, len(units) * h_kv)
    if tc and unit_heads < cand_slots:
        for k in range(1, 7):
            n0 = (k * cand_slots + unit_heads // 2) // unit_heads
            for n in range(max(1, n0 - 1), min(32, n0 + 1) + 1):
                add(max(min_chunk, cdiv(cdiv(longest, n), tk) * tk), True)
    best, chunk = -1.0, chunk_for(cand_slots)
    for c, eq in cands:
        costs = []
        for nrows, kv_end in units:
            n = max(cdiv(kv_end, c), 1)
            cu = cdiv(cdiv(kv_end, n), tk) * tk if (eq or n * c < kv_end) else c
            n = cdiv(kv_end, cu)
            for s_ in range(n):
                keys = min(cu, kv_end - s_ * cu)
                costs += [fixed + keys * key_bytes + (nrows * 4 * d if n > 1 else 0)] * h_kv
        costs.sort(reverse=True)
        loads = costs[:cand_slots]
        finish = max(costs)
        heapq.heapify(loads)
        for x in costs[cand_slots:]:
            lo = heapq.heappop(loads) + x
            finish = max(finish, lo)
            heapq.heappush(loads, lo)
        if best < 0 or finish < best * 0.97:
            best, chunk = float(finish), c
    return chunk


@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER + ["rand0", "rand1", "rand2"])
def test_split_size_is_the_cost_models_choice(va, name):
    """The plan's split size equals the cost model's choice restated above
    (the planner scores candidates on grouped items; the choice must be the
    same as placing every item one by one)."""
    if name.startswith("rand"):
        rng = np.random.default_rng(int(name[-1]) + 20)
        batch = int(rng.integers(1, 40))
        G, hkv = int(rng.choice([1, 4, 8])), int(rng.choice([2, 8]))
        L = rng.integers(1, int(rng.choice([10, 80])), batch)
        kv = rng.integers(0, int(rng.choice([600, 9000])), batch) + L
        pages = (kv + 15) // 16
        kvp = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
        qop = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
        lpl = (kv - (pages - 1) * 16).astype(np.int32)
        tabs = (kvp, qop, lpl, None, hkv * G, hkv, 128, 16)
        kvd = "fp8_e4m3" if name == "rand2" else "bf16"
    else:
        wl = synthetic.make_workload(name, with_values=False)
        tabs = (wl.kv_indptr, wl.qo_indptr, wl.last_page_len, wl.mask_indptr, wl.h_q, wl.h_kv,
                wl.d, wl.page_size)
        kvd = wl.kv_dtype
    plan = va.verify_attn_plan_host(*tabs, kv_dtype=kvd, num_sms=152)
    hd = plan.header()
    assert hd["chunk"] == _model_chunk(tabs[0], tabs[1], tabs[2], tabs[3] is not None, tabs[4],
                                       tabs[5], tabs[6], tabs[7], kvd != "bf16", 152, hd["kernel"])


def test_warp_level_plans_have_no_chains(va):
    wl = synthetic.make_workload("llama3_8b_tree_verify", with_values=False)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                    wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                    num_sms=152, kernel=2)
    assert plan.header()["n_ctas"] == 0 and np.all(plan.items()[:, 7] == -1)


def test_plan_items_sorted_longest_first(va):
    # the warp-level variant's list (the hardware hands it to SMs in order)
    wl = synthetic.make_workload("codellama34b_chain_verify", with_values=False)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, None,
                                    wl.h_q, wl.h_kv, wl.d, wl.page_size, num_sms=152, kernel=1)
    it = plan.items()
    cost = (it[:, 5] - it[:, 4]) * (it[:, 3] + 16)
    assert np.all(np.diff(cost) <= 0)


@pytest.mark.parametrize("name", synthetic.WORKLOAD_ORDER)
def test_workspace_size_covers_the_named_workloads(va, name):
    """verify_attn_workspace_size(batch, heads, head_dim, max_qo_len, SMs),
    through the C ABI, is at least what the planner needs for each named
    workload, whatever kernel variant or split option the plan takes."""
    wl = synthetic.make_workload(name, with_values=False)
    n = ctypes.c_size_t(0)
    rc = va.lib().verify_attn_workspace_size(wl.batch, wl.h_q, wl.h_kv, wl.d,
                                             int(wl.qo_lens.max()), 152, ctypes.byref(n))
    assert rc == 0 and n.value > 0
    kernels = [0, 1, 2] + ([3, 4] if wl.d == 128 and 128 % wl.group == 0 else [])
    for kernel in kernels:
        for opts in (dict(), dict(max_splits=1), dict(target_ctas=5000, min_chunk=64)):
            plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                            wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                            kv_dtype=wl.kv_dtype, num_sms=152, kernel=kernel,
                                            **opts)
            assert plan.workspace_bytes <= n.value
    assert va.verify_attn_workspace_size(wl.batch, wl.h_q, wl.h_kv, wl.d,
                                         int(wl.qo_lens.max()), 152) == n.value
    assert va.lib().verify_attn_workspace_size(-1, 4, 2, 128, 1, 152, ctypes.byref(n)) == -1
    assert va.lib().verify_attn_workspace_size(1, 5, 2, 128, 1, 152, ctypes.byref(n)) == -1
    assert va.lib().verify_attn_workspace_size(1, 4, 2, 128, 1, 152, None) == -1


# ------------------------------------------------------------------ validation

def _plan_rc(va, kv_indptr, qo_indptr, last, mask_indptr, h_q=4, h_kv=2, d=128, P=16,
             kv_dtype=0, has_mask=None, plan_bytes=1 << 16, **opts):
    lib = va.lib()
    host = np.zeros(plan_bytes, np.uint8)
    need = ctypes.c_size_t(0)
    o = va._options(**opts)
    arrs = [None if a is None else np.ascontiguousarray(a, np.int32)
            for a in (kv_indptr, qo_indptr, last, mask_indptr)]
    if has_mask is None:
        has_mask = mask_indptr is not None
    return lib.verify_attn_plan_host(*[va._hp(a) for a in arrs], len(arrs[1]) - 1, h_q, h_kv, d,
                                     P, 0, kv_dtype, int(has_mask), 152, ctypes.byref(o),
                                     va._hp(host), plan_bytes, ctypes.byref(need))


def test_plan_validation_codes(va):
    ok = ([0, 2], [0, 3], [5], None)
    assert _plan_rc(va, *ok) == 0
    assert _plan_rc(va, *ok, h_q=5, h_kv=2) == -1          # h_q % h_kv
    assert _plan_rc(va, *ok, d=96) == -2                   # head_dim
    assert _plan_rc(va, *ok, P=12) == -2                   # page size not a power of two
    assert _plan_rc(va, *ok, P=512) == -2
    assert _plan_rc(va, *ok, kv_dtype=7) == -2
    assert _plan_rc(va, [0, 1], [0, 3], [2], None) == -1   # kv_len 2 < L 3
    assert _plan_rc(va, [0, 2], [0, 3], [0], None) == -1   # last_page_len 0 with pages
    assert _plan_rc(va, [0, 2], [0, 3], [17], None) == -1  # last_page_len > page size
    assert _plan_rc(va, [0, 2], [0, 3], [5], [0, 8]) == -1  # mask block != L*L
    assert _plan_rc(va, [0, 2], [0, 3], [5], [0, 9]) == 0
    assert _plan_rc(va, [0, 2], [0, 3], [5], None, has_mask=1) == -1
    assert _plan_rc(va, *ok, plan_bytes=64) == -7
    assert _plan_rc(va, [0, 2, 1], [0, 3, 3], [5, 1], None) == -1  # decreasing indptr
    assert _plan_rc(va, *ok, max_splits=-1) == -1
    assert _plan_rc(va, *ok, kernel=9) == -1
    assert _plan_rc(va, *ok, kernel=4) == 0
    assert _plan_rc(va, *ok, kernel=4, d=64) == -2         # tcgen05 variants: head_dim 128 only
    assert _plan_rc(va, *ok, kernel=3, P=8) == -2          # page boxes of 16 rows
    # e4m3 queries: an fp8 cache and a tcgen05 variant (auto picks one)
    assert _plan_rc(va, *ok, kv_dtype=1, q_fp8=True) == 0
    assert _plan_rc(va, *ok, kv_dtype=1, q_fp8=True, kernel=4) == 0
    assert _plan_rc(va, *ok, kv_dtype=0, q_fp8=True) == -2     # bf16 cache
    assert _plan_rc(va, *ok, kv_dtype=1, q_fp8=True, kernel=2) == -2   # warp-level variant
    assert _plan_rc(va, *ok, kv_dtype=1, q_fp8=True, d=64) == -2
    # a value width of its own: 64 or 128, warp-level variants only
    assert _plan_rc(va, *ok, head_dim_v=64) == 0
    assert _plan_rc(va, *ok, d=64, head_dim_v=128) == 0
    assert _plan_rc(va, *ok, head_dim_v=96) == -2
    assert _plan_rc(va, *ok, head_dim_v=-1) == -1
    assert _plan_rc(va, *ok, head_dim_v=64, kernel=3) == -2
    assert _plan_rc(va, *ok, head_dim_v=64, kernel=4) == -2
    assert _plan_rc(va, *ok, head_dim_v=64, kv_dtype=1, q_fp8=True) == -2
    assert _plan_rc(va, *ok, head_dim_v=128) == 0            # = head_dim: the ordinary plan


def test_empty_batches_plan_to_nothing(va):
    plan = va.verify_attn_plan_host([0], [0], [], None, 4, 2, 64, 16, num_sms=152)
    assert plan.header()["n_items"] == 0 and plan.launches() == 0
    plan = va.verify_attn_plan_host([0, 3, 3], [0, 0, 0], [7, 0], None, 4, 2, 64, 16,
                                    num_sms=152)
    assert plan.header()["n_items"] == 0


def test_run_rejects_mismatched_plan_without_touching_the_device(va):
    lib = va.lib()
    plan = va.verify_attn_plan_host([0, 2], [0, 3], [5], None, 4, 2, 128, 16, num_sms=152)
    fake = ctypes.c_void_p(4096)  # never dereferenced: the checks fail first
    args = [fake] * 9
    args[7] = None  # mask
    args[8] = None
    rc = lib.verify_attn_run(*args, 8, 2, 128, 16, 0.0, 1.0, 1.0, fake, None, 10,
                             va._hp(plan.host), fake, 1 << 30, None)
    assert rc == -4  # num_qo_heads differs from the plan
    rc = lib.verify_attn_run(*args, 4, 2, 128, 16, 0.0, 1.0, 1.0, fake, None, 10,
                             None, fake, 1 << 30, None)
    assert rc == -1  # no plan
    rc = lib.verify_attn_run(*args, 4, 2, 128, 16, 0.0, 1.0, 1.0, fake, None, 10,
                             va._hp(plan.host), fake, 16, None)
    assert rc == -3  # workspace too small
    rc = lib.verify_attn_run(*args, 4, 2, 128, 16, 0.0, float("nan"), 1.0, fake, None, 10,
                             va._hp(plan.host), fake, 1 << 30, None)
    assert rc == -1  # non-finite scale
    rc = lib.verify_attn_run(*args, 4, 2, 128, 16, 0.0, 1.0, -2.0, fake, None, 10,
                             va._hp(plan.host), fake, 1 << 30, None)
    assert rc == -1  # negative scale
    margs = list(args)
    margs[7] = fake
    rc = lib.verify_attn_run(*margs, 4, 2, 128, 16, 0.0, 1.0, 1.0, fake, None, 10,
                             va._hp(plan.host), fake, 1 << 30, None)
    assert rc == -4  # mask given to a maskless plan


def test_append_validation_without_device(va):
    lib = va.lib()
    fake = ctypes.c_void_p(4096)
    P = [fake] * 8
    assert lib.paged_kv_append(*P, 1, 2, 96, 16, 10, 0, 5, None, None) == -2   # head_dim
    assert lib.paged_kv_append(*P, 1, 2, 128, 16, 10, 3, 5, None, None) == -2  # dtype
    assert lib.paged_kv_append(*P, 1, 2, 128, 16, 10, 0, 0, None, None) == 0   # nothing to do
    assert lib.paged_kv_append(*P, 1, 2, 128, 16, 10, 0, -1, None, None) == -1
    Q = list(P)
    Q[0] = ctypes.c_void_p(4097)  # misaligned
    assert lib.paged_kv_append(*Q, 1, 2, 128, 16, 10, 0, 5, None, None) == -1


def test_accept_validation_without_device(va):
    lib = va.lib()
    fake = ctypes.c_void_p(4096)
    n = ctypes.c_size_t(0)
    assert lib.verify_accept_workspace_size(17, 128256, 152, ctypes.byref(n)) == 0 and n.value > 0
    assert lib.verify_accept_workspace_size(17, 0, 152, ctypes.byref(n)) == -1
    P = [fake] * 3
    # fp8 logits are not served
    assert lib.verify_accept_greedy(fake, 1, 4, 100, 100, fake, 1, fake, fake, *P, None, None, 152,
                                    fake, 1 << 20, None) == -2
    # row stride below the vocabulary
    assert lib.verify_accept_greedy(fake, 0, 4, 100, 50, fake, 1, fake, fake, *P, None, None, 152,
                                    fake, 1 << 20, None) == -1
    # workspace too small
    assert lib.verify_accept_greedy(fake, 0, 4, 100, 100, fake, 1, fake, fake, *P, None, None, 152,
                                    fake, 8, None) == -3
    # nothing to do
    assert lib.verify_accept_greedy(fake, 0, 0, 100, 100, fake, 0, fake, fake, *P, None, None, 152,
                                    fake, 8, None) == 0


def test_latency_regime_aims_at_two_thirds_of_the_sms(va):
    """Few key tiles per SM (the Llama-3-8B tree verify: 8 KV heads, 4113
    keys): the split candidates aim at two thirds of the SMs, so the plan uses
    at most that many CTAs (plus the drafts' own items) and every chain holds
    one item; a plan forced to all SMs (target_ctas) uses more."""
    wl = synthetic.make_workload("llama3_8b_tree_verify", with_values=False)
    args = (wl.kv_indptr, wl.qo_indptr, wl.last_page_len, wl.mask_indptr, wl.h_q, wl.h_kv, wl.d,
            wl.page_size)
    auto = va.verify_attn_plan_host(*args, num_sms=152).header()
    full = va.verify_attn_plan_host(*args, num_sms=152, target_ctas=152).header()
    assert auto["n_ctas"] <= 2 * 152 // 3 + wl.h_kv
    assert full["n_ctas"] > auto["n_ctas"]
    # a large batch is not in that regime: every SM gets a chain
    wl = synthetic.make_workload("codellama34b_chain_verify", with_values=False)
    p = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, None, wl.h_q,
                                 wl.h_kv, wl.d, wl.page_size, num_sms=152).header()
    assert p["n_ctas"] == 152


def test_stream_cut_of_the_wide_tree(va):
    """The two-Q-tile plan of the fp8 wide tree cuts the units' key tiles
    into one equal run per CTA: 152 chains whose key tiles differ by at most
    one, items that tile each unit's kv range (checked by the cover test),
    and far fewer partial rows than cutting every unit seven ways."""
    wl = synthetic.make_workload("wide_tree_fp8_verify", with_values=False)
    plan = va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                    wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                    kv_dtype=wl.kv_dtype, num_sms=152)
    hd = plan.header()
    assert hd["kernel"] == 4 and hd["n_ctas"] == 152
    t = dict(masked=True, prefix=wl.prefix_lens, L=wl.qo_lens, G=wl.group, h_kv=wl.h_kv)
    _check_cover(va, t, plan)
    items = plan.items()
    tiles = []
    for c in range(152):
        i, n = c, 0
        while i >= 0:
            n += (int(items[i][5]) - int(items[i][4]) + 127) // 128
            i = int(items[i][7])
        tiles.append(n)
    assert max(tiles) - min(tiles) <= 1
    assert hd["part_rows"] < 64 * 256 * 4


def test_step_host_validation_without_device(va):
    """verify_attn_step_host checks its staging offsets, the arrays its host
    tables size, and the result buffer before any CUDA call."""
    lib = va.lib()
    stage = np.zeros(8192, np.uint8)
    i32 = stage.view(np.int32)
    # batch 1: 5 query tokens, 2 pages, last page 3 slots; 4 q / 2 kv heads, d 64
    i32[0:2] = [0, 5]          # qo_indptr at byte 0
    i32[64:66] = [0, 2]        # kv_indptr at byte 256
    i32[128] = 3               # last_page_len at byte 512
    i32[192:194] = [0, 1]      # kv_indices at byte 768
    base = dict(q=1024, k_new=3584, v_new=4864, kv_indptr=256, kv_indices=768,
                last_page_len=512, qo_indptr=0)
    fake = 1 << 20
    res = np.zeros(4096, np.uint8)
    plan = np.zeros(1 << 16, np.uint8)

    def call(offs, staging_bytes=stage.nbytes, result_bytes=res.nbytes):
        o = va.step_offsets(**offs)
        return lib.verify_attn_step_host(stage.ctypes.data, fake, staging_bytes, ctypes.byref(o),
                                         1, 4, 2, 64, 16, 0, 152, None, plan.ctypes.data,
                                         plan.nbytes, fake, 1 << 20, None, fake, fake, 8, 0.0,
                                         1.0, 1.0, fake, fake + 4096, res.ctypes.data,
                                         result_bytes, None, 1, None)

    assert call(dict(base, kv_indices=8190)) == -1               # indices past the buffer
    assert call(dict(base, v_new=7000)) == -1                    # v_new needs 1280 bytes
    assert call(dict(base), staging_bytes=4096) == -1            # arrays past staging_bytes
    assert call(dict(base, kv_indptr=258)) == -1                 # misaligned table
    assert call(dict(base, qo_indptr=-256)) == -1                # negative offset
    assert call(dict(base), result_bytes=2559) == -1             # out + LSE need 2560 + 80
    assert call(dict(base, mask=6144)) == -1                     # mask without mask_indptr
    i32[1] = -5
    assert call(dict(base)) == -1                                # negative total_qo

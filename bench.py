"""Benchmark of paged-KV GQA verify attention on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-configs] [--no-e2e]

One step is one pass of the hot path over one batch: the paged append of
the batch's draft K/V into the cache, then verify attention (split kernel +
LSE merge), in one verify_attn_append_run call.  The plan (host) is built once before the timed region and
reused, as a serving step shares it across layers; the end-to-end number
re-plans every step.  Inputs are synthetic (seeded, shaped like the
workload) and resident in HBM when the timed region starts.  L2 (129 MB) is
defeated by rotating over copies of the KV pool totalling >= 4x L2.

Prints ONE JSON line.  The default workload is the Llama-3-8B-shaped tree
verify (batch 1, 32 q / 8 kv heads, d 128, 4096-token prefix, 17-node tree).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

HEADLINE = "llama3_8b_tree_verify"
METRIC = "verify-attn tokens/s and achieved HBM GB/s (% of GB300 peak) per config"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GRAPH_STEPS = 128


# ---------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(wl):
    """Algorithmic bytes and FLOPs of one verify-attention call.
    Bytes: K and V of every (request, KV head, kv token) read once, Q read
    once, out and LSE written once, page-table, qo_indptr and mask bytes.
    FLOPs: 4 * d per visible (query row, key) pair per query head."""
    es = wl.kv_elem_bytes
    kv = int(wl.kv_lens.sum()) * wl.h_kv * wl.d * es * 2
    q = wl.total_qo * wl.h_q * wl.d * 2
    out = q
    lse = wl.total_qo * wl.h_q * 4
    idx = 4 * (2 * (wl.batch + 1) + wl.batch + len(wl.kv_indices))
    mask = 0
    if wl.mask is not None:
        mask = int(math.ceil(int(wl.mask_indptr[-1]) / 8)) + 4 * (wl.batch + 1)
    visible = 0
    for b in range(wl.batch):
        L = int(wl.qo_lens[b])
        pre = int(wl.prefix_lens[b])
        if wl.mask_dense is not None:
            draft = int(wl.mask_dense[b].sum())
        else:
            draft = L * (L + 1) // 2
        visible += L * pre + draft
    flops = 4 * wl.d * visible * wl.h_q
    return dict(kv_bytes=kv, read_bytes=kv + q + idx + mask,
                total_bytes=kv + q + out + lse + idx + mask, flops=flops, tokens=wl.total_qo)


def kernel_source_sha(kernel=0):
    """sha256 prefix of the sources of the split-kernel variant (1, 2: warp
    level; 3, 4: tcgen05)."""
    h = hashlib.sha256()
    files = ("k_partial_tc.cu", "va_tc.cuh") if kernel in (3, 4) else ("k_partial_mma.cu",)
    for f in files + ("va_device.cuh", "va_kernels.h"):
        with open(os.path.join(ROOT, "speculative_decoding_verify_gqa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel=0):
    """DRAM bytes per launch of the split kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic_per_launch.md")
    sha = kernel_source_sha(kernel)
    try:
        for line in open(path):
            parts = line.strip().strip("|").split("|")
            parts = [p.strip() for p in parts]
            if len(parts) >= 4 and parts[0] == workload and parts[2] == sha:
                return float(parts[1])
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self, background=None, seconds=0.5):
        """Start sampling; `background` (one short unit of GPU work) is
        replayed meanwhile for about `seconds`, so the first samples are
        taken under load."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        t0 = time.perf_counter()
        if background is None:
            time.sleep(seconds)
            return
        import torch
        while time.perf_counter() - t0 < seconds:
            background()
            torch.cuda.synchronize()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            n += 1
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def make_event(torch):
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


# ---------------------------------------------------------------- our arm

class Bench:
    def __init__(self, name, device, seed=0, plan_opts=None, early_reads=True):
        import torch
        import speculative_decoding_verify_gqa_gb300 as va
        self.torch, self.va = torch, va
        self.name = name
        self.dev = device
        self.plan_opts = dict(plan_opts or {})
        # q and the tables are written once, before any timed step, and no
        # kernel of a step writes them or a prefix slot: the early-reads
        # promise of va_run_options_t holds
        self.early_reads = early_reads
        wl = synthetic.make_workload(name, seed=seed)
        self.wl = wl
        fp8 = wl.kv_dtype == synthetic.FP8
        self.kvd = torch.float8_e4m3fn if fp8 else torch.bfloat16
        raw = np.uint8 if fp8 else np.int16

        def dt(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device)

        def dkv(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(raw)).to(device).view(self.kvd)

        self.q = dt(wl.q.view(np.int16)).view(torch.bfloat16)
        kn, vn = wl.new_tokens()
        self.k_new, self.v_new = dkv(kn), dkv(vn)
        self.kv_indptr, self.kv_indices = dt(wl.kv_indptr), dt(wl.kv_indices)
        self.last_page_len, self.qo_indptr = dt(wl.last_page_len), dt(wl.qo_indptr)
        self.mask = None if wl.mask is None else dt(wl.mask)
        self.mask_indptr = None if wl.mask_indptr is None else dt(wl.mask_indptr)
        shape = (wl.num_pages, wl.h_kv, wl.page_size, wl.d)
        k0 = torch.full(shape, 0xFF, dtype=torch.uint8, device=device).view(self.kvd)
        v0 = torch.full(shape, 0xFF, dtype=torch.uint8, device=device).view(self.kvd)
        if not fp8:
            k0 = torch.full(shape, -1, dtype=torch.int16, device=device).view(self.kvd)
            v0 = torch.full(shape, -1, dtype=torch.int16, device=device).view(self.kvd)
        k_tok, v_tok = dkv(wl.k_tok), dkv(wl.v_tok)
        va.paged_kv_append(k_tok, v_tok, dt(wl.tok_indptr.astype(np.int32)), self.kv_indptr,
                           self.kv_indices, self.last_page_len, k0, v0)
        del k_tok, v_tok
        pool_bytes = 2 * k0.numel() * k0.element_size()
        self.n_copies = int(min(64, max(2, math.ceil(4 * L2_BYTES / pool_bytes))))
        self.pool_bytes = pool_bytes
        self.pools = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(self.n_copies - 1)]
        self.plan = va.verify_attn_plan(wl.kv_indptr, wl.qo_indptr, wl.last_page_len,
                                        wl.mask_indptr, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                                        kv_dtype=wl.kv_dtype, device=device, **self.plan_opts)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=device)
        self.launches_per_step = 1 + self.plan.launches()   # append, split, merge
        torch.cuda.synchronize()

    # one step on pool copy i: the drafts appended and attended in one call
    # (verify_attn_append_run); verify_only: the attention call alone;
    # ev: the three kernels as separate calls with 4 events around them
    def step(self, i, ev=None, verify_only=False):
        va, wl = self.va, self.wl
        kc, vc = self.pools[i % self.n_copies]
        if not verify_only and not ev:
            va.verify_attn_append_run(self.k_new, self.v_new, self.q, kc, vc, self.kv_indptr,
                                      self.kv_indices, self.last_page_len, self.qo_indptr,
                                      self.mask, self.mask_indptr, self.plan,
                                      sm_scale=wl.sm_scale, k_scale=wl.k_scale,
                                      v_scale=wl.v_scale, out=self.out, lse=self.lse,
                                      early_reads=self.early_reads)
            return
        if ev:
            ev[0].record()
        if not verify_only:
            va.paged_kv_append(self.k_new, self.v_new, self.qo_indptr, self.kv_indptr,
                               self.kv_indices, self.last_page_len, kc, vc)
        if ev:
            ev[1].record()
        va.verify_attn_partial(self.q, kc, vc, self.kv_indptr, self.kv_indices,
                               self.last_page_len, self.qo_indptr, self.mask, self.mask_indptr,
                               self.plan, sm_scale=wl.sm_scale, k_scale=wl.k_scale,
                               v_scale=wl.v_scale, out=self.out, lse=self.lse,
                               early_reads=self.early_reads)
        if ev:
            ev[2].record()
        va.verify_attn_merge(self.qo_indptr, self.plan, self.out, self.lse)
        if ev:
            ev[3].record()

    def capture(self, n, start=0, events=None, verify_only=False, rotate=True):
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(2):
                self.step(start + i if rotate else 0, verify_only=verify_only)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                self.step(start + i if rotate else 0, events[i] if events else None,
                          verify_only=verify_only)
        return g

    def time_steps(self, k, warmup, sampler=None, barrier=None, verify_only=False, rotate=True):
        """Exactly k steps, timed with CUDA events around replays of captured
        graphs (k // GRAPH_STEPS replays of a GRAPH_STEPS-step graph and one
        of a k % GRAPH_STEPS-step graph).  The warm-up replays THOSE graphs
        (each at least once, so no graph upload or first launch lands in the
        timed region) for at least `warmup` steps, then keeps the GPU busy
        with them for about half a second while the clock sampler starts, so
        its samples see the part under load."""
        torch = self.torch
        n_full, rem = divmod(k, GRAPH_STEPS)
        full = self.capture(GRAPH_STEPS, verify_only=verify_only, rotate=rotate) if n_full else None
        part = self.capture(rem, verify_only=verify_only, rotate=rotate) if rem else None
        graphs = [(g, n) for g, n in ((full, GRAPH_STEPS), (part, rem)) if g is not None]
        done = 0
        for g, n in graphs:
            g.replay()
            done += n
        small, n_small = graphs[-1]
        while done < warmup:
            small.replay()
            done += n_small
        torch.cuda.synchronize()
        if barrier:
            barrier()
        if sampler:
            sampler.start(background=lambda: small.replay())
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n_full):
            full.replay()
        if part is not None:
            part.replay()
        e1.record()
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        if barrier:
            barrier()
        return e0.elapsed_time(e1) / k, clocks

    def kernel_times(self, n=64):
        """Average duration (ms) of each kernel of the step: CUDA events
        around a captured graph of n back-to-back launches of that kernel
        alone (its own calls: verify_attn_partial with the step's
        early-reads mode, verify_attn_merge, paged_kv_append), divided by n,
        on pool copies rotated as in the step; median of 5 replays."""
        torch, va, wl = self.torch, self.va, self.wl

        def one(kind, i):
            kc, vc = self.pools[i % self.n_copies]
            if kind == "append":
                va.paged_kv_append(self.k_new, self.v_new, self.qo_indptr, self.kv_indptr,
                                   self.kv_indices, self.last_page_len, kc, vc)
            elif kind == "partial":
                va.verify_attn_partial(self.q, kc, vc, self.kv_indptr, self.kv_indices,
                                       self.last_page_len, self.qo_indptr, self.mask,
                                       self.mask_indptr, self.plan, sm_scale=wl.sm_scale,
                                       k_scale=wl.k_scale, v_scale=wl.v_scale, out=self.out,
                                       lse=self.lse, early_reads=self.early_reads)
            else:
                va.verify_attn_merge(self.qo_indptr, self.plan, self.out, self.lse)

        res = {}
        for kind in ("append", "partial", "merge"):
            if kind == "merge" and self.plan.header()["n_merge"] == 0:
                res["merge_ms"] = 0.0
                continue
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                for i in range(2):
                    one(kind, i)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(n):
                    one(kind, i)
            g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(5):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) / n)
            res[kind + "_ms"] = statistics.median(ts)
        return res

    def e2e(self, steps):
        """End to end through the public API: one verify_attn_step_host call
        per step -- the step's inputs (q, the drafts' K/V, the index tables,
        the mask) copied in from one pinned host buffer, the plan made on the
        host from those tables, append and attention, out and LSE copied back
        into one pinned host buffer, the stream synchronised.  Each array sits
        at a 256-byte offset, the device side carved the same way; out and LSE
        share one device buffer and come back in one copy."""
        torch, va, wl = self.torch, self.va, self.wl

        src = dict(q=self.q, k_new=self.k_new, v_new=self.v_new, kv_indptr=self.kv_indptr,
                   kv_indices=self.kv_indices, last_page_len=self.last_page_len,
                   qo_indptr=self.qo_indptr)
        if self.mask is not None:
            src["mask"], src["mask_indptr"] = self.mask, self.mask_indptr
        offs, total = {}, 0
        for k, t in src.items():
            offs[k] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
        stage_d = torch.empty(total, dtype=torch.uint8, device=self.dev)
        for k, t in src.items():
            n = t.numel() * t.element_size()
            stage_h[offs[k]:offs[k] + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
        n_out = self.out.numel() * self.out.element_size()
        n_lse = self.lse.numel() * self.lse.element_size()
        lse_off = (n_out + 255) // 256 * 256
        res_d = torch.empty(lse_off + n_lse, dtype=torch.uint8, device=self.dev)
        res_h = torch.empty(lse_off + n_lse, dtype=torch.uint8).pin_memory()
        out_d = res_d[:n_out].view(self.out.dtype).view(self.out.shape)
        lse_d = res_d[lse_off:].view(self.lse.dtype).view(self.lse.shape)
        h2d, d2h = int(total), int(lse_off + n_lse)
        ws = self.plan.workspace
        n_sms = self.plan.header()["num_sms"]
        plan_buf = torch.zeros(self.plan.host.nbytes, dtype=torch.uint8).pin_memory()
        kc0, vc0 = self.pools[0]
        # the inputs arrive by a host copy on the stream (not a kernel): the
        # early-reads promise holds
        step = va.HostStep(stage_h, stage_d, offs, wl.batch, wl.h_q, wl.h_kv, wl.d, wl.page_size,
                           kc0, vc0, out_d, lse_d, res_h, ws, plan_buf, kv_dtype=wl.kv_dtype,
                           num_sms=n_sms, sm_scale=wl.sm_scale, k_scale=wl.k_scale,
                           v_scale=wl.v_scale, early_reads=True, synchronize=True,
                           **self.plan_opts)

        def one(i):
            kc, vc = self.pools[i % self.n_copies]
            step(kc, vc)

        for i in range(5):
            one(i)
        t0 = time.perf_counter()
        for i in range(steps):
            one(i)
        dt_s = (time.perf_counter() - t0) / steps
        return dict(value=wl.total_qo / dt_s, unit="tokens/s", h2d_bytes_per_step=h2d,
                    d2h_bytes_per_step=d2h, ms_per_step=dt_s * 1e3,
                    api="verify_attn_step_host (one call per step, host buffers, "
                        "arguments marshalled once by the binding's HostStep)")

    def plan_us(self, n=50):
        va, wl = self.va, self.wl
        t0 = time.perf_counter()
        for _ in range(n):
            va.verify_attn_plan_host(wl.kv_indptr, wl.qo_indptr, wl.last_page_len, wl.mask_indptr,
                                     wl.h_q, wl.h_kv, wl.d, wl.page_size, kv_dtype=wl.kv_dtype,
                                     num_sms=self.plan.header()["num_sms"], **self.plan_opts)
        return (time.perf_counter() - t0) / n * 1e6


KERNEL_NAMES = {1: "verify_partial_mma_kernel<4 warps>", 2: "verify_partial_mma_kernel<8 warps>",
                3: "verify_partial_tc_kernel<one Q tile>", 4: "verify_partial_tc_kernel<two Q tiles>"}


# dense e4m3 over dense bf16 tensor throughput, from the nominal rates
# (4.5 vs 2.25 PFLOP/s per GPU)
E4M3_OVER_BF16 = 2.0


def roofline_for(wl, kt, peaks, peak_kind, kernel=0, e4m3=False):
    """Roofline of the split-attention kernel: algorithmic bytes (K + V + Q
    read once, out + LSE written once, tables and mask) or FLOPs per launch
    over its CUDA-event duration, against the measured copy bandwidth or
    tensor throughput: measured bf16, or for e4m3 MMAs (plan option q_fp8)
    measured bf16 times the nominal e4m3 / bf16 ratio.  The bound is the one
    the workload's arithmetic intensity selects."""
    alg = algorithmic(wl)
    t = kt["partial_ms"] * 1e-3
    hbm = alg["total_bytes"] / t / 1e9
    tfl = alg["flops"] / t / 1e12
    rows_per_kv_head = int((wl.group * wl.qo_lens).max())
    tpeak = peaks["bf16_tflops"] * (E4M3_OVER_BF16 if e4m3 else 1.0)
    ridge = tpeak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor_bound = alg["flops"] / alg["total_bytes"] > ridge
    if tensor_bound:
        rf = {"bound": "tensor", "achieved": round(tfl, 2), "peak": round(tpeak, 1),
              "unit": "TFLOP/s", "frac": round(tfl / tpeak, 4)}
    else:
        rf = {"bound": "hbm", "achieved": round(hbm, 1), "peak": peaks["hbm_gbs"],
              "unit": "GB/s", "frac": round(hbm / peaks["hbm_gbs"], 4)}
    rf.update({"kernel": KERNEL_NAMES.get(kernel, "verify_partial") + ("_e4m3" if e4m3 else ""),
               "peak_source": ("MEASURED_PEAKS.json (of %s)" % peak_kind
                               + (", bf16 x %.0f nominal e4m3 ratio" % E4M3_OVER_BF16 if e4m3 else "")),
               "algorithmic_bytes_per_launch": alg["total_bytes"],
               "algorithmic_flops_per_launch": alg["flops"],
               "kernel_ms": round(kt["partial_ms"], 5),
               "hbm_gbs": round(hbm, 1), "hbm_frac": round(hbm / peaks["hbm_gbs"], 4),
               "tflops": round(tfl, 2), "tensor_frac": round(tfl / tpeak, 4),
               "rows_per_kv_head_max": rows_per_kv_head})
    return rf


def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def reduce_max(x, world):
    """Max over ranks of a float (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier_fn(world):
    if world == 1:
        return None
    import torch.distributed as dist
    return dist.barrier


def cpu_baseline(wl, seconds=10.0, nthreads=None, q_fp8=False):
    """The oracle as it stands, on the host cores, on the workload's full call
    (every row), repeated for about `seconds`; q_fp8: with e4m3 queries."""
    import oracle
    nthreads = nthreads or oracle.default_threads()
    caches = oracle.build_cache(wl)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.verify_attn_workload(wl, caches=caches, nthreads=nthreads, q_fp8=q_fp8)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or (n >= 1 and el * (n + 1) / n > 3 * seconds):
            break
    per = el / n
    return {"value": wl.total_qo / per, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": "%d full calls of the workload (%d tokens x %d heads each), %.2f s per call"
                      % (n, wl.total_qo, wl.h_q, per)}


def workload_config(wl, bench=None):
    cfg = {"workload": wl.name, "batch": wl.batch, "num_qo_heads": wl.h_q,
           "num_kv_heads": wl.h_kv, "head_dim": wl.d, "page_size": wl.page_size,
           "kv_dtype": wl.kv_dtype, "mask": wl.mask_kind,
           "prefix_tokens": int(wl.prefix_lens.sum()), "draft_tokens": wl.total_qo,
           "kv_tokens": int(wl.kv_lens.sum())}
    if bench is not None and bench.plan_opts.get("q_fp8"):
        cfg["mma"] = "e4m3 queries (per-row amax scale) and e4m3 P: kind::f8f6f4"
    if bench is not None:
        cfg["l2"] = ("inputs rotate over %d KV-pool copies of %.1f MB (%.0f MB total vs 129 MB L2)"
                     % (bench.n_copies, bench.pool_bytes / 1e6,
                        bench.n_copies * bench.pool_bytes / 1e6))
        cfg["timing"] = "CUDA-graph replays of %d-step graphs, CUDA events on the launch stream" % GRAPH_STEPS
    return cfg


def timing_block(bench, peaks, peak_kind, steps, warmup, sampler=None, barrier=None):
    """Times one workload: the step (append + attention), the attention call
    alone (append excluded: verify-attn tokens/s), per-kernel CUDA-event
    durations, and the split kernel's roofline."""
    wl = bench.wl
    ms, clocks = bench.time_steps(steps, warmup, sampler=sampler, barrier=barrier)
    ms_v, _ = bench.time_steps(steps, warmup, verify_only=True)
    kt = bench.kernel_times()
    kernel = bench.plan.header()["kernel"]
    e4m3 = bool(bench.plan_opts.get("q_fp8"))
    rf = roofline_for(wl, kt, peaks, peak_kind, kernel, e4m3=e4m3)
    rf["traffic"] = profiled_traffic(wl.name + ("+q_fp8" if e4m3 else ""), kernel)
    alg = algorithmic(wl)
    return ms, clocks, {
        "verify_only": {"tokens_per_s": round(wl.total_qo / (ms_v * 1e-3), 1),
                        "us_per_call": round(ms_v * 1e3, 3),
                        "hbm_gbs": round(alg["total_bytes"] / (ms_v * 1e-3) / 1e9, 1),
                        "note": "split attention + merge per call, paged append excluded"},
        "kernel_us": {k.replace("_ms", ""): round(v * 1e3, 3) for k, v in kt.items()},
        "roofline": rf,
    }


def accept_timing(wl, dev, vocab=128256, n=64):
    """The step after verification on this workload's drafts: greedy
    acceptance over [total_qo, vocab] bf16 target logits (N(0, 1), the
    Llama-3 vocabulary size), trees from the workload's parents (chains when
    it has none).  Bytes: the logits rows read once, plus the small tables."""
    import torch
    import speculative_decoding_verify_gqa_gb300 as va
    gen = torch.Generator().manual_seed(3)
    total = wl.total_qo
    logits = torch.randn((total, vocab), generator=gen).to(torch.bfloat16).to(dev)
    parents = []
    for b in range(wl.batch):
        L = int(wl.qo_lens[b])
        par = wl.parents[b] if wl.parents is not None and wl.parents[b] is not None else \
            [i - 1 for i in range(L)]
        parents += list(par)
    parents = torch.tensor(parents, dtype=torch.int32, device=dev)
    toks = torch.randint(0, vocab, (total,), generator=gen, dtype=torch.int32).to(dev)
    qo = torch.from_numpy(wl.qo_indptr).to(dev)
    va.verify_accept_greedy(logits, qo, toks, parents)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        va.verify_accept_greedy(logits, qo, toks, parents)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    ws = torch.empty(1 << 22, dtype=torch.uint8, device=dev)
    with torch.cuda.graph(g):
        for _ in range(n):
            va.verify_accept_greedy(logits, qo, toks, parents, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / n)
    ms = statistics.median(ts)
    nbytes = total * vocab * 2 + 4 * (3 * total + 2 * (wl.batch + 1))
    return {"us_per_call": round(ms * 1e3, 3), "vocab": vocab, "rows": total,
            "bytes_per_call": nbytes, "hbm_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
            "note": "greedy acceptance of the drafts (argmax kernel + tree walk), logits bf16, "
                    "L2 not flushed between calls"}


def run_ours(args):
    import torch
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    plan_opts = {k: v for k, v in (("kernel", args.kernel), ("target_ctas", args.target_ctas),
                                   ("min_chunk", args.min_chunk), ("q_fp8", args.q_fp8)) if v}
    bench = Bench(args.workload, dev, seed=0, plan_opts=plan_opts)
    wl = bench.wl
    sampler = ClockSampler(local)
    ms, clocks, extra = timing_block(bench, peaks, peak_kind, args.steps, args.warmup,
                                     sampler=sampler, barrier=barrier_fn(world))
    ms_max = reduce_max(ms, world)
    value = world * wl.total_qo / (ms_max * 1e-3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 q/out, %s kv, fp32 accumulate" % wl.kv_dtype, "data": "synthetic",
        "config": workload_config(wl, bench),
        "gpu_launches": args.steps * bench.launches_per_step,
        "roofline": extra["roofline"], "clocks": clocks,
        "verify_only": extra["verify_only"], "kernel_us": extra["kernel_us"],
        "plan_host_us": round(bench.plan_us(), 2),
    }
    # L2-warm: the same pool copy every step (its 21 MB stay in the 129 MB L2)
    ms_w, _ = bench.time_steps(args.steps, args.warmup, rotate=False)
    ms_wv, _ = bench.time_steps(args.steps, args.warmup, rotate=False, verify_only=True)
    line["l2_warm"] = {"ms_per_step": round(ms_w, 6),
                       "tokens_per_s": round(wl.total_qo / (ms_w * 1e-3), 1),
                       "verify_only_us_per_call": round(ms_wv * 1e3, 3),
                       "note": "every step on one KV-pool copy, which stays resident in L2"}
    line["accept_greedy"] = accept_timing(wl, dev)
    if not args.no_e2e:
        line["e2e"] = bench.e2e(args.e2e_steps)
        line["e2e"]["value"] = round(world * line["e2e"]["value"], 1)
    del bench
    torch.cuda.empty_cache()
    if not args.no_configs and world == 1:
        others = {}
        runs = []
        for name in synthetic.WORKLOAD_ORDER:
            if name != args.workload or plan_opts:
                runs.append((name, {}))
            # fp8 caches once more with e4m3 queries: both MMAs on e4m3 operands
            if synthetic.WORKLOADS[name]["kv_dtype"] == synthetic.FP8:
                runs.append((name, {"q_fp8": True}))
        for name, opts in runs:
            b = Bench(name, dev, seed=0, plan_opts=opts)
            steps = 256 if name != "tiny_verify" else 1024
            ms_o, _, ex = timing_block(b, peaks, peak_kind, steps, 16)
            entry = {"tokens_per_s": round(b.wl.total_qo / (ms_o * 1e-3), 1),
                     "ms_per_step": round(ms_o, 6)}
            entry.update(ex)
            entry["config"] = workload_config(b.wl, b)
            others[name + ("+q_fp8" if opts else "")] = entry
            del b
            torch.cuda.empty_cache()
        if rank == 0 and not args.no_cpu_baseline:
            for key, entry in others.items():
                name, _, variant = key.partition("+")
                entry["cpu_baseline"] = cpu_baseline(synthetic.make_workload(name),
                                                     seconds=args.cpu_seconds_per_config,
                                                     q_fp8=variant == "q_fp8")
        line["configs"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle (fp64 C on the host cores) as the reference implementation:
    rank 0 alone; each step is one bounded sample (a seeded subset of the
    workload's rows, or the whole call when it fits) of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    wl = synthetic.make_workload(args.workload)
    nthreads = oracle.default_threads()
    caches = oracle.build_cache(wl)
    total_rows = wl.total_qo * wl.h_q
    t0 = time.perf_counter()
    oracle.verify_attn_workload(wl, caches=caches, nthreads=nthreads)
    t_full = time.perf_counter() - t0
    budget = 120.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, budget / max(t_full, 1e-9))
    n_rows = max(wl.h_q, int(total_rows * frac))
    rows = None if n_rows >= total_rows else synthetic.sample_rows(wl, n_rows)
    if rows is not None:
        n_rows = len(rows)
    for _ in range(args.warmup):
        oracle.verify_attn_workload(wl, rows=rows, caches=caches, nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify_attn_workload(wl, rows=rows, caches=caches, nthreads=nthreads)
    per = (time.perf_counter() - t0) / args.steps
    tokens = n_rows / wl.h_q
    value = tokens / per
    sample = ("%s per step: %d of %d (token, head) rows (%.1f tokens' worth), fp64, %d threads"
              % ("whole call" if rows is None else "seeded row sample", n_rows, total_rows,
                 tokens, nthreads))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": nthreads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=synthetic.WORKLOAD_ORDER)
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' summary")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-seconds-per-config", type=float, default=3.0,
                    help="oracle time per other workload (at least one full call)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--kernel", type=int, default=0,
                    help="force a split-kernel variant (1: mma 64 rows, 2: mma 128 rows, "
                         "3: tcgen05); 0 = the planner's choice")
    ap.add_argument("--target-ctas", type=int, default=0, help="planner option (0 = auto)")
    ap.add_argument("--min-chunk", type=int, default=0, help="planner option (0 = auto)")
    ap.add_argument("--q-fp8", action="store_true",
                    help="planner option for fp8 caches: e4m3 queries, kind::f8f6f4 MMAs")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

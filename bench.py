"""Benchmark of the paged-KV attention path on one GB300 (or N replicas).

Headline workload: batch decode, batch 64, one query row per request, kv_len
uniform in [512, 8192], 32 q / 8 kv heads, head_dim 128, bf16, page 16 (pages
scattered by a seeded permutation), window -1, with LSE. A step is one
run() of the planned batch (the decode kernel and the split-KV merge); the
plan is made once, as a graph-replayed serving step would. ``value`` is KV
GB/s (algorithmic bytes: each live K/V row once, plus q, o, lse and the page
indices) with every input resident in HBM; ``e2e`` repeats the step through
the public API with host buffers: plan + host-to-device copy of q and the
page table + run + device-to-host copy of o and lse, every step.

The other workloads (prefill, verify, long-context split-KV, the 64x256
paged prefill) are timed the same way and reported under ``workloads``.

``--impl reference`` times the CPU oracle on the host cores (the same oracle
source built with fp32 accumulation and OpenMP, on every core of the process's
affinity), one measured pass over the batch per step, and prints the same
line with ``"impl": "reference"``.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "prefill/verify TFLOPS and decode KV GB/s on 1 GB300, % of tensor/HBM roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
REF_STEP_S = 2.0  # longest pass of the CPU reference arm over the batch


# ------------------------------------------------------------------ accounting
def valid_counts(lq, lk, causal, wl):
    """Valid keys per query row under the bottom-right causal mask and the
    left-only window (closed form of the mask, for FLOP accounting)."""
    i = np.arange(lq, dtype=np.int64)
    hi = np.minimum(lk - 1, i + lk - lq) if causal else np.full(lq, lk - 1)
    lo = np.maximum(0, lk - lq + i - wl) if wl >= 0 else np.zeros(lq, np.int64)
    return np.maximum(0, hi - lo + 1)


def accounting(pb, causal, wl):
    """(masked FLOPs, algorithmic bytes) of one run over the batch."""
    d, Hq, Hk = pb.head_dim, pb.num_qo_heads, pb.num_kv_heads
    es = 2
    flops = 0
    kv_rows = 0
    pages = 0
    masks = pb.extra.get("masks")  # custom (tree) masks, ANDed in
    for b, (lq, lk) in enumerate(zip(pb.q_lens, pb.kv_lens)):
        if lq == 0 or lk == 0:
            continue
        cnt = valid_counts(lq, lk, causal, wl)
        if masks is not None:
            i = np.arange(lq)[:, None]
            j = np.arange(lk)[None, :]
            std = np.ones((lq, lk), bool)
            if causal:
                std &= j <= i + lk - lq
            if wl >= 0:
                std &= j + lq + wl >= lk + i
            cnt = (std & np.asarray(masks[b], bool)).sum(axis=1)
        flops += 4 * d * Hq * int(cnt.sum())
        # distinct live keys: union of the rows' ranges [lo_i, hi_i]
        i = np.arange(lq)
        hi = np.minimum(lk - 1, i + lk - lq) if causal else np.full(lq, lk - 1)
        lo = np.maximum(0, lk - lq + i - wl) if wl >= 0 else np.zeros(lq, np.int64)
        live = np.zeros(lk, bool)
        for r0, r1 in zip(lo, hi):
            if r1 >= r0:
                live[r0:r1 + 1] = True
        n_live = int(live.sum())
        kv_rows += n_live
        pages += len({j // pb.page_size for j in np.nonzero(live)[0]}) if n_live < lk else \
            (lk + pb.page_size - 1) // pb.page_size
    T = sum(pb.q_lens)
    byts = kv_rows * Hk * d * 2 * es + T * Hq * d * es * 2 + T * Hq * 4 + 4 * pages
    return flops, byts


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            pk = json.load(open(path))
            hbm = pk.get("hbm_gbs") or pk.get("hbm_GBs") or pk.get("hbm")
            bf = pk.get("bf16_tflops")
            bfs = pk.get("bf16_tflops_sustained") or bf
            if hbm and bf:
                return float(hbm), float(bf), float(bfs), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "fi_clocks_%d_%d.csv" % (os.getpid(), index))

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm
class Runner:
    """One planned workload resident on the device."""

    def __init__(self, pb, causal, wl, mode, dev, force_kv_chunks=0, ws=None, graph=False):
        import paged_kv_attention_13_gb300 as fi
        self.fi = fi
        self.pb, self.causal, self.wl, self.mode = pb, causal, wl, mode
        self.dev = dev
        self.q = pb.q.to(dev)
        if mode == "ragged":  # contiguous K/V rows (a page-size-1, unpermuted cache)
            rows = pb.k_cache.shape[0]
            self.k = pb.k_cache.reshape(rows, pb.num_kv_heads, pb.head_dim).to(dev)
            self.v = pb.v_cache.reshape(rows, pb.num_kv_heads, pb.head_dim).to(dev)
        else:
            self.k = pb.k_cache.to(dev)
            self.v = pb.v_cache.to(dev)
        self.idx = pb.kv_indices.to(dev)
        self.mask = pb.extra["mask"].to(dev) if mode == "masked" else None
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:2], dtype=torch.float32, device=dev)
        self.ws = ws if ws is not None else torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        T = int(self.q.shape[0])
        self.plan = fi.Plan(self.ws, enable_graph_capture=graph, max_batch=len(pb.kv_lens),
                            max_total_rows=T) if graph else fi.Plan(self.ws)
        self.force = force_kv_chunks
        self.do_plan()
        self.flops, self.bytes = accounting(pb, causal or mode == "verify", wl)
        self.graph = None
        if graph:  # planned once, captured once, replayed every step
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                for _ in range(2):
                    self._launch()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._launch()
            torch.cuda.synchronize()
            self.graph = g

    def do_plan(self):
        pb = self.pb
        dt = workloads.TORCH_DTYPE[pb.dtype]
        if self.mode == "masked":
            self.plan.plan_masked(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, pb.page_size,
                                  pb.num_qo_heads, pb.num_kv_heads, pb.head_dim,
                                  pb.extra["mask_indptr"], causal=self.causal,
                                  window_left=self.wl, dtype=dt, force_kv_chunks=self.force)
        elif self.mode == "ragged":
            self.plan.plan_ragged(pb.qo_indptr, pb.kv_indptr, pb.num_qo_heads, pb.num_kv_heads,
                                  pb.head_dim, causal=self.causal, window_left=self.wl, dtype=dt,
                                  force_kv_chunks=self.force)
        elif self.mode == "prefill":
            self.plan.plan(pb.qo_indptr, pb.kv_indptr, pb.last_page_len, pb.page_size,
                           pb.num_qo_heads, pb.num_kv_heads, pb.head_dim, causal=self.causal,
                           window_left=self.wl, dtype=dt, force_kv_chunks=self.force)
        else:
            qlpr = 1 if self.mode == "decode" else pb.extra["q_len_per_req"]
            self.plan.plan(None, pb.kv_indptr, pb.last_page_len, pb.page_size, pb.num_qo_heads,
                           pb.num_kv_heads, pb.head_dim, causal=self.causal, window_left=self.wl,
                           dtype=dt, q_len_per_req=qlpr, force_kv_chunks=self.force)
        self.info = self.plan.info()

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self._launch()

    def _launch(self):
        if self.mode == "masked":
            self.fi.fi_batch_prefill_paged_masked(self.plan, self.q, self.k, self.v, self.idx,
                                                  self.mask, self.pb.sm_scale, out=self.out,
                                                  lse=self.lse)
            return
        if self.mode == "ragged":
            self.fi.fi_batch_prefill_ragged(self.plan, self.q, self.k, self.v, self.pb.sm_scale,
                                            out=self.out, lse=self.lse)
            return
        f = self.fi.fi_batch_prefill_paged if self.mode == "prefill" else self.fi.fi_batch_decode_paged
        f(self.plan, self.q, self.k, self.v, self.idx, self.pb.sm_scale, out=self.out, lse=self.lse)

    def launches_per_step(self):
        return 1 + (1 if self.info["num_merge_rows"] > 0 else 0)

    def time(self, steps, warmup, flush=False):
        """Mean and median device time of one run (CUDA events on the
        launching stream); with ``flush`` a 256 MB buffer is rewritten before
        every run so the inputs start out of L2."""
        buf = torch.empty(256 << 20, dtype=torch.uint8, device=self.dev) if flush else None
        for _ in range(warmup):
            self.run()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        st = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            if buf is not None:
                buf.fill_(i & 0xFF)
            st[i].record(s)
            self.run()
            en[i].record(s)
        torch.cuda.synchronize()
        if self.plan.device_error():
            raise RuntimeError("a kernel gave up an expired bounded wait: timings are not valid")
        ms = [a.elapsed_time(b) for a, b in zip(st, en)]
        return float(np.mean(ms)), float(np.median(ms))

    def time_e2e(self, steps, warmup):
        """End to end through the public API, every step: fi_plan (its metadata
        upload included), one host-to-device copy of the step's inputs (q and
        the page table, packed in one pinned host buffer), run(), one
        device-to-host copy of the result (o and lse, packed in one device
        buffer) into pinned host memory, and the wait for that result. The KV
        cache stays resident, as in a serving engine.

        Two schedules, both timed on the wall clock:
          serial     each step's plan, copies, run and wait in turn;
          pipelined  a serving loop that keeps one step in flight: it plans
                     and enqueues step n+1 (inputs and outputs double-
                     buffered), then waits for step n's result. The plan's
                     upload is stream-ordered after run n.
        Returns (pipelined ms, serial ms, h2d bytes, d2h bytes, breakdown)."""
        pb = self.pb
        dev = self.dev
        q_bytes = self.q.numel() * self.q.element_size()
        idx_off = (q_bytes + 255) // 256 * 256
        in_bytes = idx_off + self.idx.numel() * 4
        o_bytes = self.out.numel() * self.out.element_size()
        lse_off = (o_bytes + 255) // 256 * 256
        res_bytes = lse_off + self.lse.numel() * 4

        def buffers():
            in_h = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
            in_h[:q_bytes].copy_(pb.q.contiguous().view(-1).view(torch.uint8))
            in_h[idx_off:].copy_(pb.kv_indices.contiguous().view(torch.uint8))
            in_d = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
            res_d = torch.empty(res_bytes, dtype=torch.uint8, device=dev)
            return dict(
                in_h=in_h, in_d=in_d, res_d=res_d,
                res_h=torch.empty(res_bytes, dtype=torch.uint8).pin_memory(),
                q=in_d[:q_bytes].view(self.q.dtype).view(self.q.shape),
                idx=in_d[idx_off:].view(torch.int32),
                out=res_d[:o_bytes].view(self.out.dtype).view(self.out.shape),
                lse=res_d[lse_off:].view(torch.float32).view(self.lse.shape))

        bufs = [buffers(), buffers()]
        meta = 4 * (len(pb.kv_indptr) + len(pb.last_page_len) + len(pb.qo_indptr))
        fn = self.fi.fi_batch_decode_paged if self.mode in ("decode", "verify") else \
            self.fi.fi_batch_prefill_paged
        sm = self.pb.sm_scale
        s = torch.cuda.current_stream()

        def enqueue(b):
            b["in_d"].copy_(b["in_h"], non_blocking=True)
            fn(self.plan, b["q"], self.k, self.v, b["idx"], sm, out=b["out"], lse=b["lse"])
            b["res_h"].copy_(b["res_d"], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s)
            return ev

        def serial_step():
            self.do_plan()
            enqueue(bufs[0]).synchronize()

        for _ in range(warmup):
            serial_step()
        t0 = time.perf_counter()
        for _ in range(steps):
            serial_step()
        serial_ms = (time.perf_counter() - t0) / steps * 1e3

        def pipelined(n):
            self.do_plan()
            prev = enqueue(bufs[0])
            for i in range(1, n):
                self.do_plan()
                ev = enqueue(bufs[i & 1])
                prev.synchronize()  # step i-1's result is on the host
                prev = ev
            prev.synchronize()

        pipelined(warmup + 1)
        t0 = time.perf_counter()
        pipelined(steps)
        pipe_ms = (time.perf_counter() - t0) / steps * 1e3

        # where the serial step's time goes (host wall clock per phase)
        n = max(steps, 5)
        b = bufs[0]
        acc = {"plan_us": 0.0, "h2d_enqueue_us": 0.0, "run_call_us": 0.0, "d2h_enqueue_us": 0.0,
               "wait_us": 0.0}
        for _ in range(n):
            t = time.perf_counter()
            self.do_plan()
            t1 = time.perf_counter()
            b["in_d"].copy_(b["in_h"], non_blocking=True)
            t2 = time.perf_counter()
            fn(self.plan, b["q"], self.k, self.v, b["idx"], sm, out=b["out"], lse=b["lse"])
            t3 = time.perf_counter()
            b["res_h"].copy_(b["res_d"], non_blocking=True)
            t4 = time.perf_counter()
            s.synchronize()
            t5 = time.perf_counter()
            for k_, a_, b_ in (("plan_us", t, t1), ("h2d_enqueue_us", t1, t2),
                               ("run_call_us", t2, t3), ("d2h_enqueue_us", t3, t4),
                               ("wait_us", t4, t5)):
                acc[k_] += (b_ - a_) * 1e6 / n
        brk = {k_: round(v, 1) for k_, v in acc.items()}
        return pipe_ms, serial_ms, in_bytes + meta, res_bytes, brk


# the sources each profiled kernel is built from (their digest is recorded
# with the profile; a profile of other sources is not reported)
KERNEL_SOURCES = {
    "decode": ["decode_kernel.cuh", "decode.cu", "tma.cuh", "common.cuh", "fi_internal.h"],
    "prefill_tc": ["prefill_tc.cu", "tma.cuh", "common.cuh", "fi_internal.h"],
}


def source_digest(kernel):
    """First 16 hex digits of the SHA-256 of the kernel's sources, in order."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "paged_kv_attention_13_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profile_record(kernel, name):
    """The key: value lines of a committed ncu summary under profiles/, if the
    kernel's sources are unchanged since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.lstrip().startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != source_digest(kernel):
        return None
    return vals


def traffic_from_profile(kernel, name):
    """Per-launch DRAM bytes from the committed ncu summary (None when the
    kernel changed since)."""
    vals = profile_record(kernel, name)
    try:
        return float(vals["dram_bytes_per_launch"]) if vals else None
    except (KeyError, ValueError):
        return None


def host_cores():
    """CPU cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_oracle_pass(pb, causal, wl, requests=None):
    """One timed pass of the oracle's fp32-accumulate OpenMP build over every
    (token, head) row of the batch, or of its first `requests` requests, on
    all the host's cores. Returns (seconds, threads, algorithmic bytes of the
    rows computed)."""
    from oracle.reference import attention_rows, fp32omp_threads
    threads = fp32omp_threads(host_cores())
    H = pb.num_qo_heads
    nb = len(pb.kv_lens) if requests is None else int(requests)
    T = int(pb.qo_indptr[nb])
    toks = np.repeat(np.arange(T, dtype=np.int64), H)
    heads = np.tile(np.arange(H, dtype=np.int32), T)
    args = pb.oracle_args()
    t0 = time.perf_counter()
    attention_rows(*args, causal, wl, pb.sm_scale, toks, heads, dtype=pb.dtype, fp32omp=True)
    dt = time.perf_counter() - t0
    if requests is None:
        byts = accounting(pb, causal, wl)[1]
    else:
        sub = workloads.make_paged_batch(pb.q_lens[:nb], pb.kv_lens[:nb], pb.num_qo_heads,
                                         pb.num_kv_heads, pb.head_dim, pb.page_size, pb.dtype, 0)
        byts = accounting(sub, causal, wl)[1]
    return dt, threads, byts


def aggregate_ranks(ms_local, bytes_per_rank, world, device):
    """Whole-job rate of N replicas: the step time is the max over ranks, the
    bytes are every rank's. Returns (ms_max, GB/s)."""
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    return ms, world * bytes_per_rank / (ms * 1e-3) / 1e9


def run_ours(args):
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    hbm_peak, bf16_peak, bf16_sus, peak_kind = peaks()

    # ---- headline: batch decode
    pb = workloads.batch_decode()
    ws = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    r = Runner(pb, False, -1, "decode", dev, ws=ws)
    for _ in range(args.warmup):
        r.run()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms_mean, ms_med = r.time(args.steps, args.warmup)
    if world > 1:
        dist.barrier()
    ms_step, value = aggregate_ranks(ms_mean, r.bytes, world, dev)
    e2e_ms, e2e_serial_ms, h2d, d2h, e2e_brk = r.time_e2e(max(5, args.steps), 3)
    e2e_value = world * r.bytes / (e2e_ms * 1e-3) / 1e9
    achieved = r.bytes / (ms_step * 1e-3) / 1e9
    traffic = traffic_from_profile("decode", "decode_tma_kernel_batch64.txt")
    roof = {"bound": "hbm", "kernel": "decode_tma_kernel (+ split-KV merge, timed together)",
            "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
            "frac_of_nominal_8000": round(achieved / 8000.0, 4),
            "algorithmic_bytes_per_launch": r.bytes,
            "traffic": traffic}
    launches = r.launches_per_step() * args.steps
    clocks = clk.summary()

    extra = {}
    if rank == 0 and not args.headline_only:
        extra = other_workloads(args, dev, ws, hbm_peak, bf16_peak)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        times, threads = [], 1
        t_all = time.perf_counter()
        while len(times) < 3 and (not times or time.perf_counter() - t_all < args.cpu_budget):
            dt, threads, _ = cpu_oracle_pass(pb, False, -1)
            times.append(dt)
        full_s = float(np.median(times))
        cpu = {"value": round(r.bytes / full_s / 1e9, 4), "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "ms_per_pass": round(full_s * 1e3, 2),
               "sample": "the whole batch (all %d (token, head) rows), %d timed passes, median; "
                         "the oracle's source built with fp32 accumulation, -O3 and OpenMP over "
                         "the rows, on the %d cores of the process's CPU affinity" % (
                             64 * 32, len(times), threads)}
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v, seeded page permutation)",
                "config": {"workload": "batch decode: batch 64, q_len 1, kv_len U[512,8192], "
                                       "32 q / 8 kv heads, head_dim 128, bf16, page 16, "
                                       "window -1, lse",
                           "total_kv_tokens": int(sum(pb.kv_lens)),
                           "l2": "inputs larger than L2 (KV cache %.2f GB > 129 MB)" % (
                               2 * sum(pb.kv_lens) * 8 * 128 * 2 / 1e9),
                           "plan": {k: r.info[k] for k in ("kernel_name", "num_items", "grid",
                                                            "max_chunks", "num_merge_rows")},
                           "parallelism": "replicas" if world > 1 else "single GPU"},
                "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                        "ms_per_step": round(e2e_ms, 4),
                        "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                        "serial": {"value": round(world * r.bytes / (e2e_serial_ms * 1e-3) / 1e9, 1),
                                   "ms_per_step": round(e2e_serial_ms, 4),
                                   "breakdown_host_us": e2e_brk},
                        "note": "every step: fi_plan (metadata upload) + one H2D copy of q and "
                                "the page table from pinned memory + run + one D2H copy of o "
                                "and lse + the wait for it; the KV cache stays resident. value: "
                                "a serving loop with one step in flight (plan and enqueue step "
                                "n+1, then wait for step n's result; double-buffered inputs "
                                "and outputs); serial: each step's phases in turn"},
                "gpu_launches": launches, "clocks": clocks, "roofline": roof,
                "cpu_baseline": cpu, "workloads": extra}
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def spec_sampling_entry(dev, steps, hbm_peak, batch=64, n_draft=4, vocab=128256):
    """The chain speculative-sampling step (acceptance + one draw per request).
    Algorithmic bytes: the n acceptance lookups and the drawn row (p, and q
    when a draft was rejected) of every request, plus the outputs; counted
    from the step's own acceptance result."""
    import paged_kv_attention_13_gb300 as fi
    d = workloads.spec_sampling_batch(batch=batch, n_draft=n_draft, vocab=vocab)
    t = {k: v.to(dev) for k, v in d.items()}
    outs = (torch.empty((batch, n_draft + 1), dtype=torch.int32, device=dev),
            torch.empty(batch, dtype=torch.int32, device=dev),
            torch.empty(batch, dtype=torch.int32, device=dev))

    def step():
        fi.fi_chain_speculative_sampling(t["draft_probs"], t["draft_ids"], t["target_probs"],
                                         t["u_accept"], t["u_sample"], *outs)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    acc = outs[1].cpu().numpy()
    byts = int(sum(vocab * 4 * (2 if a < n_draft else 1) for a in acc)) + \
        batch * n_draft * (4 + 4 + 4 + 4) + batch * 4 + batch * (n_draft + 1) * 4 + 8 * batch
    buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()
    ms = []
    for i in range(steps):
        buf.fill_(i & 0xFF)  # the rows start out of L2
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        step()
        b.record(s)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    m = float(np.median(ms))
    gbs = byts / (m * 1e-3) / 1e9
    return {"ms": round(m, 4), "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_peak, 4),
            "kernel": "chain_spec_kernel", "accepted_mean": round(float(acc.mean()), 3)}


def other_workloads(args, dev, ws, hbm_peak, bf16_peak):
    res = {}
    steps = max(3, min(args.steps, 10))

    def one(name, pb, causal, wl, mode, force=0, bound="hbm", graph=False):
        r = Runner(pb, causal, wl, mode, dev, force_kv_chunks=force, ws=ws, graph=graph)
        ms, med = r.time(steps, 3, flush=r.bytes < (512 << 20))
        tf = r.flops / (ms * 1e-3) / 1e12
        gbs = r.bytes / (ms * 1e-3) / 1e9
        ent = {"ms": round(ms, 4), "TFLOPS": round(tf, 2), "GB/s": round(gbs, 1),
               "kernel": r.info["kernel_name"], "items": r.info["num_items"],
               "chunks": r.info["max_chunks"], "bytes_per_launch": int(r.bytes)}
        if graph:
            ent["replay"] = "CUDA graph (planned once, captured, replayed)"
        if bound == "tensor":
            ent["frac_of_bf16_peak"] = round(tf / bf16_peak, 4)
        else:
            ent["frac_of_hbm"] = round(gbs / hbm_peak, 4)
        res[name] = ent
        del r

    pb = workloads.speculative_verify(batch=32)
    one("verify_b32", pb, True, -1, "verify", graph=True)
    one("verify_b32_eager", pb, True, -1, "verify")
    pb = workloads.speculative_verify(batch=4)
    one("verify_b4", pb, True, -1, "verify", graph=True)
    one("verify_b4_eager", pb, True, -1, "verify")
    for P in (16, 1024):
        pb = workloads.batch_prefill(page_size=P)
        one("prefill_p%d_causal" % P, pb, True, -1, "prefill", bound="tensor")
        if P == 16:
            # the ncu capture of this launch (its tensor-pipe share and DRAM
            # traffic), when the kernel is the one that was captured
            rec = profile_record("prefill_tc", "prefill_tc_kernel_prefill_b16_causal.txt")
            if rec:
                ent = res["prefill_p16_causal"]
                prof = {"source": "profiles/prefill_tc_kernel_prefill_b16_causal.txt"}
                for k in ("tensor_pipe_active_pct", "dram_bytes_per_launch",
                          "duration_us_under_ncu"):
                    if k in rec:
                        prof[k] = float(rec[k])
                if "dram_bytes_per_launch" in prof:
                    prof["traffic_over_algorithmic"] = round(
                        prof["dram_bytes_per_launch"] / ent["bytes_per_launch"], 3)
                ent["profile"] = prof
            one("prefill_p16_noncausal", pb, False, -1, "prefill", bound="tensor")
            one("prefill_p16_causal_wl127", pb, True, 127, "prefill")
    pb = workloads.batch_prefill_hd64()
    one("prefill_hd64_f16_p16_causal", pb, True, -1, "prefill", bound="tensor")
    pb = workloads.batch_prefill(page_size=48)
    one("prefill_p48_causal", pb, True, -1, "prefill", bound="tensor")
    pb = workloads.ragged_prefill()
    one("ragged_prefill_causal", pb, True, -1, "ragged", bound="tensor")
    pb = workloads.tree_verify(batch=32)
    one("tree_verify_b32", pb, True, -1, "masked")
    res["spec_sampling_b64_n4_v128256"] = spec_sampling_entry(dev, steps, hbm_peak)
    pb = workloads.long_context()
    one("longctx_causal_split", pb, True, -1, "prefill")
    one("longctx_causal_force32", pb, True, -1, "prefill", force=32)
    one("longctx_causal_wl127", pb, True, 127, "prefill")
    pb = workloads.pr1_reference()
    one("pr1_64x256_causal", pb, True, -1, "prefill")
    return res


def run_reference(args):
    """The CPU oracle as it stands, on the host cores, same metric and unit.

    Each step is one measured pass of the oracle's fp32-accumulate OpenMP
    build over the decode batch on every core of the process's affinity:
    the whole batch when a pass takes at most REF_STEP_S seconds, else the
    batch's first requests, as many as fit that time (the first warm-up pass
    decides). ms_per_step is the measured time of one such pass, nothing is
    scaled, so steps x ms_per_step is the time the timed steps took."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle.build import build_all
    build_all()
    pb = workloads.batch_decode()
    requests = None
    dt, threads, byts = cpu_oracle_pass(pb, False, -1)  # calibration (first warm-up)
    if dt > REF_STEP_S:
        frac = REF_STEP_S / dt
        kv = np.cumsum(pb.kv_lens) / float(sum(pb.kv_lens))
        requests = max(1, int(np.searchsorted(kv, frac)))
    for _ in range(max(0, args.warmup - 1)):
        cpu_oracle_pass(pb, False, -1, requests)
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        dt, threads, byts = cpu_oracle_pass(pb, False, -1, requests)
        times.append(dt)
    wall = time.perf_counter() - t_all
    step_s = float(np.mean(times))
    value = byts / step_s / 1e9
    what = "the whole batch (64 requests)" if requests is None else \
        "the batch's first %d of 64 requests" % requests
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "batch decode: batch 64, q_len 1, kv_len U[512,8192], 32 q / "
                                   "8 kv heads, head_dim 128, bf16, page 16, window -1, lse"},
            "timed_wall_s": round(wall, 3),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle",
                             "sample": "each step one pass over %s, every (token, head) row; the "
                                       "oracle's source built with fp32 accumulation, -O3 and "
                                       "OpenMP over the rows" % what},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line))


PROFILE_CASES = {
    # name: (batch factory, causal, window_left, mode)
    "decode_b16": (lambda: workloads.batch_decode(batch=16), False, -1, "decode"),
    "decode_b64": (lambda: workloads.batch_decode(), False, -1, "decode"),
    "verify_b32": (lambda: workloads.speculative_verify(batch=32), True, -1, "verify"),
    "prefill_p16_causal": (lambda: workloads.batch_prefill(page_size=16), True, -1, "prefill"),
    "prefill_b4_causal": (lambda: workloads.batch_prefill(page_size=16, batch=4), True, -1, "prefill"),
    "prefill_p1024_causal": (lambda: workloads.batch_prefill(page_size=1024), True, -1, "prefill"),
    "prefill_p16_noncausal": (lambda: workloads.batch_prefill(page_size=16), False, -1, "prefill"),
    "prefill_p16_causal_wl127": (lambda: workloads.batch_prefill(page_size=16), True, 127, "prefill"),
    "prefill_hd64_f16_causal": (lambda: workloads.batch_prefill_hd64(), True, -1, "prefill"),
    "prefill_p48_causal": (lambda: workloads.batch_prefill(page_size=48), True, -1, "prefill"),
    "longctx_causal": (lambda: workloads.long_context(), True, -1, "prefill"),
    "longctx_causal_wl127": (lambda: workloads.long_context(), True, 127, "prefill"),
    "ragged_prefill_causal": (lambda: workloads.ragged_prefill(), True, -1, "ragged"),
    "tree_verify_b32": (lambda: workloads.tree_verify(batch=32), True, -1, "masked"),
    "spec_sampling_b64": None,  # the sampling step (spec_sampling_entry)
}


def run_case(args):
    """One workload alone (for profiler captures): warm-up, then timed runs."""
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.case == "spec_sampling_b64":
        print(json.dumps({"case": args.case,
                          **spec_sampling_entry(dev, args.steps, peaks()[0])}))
        return
    make, causal, wl, mode = PROFILE_CASES[args.case]
    pb = make()
    r = Runner(pb, causal, wl, mode, dev)
    ms, med = r.time(args.steps, args.warmup)
    print(json.dumps({"case": args.case, "ms_mean": round(ms, 4), "ms_median": round(med, 4),
                      "GB/s": round(r.bytes / (ms * 1e-3) / 1e9, 1),
                      "TFLOPS": round(r.flops / (ms * 1e-3) / 1e12, 2), "plan": r.info}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None, choices=sorted(PROFILE_CASES))
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

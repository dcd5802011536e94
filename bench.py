"""Decode-step benchmark of the NOSA hot path on GB300.

One step = one nosa_decode_step over every request of the workload (append +
pooling, block scoring, dual selection, set-difference, UVA gather, split-K
attention, combine). Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl nosa|reference]

Under torchrun every rank runs its own copy of the workload on its own GPU
(weak scaling: units are independent, no collective on the data path); the
value is all ranks' tokens over the max-over-ranks time.

--impl reference times the fp64 CPU oracle (the only reference this method has)
on a bounded sample of units per step, on the host cores.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s per layer step; attn HBM GB/s & recall H2D GB/s vs peak"
DEFAULT_WORKLOAD = "8b-offload-bf16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20


# ---------------------------------------------------------------------------
# distributed plumbing (host logic; tested with gloo on CPU)
# ---------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(seconds: float, tokens: int, world: int):
    """(max seconds over ranks, total tokens over ranks). Plain values at world 1."""
    if world == 1:
        return seconds, tokens
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def arm_config(w, world, budget=None):
    """The `config` object of a decode line (both arms): the workload and how it
    is laid out and run."""
    n_cand = w.prompt // w.block
    slot_mib = w.units * w.k * (64 * w.head_dim * 2 * (4 if w.dtype == "f32" else 2) + 256) / 2 ** 20
    pk_mib = w.units * n_cand * 4 * w.head_dim * 4 / 2 ** 20
    big = (slot_mib + pk_mib) * 2 ** 20 > L2_BYTES
    return {"workload": w.name, "batch": w.batch, "n_q_heads": w.n_q_heads,
            "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "k": w.k, "k_e": w.k_e,
            "context_start": w.prompt,
            "l2": ("inputs larger than L2 (slot pool %.0f MiB, pooled keys %.0f MiB > %d MiB)"
                   if big else
                   "inputs within L2 (slot pool %.1f MiB, pooled keys %.1f MiB < %d MiB): "
                   "steps run with a warm L2") % (slot_mib, pk_mib, L2_BYTES >> 20),
            "parallelism": f"replicas x{world} (independent requests per GPU)",
            "queries": "AR(1), rho %g, %s" % (w.rho, "stationary start" if w.q_stationary
                                              else "started from one innovation"),
            **(budget or {})}


def rank_requests(batch: int, world: int, rank: int):
    """Requests (first, count) of the job's world * batch that rank runs: weak
    scaling, every rank its own batch of requests, disjoint, covering the job."""
    import synth
    if world * batch > synth.MAX_REQUESTS:
        raise ValueError(f"{world} ranks x {batch} requests exceed the generator's "
                         f"{synth.MAX_REQUESTS} requests")
    return rank * batch, batch


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.lines, self.proc, self.windows = [], None, []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            inside = any(a - 0.06 <= ts <= b + 0.06 for a, b in self.windows)
            rows.append((inside, parts))
        use = [p for ins, p in rows if ins] or [p for _, p in rows]
        if not use:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for p in use if num(p[2]) is not None]
        mx = [num(p[3]) for p in use if num(p[3]) is not None]
        reasons = sorted({name for p in use for name, v in zip(self.REASONS, p[6:10])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": sum(1 for i, _ in rows if i)}


def pct(sorted_vals, q):
    """q-th percentile (linear interpolation) of an ascending list."""
    if not sorted_vals:
        return 0.0
    x = (len(sorted_vals) - 1) * q / 100.0
    lo = int(math.floor(x))
    hi = min(lo + 1, len(sorted_vals) - 1)
    return sorted_vals[lo] + (sorted_vals[hi] - sorted_vals[lo]) * (x - lo)


def gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v for v in vis.split(",") if v.strip() != ""]
    if ids and all(v.strip().isdigit() for v in ids):
        return int(ids[min(local_rank, len(ids) - 1)])
    return local_rank


# ---------------------------------------------------------------------------
# roofline bookkeeping
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def attn_bytes_per_launch(w, n_cand, tail_len):
    """Algorithmic bytes of one attention launch: every attended token's K, V and e,
    plus the queries and the outputs."""
    elt = 4 if w.dtype == "f32" else 2
    per_tok = 2 * w.head_dim * elt + 4
    toks = min(w.k, n_cand) * w.block + tail_len
    return w.units * (toks * per_tok + 2 * w.group * w.head_dim * elt)


def score_bytes_per_launch(w, n_cand, pk_elt=4):
    """Algorithmic bytes of one scoring launch: all pooled keys (fp32, or bf16 in
    the pooled-bf16 variant), the scores written, and the queries."""
    elt = 4 if w.dtype == "f32" else 2
    return w.units * (n_cand * 4 * w.head_dim * pk_elt + n_cand * 4 + w.group * w.head_dim * elt)


def frontend_bytes_per_launch(w, D):
    """Algorithmic bytes of one fused front-end launch: the packed weights and the
    hidden states read once, every projected value written once (bf16)."""
    F = (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim + w.n_kv_heads
    return F * D * 2 + w.batch * D * 2 + w.batch * F * 2


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


ATTN_SOURCES = ["trainable_sparse_attention_decode_gb300/csrc/k_attn.cuh",
                "trainable_sparse_attention_decode_gb300/csrc/k_attn_bf16.cu"]
TILE_SOURCES = ["trainable_sparse_attention_decode_gb300/csrc/k_prefill_tc.cu",
                "trainable_sparse_attention_decode_gb300/csrc/tcgen05.cuh"]


def ncu_traffic(workload_name, kernel="attn_streamk_kernel", sources=None):
    """Per-launch DRAM bytes of a kernel from its committed ncu summary, or None when
    the summary is missing or the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload_name}.md")
    if not os.path.exists(p):
        return None
    src_hash = kernel_source_hash(sources or ATTN_SOURCES)
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_hash") != src_hash:
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def pinned_kb():
    """VmPin + VmLck of this process in kB (None where the kernel does not say)."""
    try:
        tot, seen = 0, False
        with open("/proc/self/status") as f:
            for line in f:
                if line.startswith(("VmPin:", "VmLck:")):
                    tot += int(line.split()[1])
                    seen = True
        return tot if seen else None
    except OSError:
        return None


def anon_huge_kb():
    """AnonHugePages of this process in kB (None where the kernel does not say)."""
    try:
        with open("/proc/self/smaps_rollup") as f:
            for line in f:
                if line.startswith("AnonHugePages:"):
                    return int(line.split()[1])
    except OSError:
        pass
    return None


VM_EVENTS = ("thp_fault_alloc", "thp_fault_fallback", "thp_collapse_alloc",
             "thp_collapse_alloc_failed", "thp_split_page", "thp_split_page_failed",
             "thp_deferred_split_page", "thp_underused_split_page", "thp_migration_split",
             "thp_migration_success", "thp_migration_fail", "thp_split_pmd", "thp_swpout",
             "thp_swpout_fallback", "pswpout", "pgsteal_anon", "compact_stall",
             "compact_migrate_scanned", "pgmigrate_success", "pgmigrate_fail",
             "numa_hint_faults", "numa_pages_migrated")


def vm_events():
    """A few of the kernel's memory-management event counters (/proc/vmstat), or
    None where the kernel does not say: their change over the timed region tells
    whether the host rearranged pages (huge-page collapse, compaction, migration)
    while the GPU was reading the host store."""
    try:
        out = {}
        with open("/proc/vmstat") as f:
            for line in f:
                k, _, v = line.partition(" ")
                if k in VM_EVENTS:
                    out[k] = int(v)
        return out
    except OSError:
        return None


STORE_LAYOUTS = {0: "cudaHostAlloc", 1: "mapping bound to the GPU's node",
                 2: "transparent huge pages"}


def host_store_report(st, huge_kb, huge_kb_after, pin_kb, vm_created, vm_t0, vm_t1):
    """How the host store was laid out, how much of the process was in huge pages
    and pinned after the create and after the timed steps, and the host's
    memory-management events during the setup and the timed steps."""
    mb = lambda kb: round(kb / 1024) if kb is not None else None
    delta = lambda a, b: {k_: b[k_] - a.get(k_, 0) for k_ in b if b[k_] != a.get(k_, 0)}
    return {"layout": STORE_LAYOUTS.get(st["host_store_kind"], st["host_store_kind"]),
            "long_term_pins": bool(st["host_store_pinned"]),
            "huge_pages_mb": mb(huge_kb), "huge_pages_mb_after_timed": mb(huge_kb_after),
            "pinned_mb": mb(pin_kb),
            "vm_events": ({"setup": delta(vm_created, vm_t0), "timed": delta(vm_t0, vm_t1)}
                          if vm_created and vm_t0 and vm_t1 else None)}


def h2d_peak_gbs(torch, nbytes=1 << 30, reps=5, median=False):
    """Pinned host -> device copy rate (GB/s): the best of `reps` copies, or their
    median."""
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    del src, dst
    t = sorted(times)[len(times) // 2] if median else min(times)
    return nbytes / t / 1e9


def attention_alone(nosa, torch, w, n_cand, tail_len, reps=20, classic=False):
    """Times the split-K attention kernel alone on the step's shape: every unit
    attends over min(k, N) full blocks plus a tail of tail_len tokens, all block
    units fresh in HBM (more than L2). classic: the classic split the decode step
    launches (attn_split_kernel; the planner's split count for one launch over
    every unit: the step launches it per unit chunk), else the standalone call's
    own plan (stream-K when it fits).
    Returns (seconds per launch, algorithmic bytes per launch)."""
    saved = os.environ.get("NOSA_ATTN_STREAMK")
    if classic:
        os.environ["NOSA_ATTN_STREAMK"] = "0"
    try:
        return _attention_alone(nosa, torch, w, n_cand, tail_len, reps)
    finally:
        if classic:
            if saved is None:
                os.environ.pop("NOSA_ATTN_STREAMK", None)
            else:
                os.environ["NOSA_ATTN_STREAMK"] = saved


def _attention_alone(nosa, torch, w, n_cand, tail_len, reps):
    # the standalone call uses only the shape fields of the config (k is capped to
    # the decode step's limit for validation; the block table sets the blocks)
    kk = min(w.k, 256)
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, kk,
                           min(w.k_e, kk), w.max_context)
    payload = nosa.nosa_payload_bytes(cfg)
    nb = min(w.k, n_cand)
    U = w.units
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    # finite random contents: normals of the storage dtype, viewed as bytes
    elems = (U * nb + U) * payload // (4 if w.dtype == "f32" else 2)
    units = torch.randn(elems, dtype=dt, device="cuda").view(torch.uint8)
    body, tail = units[: U * nb * payload], units[U * nb * payload:]
    tab = torch.arange(U * nb, dtype=torch.int32, device="cuda").view(U, nb)
    q = torch.randn((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
    ws = torch.empty(nosa.nosa_attention_workspace_bytes(cfg, nb), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        nosa.nosa_sparse_attention(cfg, body, tab, tail, tail_len, q, out, lse, ws)
    # The units (hundreds of MB) exceed L2, so back-to-back launches read HBM; queueing
    # them hides the host's per-call work.
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        nosa.nosa_sparse_attention(cfg, body, tab, tail, tail_len, q, out, lse, ws)
    b.record()
    b.synchronize()
    del units
    return a.elapsed_time(b) / 1e3 / reps, attn_bytes_per_launch(w, n_cand, tail_len)


def budget_batch(args, w, mode):
    """Largest batch whose GPU-resident state fits the HBM budget (--hbm-budget GB).

    fullattn: the whole cache of a request in HBM, every complete block and the
    tail as block units. nosa / infllmv2: the handle's device state of a request
    (slot pool, tail buffers, pooled metadata, bitmasks, split-K partials),
    measured on a 4-request handle; capped so that the pinned host store stays
    within --host-budget GB."""
    import torch
    import trainable_sparse_attention_decode_gb300 as nosa
    budget = args.hbm_budget * 1e9
    cfg1 = nosa.nosa_config(1, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                            w.max_context)
    payload = nosa.nosa_payload_bytes(cfg1)
    if mode == "fullattn":
        per_req = w.n_kv_heads * (w.prompt // w.block + 1) * payload
        return max(1, int(budget // per_req)), per_req, 0
    probe = 4
    cfg = nosa.nosa_config(probe, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                           w.max_context)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    h = nosa.nosa_create(cfg)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    nosa.nosa_destroy(h)
    per_req = (free0 - free1) / probe
    host_req = w.n_kv_heads * ((w.max_context + w.block - 1) // w.block) * payload
    b = int(budget // per_req)
    b = min(b, int(args.host_budget * 1e9 // host_req), 65535 // w.n_kv_heads)
    return max(1, b), per_req, host_req


def run_fullattn(args, rank, world, local_rank):
    """Comparator: dense decode attention with the whole KV cache resident in HBM
    (no selection, no recall), on the same split-K kernel: every unit attends
    over all N complete blocks plus the tail. One step = one attention launch
    for the batch."""
    import torch
    import synth
    import trainable_sparse_attention_decode_gb300 as nosa
    torch.cuda.set_device(local_rank)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(batch=args.batch)
    budget = None
    if args.hbm_budget:
        b, per_req, _ = budget_batch(args, w, "fullattn")
        w = w.with_(batch=b)
        budget = {"hbm_budget_gb": args.hbm_budget, "hbm_bytes_per_request": per_req,
                  "batch_from_budget": b}
    n_cand = w.prompt // w.block
    wf = w.with_(k=n_cand)               # attend to every block
    W, K = args.warmup, args.steps
    barrier(world)
    secs_w, _ = attention_alone(nosa, torch, wf, n_cand, 33, reps=W)
    barrier(world)
    secs, nbytes = attention_alone(nosa, torch, wf, n_cand, 33, reps=K)
    max_secs, tokens = aggregate(secs * K, w.batch * K, world)
    if rank != 0:
        return None
    peak, kind = measured_peaks()
    gbs = nbytes / secs / 1e9
    return {"metric": METRIC, "value": round(tokens / max_secs, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(secs * 1e3, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "mode": "fullattn",
            "config": {"workload": w.name + "-fullattn", "batch": w.batch,
                       "context": w.prompt, "blocks_per_unit": n_cand,
                       "kv_bytes_in_hbm": w.units * (n_cand + 1) * 33024,
                       "l2": "inputs larger than L2", **(budget or {})},
            "roofline": {"bound": "hbm", "kernel": "attn_split_kernel (dense)",
                         "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None, "peak_source": kind,
                         "algorithmic_bytes_per_launch": nbytes},
            "gpu_launches": K}


def run_prefill(args, rank, world, local_rank):
    """Training-time forward (causal dual selection at every position, then the
    block-sparse attention) over whole sequences of the workload's shape. One step
    = one nosa_prefill_forward over batch x L tokens."""
    import torch
    import synth
    import synth.gpu
    import trainable_sparse_attention_decode_gb300 as nosa
    torch.cuda.set_device(local_rank)
    w = synth.WORKLOADS[args.workload].with_(batch=args.batch or 1)
    L = args.prompt or 32768
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e, L,
                           device=local_rank)
    k, v, e = synth.gpu.kv(w, 0, L)
    q = synth.gpu.queries(w, L).permute(1, 0, 2, 3).contiguous()
    out = torch.empty_like(q)
    lse = torch.empty((w.batch, L, w.n_q_heads), dtype=torch.float32, device="cuda")
    ws = torch.empty(nosa.nosa_prefill_workspace_bytes(cfg, L), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    W, K = args.warmup, max(1, min(args.steps, 20))
    for _ in range(W):
        nosa.nosa_prefill_forward(cfg, q, k, v, e, out, lse, workspace=ws, stream=stream)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(K):
        nosa.nosa_prefill_forward(cfg, q, k, v, e, out, lse, workspace=ws, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    secs = ev0.elapsed_time(ev1) / 1e3 / K
    # per-phase device time (events the library records on the stream when the
    # config asks for it), on the same inputs right after the timed region
    cfg_t = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                             L, device=local_rank, flags=nosa.NOSA_FLAG_TIMING)
    front_ms, attn_ms = [], []
    for _ in range(K):
        nosa.nosa_prefill_forward(cfg_t, q, k, v, e, out, lse, workspace=ws, stream=stream)
        f_ms, a_ms = nosa.nosa_prefill_timing()
        front_ms.append(f_ms)
        attn_ms.append(a_ms)
    max_secs, tokens = aggregate(secs, w.batch * L, world)
    if rank != 0:
        return None
    elt = 2 if w.dtype == "bf16" else 4
    payload = nosa.nosa_payload_bytes(cfg)
    nblk = (L + 63) // 64
    attn_s = sum(attn_ms) / len(attn_ms) / 1e3
    # tokens each position attends: its selected blocks and its own block up to itself
    att_tokens = sum(min(w.k, t // 64) * 64 + t % 64 + 1 for t in range(L)) * w.batch
    # bytes that must cross HBM at least once: inputs, block units written and read,
    # pooled keys, outputs
    hbm_bytes = (w.batch * L * (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim * elt
                 + w.batch * L * w.n_kv_heads * 4
                 + 2 * w.units * nblk * payload + w.units * nblk * 4 * w.head_dim * 4
                 + w.batch * L * w.n_q_heads * (w.head_dim * elt + 4))
    tiled = (w.dtype == "bf16" and w.group in (1, 2, 4) and w.head_dim in (64, 128)
             and os.environ.get("NOSA_PREFILL_TILED", "1") != "0")
    if tiled:
        # useful work of the tensor-core attention: Q K^T and P V over every
        # position's attended tokens, per query head (the kernel also computes the
        # masked entries of the union of a query block's selections)
        flops = 4.0 * w.head_dim * w.n_q_heads * att_tokens
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk_d = json.load(f)
        peak_t, kind = float(pk_d["bf16_tflops"]), "measured bf16 burst (P V runs in fp16, same rate)"
        ach = flops / attn_s / 1e12
        roof = {"bound": "tensor", "kernel": "prefill_tile_kernel (tcgen05 attention per query block)",
                "achieved": round(ach, 1), "peak": peak_t, "unit": "TFLOP/s",
                "frac": round(ach / peak_t, 4),
                # DRAM bytes of one launch from the committed capture of this
                # sequence length (the union of a block's selections, and so the
                # traffic, does not scale with L)
                "traffic": ncu_traffic(f"8b-L{L}", "prefill_tile_kernel", TILE_SOURCES)
                if w.name == "8b-offload-bf16" and w.batch == 1 else None,
                "peak_source": kind,
                "algorithmic_flops_per_launch": flops,
                "kernel_ms": round(attn_s * 1e3, 4)}
    else:
        peak, kind = measured_peaks()
        attn_bytes = sum(min(w.k, t // 64) + 1 for t in range(L)) * w.batch * w.n_kv_heads * payload
        gbs = attn_bytes / attn_s / 1e9
        roof = {"bound": "hbm", "kernel": "attn_split_kernel (a virtual unit per position)",
                "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(gbs / peak, 4), "traffic": None, "peak_source": kind,
                "algorithmic_bytes_per_launch": attn_bytes, "kernel_ms": round(attn_s * 1e3, 4),
                "note": "bytes gathered per position (mostly served by L2)"}
    # the selection on the tensor cores adds the key-split launch
    select_tc = (w.head_dim in (64, 128) and w.k - w.k_e <= 32
                 and os.environ.get("NOSA_PREFILL_SELECT_TC", "1") != "0")
    launches = (5 if tiled else 3 + -(-w.batch * L * w.n_kv_heads // 65535)) + (1 if select_tc else 0)
    return {"metric": "training-time forward tokens/s per layer (causal dual selection + "
                      "block-sparse attention)",
            "value": round(tokens / max_secs, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(secs * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "mode": "prefill",
            "config": {"workload": w.name + f"-prefill-L{L}", "batch": w.batch, "seq_len": L,
                       "k": w.k, "k_e": w.k_e, "n_q_heads": w.n_q_heads,
                       "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
                       "attention": "tiled tensor-core" if tiled else "split-K per position",
                       "selection": "tensor-core (fp32 operands split in 3 bf16 terms)" if select_tc
                       else "CUDA-core fp32"},
            "roofline": roof,
            "phase_ms": {"front": round(sum(front_ms) / len(front_ms), 4),
                         "attention": round(attn_s * 1e3, 4)},
            "hbm_unique_bytes_per_call": hbm_bytes,
            "gpu_launches": launches * K}


def run_gpu(args, rank, world, local_rank):
    import torch
    import synth
    import synth.gpu
    import trainable_sparse_attention_decode_gb300 as nosa

    torch.cuda.set_device(local_rank)
    w0 = synth.WORKLOADS[args.workload].with_(q_stationary=not args.q_innovation_start)
    budget = None
    if args.hbm_budget:
        wb = w0.with_(k_e=0) if args.mode == "infllmv2" else w0
        b, per_req, host_req = budget_batch(args, wb.with_(steps=args.warmup + args.steps
                                                           + args.e2e_steps + args.phase_steps),
                                            args.mode)
        args.batch = b
        budget = {"hbm_budget_gb": args.hbm_budget, "host_budget_gb": args.host_budget,
                  "hbm_bytes_per_request": round(per_req), "host_bytes_per_request": host_req,
                  "batch_from_budget": b}
    if args.batch:
        w0 = w0.with_(name=f"{w0.name}-b{args.batch}", batch=args.batch)
    if world > 1:  # this rank's own requests of the job
        w0 = w0.with_(request_base=rank_requests(w0.batch, world, rank)[0])
    if args.prompt:
        w0 = w0.with_(name=f"{w0.name}-p{args.prompt}", prompt=args.prompt)
    if args.mode == "infllmv2":
        # comparator: no query-agnostic part, every block chosen by the query
        w0 = w0.with_(name=f"{w0.name}-ke0", k_e=0)
    W, K = args.warmup, args.steps
    KE = args.e2e_steps
    KT = 0 if args.no_timing else args.phase_steps  # per-phase event timing window
    total_steps = W + K + KE + KT
    w = w0.with_(steps=total_steps)
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                           w.max_context, device=local_rank,
                           flags=(nosa.NOSA_FLAG_POOLED_BF16 if args.pooled_bf16 else 0))
    h = nosa.nosa_create(cfg)
    huge_kb = anon_huge_kb()  # how much of the process is backed by huge pages (Linux)
    pin_kb = pinned_kb()  # how much of it is pinned or locked by the process itself
    vm_created = vm_events()
    # prompt, appended in chunks generated on the device
    chunk = 4096
    t = 0
    while t < w.prompt:
        n = min(chunk, w.prompt - t)
        k, v, e = synth.gpu.kv(w, t, n)
        nosa.nosa_append_kv(h, k, v, e)
        t += n
        del k, v, e
    torch.cuda.synchronize()
    # per-step inputs staged in HBM before the timed region
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device="cuda")
    lse = torch.empty((w.batch, w.n_q_heads), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    peak_h2d = h2d_peak_gbs(torch) if rank == 0 else None
    out_p, lse_p, stream_p = out.data_ptr(), lse.data_ptr(), stream.cuda_stream
    D = synth.hidden_width(w)
    if args.frontend:
        # the step starts from hidden states: the fused front-end projects them
        Wf = nosa.nosa_frontend_pack(cfg, synth.gpu.proj_weights(w, D))  # packed once
        x_all = synth.gpu.hidden(w, w.prompt, total_steps, D)
        def warm_step(s):
            nosa.nosa_decode_step_hidden(h, x_all[s], Wf, out, lse, stream=stream)
        ptrs = [x_all[s].data_ptr() for s in range(total_steps)]
        w_p = Wf.data_ptr()
        step_fn = nosa.lib.nosa_decode_step_hidden

        def raw_step(s):
            r = step_fn(h, ptrs[s], D, w_p, None, out_p, lse_p, stream_p)
            if r:
                raise nosa.NosaError(r, nosa.nosa_last_error(h))
        e2e_hosts = lambda: [x_all[W + K:W + K + KE].cpu().pin_memory()]
        e2e_step = lambda devs, o: nosa.nosa_decode_step_hidden(h, devs[0], Wf, o, None, stream=stream)
    else:
        q_all = synth.gpu.queries(w, total_steps)
        k_all, v_all, e_all = synth.gpu.kv(w, w.prompt, total_steps, step_major=True)
        def warm_step(s):
            nosa.nosa_decode_step(h, q_all[s], k_all[s], v_all[s], e_all[s], out, lse, stream)
        # raw pointers for the timed loop (shapes were checked by the warm-up calls)
        ptrs = [(q_all[s].data_ptr(), k_all[s].data_ptr(), v_all[s].data_ptr(), e_all[s].data_ptr())
                for s in range(total_steps)]
        step_fn = nosa.lib.nosa_decode_step

        def raw_step(s):
            p_ = ptrs[s]
            r = step_fn(h, p_[0], p_[1], p_[2], p_[3], out_p, lse_p, stream_p)
            if r:
                raise nosa.NosaError(r, nosa.nosa_last_error(h))
        e2e_hosts = lambda: [x[W + K:W + K + KE].cpu().pin_memory() for x in (q_all, k_all, v_all, e_all)]
        e2e_step = lambda devs, o: nosa.nosa_decode_step(h, *devs, o, None, stream)
    # Step 0 is the cold start (every slot empty: min(k, N) blocks per unit come
    # from the host store). It runs with the library's phase events, so its recall
    # rate is reported on its own; the other warm-up steps follow untimed.
    torch.cuda.synchronize()
    nosa.nosa_stats_reset(h)
    nosa.nosa_set_timing(h, True)
    warm_step(0)
    st_cold = nosa.nosa_stats(h)
    nosa.nosa_set_timing(h, False)
    for s in range(1, W):
        warm_step(s)
    torch.cuda.synchronize()
    nosa.nosa_stats_reset(h)
    sampler = ClockSampler(gpu_index(local_rank)) if rank == 0 else None
    time.sleep(0.15 if sampler else 0)
    barrier(world)
    torch.cuda.synchronize()
    # one event before every timed step (and one after the last): the whole-run
    # time is first to last, and the per-step times give the median and spread
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    vm_t0 = vm_events()
    w0t = time.time()
    torch.cuda.nvtx.range_push("timed")
    h0 = time.perf_counter()
    for i, s in enumerate(range(W, W + K)):
        evs[i].record(stream)
        raw_step(s)
    host_enqueue_us = (time.perf_counter() - h0) / K * 1e6
    evs[K].record(stream)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    w1t = time.time()
    vm_t1 = vm_events()
    huge_kb_after = anon_huge_kb()
    barrier(world)
    if sampler:
        sampler.mark(w0t, w1t)
    secs = evs[0].elapsed_time(evs[K]) / 1e3
    step_us = [evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(K)]
    st = nosa.nosa_stats(h)
    context_after = st["context"]
    # the pinned-copy rate again, right after the timed steps: a diagnostic of the
    # host link's state during them (the one before the setup is `h2d_peak_gbs`)
    h2d_after = h2d_peak_gbs(torch, nbytes=256 << 20, reps=3, median=True) if rank == 0 else None

    # end to end: pinned host inputs -> device, step, result -> pinned host, every
    # step, as a server pipelines them: double-buffered device inputs and outputs,
    # the copies on a copy stream overlapping the previous step's kernels
    hosts = e2e_hosts()
    devs = [[torch.empty_like(x[0], device="cuda") for x in hosts] for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    out_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    cs = torch.cuda.Stream()      # host -> device inputs
    cs_out = torch.cuda.Stream()  # device -> host results (never ahead of the next inputs)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0t = time.time()
    e0.record(stream)
    cs.wait_event(e0)
    cs_out.wait_event(e0)
    for s in range(KE):
        i = s % 2
        with torch.cuda.stream(cs):
            if s >= 2:
                cs.wait_event(ev_done[i])  # step s - 2 has read these inputs
            for d_, h_ in zip(devs[i], hosts):
                d_.copy_(h_[s], non_blocking=True)
            ev_in[i].record(cs)
        stream.wait_event(ev_in[i])
        if s >= 2:
            stream.wait_event(ev_out[i])  # step s - 2's output is on the host
        e2e_step(devs[i], outs[i])
        ev_done[i].record(stream)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(ev_done[i])
            out_h[i].copy_(outs[i], non_blocking=True)
            ev_out[i].record(cs_out)
    for ev in ev_out:
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    x1t = time.time()
    if sampler:
        sampler.mark(x0t, x1t)
    e2e_secs = e0.elapsed_time(e1) / 1e3
    bi = sum(x[0].numel() * x.element_size() for x in hosts)
    bo = out_h[0].numel() * out_h[0].element_size()
    clocks = sampler.stop() if sampler else None

    # Per-phase device times from the library's events, in a window of their own
    # (the events cost some device time, so the timed loops above run without).
    st_ph = None
    if KT > 0:
        nosa.nosa_set_timing(h, True)
        torch.cuda.synchronize()
        nosa.nosa_stats_reset(h)
        for s in range(W + K + KE, W + K + KE + KT):
            raw_step(s)
        st_ph = nosa.nosa_stats(h)
    nosa.nosa_destroy(h)
    del ptrs
    n_mid = (w.prompt + W + K // 2) // w.block
    tail_alone = (w.prompt + W + K // 2) % w.block + 1
    alone_secs, alone_bytes = attention_alone(nosa, torch, w, n_mid, tail_alone, classic=True)
    sk_secs, _ = attention_alone(nosa, torch, w, n_mid, tail_alone)

    max_secs, tokens = aggregate(secs, w.batch * K, world)
    e2e_max, e2e_tokens = aggregate(e2e_secs, w.batch * KE, world)
    if rank != 0:
        return None

    n_cand = (w.prompt + W + K // 2) // w.block       # mid-region candidate count
    tail_mid = (w.prompt + W + K // 2) % w.block + 1
    tu = st_ph["t_us"] if st_ph else [0.0] * 8
    nt = max(st_ph["t_count"], 1) if st_ph else 1
    # phases of nosa_stats: append+pool, score, select+set-difference, attention
    # over the slots kept from the previous step (runs while the gather runs on a
    # side stream), gather, attention over the filled slots (waits for the gather)
    # phases of nosa_stats (the step is pipelined over unit chunks, so they overlap;
    # each spans its first start to its last end)
    phase_us = {name: tu[i] / nt for i, name in enumerate(
        ["append_pool", "score_select", "unused2", "attention_kept", "gather",
         "after_kept", "unused6", "step"])}
    phase_us.pop("unused2")
    phase_us.pop("unused6")
    loads_per_unit = (st["host_loads"] + st["tail_loads"]) / max(K * w.units, 1)
    elt = 4 if w.dtype == "f32" else 2
    per_block = w.block * (2 * w.head_dim * elt + 4)
    attn_bytes = attn_bytes_per_launch(w, n_cand, tail_mid)
    attn_kept_bytes = attn_bytes - w.units * loads_per_unit * per_block
    score_bytes = score_bytes_per_launch(w, n_cand, 2 if args.pooled_bf16 else 4)
    peak, peak_kind = measured_peaks()
    def rate(nbytes, us):
        return nbytes / (us * 1e-6) / 1e9 if us > 0 else 0.0
    attn_gbs = rate(attn_kept_bytes, phase_us["attention_kept"])
    score_gbs = rate(score_bytes, phase_us["score_select"])  # includes the selection
    host_bytes_step = st["host_bytes"] / K
    host_bytes_window = st_ph["host_bytes"] / KT if st_ph else 0.0
    recall_gbs = (host_bytes_window / (phase_us["gather"] * 1e-6) / 1e9) if phase_us["gather"] else 0.0
    # Roofline kernel: the attention kernel the step launches (attn_split_kernel,
    # the classic split with the step's split count per unit), timed alone on the
    # step's shape; inside the step it runs at low priority beside the gather and
    # the scoring, so its in-step rate (attn_kept_in_step_gbs) measures sharing,
    # not the kernel. The stream-K form of the standalone call is reported apart.
    dominant = "attn_split_kernel (alone, the step's shape, one launch over every unit)"
    dom_bytes, dom_us = alone_bytes, alone_secs * 1e6
    traffic = ncu_traffic(w0.name, kernel="attn_split_kernel")
    value = tokens / max_secs
    srt = sorted(step_us)
    t_step = {"median": round(pct(srt, 50), 3), "p10": round(pct(srt, 10), 3),
              "p90": round(pct(srt, 90), 3), "mean": round(sum(srt) / len(srt), 3),
              "tokens_per_s_at_median": round(w.batch / (pct(srt, 50) * 1e-6), 3)}
    cold_gather_us = st_cold["t_us"][4] / max(st_cold["t_count"], 1)
    cold = {"step_us": round(st_cold["t_us"][7] / max(st_cold["t_count"], 1), 3),
            "host_bytes": st_cold["host_bytes"],
            "gather_us": round(cold_gather_us, 3),
            "recall_h2d_gbs": round(st_cold["host_bytes"] / (cold_gather_us * 1e-6) / 1e9, 2)
            if cold_gather_us > 0 else None}
    if peak_h2d and cold["recall_h2d_gbs"]:
        cold["recall_frac_of_h2d_peak"] = round(cold["recall_h2d_gbs"] / peak_h2d, 4)
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(max_secs / K * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded counter-based generator; shapes of the workload)",
        "mode": args.mode + ("+pooled_bf16" if args.pooled_bf16 else "")
                + ("+frontend" if args.frontend else ""),
        "config": arm_config(w0, world, budget),
        "context_end": context_after,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(dom_bytes / (dom_us * 1e-6) / 1e9, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(dom_bytes / (dom_us * 1e-6) / 1e9 / peak, 4),
                     "traffic": traffic, "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": dom_bytes},
        "attn_hbm_gbs": round(dom_bytes / (dom_us * 1e-6) / 1e9, 1),
        "attn_frac_of_peak": round(dom_bytes / (dom_us * 1e-6) / 1e9 / peak, 4),
        "attn_kept_in_step_gbs": round(attn_gbs, 1),
        "attn_streamk_alone": {"kernel": "attn_streamk_kernel (the standalone call's plan)",
                               "us": round(sk_secs * 1e6, 2),
                               "gbs": round(alone_bytes / sk_secs / 1e9, 1),
                               "frac_of_peak": round(alone_bytes / sk_secs / 1e9 / peak, 4)},
        **({"frontend": {"hidden": D, "rows": (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim
                         + w.n_kv_heads,
                         "kernel_us": round(phase_us["append_pool"], 3),
                         "hbm_gbs": round(rate(frontend_bytes_per_launch(w, D),
                                               phase_us["append_pool"]), 1),
                         "frac_of_peak": round(rate(frontend_bytes_per_launch(w, D),
                                                    phase_us["append_pool"]) / peak, 4),
                         "algorithmic_bytes_per_launch": frontend_bytes_per_launch(w, D)}}
           if args.frontend else {}),
        "score_hbm_gbs": round(score_gbs, 1),
        "recall_h2d_gbs": round(recall_gbs, 2),
        "h2d_peak_gbs": round(peak_h2d, 2) if peak_h2d else None,
        "h2d_after_timed_gbs": round(h2d_after, 2) if h2d_after else None,
        "host_store": host_store_report(st, huge_kb, huge_kb_after, pin_kb,
                                        vm_created, vm_t0, vm_t1),
        "recall_frac_of_h2d_peak": round(recall_gbs / peak_h2d, 4) if peak_h2d else None,
        "host_bytes_per_step": round(host_bytes_step),
        "phase_us": {k_: round(v_, 3) for k_, v_ in phase_us.items()},
        "t_step_us": t_step,
        "cold_step": cold,
        "gamma_mean": round(st["gamma_mean"], 4), "gamma_min": st["gamma_min"],
        "near_ties": st["near_ties"],
        "e2e": {"value": round(e2e_tokens / e2e_max, 3), "unit": "tokens/s",
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": KE,
                "copies": "every step; double-buffered, on copy streams overlapping the "
                          "previous step"},
        "gpu_launches": st["launches"],
        "loads_per_unit_step": round(loads_per_unit, 3),
        "host_enqueue_us_per_step": round(host_enqueue_us, 2),
        "step_graphs": os.environ.get("NOSA_GRAPHS", "1") != "0",
        "phase_window_steps": KT,
        "clocks": clocks,
    }
    return line


def run_horizon(args, rank, world, local_rank):
    """The workload's whole decode horizon (every step of `steps`), graph-replayed
    back to back; `args.horizon` windows of `window` steps, spread from the first
    warm step to the last, are timed with an event before every step and their
    counters read (host loads, locality). Reports each window's median step time,
    tokens/s, host bytes per step and the recall rate those bytes need."""
    import torch
    import synth
    import synth.gpu
    import trainable_sparse_attention_decode_gb300 as nosa
    torch.cuda.set_device(local_rank)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(batch=args.batch)
    n = w.steps
    win = max(16, min(256, n // (2 * args.horizon)))
    starts = [1 + round(i * (n - 1 - win) / max(1, args.horizon - 1)) for i in range(args.horizon)]
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                           w.max_context, device=local_rank)
    h = nosa.nosa_create(cfg)
    t = 0
    while t < w.prompt:
        m = min(4096, w.prompt - t)
        k, v, e = synth.gpu.kv(w, t, m)
        nosa.nosa_append_kv(h, k, v, e)
        t += m
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device="cuda")
    stream = torch.cuda.current_stream()
    q_all = synth.gpu.queries(w, n)
    k_all, v_all, e_all = synth.gpu.kv(w, w.prompt, n, step_major=True)
    peak_h2d = h2d_peak_gbs(torch)
    step_fn = nosa.lib.nosa_decode_step
    out_p, s_p = out.data_ptr(), stream.cuda_stream
    ptrs = [(q_all[s].data_ptr(), k_all[s].data_ptr(), v_all[s].data_ptr(), e_all[s].data_ptr())
            for s in range(n)]
    windows = []
    s = 0
    torch.cuda.synchronize()
    t_wall = time.time()
    for w0s in starts + [n]:
        while s < w0s:  # untimed steps up to the window
            p_ = ptrs[s]
            if step_fn(h, p_[0], p_[1], p_[2], p_[3], out_p, None, s_p):
                raise nosa.NosaError(0, nosa.nosa_last_error(h))
            s += 1
        if w0s == n:
            break
        nosa.nosa_stats_reset(h)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(win + 1)]
        for i in range(win):
            evs[i].record(stream)
            p_ = ptrs[s]
            if step_fn(h, p_[0], p_[1], p_[2], p_[3], out_p, None, s_p):
                raise nosa.NosaError(0, nosa.nosa_last_error(h))
            s += 1
        evs[win].record(stream)
        st = nosa.nosa_stats(h)
        us = sorted(evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(win))
        med = pct(us, 50)
        hb = st["host_bytes"] / win
        windows.append({"steps": [w0s, w0s + win], "context": [w.prompt + w0s + 1, w.prompt + w0s + win],
                        "t_step_us_median": round(med, 2), "t_step_us_p10": round(pct(us, 10), 2),
                        "t_step_us_p90": round(pct(us, 90), 2),
                        "tokens_per_s": round(w.batch / (med * 1e-6), 1),
                        "host_bytes_per_step": round(hb),
                        "link_time_frac": round(hb / (peak_h2d * 1e9) / (med * 1e-6), 4),
                        "gamma_mean": round(st["gamma_mean"], 4), "gamma_min": st["gamma_min"],
                        "max_host_loads_unit": st["max_host_loads_unit"]})
    wall = time.time() - t_wall
    nosa.nosa_destroy(h)
    if rank != 0:
        return None
    return {"metric": METRIC, "mode": "horizon", "unit": "tokens/s", "n_gpus": world,
            "config": {"workload": w.name, "batch": w.batch, "steps": n, "window_steps": win,
                       "context_start": w.prompt, "context_end": w.prompt + n},
            "h2d_peak_gbs": round(peak_h2d, 2), "windows": windows, "wall_s": round(wall, 1),
            "note": "link_time_frac = host bytes per step / measured pinned-copy peak / median "
                    "step time: the share of a step the recall alone needs on the host link"}


def run_trace(args, rank, world, local_rank):
    """Timeline of isolated decode steps from the library's step trace
    (NOSA_TRACE=1): after the warm-up, `args.trace` steps each followed by a
    synchronisation; per traced launch the first CTA's start and the last CTA's
    end (us from the step's first start), and the step's host bytes."""
    os.environ["NOSA_TRACE"] = "1"
    import numpy as np
    import torch
    import synth
    import synth.gpu
    import trainable_sparse_attention_decode_gb300 as nosa
    torch.cuda.set_device(local_rank)
    w = synth.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(batch=args.batch)
    n = args.warmup + args.trace
    w = w.with_(steps=n + 1)
    cfg = nosa.nosa_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.dtype, w.k, w.k_e,
                           w.max_context, device=local_rank)
    h = nosa.nosa_create(cfg)
    t = 0
    while t < w.prompt:
        m = min(4096, w.prompt - t)
        k, v, e = synth.gpu.kv(w, t, m)
        nosa.nosa_append_kv(h, k, v, e)
        t += m
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device="cuda")
    if args.frontend:  # steps from hidden states: the first kernel is the fused front-end
        D = synth.hidden_width(w)
        Wf = nosa.nosa_frontend_pack(cfg, synth.gpu.proj_weights(w, D))
        x = synth.gpu.hidden(w, w.prompt, n, D)
        step = lambda s_: nosa.nosa_decode_step_hidden(h, x[s_], Wf, out, None)
    else:
        q = synth.gpu.queries(w, n)
        kk, vv, ee = synth.gpu.kv(w, w.prompt, n, step_major=True)
        step = lambda s_: nosa.nosa_decode_step(h, q[s_], kk[s_], vv[s_], ee[s_], out)
    for s_ in range(args.warmup):
        step(s_)
    names = {0: "front-end" if args.frontend else "append", 41: "front-end main loop done",
             42: "front-end epilogue done", 43: "chunk 0 selection begins",
             44: "chunk 0 selection done", 45: "chunk 0 Gamma_e done",
             46: "chunk 0 Gamma_q done", 47: "chunk 0 lists written"}
    for c in range(8):
        names.update({1 + c: f"score+select {c}", 9 + c: f"select {c}", 17 + c: f"gather {c}",
                      25 + c: f"attention kept {c}", 33 + c: f"attention filled {c}"})
    steps = []
    for s_ in range(args.warmup, n):
        hb0 = nosa.nosa_stats(h)["host_bytes"]
        step(s_)
        torch.cuda.synchronize()
        hb = nosa.nosa_stats(h)["host_bytes"] - hb0
        tr = np.frombuffer(nosa.nosa_debug_read(h, "TRACE").tobytes(), np.uint64).reshape(-1, 2)
        used = [i for i in range(tr.shape[0]) if int(tr[i, 0]) != 0xFFFFFFFFFFFFFFFF]
        t0 = min(int(tr[i, 0]) for i in used)
        launches = sorted(((names.get(i, f"slot {i}"), round((int(tr[i, 0]) - t0) / 1e3, 1),
                            round((int(tr[i, 1]) - t0) / 1e3, 1)) for i in used), key=lambda x: x[1])
        steps.append({"step": s_, "span_us": max(x[2] for x in launches), "host_bytes": hb,
                      "launches": launches})
    nosa.nosa_destroy(h)
    line = {"mode": "trace" + ("+frontend" if args.frontend else ""),
            "config": {"workload": w.name, "batch": w.batch}, "steps": steps}
    if args.frontend:
        # the front-end kernel's own span (first CTA start to last CTA end) per
        # traced step, and its rate on the algorithmic bytes of one launch
        us = [dict((x[0], x[2] - x[1]) for x in st["launches"])["front-end"] for st in steps]
        phases = []
        for st in steps:
            at = {x[0]: (x[1], x[2]) for x in st["launches"]}
            f0 = at["front-end"][0]
            phases.append({k.replace("front-end ", ""): [round(a - f0, 1), round(b - f0, 1)]
                           for k, (a, b) in at.items() if k.startswith("front-end ")})
        nbytes = frontend_bytes_per_launch(w, synth.hidden_width(w))
        peak, kind = measured_peaks()
        med = float(np.median(us))
        line["frontend"] = {"kernel_us": us, "median_us": med, "bytes": nbytes,
                            "phases_us (earliest, latest CTA)": phases,
                            "hbm_gbs": round(nbytes / (med * 1e-6) / 1e9, 1),
                            "frac_of_" + kind + "_peak": round(nbytes / (med * 1e-6) / 1e9 / peak, 4)}
    return line


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def _oracle_proc(workload, units, warm, steps, batch, barrier, out_q):
    """One process of the oracle pool: builds its units (prompt appended, the
    step inputs generated), runs `warm` untimed decode steps, waits for the other
    processes, then times `steps` decode steps of all its units in lock-step."""
    import synth
    from oracle import nosa_oracle as O
    try:
        w = synth.WORKLOADS[workload]
        if batch:
            w = w.with_(batch=batch)
        w = w.with_(steps=max(w.steps, warm + steps))
        G = w.group
        state = []
        for u in units:
            b, h = divmod(u, w.n_kv_heads)
            uo = O.UnitOracle(w.head_dim, w.dtype, w.k, w.k_e, w.max_context, w.block, w.sub_block)
            uo.append(synth.keys(w, b, h, 0, w.prompt), synth.values(w, b, h, 0, w.prompt),
                      synth.evict(w, b, h, 0, w.prompt))
            q = synth.queries(w, b, range(h * G, (h + 1) * G), warm + steps)
            kk = synth.keys(w, b, h, w.prompt, warm + steps)
            vv = synth.values(w, b, h, w.prompt, warm + steps)
            ee = synth.evict(w, b, h, w.prompt, warm + steps)
            state.append((uo, q, kk, vv, ee))
        for s in range(warm):
            for uo, q, kk, vv, ee in state:
                uo.decode_step(q[s], kk[s], vv[s], ee[s])
        barrier.wait()
        t0 = time.perf_counter()
        for s in range(warm, warm + steps):
            for uo, q, kk, vv, ee in state:
                uo.decode_step(q[s], kk[s], vv[s], ee[s])
        out_q.put(("ok", time.perf_counter() - t0))
    except Exception as exc:  # reported to the parent, which prints the reason
        out_q.put(("error", repr(exc)))
        try:
            barrier.abort()
        except Exception:
            pass


def oracle_timing(workload, units, warm, steps, batch=0, procs=None):
    """Times the fp64 oracle on the host cores: `units` split over `procs` spawned
    processes (default: every core; BLAS pinned to one thread each), `warm`
    untimed steps, then `steps` timed ones. Returns (seconds of the timed steps,
    the slowest process; processes used)."""
    import multiprocessing as mp
    procs = min(procs or os.cpu_count() or 1, len(units))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                            "MKL_NUM_THREADS")}
    os.environ.update({k: "1" for k in saved})
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(procs)
    out_q = ctx.Queue()
    ps = [ctx.Process(target=_oracle_proc,
                      args=(workload, units[i::procs], warm, steps, batch, barrier, out_q))
          for i in range(procs)]
    try:
        for p_ in ps:
            p_.start()
        res = [out_q.get(timeout=3000) for _ in ps]
    finally:
        for p_ in ps:
            p_.join(timeout=60)
            if p_.is_alive():
                p_.kill()
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    errs = [r[1] for r in res if r[0] != "ok"]
    if errs:
        raise RuntimeError("oracle process failed: " + errs[0])
    return max(r[1] for r in res), procs


def cpu_baseline(workload, batch=0, n_units=64, steps=20):
    """The oracle on all host cores over a bounded sample of the workload's units
    (spread over the batch), scaled to the whole batch."""
    import synth
    w = synth.WORKLOADS[workload]
    if batch:
        w = w.with_(batch=batch)
    n_units = min(n_units, w.units)
    units = [i * w.units // n_units for i in range(n_units)]
    try:
        secs, procs = oracle_timing(workload, units, 1, steps, batch)
    except Exception as exc:
        return {"value": None, "unit": "tokens/s", "kind": "oracle", "error": str(exc)[:200]}
    per_step_batch = secs / steps * w.units / n_units
    return {"value": round(w.batch / per_step_batch, 4), "unit": "tokens/s", "cores": procs,
            "kind": "oracle",
            "sample": f"{n_units} of {w.units} units x {steps} decode steps (after 1 untimed step), "
                      f"{procs} processes (one per core, BLAS one thread each), scaled to the full "
                      f"batch; fp64 numpy"}


def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle times the whole batch of the workload on
    every host core: W untimed decode steps (the first is the cold step), then
    exactly K timed ones; rank 0 only."""
    if rank != 0:
        return None
    import synth
    w = synth.WORKLOADS[args.workload].with_(q_stationary=not args.q_innovation_start)
    if args.batch:
        w = w.with_(name=f"{w.name}-b{args.batch}", batch=args.batch)
    K, W = args.steps, args.warmup
    units = list(range(w.units))
    t0 = time.time()
    try:
        secs, procs = oracle_timing(args.workload, units, W, K, args.batch)
    except Exception as exc:
        return {"impl": "reference", "unavailable": "oracle pool failed: " + str(exc)[:200]}
    wall = time.time() - t0
    value = w.batch * K / secs
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(secs / K * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": arm_config(w, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": procs,
                             "kind": "oracle",
                             "sample": f"the whole batch ({w.units} units) x {K} timed decode "
                                       f"steps after {W} untimed, {procs} processes"},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 1)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="nosa", choices=["nosa", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", default="nosa", choices=["nosa", "infllmv2", "fullattn", "prefill"],
                    help="nosa (the method); comparators: infllmv2 = k_e 0 (no query-agnostic "
                         "part), fullattn = dense attention over the whole cache in HBM; "
                         "prefill = the training-time forward over whole sequences "
                         "(--prompt sets the length, default 32768)")
    ap.add_argument("--attention-only", action="store_true",
                    help="time only the split-K attention on the step shape (profiling aid)")
    ap.add_argument("--classic", action="store_true",
                    help="with --attention-only: the classic split the decode step launches "
                         "(attn_split_kernel) instead of the standalone plan")
    ap.add_argument("--pooled-bf16", action="store_true",
                    help="variant: pooled keys stored in bf16 (halves the scoring traffic)")
    ap.add_argument("--frontend", action="store_true",
                    help="steps start from hidden states: the fused front-end (projection on the "
                         "tensor cores + QKV split + append and pooling) runs first")
    ap.add_argument("--no-timing", action="store_true",
                    help="skip the per-phase timing window")
    ap.add_argument("--phase-steps", type=int, default=64,
                    help="decode steps of the per-phase timing window (after the timed loops)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch")
    ap.add_argument("--hbm-budget", type=float, default=0.0,
                    help="GB of HBM for the GPU-resident state: the batch is the largest that "
                         "fits (fullattn: the whole cache; nosa/infllmv2: the handle's state)")
    ap.add_argument("--host-budget", type=float, default=96.0,
                    help="GB of pinned host memory the host store may take (with --hbm-budget)")
    ap.add_argument("--trace", type=int, default=0,
                    help="print the launch timeline of this many isolated decode steps after "
                         "the warm-up (the library's step trace)")
    ap.add_argument("--horizon", type=int, default=0,
                    help="run the workload's whole decode horizon and report this many "
                         "windows along it (tokens/s, recall, locality)")
    ap.add_argument("--prompt", type=int, default=0, help="override the workload's prompt")
    ap.add_argument("--q-innovation-start", action="store_true",
                    help="AR(1) queries from q_0 = eps_0 instead of their stationary distribution")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.attention_only:
        # Profiling aid: only the split-K attention on the workload's step shape,
        # inside an NVTX range "attention" (for ncu --nvtx-include attention/).
        import torch
        import synth
        import trainable_sparse_attention_decode_gb300 as nosa
        torch.cuda.set_device(local_rank)
        w = synth.WORKLOADS[args.workload]
        if args.batch:
            w = w.with_(batch=args.batch)
        n_cand = w.prompt // w.block
        torch.cuda.nvtx.range_push("attention")
        secs, nbytes = attention_alone(nosa, torch, w, n_cand, 33, reps=args.steps,
                                       classic=args.classic)
        torch.cuda.nvtx.range_pop()
        peak, kind = measured_peaks()
        print(json.dumps({"attention_alone_us": round(secs * 1e6, 2), "bytes": nbytes,
                          "gbs": round(nbytes / secs / 1e9, 1),
                          "frac_of_" + kind + "_peak": round(nbytes / secs / 1e9 / peak, 4)}))
        return
    if args.trace:
        line = run_trace(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.horizon:
        line = run_horizon(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.mode in ("fullattn", "prefill"):
        line = (run_fullattn if args.mode == "fullattn" else run_prefill)(args, rank, world,
                                                                           local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    line = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(args.workload, args.batch)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark: µs per split-KV decode-attention call on one GB300 (or N replicas).

Default workload: long single-stream GQA decode -- batch 1, one query token,
16 query / 2 KV heads, head dim 128, context 5,900, BF16 KV in 16-token pages
behind a shuffled block table, split count chosen by the planner.  ("vLLM
0.30.0 FA4 SplitKV Bug: H100 Decode Can Be 48% Slower": the ~5.9k-context
global-layer decode with two KV heads.)

Protocol
  * One step = one ``splitkv_decode`` call (all kernels of the path) over one
    batch.  Steps are captured in CUDA graphs and replayed; the timed region
    is bracketed by a barrier and ``torch.cuda.synchronize()`` and timed with
    CUDA events on the launching stream.
  * The KV inputs rotate over R copies of the page pool whose total exceeds 4x
    the L2 size, so no step starts with its pages in L2.
  * ``value`` = timed-region time / steps (whole-job: / (steps x ranks)).
  * ``roofline``: algorithmic bytes of one launch of the split-KV kernel (KV
    bytes of the visible keys + Q bytes) / its average launch duration,
    against the measured HBM copy bandwidth.  With the fused combine the
    kernel is the only launch of a step, so its average duration is taken as
    timed-region time / launches (this includes inter-launch gaps and so
    understates the kernel's own bandwidth).
  * ``e2e``: the same call with host buffers -- pinned-host -> device copies
    of every input, the decode, and device -> host copies of out and lse,
    all inside the timed region.
  * ``cpu_baseline``: the fp64 oracle, single-threaded, on a bounded sample.
  * Clocks: ``nvidia-smi`` samples every 200 ms while the same work runs
    (a >= 1 s soak immediately followed by the timed region).

``--impl reference`` times the fp64 CPU oracle on the same workload (the
reference arm: the pages ship no code of their own).
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "µs per decode-attention call; achieved HBM GB/s as fraction of GB300 peak"
NOMINAL_HBM_GBS = 8000.0  # the "about 8 TB/s" HBM figure the metric also reports against

# DRAM bytes (read + write) of one launch of each workload's dominant kernel,
# from the ncu captures summarised under profiles/.  An entry is removed
# whenever that kernel changes after its capture.
PROFILED_TRAFFIC = {
    "gqa_ctx5900": (6115328, "profiles/gqa_splitkv_kernel_gqa_ctx5900.md"),
    "fp8_batch8_ctx32k": (253606400, "profiles/gqa_splitkv_kernel_fp8_batch8_ctx32k.md"),
    "mla_t6_ctx64k": (79173632, "profiles/mla_splitkv_kernel_mla_t6_ctx64k.md"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa_ctx5900", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--splits", type=int, default=0, help="num_splits (0 = planner)")
    ap.add_argument("--fixed", action="store_true",
                    help="capacity plan whose kernels derive the items from the device "
                         "lengths every step (needs --splits)")
    ap.add_argument("--combine", default="separate", choices=["fused", "separate"])
    ap.add_argument("--page-size", type=int, default=0,
                    help="page size in keys (0 = the workload's own)")
    ap.add_argument("--layout", default="hnd", choices=["hnd", "nhd"],
                    help="page layout of the KV pools: [N][Hkv][P][D] or [N][P][Hkv][D]")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=1.5)
    return ap.parse_args()


# ----------------------------------------------------------------- distributed

def dist_init(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- helpers

def algorithmic_bytes(w: workloads.Workload, lens: np.ndarray) -> int:
    """KV bytes of the visible keys plus Q bytes of one call."""
    elt = 1 if w.kv_dtype == "fp8_e4m3" else 2
    row = w.qk_dim * elt + (0 if w.v_shares_k else w.v_dim * elt)
    kv = int(lens.astype(np.int64).sum()) * w.num_kv_heads * row
    q = w.batch * w.q_tokens * w.num_q_heads * w.qk_dim * 2
    return kv + q


def algorithmic_flops(w: workloads.Workload, lens: np.ndarray) -> float:
    """Multiply-add FLOPs of QK^T and PV over the visible keys of one call
    (query token t of a sequence of length L sees L - T + 1 + t keys)."""
    vis = 0
    for L in lens.astype(np.int64):
        for t in range(w.q_tokens):
            vis += max(0, int(L) - w.q_tokens + 1 + t)
    return 2.0 * w.num_q_heads * vis * (w.qk_dim + w.v_dim)


def is_tensor_bound(w: workloads.Workload) -> bool:
    """The MLA shape (128 heads x T tokens on one latent head) is a dense
    contraction (about 1,450 FLOP per KV byte); the GQA shapes stream KV."""
    return w.num_kv_heads == 1 and w.num_q_heads >= 64 and w.qk_dim > w.v_dim


def measured_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, kind)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows),
                "power_w_max": max(r["power"] for r in rows),
                "samples": len(rows), "reasons": sorted(reasons)}


def time_oracle(w, x, seconds, threads=1, calls=0, warmup=0):
    """Runs the oracle on the full call in a clean single-threaded subprocess:
    `warmup` untimed calls, then exactly `calls` timed ones, or (calls = 0)
    timed ones until `seconds` have passed (at least one); returns (µs per
    call, timed calls)."""
    import pickle
    payload = dict(q=workloads.bits(x.q), k=workloads.bits(x.k_pages),
                   v=None if x.v_pages is None else workloads.bits(x.v_pages),
                   table=x.block_table.cpu().numpy(), lens=x.seq_lens_host, scale=x.scale,
                   kv_dtype=w.kv_dtype, kv_scale=x.kv_scale, v_dim=w.v_dim,
                   v_shares_k=w.v_shares_k, seconds=seconds, calls=calls, warmup=warmup)
    with tempfile.NamedTemporaryFile(suffix=".pkl", delete=False) as f:
        pickle.dump(payload, f)
        path = f.name
    code = (
        "import pickle, sys, time, json\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import oracle\n"
        f"d = pickle.load(open({path!r}, 'rb'))\n"
        "def call():\n"
        "    oracle.attention_direct(d['q'], d['k'], d['v'], d['table'], d['lens'], scale=d['scale'],\n"
        "        kv_dtype=d['kv_dtype'], kv_scale=d['kv_scale'], v_dim=d['v_dim'], v_shares_k=d['v_shares_k'])\n"
        "for _ in range(d['warmup']): call()\n"
        "n = 0; t0 = time.perf_counter()\n"
        "while True:\n"
        "    call()\n"
        "    n += 1\n"
        "    if n == d['calls'] or (not d['calls'] and time.perf_counter() - t0 >= d['seconds']): break\n"
        "print(json.dumps({'us': (time.perf_counter() - t0) / n * 1e6, 'n': n}))\n")
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    os.unlink(path)
    if r.returncode != 0:
        raise RuntimeError(r.stderr)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d["us"], d["n"]


def oracle_sample_desc(w, n):
    return (f"fp64 oracle (numpy, 1 thread) on the full {w.name} call "
            f"({w.batch} seq x {w.num_q_heads} q heads x {w.lens} keys), repeated {n} times")


# ----------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    if args.page_size:
        w = dataclasses.replace(w, page_size=args.page_size)
    x = workloads.make_inputs(w, device="cpu")
    # Each step is one full oracle call; the run is bounded by --cpu-seconds
    # (so at most --steps calls, at least one).
    per_call, _ = time_oracle(w, x, 0.0)
    steps = max(1, min(args.steps, int(args.cpu_seconds * 1e6 / max(per_call, 1.0))))
    warm = max(1, min(args.warmup, steps))
    us, n = time_oracle(w, x, 0.0, calls=steps, warmup=warm)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us", "n_gpus": args.gpus,
        "steps": n, "warmup": warm, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "page_size": w.page_size},
        "cpu_baseline": {"value": us, "unit": "us", "cores": 1, "kind": "oracle",
                         "sample": oracle_sample_desc(w, n)},
        "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import split_kv_paged_splitkv_gb300 as skv
    from split_kv_paged_splitkv_gb300.runner import DecodeSession

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    if args.page_size:
        w = dataclasses.replace(w, page_size=args.page_size)
    x = workloads.make_inputs(w, device=dev, layout=args.layout.upper())
    mode = skv.SPLITKV_COMBINE_FUSED if args.combine == "fused" else skv.SPLITKV_COMBINE_SEPARATE
    # Everything runs on torch's current stream: graphs are captured on a side
    # stream by torch.cuda.graph and replayed on the current stream.
    if args.fixed and args.splits < 1:
        raise SystemExit("--fixed needs --splits >= 1")
    sess = DecodeSession(x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens, x.seq_lens_host,
                         scale=x.scale, kv_scale=x.kv_scale, num_splits=args.splits,
                         v_dim=w.v_dim, v_shares_k=w.v_shares_k, combine_mode=mode,
                         fixed=args.fixed,
                         kv_layout=skv.SPLITKV_LAYOUT_NHD if args.layout == "nhd" else skv.SPLITKV_LAYOUT_HND)
    items = skv.splitkv_plan_get_items(sess.plan)
    n_groups = len(np.unique(items[items[:, 3] > 1][:, 7])) if len(items) else 0
    launches_per_step = skv.splitkv_plan_launches_per_call(sess.plan)

    # rotating KV pools: total > 4x L2
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    pool_bytes = x.k_pages.numel() * x.k_pages.element_size() + (
        0 if x.v_pages is None else x.v_pages.numel() * x.v_pages.element_size())
    R = max(2, min(256, math.ceil(4 * l2 / pool_bytes)))
    pools = [(x.k_pages.clone(), None if x.v_pages is None else x.v_pages.clone()) for _ in range(R - 1)]
    pools.insert(0, (x.k_pages, x.v_pages))

    def step(i):
        k, v = pools[i % R]
        sess.run(tensors=(x.q, k, v, x.block_table, x.seq_lens))

    # eager warm-up (also sets up per-process kernel attributes before capture)
    for i in range(max(3, min(args.warmup, R))):
        step(i)
    torch.cuda.synchronize()
    log, status = sess.stats()
    assert status == 0, f"device status {status}"
    nonempty = float((log[:, 2] > 0).mean()) if len(log) else 1.0

    def capture(n, start):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                step(start + i)
        return g

    cycle = capture(R, 0)
    K = args.steps
    reps, rem = divmod(K, R)
    tail = capture(rem, 0) if rem else None

    # graph warm-up + clock soak (same work), then the timed region
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(max(1, math.ceil(args.warmup / R))):
        cycle.replay()
    torch.cuda.synchronize()
    t_end = time.perf_counter() + args.soak_seconds
    while time.perf_counter() < t_end:
        for _ in range(20):
            cycle.replay()
        torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    # The split-KV kernel alone (splitkv_decode_partials, the first launch of
    # each call), timed the same way on the same stream: its average launch
    # duration is the roofline's denominator.  With the fused combine the
    # split kernel is the step's only launch and the step time is used.
    kernel_us = None
    if args.combine == "separate":
        def step_partials(i):
            k, v = pools[i % R]
            sess.run_partials(tensors=(x.q, k, v, x.block_table, x.seq_lens))

        pg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pg):
            for i in range(R):
                step_partials(i)
        for _ in range(3):
            pg.replay()
        torch.cuda.synchronize()
        p_reps = max(1, min(max(1, K // R), math.ceil(2000 / R)))
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(p_reps):
            pg.replay()
        p1.record(stream)
        p1.synchronize()
        kernel_us = p0.elapsed_time(p1) * 1e3 / (p_reps * R)
        del pg

    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        cycle.replay()
    if tail is not None:
        tail.replay()
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms_local = e0.elapsed_time(e1)
    ms = max_over_ranks(ms_local, world)
    us_per_call_local = ms_local * 1e3 / K
    value = ms * 1e3 / (K * world)

    log, status = sess.stats()
    assert status == 0, f"device status {status} after the timed region"

    # roofline of the split-KV kernel
    nbytes = algorithmic_bytes(w, x.seq_lens_host)
    nflops = algorithmic_flops(w, x.seq_lens_host)
    hbm_peak, tc_peak, peak_kind = measured_peaks()
    launch_us = kernel_us if kernel_us is not None else us_per_call_local
    if is_tensor_bound(w):
        roof = {"bound": "tensor", "achieved": nflops / (launch_us * 1e-6) / 1e12, "peak": tc_peak,
                "unit": "TFLOP/s", "algorithmic_flops": nflops,
                "hbm_gbs": nbytes / (launch_us * 1e-6) / 1e9, "kernel": "mla_splitkv_kernel"}
    else:
        achieved = nbytes / (launch_us * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac_of_8tbs": achieved / NOMINAL_HBM_GBS, "kernel": "gqa_splitkv_kernel"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # the captures ran the default configuration (planner splits, separate
    # combine, host plan, HND pages); other configurations report no traffic
    default_cfg = (args.splits == 0 and not args.fixed and args.combine == "separate"
                   and args.layout == "hnd"
                   and args.page_size in (0, workloads.WORKLOADS[args.workload].page_size))
    traffic, traffic_src = PROFILED_TRAFFIC.get(w.name, (None, None)) if default_cfg else (None, None)
    roof.update({"traffic": traffic, "traffic_source": traffic_src,
                 "duration_basis": ("split-KV kernel alone (splitkv_decode_partials), CUDA-graph "
                                    "replay, CUDA events on the launching stream"
                                    if kernel_us is not None else
                                    "timed-region time per call (the split kernel is the only launch)"),
                 "kernel_us": launch_us, "step_us": us_per_call_local,
                 "peak_kind": peak_kind, "algorithmic_bytes": nbytes})

    # cold calls: L2 flushed (a buffer of twice its size written) before each
    # call, events around the call only; the median of a few, for context
    cold_us = run_cold(x, sess, l2, stream)

    # end to end: host buffers, copies inside the timed region
    e2e = run_e2e(args, x, sess, dev)

    line = {
        "metric": METRIC, "value": value, "unit": "us", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == "bf16" else "f16",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "q_tokens": w.q_tokens,
                   "heads_q_kv": [w.num_q_heads, w.num_kv_heads], "head_dim": w.qk_dim,
                   "context": w.lens, "page_size": w.page_size, "kv_dtype": w.kv_dtype,
                   "kv_layout": args.layout.upper(),
                   "num_splits": args.splits, "planned_items": int(len(items)),
                   "plan": "capacity plan, items derived from the device lengths each step" if args.fixed else "host",
                   "combine": args.combine, "parallelism": f"replicas{world}",
                   "l2": f"inputs rotate over {R} KV pools ({R * pool_bytes / 2**20:.0f} MiB > 4x L2 {l2 / 2**20:.0f} MiB)",
                   "timing": "CUDA-graph replay of back-to-back calls, CUDA events on the launching stream"},
        "roofline": roof,
        "nonempty_cta_fraction": nonempty,
        "cold_us_per_call": cold_us,
        "gpu_launches": K * launches_per_step,
        "e2e": e2e,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        us, n = time_oracle(w, x, args.cpu_seconds)
        line["cpu_baseline"] = {"value": us, "unit": "us", "cores": 1, "kind": "oracle",
                                "sample": oracle_sample_desc(w, n)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_cold(x, sess, l2, stream, n=30):
    """Median device µs of single calls that each start with a cold L2 (a
    buffer of twice its size is written between calls).  The call is a
    one-call CUDA graph, so the events time the GPU work, not the host's
    enqueueing of an eager call."""
    flush = torch.empty(2 * l2 // 4, dtype=torch.int32, device=x.q.device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sess.run()
    times = []
    for _ in range(n):
        flush.fill_(1)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    del flush, g
    return float(np.median(times))


def run_e2e(args, x, sess, dev):
    """Pinned host inputs -> device, decode, out/lse -> pinned host, every step.

    The inputs are double-buffered on the device: step i + 1's host-to-device
    copies run on a copy stream while step i decodes on the compute stream
    (events order each buffer's reuse), and every step's out/lse are copied
    back to pinned host memory on the compute stream.  The steps are captured
    in a CUDA graph (copies, kernels and read-backs alike) and replayed, as a
    serving loop would; the timed region starts before the first copy and
    ends after the last read-back.
    """
    host_in = [t.cpu().pin_memory() for t in (x.q, x.k_pages, x.v_pages, x.block_table, x.seq_lens)
               if t is not None]
    dev_in = [[torch.empty_like(t, device=dev) for t in host_in] for _ in range(2)]
    out_h = torch.empty(sess.out.shape, dtype=sess.out.dtype).pin_memory()
    lse_h = torch.empty(sess.lse.shape, dtype=sess.lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    copy = torch.cuda.Stream(device=dev)

    def steps(n):
        compute = torch.cuda.current_stream()
        copied = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        copy.wait_stream(compute)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(free[b])  # decode i - 2 has read this buffer
                for d, h in zip(dev_in[b], host_in):
                    d.copy_(h, non_blocking=True)
                copied[b].record(copy)
            compute.wait_event(copied[b])
            if x.v_pages is None:
                q, k, table, lens = dev_in[b]
                v = None
            else:
                q, k, v, table, lens = dev_in[b]
            out, lse = sess.run(tensors=(q, k, v, table, lens))
            free[b].record(compute)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        compute.wait_stream(copy)

    steps(3)  # eager warm-up
    torch.cuda.synchronize()
    n_cap = max(1, min(args.e2e_steps, 16))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        steps(n_cap)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, math.ceil(args.e2e_steps / n_cap))
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    n = reps * n_cap
    us = e0.elapsed_time(e1) * 1e3 / n
    return {"value": us, "unit": "us", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": n,
            "note": "CUDA-graph replay of the steps; inputs double-buffered on the device, "
                    "step i+1's host-to-device copies overlap step i's decode"}


def main():
    args = parse()
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

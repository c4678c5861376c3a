"""Benchmark: split-KV paged decode attention on GB300.

A step is one call of the whole path (partial kernel + combine kernel, through the C
ABI) over one batch of synthetic inputs already resident in HBM. The default workload
is the batch-200 x 200,000-token MTP4 FP8 paged decode (Hq16/Hkv1/D128, block 16), the
configuration whose effective bandwidth the pages report ("[FlyDSL] perf(pa_decode):
tune MTP work budgets and planned reduction", Performance table).

value = effective TB/s over all ranks: logical bytes (query and output, KV and scales
of every visible token, referenced page-table entries and context lengths, counted
once; same paper, the paragraph under the table) / device time per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
Under torchrun each rank runs its own batch (weak scaling); rank 0 prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from split_kv_paged_gb300 import workloads as W  # noqa: E402

METRIC = "µs/call + effective HBM TB/s (% of GB300 peak), split-KV paged decode attention"
UNIT = "TB/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mtp4_fp8_long", choices=sorted(W.ALL_WORKLOADS))
    ap.add_argument("--kernel", default="auto", choices=["auto", "generic", "simt", "tc_fp8", "tc_i8", "tc_b16"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="shrink the batch (profiling a smaller case)")
    ap.add_argument("--ctx", type=int, default=0, help="override every context length (profiling)")
    ap.add_argument("--bs", type=int, default=0, help="override the block size (profiling)")
    ap.add_argument("--splits", type=int, default=0, help="override the planner's split count (0: plan it)")
    ap.add_argument("--record", default="f32", choices=["f32", "bf16", "f16"], help="split-record element type")
    ap.add_argument("--v-layout", default="token_major", choices=["token_major", "dim_major"],
                    help="V cache layout of the timed workload (dim_major: [pages, Hkv, D, bs])")
    ap.add_argument("--no-other-configs", action="store_true", help="time only the headline workload")
    ap.add_argument("--other-steps", type=int, default=50, help="timed replays of each other workload")
    return ap.parse_args()


def workload(args):
    wl = W.ALL_WORKLOADS[args.workload]()
    ctx = list(wl.ctx)
    if args.batch > 0:
        ctx = (ctx * ((args.batch + len(ctx) - 1) // len(ctx)))[:args.batch]
    if args.ctx > 0:
        ctx = [args.ctx] * len(ctx)
    if ctx != wl.ctx:
        wl = wl.replace(ctx=ctx, name=f"{wl.name}_b{len(ctx)}_ctx{max(ctx)}")
    if args.bs > 0 and args.bs != wl.bs:
        wl = wl.replace(bs=args.bs, name=f"{wl.name}_bs{args.bs}")
    return wl


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def rank_seed(rank: int) -> int:
    """Input seed of a rank: every rank draws its own batch (weak scaling, no shared data)."""
    return 1003 + 7919 * rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over the ranks (the slowest rank sets the job's time); x itself for one
    rank. A collective: every rank calls it with its own value."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tbps(nbytes_per_rank: int, world: int, ms: float) -> float:
    """Whole-job effective TB/s: the logical bytes all ranks processed over the job's time."""
    return nbytes_per_rank * world / (ms * 1e-3) / 1e12


# DRAM traffic of the dominant kernel, from the record written next to its ncu capture: valid
# only while the kernel's sources hash to the value recorded with the capture.
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "traffic_record.json")


def source_hash(sources):
    import hashlib
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "split_kv_paged_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(kernel, workload_name, nbytes):
    """Bytes read + written by one partial launch (ncu's dram__bytes_read.sum +
    dram__bytes_write.sum), scaled from the recorded traffic / algorithmic ratio; None when the
    kernel, the workload or the kernel sources differ from the capture."""
    from split_kv_paged_gb300 import binding as B
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    names = {"partial_tc_fp8": B.TLLM_KERNEL_TC_FP8}
    if names.get(rec.get("kernel")) != kernel or rec.get("workload") != workload_name:
        return None
    if source_hash(rec["sources"]) != rec.get("source_sha256"):
        return None
    return float(rec["traffic_over_algorithmic"]) * nbytes


def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            c = [x.strip() for x in ln.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                mx = float(c[2])
            except ValueError:
                continue
            for name, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def kernel_code(name):
    from split_kv_paged_gb300 import binding as B
    return {"auto": B.TLLM_KERNEL_AUTO, "generic": B.TLLM_KERNEL_GENERIC, "simt": B.TLLM_KERNEL_SIMT, "tc_i8": B.TLLM_KERNEL_TC_I8,
            "tc_fp8": B.TLLM_KERNEL_TC_FP8, "tc_b16": B.TLLM_KERNEL_TC_B16}[name]


def cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_sample(wl, seed, budget_s, device_inp=None):
    """Time the CPU oracle on a bounded sample of ``wl``: the first n requests (or one
    request truncated to T tokens), sized to about ``budget_s`` seconds. Returns
    (TB/s, seconds, description, threads)."""
    import oracle
    oracle.build()
    nthreads = cores()

    def sample_inputs(ctx_list):
        sub = wl.replace(ctx=ctx_list)
        if device_inp is not None and len(ctx_list) <= wl.B and ctx_list == wl.ctx[:len(ctx_list)]:
            return W.gather_requests(device_inp, list(range(len(ctx_list)))).to("cpu")
        return W.make_inputs(sub, seed, device="cpu")

    def run(ctx_list):
        h = sample_inputs(ctx_list)
        t = time.perf_counter()
        oracle.attention(h.q, h.k_cache, h.v_cache, h.kv_scales, h.block_table, h.context_lens, h.sinks,
                         q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype, window=wl.window, scale=wl.scale or None,
                         nthreads=nthreads)
        dt = time.perf_counter() - t
        return dt, W.effective_bytes(wl.replace(ctx=ctx_list))

    # calibrate on a short slice of request 0, then size the sample to the budget
    c0 = min(wl.ctx[0], 4096)
    dt, _ = run([c0])
    per_token = dt / max(1, c0)
    tokens = max(1, int(budget_s / max(per_token, 1e-9)))
    ctx_list = []
    for c in wl.ctx:
        if tokens <= 0:
            break
        if c <= tokens:
            ctx_list.append(c)
            tokens -= c
        else:
            if not ctx_list:
                ctx_list.append(max(1, tokens))
            break
    dt, nbytes = run(ctx_list)
    desc = (f"oracle over {len(ctx_list)} of {wl.B} requests ({sum(ctx_list)} tokens of "
            f"{sum(wl.ctx)}), {nthreads} threads")
    return nbytes / dt / 1e12, dt, desc, nthreads, nbytes


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, each step a bounded sample."""
    if rank != 0:
        return
    wl = workload(args)
    import oracle
    oracle.build()
    steps, warm = args.steps, args.warmup
    per_step_budget = max(0.2, 150.0 / max(1, steps + warm))
    # sample: request 0 truncated so that one step takes about per_step_budget
    c0 = min(wl.ctx[0], 2048)
    sub = wl.replace(ctx=[c0])
    h = W.make_inputs(sub, 1000 + 3, device="cpu")
    t = time.perf_counter()
    oracle.attention(h.q, h.k_cache, h.v_cache, h.kv_scales, h.block_table, h.context_lens, h.sinks,
                     q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype, window=wl.window, scale=wl.scale or None,
                     nthreads=cores())
    per_tok = (time.perf_counter() - t) / c0
    T = int(min(wl.ctx[0], max(256, per_step_budget / max(per_tok, 1e-9))))
    sub = wl.replace(ctx=[T])
    h = W.make_inputs(sub, 1000 + 3, device="cpu")
    nbytes = W.effective_bytes(sub)

    def step():
        oracle.attention(h.q, h.k_cache, h.v_cache, h.kv_scales, h.block_table, h.context_lens, h.sinks,
                         q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype, window=wl.window, scale=wl.scale or None,
                         nthreads=cores())
    for _ in range(warm):
        step()
    t = time.perf_counter()
    for _ in range(steps):
        step()
    dt = (time.perf_counter() - t) / steps
    value = nbytes / dt / 1e12
    sample = f"request 0 of {wl.name} truncated to {T} tokens ({nbytes} logical bytes) per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.B, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class Measured:
    """One workload on the device: its inputs, plan, workspace and output, and CUDA-graph
    timings of the whole call, the partial kernel alone and the combine kernel alone.

    Each timed unit is one call captured as a CUDA graph and replayed ("[FlyDSL]
    perf(pa_decode)", Performance: CUDA events around a graph of one call), so the host's
    launch work never sits between the events. Inputs smaller than twice the L2 would be
    served from L2 on the next step: then every timed replay is preceded (outside its events)
    by a write of a buffer twice the L2 size."""

    def __init__(self, wl, seed, dev, stream, kernel, splits=0, record="f32", v_dim_major=False):
        from split_kv_paged_gb300 import binding as B
        self.B = B
        self.wl, self.dev, self.stream = wl, dev, stream
        self.inp = W.make_inputs(wl, seed, device=dev)
        if v_dim_major:
            # the same V values, stored [pages, Hkv, D, bs]
            self.inp.v_cache = self.inp.v_cache.transpose(-1, -2).contiguous()
        rec = {"f32": B.TLLM_RECORD_F32, "bf16": B.TLLM_RECORD_BF16, "f16": B.TLLM_RECORD_F16}[record]
        vl = B.TLLM_V_DIM_MAJOR if v_dim_major else B.TLLM_V_TOKEN_MAJOR
        desc = B.desc_for(wl, kernel, num_pages=self.inp.num_pages, record_type=rec, v_layout=vl)
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        plan_args = (desc, wl.B, wl.Lq, wl.window)
        plan_kw = dict(host_ctx_lens=wl.ctx, num_sms=n_sm, splits_override=splits)
        self.plan = B.tllm_decode_attn_plan(*plan_args, **plan_kw)
        # host time of the planner (the call a serving loop makes when the shape changes)
        reps = 200
        t = time.perf_counter()
        for _ in range(reps):
            B.tllm_decode_attn_plan(*plan_args, **plan_kw)
        self.plan_us = (time.perf_counter() - t) / reps * 1e6
        self.ws = B.Workspace(self.plan, device=dev)
        self.out = torch.empty((wl.B, wl.Lq, wl.Hq, wl.D), dtype=W.DTYPES[wl.out_dtype], device=dev)
        self.S = self.plan.num_splits
        self.nbytes = W.effective_bytes(wl)
        l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0))
        self.flush_buf = None
        if self.nbytes < 2 * l2_bytes:
            self.flush_buf = torch.empty(2 * l2_bytes // 4, dtype=torch.int32, device=dev)
            self.l2_note = (f"inputs ({self.nbytes / 1e9:.3f} GB) smaller than 2x L2: L2 flushed by a "
                            f"{2 * l2_bytes >> 20} MiB write before every timed step")
        else:
            self.l2_note = f"inputs ({self.nbytes / 1e9:.2f} GB) larger than L2; no flush"
        inp = self.inp
        self.call = (inp.q, inp.k_cache, inp.v_cache, inp.block_table, inp.context_lens, wl.Lq, inp.kv_scales,
                     inp.sinks, wl.window, self.S, self.ws, self.out)

    def capture(self, warmup):
        B, stream = self.B, self.stream
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                B.tllm_decode_attn_splitkv(*self.call, stream=stream)
            torch.cuda.synchronize(self.dev)

            def graph(fn):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn()
                return g
            self.g_call = graph(lambda: B.tllm_decode_attn_splitkv(*self.call, stream=stream))
            self.g_part = graph(lambda: B.tllm_decode_attn_partial(*self.call, stream=stream))
            self.g_comb = graph(lambda: B.tllm_decode_attn_combine(*self.call, stream=stream)) if self.S > 1 else None
            for g in (self.g_call, self.g_part, self.g_comb):
                if g is not None:
                    for _ in range(max(1, warmup)):
                        g.replay()
            torch.cuda.synchronize(self.dev)

    def timed(self, g, K):
        """K replays of g. Returns (mean ms per replay over the K, median over three
        consecutive runs of K/3 replays of each run's mean ms)."""
        stream = self.stream
        with torch.cuda.stream(stream):
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for k in range(K):
                if self.flush_buf is not None:
                    self.flush_buf.fill_(k)
                ev[k][0].record(stream)
                g.replay()
                ev[k][1].record(stream)
            e1.record(stream)
            torch.cuda.synchronize(self.dev)
        per = [x.elapsed_time(y) for x, y in ev]
        mean = e0.elapsed_time(e1) / K if self.flush_buf is None else sum(per) / K
        runs = [per[i * K // 3:(i + 1) * K // 3] for i in range(3)] if K >= 3 else [per]
        med3 = statistics.median(sum(r) / len(r) for r in runs if r)
        return mean, med3

    def timed_pair(self, ga, gb, K):
        """K rounds of one replay of ga then one of gb, each timed alone (events around it, L2
        flushed before it when the inputs are small), so that clock changes during the run
        reach both alike. Returns the mean ms per replay of each."""
        stream = self.stream
        with torch.cuda.stream(stream):
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
            for k in range(K):
                for i, g in enumerate((ga, gb)):
                    if self.flush_buf is not None:
                        self.flush_buf.fill_(k)
                    ev[k][2 * i].record(stream)
                    g.replay()
                    ev[k][2 * i + 1].record(stream)
            torch.cuda.synchronize(self.dev)
        ta = sum(e[0].elapsed_time(e[1]) for e in ev) / K
        tb = sum(e[2].elapsed_time(e[3]) for e in ev) / K
        return ta, tb

    def release(self):
        for name in ("inp", "ws", "out", "flush_buf", "g_call", "g_part", "g_comb", "call"):
            if hasattr(self, name):
                delattr(self, name)
        torch.cuda.empty_cache()


def other_config(name, wl, seed, dev, stream, peak, steps, warmup, splits=0):
    """µs per call, TB/s and fraction of the HBM peak of one more workload (graph replays,
    L2 flushed before each step when its inputs are small)."""
    from split_kv_paged_gb300 import binding as B
    m = Measured(wl, seed, dev, stream, B.TLLM_KERNEL_AUTO, splits)
    m.capture(warmup)
    call_ms, call_med = m.timed(m.g_call, steps)
    part_ms, _ = m.timed(m.g_part, steps)
    comb_ms = m.timed(m.g_comb, steps)[0] if m.g_comb is not None else 0.0
    tbps = m.nbytes / (call_ms * 1e-3) / 1e12
    rec = {"workload": wl.name, "num_splits": m.S, "kernel": int(m.plan.kernel), "logical_bytes": m.nbytes,
           "us_per_call": call_ms * 1e3, "us_per_call_median_of_3_runs": call_med * 1e3, "TBps": tbps,
           "frac": tbps * 1e3 / peak, "partial_us": part_ms * 1e3, "combine_alone_us": comb_ms * 1e3,
           "partial_frac": m.nbytes / (part_ms * 1e-3) / 1e9 / peak, "plan_host_us": m.plan_us,
           "steps": steps, "l2": m.l2_note}
    m.release()
    return name, rec


def option_config(m, record, v_dim_major, steps, warmup, peak):
    """The headline workload with one descriptor option (16-bit split records, or the V cache
    in the transposed, dimension-major layout): the same inputs (V copied into that layout),
    its own plan and workspace, timed the same way as the headline (graph replays)."""
    B, wl, inp, dev, stream = m.B, m.wl, m.inp, m.dev, m.stream
    rec = {"f32": B.TLLM_RECORD_F32, "bf16": B.TLLM_RECORD_BF16, "f16": B.TLLM_RECORD_F16}[record]
    vl = B.TLLM_V_DIM_MAJOR if v_dim_major else B.TLLM_V_TOKEN_MAJOR
    desc = B.desc_for(wl, B.TLLM_KERNEL_AUTO, num_pages=inp.num_pages, v_layout=vl, record_type=rec)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    plan = B.tllm_decode_attn_plan(desc, wl.B, wl.Lq, wl.window, host_ctx_lens=wl.ctx, num_sms=n_sm)
    ws = B.Workspace(plan, device=dev)
    out = torch.empty_like(m.out)
    v = inp.v_cache.transpose(-1, -2).contiguous() if v_dim_major else inp.v_cache
    call = (inp.q, inp.k_cache, v, inp.block_table, inp.context_lens, wl.Lq, inp.kv_scales, inp.sinks, wl.window,
            plan.num_splits, ws, out)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            B.tllm_decode_attn_splitkv(*call, stream=stream)
        torch.cuda.synchronize(dev)
        graphs = []
        for fn in (B.tllm_decode_attn_splitkv, B.tllm_decode_attn_partial):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn(*call, stream=stream)
            for _ in range(max(1, warmup)):
                g.replay()
            graphs.append(g)
        torch.cuda.synchronize(dev)
    # each replay of the option's graph alternates with one of the default descriptor's, so
    # that the two see the same clocks
    base_call_ms, call_ms = m.timed_pair(m.g_call, graphs[0], steps)
    base_part_ms, part_ms = m.timed_pair(m.g_part, graphs[1], steps)
    del graphs, v, ws, out
    torch.cuda.empty_cache()
    return {"workload": wl.name, "record": record, "v_layout": "dim_major" if v_dim_major else "token_major",
            "kernel": int(plan.kernel), "num_splits": int(plan.num_splits), "us_per_call": call_ms * 1e3,
            "partial_us": part_ms * 1e3,
            "partial_frac": m.nbytes / (part_ms * 1e-3) / 1e9 / peak, "steps": steps,
            "default_us_per_call": base_call_ms * 1e3, "default_partial_us": base_part_ms * 1e3}


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    from split_kv_paged_gb300 import binding as B
    from split_kv_paged_gb300 import build as libbuild
    libbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = workload(args)
    stream = torch.cuda.Stream(device=dev)
    m = Measured(wl, rank_seed(rank), dev, stream, kernel_code(args.kernel), args.splits, args.record,
                 args.v_layout == "dim_major")
    plan, inp, out, S, nbytes = m.plan, m.inp, m.out, m.S, m.nbytes

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    m.capture(args.warmup)
    K = args.steps
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        ms_step, ms_med3 = m.timed(m.g_call, K)
    barrier()
    partial_ms, _ = m.timed(m.g_part, K)
    combine_ms = m.timed(m.g_comb, K)[0] if m.g_comb is not None else 0.0
    ms_step = max_over_ranks(ms_step, world, dev)
    value = job_tbps(nbytes, world, ms_step)

    # end to end through the C ABI from pinned host buffers: H2D inputs, call, D2H output
    host = {}
    dev_tensors = {"q": inp.q, "k_cache": inp.k_cache, "v_cache": inp.v_cache, "kv_scales": inp.kv_scales,
                   "block_table": inp.block_table, "context_lens": inp.context_lens, "sinks": inp.sinks}
    for k, t in dev_tensors.items():
        if t is not None:
            host[k] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            host[k].copy_(t)
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(h.numel() * h.element_size() for h in host.values())
    d2h = out_host.numel() * out_host.element_size()
    E = max(1, args.e2e_steps)
    with torch.cuda.stream(stream):
        def e2e_step():
            for k, h in host.items():
                dev_tensors[k].copy_(h, non_blocking=True)
            B.tllm_decode_attn_splitkv(*m.call, stream=stream)
            out_host.copy_(out, non_blocking=True)
        e2e_step()
        torch.cuda.synchronize(dev)
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(E):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    e2e_ms = a.elapsed_time(b) / E
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    del host, out_host

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tbps, secs, desc_s, nthr, sb = oracle_sample(wl, rank_seed(0), args.cpu_budget, device_inp=inp)
        cpu = {"value": tbps, "unit": UNIT, "cores": nthr, "kind": "oracle", "sample": desc_s,
               "seconds": secs}

    peak, peak_src = peak_hbm()
    # the other measured workloads, each timed the same way (graph replays of one call), on
    # rank 0 of a single-rank run by default
    others = {}
    if rank == 0 and world == 1 and not args.no_other_configs and args.workload == "mtp4_fp8_long" \
            and args.batch == 0 and args.ctx == 0 and args.bs == 0:
        k_o, w_o = args.other_steps, max(3, min(args.warmup, 5))
        specs = [("single_decode_S1", W.single_decode(), 1001, 1), ("single_decode_S4", W.single_decode(), 1001, 4),
                 ("single_decode", W.single_decode(), 1001, 0),
                 ("verify16_int8", W.verify16_int8(), 1002, 0),
                 ("ragged_fp8_bs128", W.ragged_fp8(bs=128), 1004, 0),
                 ("ragged_fp8_bs16", W.ragged_fp8(bs=16), 1004, 0),
                 ("window_sink_bf16", W.window_sink_bf16(), 1005, 0)]
        for name, wlo, seed, splits in specs:
            k, rec = other_config(name, wlo, seed, dev, stream, peak, k_o, w_o, splits)
            others[k] = rec
    # the headline workload with each layout / record option of the descriptor (rank 0 of a
    # single-rank default run), after the other workloads: these long runs can bring the GPU to
    # its power cap, which would slow the short latency-bound workloads measured after them
    options = {}
    if rank == 0 and world == 1 and not args.no_other_configs and args.workload == "mtp4_fp8_long" \
            and args.batch == 0 and args.ctx == 0 and args.bs == 0 and args.record == "f32" and args.kernel == "auto" \
            and args.v_layout == "token_major":
        for name, record, vdm in (("record_bf16", "bf16", False), ("v_dim_major", "f32", True)):
            options[name] = option_config(m, record, vdm, args.steps, max(3, min(args.warmup, 5)), peak)

    achieved = nbytes / (partial_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_call": ms_step * 1e3,
        "us_per_call_median_of_3_runs": ms_med3 * 1e3,
        "pct_of_peak": 100.0 * value * 1e3 / world / peak, "peak_source": peak_src,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.kv_dtype,
        "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.B, "ctx": max(wl.ctx), "query_rows": wl.Lq, "Hq": wl.Hq,
                   "Hkv": wl.Hkv, "head_dim": wl.D, "block_size": wl.bs, "num_splits": S,
                   "kernel": int(plan.kernel), "record": args.record, "v_layout": args.v_layout, "logical_bytes": nbytes, "plan_host_us": m.plan_us,
                   "l2": m.l2_note, "aggregation": "mean of the K timed graph replays",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(int(plan.kernel), wl.name, nbytes), "kernel": "partial",
                     "partial_ms": partial_ms, "combine_ms": combine_ms, "peak_source": peak_src},
        "clocks": clocks.summary(),
        "e2e": {"value": job_tbps(nbytes, world, e2e_ms), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * (2 if S > 1 else 1),
    }
    if options:
        line["options"] = options
    if others:
        line["other_configs"] = others
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark of the gated delta rule prefill on one GB300 (or N independent replicas).

Workload: 74 packed prompts of 80..3,399 tokens (log-uniform), 16 q/k heads,
32 v heads, head dim 128, bf16 q/k/v and output, fp32 g/beta and final state
(the single-candidate workload shape of the System1-Omni validation page,
"Raw HF Transformers comparison"). Synthetic, seeded inputs.

One step = one gdn_prefill_varlen call over the whole batch (the prep kernel
and the chunk kernel). Inputs (about 1.6 GB) are larger than the 129 MB L2, so
no flush is needed between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]
                  [--kernel tc|simt] [--no-cpu-baseline]
  python bench.py --long | --tree | --latency | --gated-rmsnorm | --input-prep

Prints one JSON line (rank 0). Under torchrun every rank runs its own replica
batch (seed offset by rank; no collective on the data path) and the line
reports the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "GDN prefill tokens/s at 1 GB300 and % of roofline (HBM vs bf16 TC)"
UNIT = "tokens/s"
CONFIG_INDEX = 2
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_COLS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


# ---------------------------------------------------------------- workload accounting
def algorithmic_bytes(w) -> int:
    """Bytes the method must move once: q, k, v, g, beta, cu_seqlens read; o and
    the final state written; each distinct gathered initial-state slot read."""
    b = 0
    for t in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens):
        b += t.numel() * t.element_size()
    b += w.v.numel() * torch.empty((), dtype=w.out_dtype).element_size()
    b += w.num_seqs * w.h_v * w.d_k * w.d_v * 4
    if w.initial_state is not None:
        if w.state_index is None:
            slots = w.num_seqs
        else:
            si = w.state_index.numpy()
            slots = len(set(int(x) for x in si if x >= 0))
        b += slots * w.h_v * w.d_k * w.d_v * 4
    return int(b)


def chunked_tensor_flops(w, C=64) -> int:
    """Tensor-core products of the chunked form per chunk of length l:
    per q/k head 4 l^2 d_k (K K^T, Q K^T); per v head 2 l^2 d_k + 4 l^2 d_v
    (W, U, intra-chunk output) + 6 l d_k d_v (W S, Q S, K^T U')."""
    f = 0
    G = w.h_v // w.h_qk
    for L in w.lengths:
        full, rem = divmod(int(L), C)
        for l, cnt in ((C, full), (rem, 1 if rem else 0)):
            if cnt == 0:
                continue
            per_qk = 4 * l * l * w.d_k
            per_v = 2 * l * l * w.d_k + 4 * l * l * w.d_v + 6 * l * w.d_k * w.d_v
            f += cnt * (w.h_qk * per_qk + w.h_v * per_v)
    del G
    return int(f)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# the sources each profiled kernel is compiled from: a committed ncu summary holds
# for the current build only if their hash matches the one it records
KERNEL_SOURCES = {
    "gdn_tc_kernel": ["gdn_tc.cu", "tc_ptx.cuh", "gdn_internal.cuh"],
    "gated_rmsnorm_kernel": ["gdn_norm.cu", "gdn_ops.cuh"],
    "conv_silu_kernel": ["gdn_input_prep.cu", "gdn_ops.cuh"],
}


def kernel_source_hash(kernel_name: str) -> str:
    import hashlib
    src = os.path.join(ROOT, "gated_deltanet_linear_prefill_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel_name]:
        with open(os.path.join(src, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_name: str, workload_name: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel source (the summary records the sources' hash)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_name}_{workload_name}.md")
    if kernel_name not in KERNEL_SOURCES or not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k_, v_ = line[2:].split(":", 1)
                vals[k_.strip()] = v_.strip().strip("`")
    if vals.get("kernel_sources_sha256_16") != kernel_source_hash(kernel_name):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks
def clocks_path(name: str) -> str:
    """Where the raw nvidia-smi samples go (the JSON line carries their summary):
    $GDN_CLOCKS_DIR if set, else the system temporary directory."""
    import tempfile
    d = os.environ.get("GDN_CLOCKS_DIR") or tempfile.gettempdir()
    os.makedirs(d, exist_ok=True)
    return os.path.join(d, name)


class ClockSampler:
    """nvidia-smi sampling during the timed region (200 ms period)."""

    def __init__(self, gpu_index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            return summarize_clock_samples(f)


def summarize_clock_samples(lines) -> dict:
    """The clocks summary of a bench line from nvidia-smi CSV rows (CLOCK_QUERY,
    no header, no units): the median SM clock over the loaded samples (those at
    least half the highest), the maximum SM clock, every throttle reason seen
    Active, and a note when the SM clock stayed below 90% of its maximum with no
    reason (a clock lock left by someone else)."""
    sm, mx, reasons = [], [], set()
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for name, val in zip(REASON_COLS, parts[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    loaded = [x for x in sm if x >= 0.5 * max(sm)] or sm
    out = {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
           "samples": len(sm)}
    if not reasons and out["sm_mhz"] < 0.9 * out["sm_max_mhz"]:
        out["note"] = "SM clock below 90% of its maximum with no throttle reason"
    return out


# ---------------------------------------------------------------- oracle timing (CPU)
def _oracle_sample(w, target_tokens: int, seed: int = 0):
    """A fixed subset of the workload's sequences with about target_tokens rows."""
    rng = np.random.default_rng(seed)
    order = rng.permutation(w.num_seqs)
    pick, tot = [], 0
    for n in order:
        if tot >= target_tokens:
            break
        pick.append(int(n))
        tot += int(w.lengths[n])
    return sorted(pick), tot


def time_oracle(w, target_tokens: int, seed: int = 0):
    import oracle
    seqs, tokens = _oracle_sample(w, target_tokens, seed)
    sub = workloads.subset_sequences(w, seqs)
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    oracle.run_workload(sub, n_threads=threads)
    dt = time.perf_counter() - t0
    return tokens / dt, dt, len(seqs), tokens, threads


# ---------------------------------------------------------------- distributed helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(tokens_per_rank: int, times_ms, world: int, device):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    total_ms = reduce_max(float(sum(times_ms)), world, device)
    steps = len(times_ms)
    total_tokens = tokens_per_rank * world * steps
    return total_tokens / (total_ms / 1e3), total_ms / steps


def pipelined_e2e(host_in, dev_sets, run, out_sets, host_out, steps, device):
    """End-to-end steps through pinned host memory, pipelined across steps.

    Every step copies its inputs host -> device (`host_in` into dev_sets[b]), runs the
    call (`run(b)`, on the current stream) and reads its results device -> host
    (out_sets[b] into `host_out`), b = step % 2. The input copies run on one stream,
    the calls on the current stream, the result copies on a third, with events
    between them, so step i+1's inputs travel while step i computes and step i-1's
    results come back. Returns the milliseconds from the first copy's start to the
    last copy's end (CUDA events), over `steps` steps."""
    comp = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    loaded = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(s_in)
    s_out.wait_event(e0)
    comp.wait_event(e0)
    for i in range(steps):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(computed[b])  # step i-2 has read this input set
            for n, t in host_in.items():
                dev_sets[b][n].copy_(t, non_blocking=True)
            loaded[b].record(s_in)
        comp.wait_event(loaded[b])
        if i >= 2:
            comp.wait_event(drained[b])  # step i-2's results have left this output set
        run(b)
        computed[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[b])
            for dev, host in zip(out_sets[b], host_out):
                host.copy_(dev, non_blocking=True)
            drained[b].record(s_out)
    s_out.wait_stream(s_in)
    s_out.wait_stream(comp)
    e1.record(s_out)
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1)


# ---------------------------------------------------------------- arms
def run_reference(args, world, rank):
    """The oracle arm: the fp64 CPU oracle as it stands, on host cores, each step
    a bounded sample (about 1/16 of the batch's tokens) of the same workload."""
    if rank != 0:
        return
    w = workloads.config(CONFIG_INDEX)
    target = max(1, w.total_tokens // 16)
    for i in range(args.warmup):
        time_oracle(w, target, seed=i)
    rates, secs, toks = [], [], []
    for i in range(args.steps):
        r, dt, nseq, tok, threads = time_oracle(w, target, seed=1000 + i)
        rates.append(r)
        secs.append(dt)
        toks.append(tok)
    value = sum(toks) / sum(secs)
    sample = (f"per step a fixed random subset of the batch's sequences with ~{target} of "
              f"{w.total_tokens} tokens, all {w.h_v} heads; {args.steps} steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(secs) / len(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workloads.CONFIG_NAMES[CONFIG_INDEX], "num_seqs": w.num_seqs,
                   "total_tokens": w.total_tokens, "max_seqlen": w.max_seqlen, "h_qk": w.h_qk,
                   "h_v": w.h_v, "d_k": w.d_k, "d_v": w.d_v, "chunk": 64, "gates": "fp32", "out": "bf16",
                   "state": "fp32", "parallelism": f"host cores x{threads}"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gdn(args, world, rank, local):
    import gated_deltanet_linear_prefill_gb300 as gdn
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl gdn")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    gdn.load_library()
    w = workloads.config(CONFIG_INDEX, seed_offset=rank)
    workload_name = workloads.CONFIG_NAMES[CONFIG_INDEX]
    if args.subset_seqs > 0:
        # a smaller case of the same batch (profiling captures): its first K sequences
        w = workloads.subset_sequences(w, range(min(args.subset_seqs, w.num_seqs)))
        workload_name += f"_first{args.subset_seqs}"
    flags = gdn.GDN_FLAG_SIMT if args.kernel == "simt" else 0
    d = w.to(device)
    out = torch.empty(d.v.shape, dtype=d.out_dtype, device=device)
    fs = torch.empty((d.num_seqs, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device=device)
    desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=d.out_dtype,
                         max_seqlen=w.max_seqlen, flags=flags)
    ws = torch.empty(max(256, gdn.gdn_workspace_bytes(desc)), dtype=torch.uint8, device=device)
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    stream = torch.cuda.current_stream(device)
    launches_per_step = 2  # prep kernel + chunk kernel

    def step():
        rc = gdn.gdn_prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, None, None, out,
                                    fs, desc, stream)
        if rc != gdn.GDN_OK:
            raise gdn.GdnError(rc, "gdn_prefill_varlen")

    for _ in range(max(3, args.warmup)):
        step()
    rc = gdn.gdn_get_device_status(desc, stream)
    if rc != gdn.GDN_OK:
        raise gdn.GdnError(rc, "device status")
    torch.cuda.synchronize(device)

    # ---- device-resident timing, per-step events on the launching stream. The
    # clock sampler starts one second of untimed steps before the timed region
    # (its 200 ms period needs samples) and stops right after it.
    clocks = ClockSampler(local, clocks_path(f"clocks_rank{rank}.csv"))
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(8):
            step()
        torch.cuda.synchronize(device)
    barrier(world)
    torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    clk = clocks.stop()
    times = [a.elapsed_time(b) for a, b in ev]
    value, ms_per_step = aggregate(w.total_tokens, times, world, device)

    e2e_line = None
    # ---- end to end: pinned host inputs -> device, call, results -> pinned host
    if not args.no_e2e:
        host_in = {n: getattr(w, n).pin_memory() for n in ("q", "k", "v", "g", "beta", "cu_seqlens")}
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        host_fs = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = host_out.numel() * host_out.element_size() + host_fs.numel() * host_fs.element_size()

        # two device input sets and two output sets, so that copies of neighbouring
        # steps overlap the call between them
        dev_sets = [{n: getattr(d, n) for n in host_in},
                    {n: torch.empty_like(getattr(d, n)) for n in host_in}]
        out_sets = [(out, fs), (torch.empty_like(out), torch.empty_like(fs))]

        def run(b):
            x = dev_sets[b]
            rc = gdn.gdn_prefill_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], None, None,
                                        out_sets[b][0], out_sets[b][1], desc, stream)
            if rc != gdn.GDN_OK:
                raise gdn.GdnError(rc, "gdn_prefill_varlen")

        pipelined_e2e(host_in, dev_sets, run, out_sets, (host_out, host_fs), 2, device)  # warm-up
        e2e_steps = max(4, min(args.steps, 10))
        barrier(world)
        ms = pipelined_e2e(host_in, dev_sets, run, out_sets, (host_out, host_fs), e2e_steps, device)
        barrier(world)
        e2e_value, _ = aggregate(w.total_tokens, [ms], world, device)
        e2e_value *= e2e_steps
        e2e_line = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h),
                    "pipelined": "inputs of step i+1 copied in while step i computes and step i-1's "
                                 "results are copied out (three streams, two buffer sets)"}

    # ---- roofline of the dominant kernel (the chunk kernel; the step also holds
    # the one-block prep kernel, so the figure is a slight underestimate)
    hbm_peak, tc_peak, peak_kind = measured_peaks()
    B = algorithmic_bytes(w)
    F = chunked_tensor_flops(w)
    step_s = sum(times) / len(times) / 1e3  # mean launch duration over the timed region
    achieved = B / step_s / 1e9
    kernel_name = "gdn_tc_kernel" if args.kernel == "tc" else "gdn_simt_kernel"
    traffic = profiled_traffic(kernel_name, workload_name)
    roofline_time = max(B / (hbm_peak * 1e9), F / (tc_peak * 1e12))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name, "num_seqs": w.num_seqs,
                   "total_tokens": w.total_tokens, "max_seqlen": w.max_seqlen, "h_qk": w.h_qk,
                   "h_v": w.h_v, "d_k": w.d_k, "d_v": w.d_v, "chunk": 64,
                   "gates": "fp32", "out": "bf16", "state": "fp32", "kernel": args.kernel,
                   "l2_flush": "none needed: inputs (%.2f GB) exceed the 129 MB L2" % (
                       (B - w.num_seqs * w.h_v * w.d_k * w.d_v * 4) / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": B, "tensor_flops_per_launch": F,
                     "tensor_tflops_achieved": F / step_s / 1e12,
                     "frac_nominal_8tbs": achieved / 8000.0,
                     "frac_of_roofline_time": roofline_time / step_s},
        "e2e": e2e_line,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the whole batch through the fp64 oracle, repeated until at least 10 s of CPU work
        tot_tok, tot_s, passes = 0, 0.0, 0
        while tot_s < 10.0 and passes < 20:
            r, dt, nseq, tok, threads = time_oracle(w, w.total_tokens, seed=0)
            tot_tok += tok
            tot_s += dt
            passes += 1
        line["cpu_baseline"] = {
            "value": tot_tok / tot_s, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"the whole batch ({w.num_seqs} sequences, {w.total_tokens} tokens, "
                      f"{w.h_v} heads), fp64 recurrence, {passes} passes in {tot_s:.1f} s"}
    if rank == 0 and world == 1 and not args.no_long and args.kernel == "tc" and args.subset_seqs == 0:
        # the long-prompt workload (one 16,384-token prompt as one call and as 48 calls), so
        # that the default run's record holds it too; `bench.py --long` prints it in full
        la = argparse.Namespace(**vars(args))
        la.steps, la.warmup, la.soak_s, la.layers = 10, 3, 0.5, 48
        la.no_cpu_baseline = True
        ll = measure_long(la)
        line["long_prompt"] = {
            "workload": ll["config"]["workload"], "metric": ll["metric"], "unit": ll["unit"],
            "value": ll["value"], "ms_per_call": ll["ms_per_step"],
            "ms_per_call_48_layers": ll["layers48"]["ms_per_call"],
            "roofline_frac": ll["roofline"]["frac"], "segment_scan": ll["config"]["segment_scan"],
            "e2e": ll["e2e"], "gpu_launches": ll["gpu_launches"], "clocks": ll["clocks"],
            "full_line": "python bench.py --long"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_tree_bench(args):
    """Latency of the two-level prefix tree of config 3 (one shared prompt, 3
    question branches, 7 candidate tails; 11 nodes), three ways on one GPU:
    one gdn_prefill_tree launch; three gdn_prefill_varlen calls, one per level,
    each handing its final states to the next; and one call over the 7 full
    root-to-leaf paths (the replicated layout). Inputs resident on the device;
    each variant is timed over `steps` calls after `warmup`, with CUDA events
    on the launching stream. Prints one JSON line."""
    import gated_deltanet_linear_prefill_gb300 as gdn
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --tree needs a CUDA device")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    t = workloads.tree_config()
    rows = t.rows
    parent = torch.tensor([-1] + [0] * len(t.branch_lens) + [1 + b for b in t.leaf_parent],
                          dtype=torch.int32)
    n_nodes = int(parent.numel())
    d = rows.to(device)
    par = parent.to(device)
    stream = torch.cuda.current_stream(device)
    out = torch.empty(d.v.shape, dtype=d.out_dtype, device=device)
    fs = torch.empty((n_nodes, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device=device)
    desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=d.out_dtype)
    ws = torch.empty(max(256, gdn.gdn_tree_workspace_bytes(desc)), dtype=torch.uint8, device=device)
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()

    def tree_call():
        rc = gdn.gdn_prefill_tree(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, par, None, None, out, fs,
                                  desc, stream)
        if rc != gdn.GDN_OK:
            raise gdn.GdnError(rc, "gdn_prefill_tree")

    # level by level
    nb, nl = len(t.branch_lens), len(t.leaf_lens)
    levels = [workloads.take_rows(rows, [[t.segment("prefix")]], "prefix"),
              workloads.take_rows(rows, [[t.segment("branch", b)] for b in range(nb)], "branches"),
              workloads.take_rows(rows, [[t.segment("leaf", l)] for l in range(nl)], "leaves")]
    lv = [x.to(device) for x in levels]
    lv_out = [torch.empty(x.v.shape, dtype=x.out_dtype, device=device) for x in lv]
    lv_fs = [torch.empty((x.num_seqs, x.h_v, x.d_k, x.d_v), dtype=torch.float32, device=device)
             for x in lv]
    lv_sidx = [None, torch.zeros(nb, dtype=torch.int32, device=device),
               torch.tensor(t.leaf_parent, dtype=torch.int32, device=device)]
    lv_init = [None, lv_fs[0], lv_fs[1]]
    lv_desc = []
    for i, x in enumerate(lv):
        dd = gdn.make_desc(x.q, x.v, x.g, x.cu_seqlens, out_dtype=x.out_dtype,
                           initial_state=lv_init[i])
        w_ = torch.empty(max(256, gdn.gdn_workspace_bytes(dd)), dtype=torch.uint8, device=device)
        dd.workspace, dd.workspace_bytes = w_.data_ptr(), w_.numel()
        lv_desc.append((dd, w_))

    def level_calls():
        for i, x in enumerate(lv):
            rc = gdn.gdn_prefill_varlen(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, lv_init[i],
                                        lv_sidx[i], lv_out[i], lv_fs[i], lv_desc[i][0], stream)
            if rc != gdn.GDN_OK:
                raise gdn.GdnError(rc, "gdn_prefill_varlen")

    # replicated full paths
    pw = workloads.take_rows(rows, [[t.segment("prefix"), t.segment("branch", t.leaf_parent[l]),
                                     t.segment("leaf", l)] for l in range(nl)], "paths").to(device)
    p_out = torch.empty(pw.v.shape, dtype=pw.out_dtype, device=device)
    p_fs = torch.empty((pw.num_seqs, pw.h_v, pw.d_k, pw.d_v), dtype=torch.float32, device=device)
    p_desc = gdn.make_desc(pw.q, pw.v, pw.g, pw.cu_seqlens, out_dtype=pw.out_dtype)
    p_ws = torch.empty(max(256, gdn.gdn_workspace_bytes(p_desc)), dtype=torch.uint8, device=device)
    p_desc.workspace, p_desc.workspace_bytes = p_ws.data_ptr(), p_ws.numel()

    def path_call():
        rc = gdn.gdn_prefill_varlen(pw.q, pw.k, pw.v, pw.g, pw.beta, pw.cu_seqlens, None, None,
                                    p_out, p_fs, p_desc, stream)
        if rc != gdn.GDN_OK:
            raise gdn.GdnError(rc, "gdn_prefill_varlen")

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(device)
        ts = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    us_tree, us_levels, us_paths = timed(tree_call), timed(level_calls), timed(path_call)
    rc = gdn.gdn_get_device_status(desc, stream)
    if rc != gdn.GDN_OK:
        raise gdn.GdnError(rc, "device status")
    T = int(rows.q.shape[0])
    line = {
        "metric": "GDN prefix-tree prefill latency (config 3 tree, one launch)",
        "value": us_tree, "unit": "us per tree", "higher_is_better": False, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
        "variants_us": {"tree_one_launch": us_tree, "three_level_calls": us_levels,
                        "replicated_full_paths": us_paths},
        "gpu_launches": {"tree_one_launch": 2, "three_level_calls": 6, "replicated_full_paths": 2},
        "config": {"workload": "cfg3_prefix_tree", "nodes": n_nodes, "tokens": T,
                   "replicated_path_tokens": int(pw.q.shape[0]), "h_qk": d.h_qk, "h_v": d.h_v,
                   "d": d.d_k, "timing": "median of per-call CUDA events, inputs resident"},
    }
    print(json.dumps(line))


def run_latency_bench(args):
    """Per-call latency of the small, launch-bound workloads (inputs resident):
    config 0, config 1 (one 539-token prompt, 32 value heads), a batch of seven
    65-96-token candidate paths (two chunks each), and the config 3 prefix tree
    in one launch. Each is timed as plain launches and as a CUDA graph replay
    (the call captured once), median of `steps` calls after `warmup`, with
    CUDA events on the launching stream. Prints one JSON line."""
    import gated_deltanet_linear_prefill_gb300 as gdn
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --latency needs a CUDA device")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)

    def varlen_case(w):
        d = w.to(device)
        out = torch.empty(d.v.shape, dtype=d.out_dtype, device=device)
        fs = torch.empty((d.num_seqs, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device=device)
        desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=d.out_dtype,
                             initial_state=d.initial_state, max_seqlen=w.max_seqlen)
        ws = torch.empty(max(256, gdn.gdn_workspace_bytes(desc)), dtype=torch.uint8, device=device)
        desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
        keep = (d, out, fs, ws)

        def call():
            rc = gdn.gdn_prefill_varlen(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, d.initial_state,
                                        d.state_index, out, fs, desc, stream)
            if rc != gdn.GDN_OK:
                raise gdn.GdnError(rc, "gdn_prefill_varlen")
        return call, keep, int(w.q.shape[0])

    def tree_case():
        t = workloads.tree_config()
        d = t.rows.to(device)
        par = torch.tensor([-1] + [0] * len(t.branch_lens) + [1 + b for b in t.leaf_parent],
                           dtype=torch.int32, device=device)
        out = torch.empty(d.v.shape, dtype=d.out_dtype, device=device)
        fs = torch.empty((d.num_seqs, d.h_v, d.d_k, d.d_v), dtype=torch.float32, device=device)
        desc = gdn.make_desc(d.q, d.v, d.g, d.cu_seqlens, out_dtype=d.out_dtype)
        ws = torch.empty(max(256, gdn.gdn_tree_workspace_bytes(desc)), dtype=torch.uint8,
                         device=device)
        desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
        keep = (d, par, out, fs, ws)

        def call():
            rc = gdn.gdn_prefill_tree(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, par, None, None,
                                      out, fs, desc, stream)
            if rc != gdn.GDN_OK:
                raise gdn.GdnError(rc, "gdn_prefill_tree")
        return call, keep, int(t.rows.q.shape[0])

    rng = np.random.default_rng(5)
    short = workloads.random_workload([int(x) for x in rng.integers(65, 97, 7)], h_qk=16, h_v=32,
                                      d_k=128, d_v=128, seed=5)
    lone = workloads.random_workload([96], h_qk=1, h_v=1, d_k=128, d_v=128, seed=6)
    cases = {"lone_unit_T96_1head": varlen_case(lone),
             "cfg0_tiny_T128_d64": varlen_case(workloads.config(0)),
             "cfg1_single_T539": varlen_case(workloads.config(1)),
             "short_paths_7x65to96": varlen_case(short),
             "cfg3_prefix_tree_one_launch": tree_case()}

    def med(fn):
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                fn()
        stream.synchronize()
        ts = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        return statistics.median(ts)

    res = {}
    for name, (call, keep, tokens) in cases.items():
        plain = med(call)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            call()  # the library's one-time set-up happens outside the capture
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                call()
        def replay(g=g):
            with torch.cuda.stream(stream):
                g.replay()
        graph = med(replay)
        res[name] = {"tokens": tokens, "us_per_call": plain, "us_per_graph_replay": graph}
    line = {"metric": "GDN prefill latency of small workloads (per call, one GB300)",
            "value": min(res["cfg1_single_T539"]["us_per_call"], res["cfg1_single_T539"]["us_per_graph_replay"]),
            "unit": "us per call",
            "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "dtype": "bf16", "data": "synthetic", "cases": res,
            "config": {"workload": "cfg1_single_T539 (value: the faster of a plain call and a graph replay); "
                                   "all cases under 'cases'",
                       "timing": "median of per-call CUDA events, inputs resident"}}
    print(json.dumps(line))


def run_norm_bench(args):
    """The gated RMSNorm that follows the prefill, on the 74-prompt batch's
    output shape [62,875, 32, 128]: bf16 o, z and y, fp32 weight. One step =
    one gdn_gated_rmsnorm call. o and z (1.03 GB) exceed the 129 MB L2."""
    import gated_deltanet_linear_prefill_gb300 as gdn
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --gated-rmsnorm needs a CUDA device")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    gdn.load_library()
    w = workloads.config(CONFIG_INDEX)
    T, H, D = w.total_tokens, w.h_v, w.d_v
    o_h, _ = workloads.norm_inputs(T, H, D, seed=21)  # stands in for the prefill's output
    z_h, wt_h = workloads.norm_inputs(T, H, D, seed=22)
    o, z, wt = o_h.to(device), z_h.to(device), wt_h.to(device)
    y = torch.empty_like(o)
    rows = T * H
    stream = torch.cuda.current_stream(device)

    def step():
        rc = gdn.gdn_gated_rmsnorm(o, z, wt, y, rows, D, gdn.GDN_BF16, gdn.GDN_BF16, 1e-6, stream)
        if rc != gdn.GDN_OK:
            raise gdn.GdnError(rc, "gdn_gated_rmsnorm")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    clocks = ClockSampler(0, clocks_path("clocks_norm.csv"))
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(32):
            step()
        torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = sum(times) / len(times)
    B = rows * D * (2 + 2 + 2) + D * 4  # read o and z, write y, read the weights
    hbm_peak, _, peak_kind = measured_peaks()
    achieved = B / (ms / 1e3) / 1e9

    # end to end: pinned host o and z in, y out, each step
    e2e_line = None
    if not args.no_e2e:
        ho, hz = o_h.pin_memory(), z_h.pin_memory()
        hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()

        def e2e_step():
            o.copy_(ho, non_blocking=True)
            z.copy_(hz, non_blocking=True)
            step()
            hy.copy_(y, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(device)
        n_e2e = max(3, min(args.steps, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(device)
        e2e_line = {"value": T * n_e2e / (e0.elapsed_time(e1) / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": int(2 * rows * D * 2), "d2h_bytes_per_step": int(rows * D * 2)}
    line = {
        "metric": "gated RMSNorm tokens/s at 1 GB300 and % of HBM roofline", "value": T / (ms / 1e3),
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "gated_rmsnorm_cfg2_output", "tokens": T, "h_v": H, "d_v": D,
                   "o_z_y": "bf16", "weight": "fp32", "eps": 1e-6,
                   "l2_flush": "none needed: o and z (%.2f GB) exceed the 129 MB L2" % (2 * rows * D * 2 / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": profiled_traffic("gated_rmsnorm_kernel", "gated_rmsnorm_cfg2_output"),
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": B},
        "e2e": e2e_line, "gpu_launches": args.steps, "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import oracle
        idx = np.random.default_rng(0).choice(rows, min(rows, 400_000), replace=False)
        o2, z2 = o_h.reshape(rows, D)[idx].float().numpy(), z_h.reshape(rows, D)[idx].float().numpy()
        w2 = wt_h.numpy()
        tot, n = 0.0, 0
        while tot < 10.0 and n < 50:
            t0 = time.perf_counter()
            oracle.gated_rmsnorm(o2, z2, w2, 1e-6)
            tot += time.perf_counter() - t0
            n += 1
        line["cpu_baseline"] = {"value": n * idx.size / H / tot, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"{idx.size} random rows of {D} (token-heads), fp64 numpy, "
                                          f"{n} passes in {tot:.1f} s; tokens = rows / {H}"}
    print(json.dumps(line), flush=True)


def run_prep_bench(args):
    """The GDN input prep on the 74-prompt batch: x [62,875, 8,192] bf16 (q | k | v
    channels of 16 x 128, 16 x 128, 32 x 128), 4 conv taps, gate projections
    [62,875, 32]. One step = one gdn_input_prep call (the conv + SiLU kernel and
    the gate kernel). x (1.03 GB) exceeds the 129 MB L2."""
    import gated_deltanet_linear_prefill_gb300 as gdn
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --input-prep needs a CUDA device")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    gdn.load_library()
    w = workloads.config(CONFIG_INDEX)
    h_qk, d_k, h_v, d_v, K = w.h_qk, w.d_k, w.h_v, w.d_v, 4
    inp_h = workloads.prep_inputs(w.lengths.tolist(), h_qk=h_qk, d_k=d_k, h_v=h_v, d_v=d_v, K=K, seed=31)
    inp = {n: (None if t is None else t.to(device)) for n, t in inp_h.items()}
    T, C, N = w.total_tokens, 2 * h_qk * d_k + h_v * d_v, w.num_seqs
    q = torch.empty((T, h_qk, d_k), dtype=torch.bfloat16, device=device)
    k = torch.empty_like(q)
    v = torch.empty((T, h_v, d_v), dtype=torch.bfloat16, device=device)
    g = torch.empty((T, h_v), dtype=torch.float32, device=device)
    beta = torch.empty_like(g)
    cs = torch.empty((N, K - 1, C), dtype=torch.bfloat16, device=device)
    d = gdn.GdnPrepDesc()
    d.num_seqs, d.total_tokens, d.h_qk, d.h_v, d.d_k, d.d_v = N, T, h_qk, h_v, d_k, d_v
    d.conv_width, d.num_state_slots = K, 0
    stream = torch.cuda.current_stream(device)

    def step():
        rc = gdn.gdn_input_prep(inp["x"], inp["conv_w"], None, inp["cu_seqlens"], None, None, inp["a"], inp["b"],
                                inp["A_log"], inp["dt_bias"], q, k, v, g, beta, cs, d, stream)
        if rc != gdn.GDN_OK:
            raise gdn.GdnError(rc, "gdn_input_prep")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    clocks = ClockSampler(0, clocks_path("clocks_prep.csv"))
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(32):
            step()
        torch.cuda.synchronize(device)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a_, b_ in ev:
        a_.record(stream)
        step()
        b_.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    ms = sum(a_.elapsed_time(b_) for a_, b_ in ev) / len(ev)
    B = (T * C * 2 * 2 + T * h_v * (2 * 2 + 4 * 2) + C * K * 4 + 2 * h_v * 4 + N * (K - 1) * C * 2
         + (N + 1) * 4)
    hbm_peak, _, peak_kind = measured_peaks()
    achieved = B / (ms / 1e3) / 1e9
    e2e_line = None
    if not args.no_e2e:
        hx, ha, hb = inp_h["x"].pin_memory(), inp_h["a"].pin_memory(), inp_h["b"].pin_memory()
        hq, hk, hv = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (q, k, v))
        hg, hbeta = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (g, beta))

        def e2e_step():
            inp["x"].copy_(hx, non_blocking=True)
            inp["a"].copy_(ha, non_blocking=True)
            inp["b"].copy_(hb, non_blocking=True)
            step()
            for h_, t_ in ((hq, q), (hk, k), (hv, v), (hg, g), (hbeta, beta)):
                h_.copy_(t_, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(device)
        n_e2e = max(3, min(args.steps, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(device)
        e2e_line = {"value": T * n_e2e / (e0.elapsed_time(e1) / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": int(T * C * 2 + 2 * T * h_v * 2),
                    "d2h_bytes_per_step": int(T * C * 2 + 2 * T * h_v * 4)}
    line = {
        "metric": "GDN input prep tokens/s at 1 GB300 and % of HBM roofline", "value": T / (ms / 1e3),
        "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "input_prep_cfg2", "tokens": T, "num_seqs": N, "channels": C, "conv_width": K,
                   "h_qk": h_qk, "h_v": h_v, "d_k": d_k, "d_v": d_v, "x_qkv": "bf16", "gates": "fp32",
                   "l2_flush": "none needed: x (%.2f GB) exceeds the 129 MB L2" % (T * C * 2 / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": profiled_traffic("conv_silu_kernel", "input_prep_cfg2"),
                     "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": B,
                     "note": "bytes and time of the whole call (conv + SiLU kernel and gate kernel); "
                             "traffic: the conv + SiLU kernel's DRAM bytes"},
        "e2e": e2e_line, "gpu_launches": 2 * args.steps, "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import oracle
        lens = w.lengths
        cu = inp_h["cu_seqlens"].numpy().astype(np.int64)
        n = int(np.argsort(lens)[len(lens) // 2])  # a median-length sequence
        b0, e0_ = int(cu[n]), int(cu[n + 1])
        xs = inp_h["x"][b0:e0_].float().numpy()
        wc = inp_h["conv_w"].numpy()
        tot, passes = 0.0, 0
        while tot < 10.0 and passes < 50:
            t0 = time.perf_counter()
            oracle.causal_conv_silu(xs, wc, np.array([0, e0_ - b0]))
            oracle.gate_params(inp_h["a"][b0:e0_].float().numpy(), inp_h["b"][b0:e0_].float().numpy(),
                               inp_h["A_log"].numpy(), inp_h["dt_bias"].numpy())
            tot += time.perf_counter() - t0
            passes += 1
        line["cpu_baseline"] = {"value": passes * (e0_ - b0) / tot, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"sequence {n} ({e0_ - b0} tokens, all {C} channels and {h_v} gate "
                                          f"heads), fp64 numpy, {passes} passes in {tot:.1f} s"}
    print(json.dumps(line), flush=True)


def device_layer_inputs(layer: int, device, T=16384, h_qk=16, h_v=32, d=128):
    """One input set of the 16,384-token workload drawn on the device, with the same
    distributions as workloads.config(4) (q, k unit rows in bf16; v ~ N(0, 1) bf16;
    alpha ~ U(0.95, 1), g = log alpha, beta = sigmoid(N(0, 1)), both bf16; initial
    state ~ N(0, 0.02) fp32), from a torch generator seeded 4 * 1000 + layer. The
    48-call loop needs 48 distinct sets (about 20 GB); drawing them on the host
    would take minutes."""
    gen = torch.Generator(device=device)
    gen.manual_seed(4 * 1000 + int(layer))

    def unit_rows(h):
        x = torch.randn((T, h, d), generator=gen, device=device, dtype=torch.float32)
        return (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)

    q, k = unit_rows(h_qk), unit_rows(h_qk)
    v = torch.randn((T, h_v, d), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    alpha = 0.95 + 0.05 * torch.rand((T, h_v), generator=gen, device=device, dtype=torch.float64)
    g = torch.log(alpha).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((T, h_v), generator=gen, device=device, dtype=torch.float64)).to(torch.bfloat16)
    init = 0.02 * torch.randn((1, h_v, d, d), generator=gen, device=device, dtype=torch.float32)
    return q, k, v, g, beta, init


def run_long_bench(args):
    """`--long`: prints measure_long's JSON line."""
    print(json.dumps(measure_long(args)), flush=True)


def measure_long(args):
    """The long-prompt workload: one 16,384-token prompt, 16 q/k and 32 v heads, head
    dim 128, bf16 inputs and output, fp32 initial and final state. Times one call
    (layer 0's inputs, resident) and 48 back-to-back calls, one per linear-attention
    layer, each on its own input set. Returns one JSON-line dict; value = tokens/s of
    one call."""
    import gated_deltanet_linear_prefill_gb300 as gdn
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --long needs a CUDA device")
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    gdn.load_library()
    n_layers = max(1, min(48, args.layers))
    w = workloads.config(4, layer=0)
    T = w.total_tokens
    stream = torch.cuda.current_stream(device)
    cu = w.cu_seqlens.to(device)
    sidx = w.state_index.to(device)
    layers = [tuple(getattr(w, n).to(device) for n in ("q", "k", "v", "g", "beta", "initial_state"))]
    for layer in range(1, n_layers):
        layers.append(device_layer_inputs(layer, device))
    out = torch.empty((T, w.h_v, w.d_v), dtype=torch.bfloat16, device=device)
    fs = torch.empty((1, w.h_v, w.d_k, w.d_v), dtype=torch.float32, device=device)
    q0, _, v0, g0, _, init0 = layers[0]
    desc = gdn.make_desc(q0, v0, g0, cu, initial_state=init0, out_dtype=torch.bfloat16,
                         max_seqlen=w.max_seqlen)
    ws = torch.empty(max(256, gdn.gdn_workspace_bytes(desc)), dtype=torch.uint8, device=device)
    desc.workspace, desc.workspace_bytes = ws.data_ptr(), ws.numel()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    n_seg, rows0, rows = gdn.gdn_segment_plan(desc, sms)
    # kernels per call: segment scan = set-up, prep + chunk kernel (A), composition,
    # prep + chunk kernel (C); one launch = prep + chunk kernel
    launches_per_call = 6 if n_seg else 2

    def call(i):
        q, k, v, g, beta, init = layers[i]
        rc = gdn.gdn_prefill_varlen(q, k, v, g, beta, cu, init, sidx, out, fs, desc, stream)
        if rc != gdn.GDN_OK:
            raise gdn.GdnError(rc, "gdn_prefill_varlen")

    for i in range(n_layers):
        call(i)
    for _ in range(max(3, args.warmup)):
        call(0)
    rc = gdn.gdn_get_device_status(desc, stream)
    if rc != gdn.GDN_OK:
        raise gdn.GdnError(rc, "device status")
    torch.cuda.synchronize(device)
    clocks = ClockSampler(0, clocks_path("clocks_long.csv"))
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for i in range(n_layers):
            call(i)
        torch.cuda.synchronize(device)
    # one call, layer 0 (inputs 0.27 GB, larger than the L2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        call(0)
        b.record(stream)
    torch.cuda.synchronize(device)
    t_one = [a.elapsed_time(b) for a, b in ev]
    # 48 back-to-back calls, each on its own layer's inputs
    passes = max(3, args.steps // 4)
    ev48 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(passes)]
    for a, b in ev48:
        a.record(stream)
        for i in range(n_layers):
            call(i)
        b.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop()
    t48 = [a.elapsed_time(b) for a, b in ev48]
    ms_one = statistics.median(t_one)
    ms_48 = statistics.median(t48)

    e2e_line = None
    if not args.no_e2e:
        names = ("q", "k", "v", "g", "beta", "initial_state", "state_index", "cu_seqlens")
        host_in = {n: getattr(w, n).pin_memory() for n in names}
        dev_in = {n: torch.empty_like(t, device=device) for n, t in host_in.items()}
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        host_fs = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = host_out.numel() * host_out.element_size() + host_fs.numel() * host_fs.element_size()

        dev_sets = [dev_in, {n: torch.empty_like(t) for n, t in dev_in.items()}]
        out_sets = [(out, fs), (torch.empty_like(out), torch.empty_like(fs))]

        def run(b):
            x = dev_sets[b]
            rc = gdn.gdn_prefill_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                                        x["initial_state"], x["state_index"], out_sets[b][0], out_sets[b][1],
                                        desc, stream)
            if rc != gdn.GDN_OK:
                raise gdn.GdnError(rc, "gdn_prefill_varlen")

        pipelined_e2e(host_in, dev_sets, run, out_sets, (host_out, host_fs), 2, device)  # warm-up
        n_e2e = max(4, min(args.steps, 10))
        ms = pipelined_e2e(host_in, dev_sets, run, out_sets, (host_out, host_fs), n_e2e, device)
        e2e_line = {"value": T * n_e2e / (ms / 1e3), "unit": UNIT,
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "pipelined": "inputs of call i+1 copied in while call i computes and call i-1's "
                                 "results are copied out (three streams, two buffer sets)"}

    hbm_peak, tc_peak, peak_kind = measured_peaks()
    B = algorithmic_bytes(w)
    F = chunked_tensor_flops(w)
    s_one = ms_one / 1e3
    achieved = B / s_one / 1e9
    roofline_time = max(B / (hbm_peak * 1e9), F / (tc_peak * 1e12))
    line = {
        "metric": METRIC, "value": T / s_one, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_one, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "cfg4_long_T16384", "num_seqs": 1, "total_tokens": T, "h_qk": w.h_qk,
                   "h_v": w.h_v, "d_k": w.d_k, "d_v": w.d_v, "chunk": 64, "gates": "bf16", "out": "bf16",
                   "state": "fp32 (initial state gathered)", "kernel": "tc",
                   "segment_scan": ({"segments": n_seg, "rows_segment0": rows0, "rows_per_segment": rows,
                                     "units_launch_a": w.h_v * (2 * n_seg - 3), "units_launch_c": w.h_v * (n_seg - 1)}
                                    if n_seg else None),
                   "l2_flush": "none needed: one call's inputs (%.2f GB) exceed the 129 MB L2" % (
                       (B - 2 * w.h_v * w.d_k * w.d_v * 4) / 1e9),
                   "layers": n_layers,
                   "layer_inputs": "layer 0 drawn on the host (the parity case); layers 1-47 drawn on "
                                   "the device with the same distributions"},
        "layers48": {"ms_per_48_calls": ms_48, "ms_per_call": ms_48 / n_layers,
                     "tokens_per_s": n_layers * T / (ms_48 / 1e3), "passes": passes},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": None,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "frac_nominal_8tbs": achieved / 8000.0,
                     "algorithmic_bytes_per_launch": B, "tensor_flops_per_launch": F,
                     "tensor_tflops_achieved": F / s_one / 1e12,
                     "frac_of_roofline_time": roofline_time / s_one,
                     "note": ("one prompt: the segment scan runs %d segments' state maps side by side, "
                              "then the segments from their true states; bound by the chunk chains "
                              "(one unit per SM), not by bandwidth" % n_seg) if n_seg else
                             ("%d (sequence, value head) chains on %d SMs: bound by the chain length, "
                              "not by bandwidth" % (w.h_v, sms))},
        "e2e": e2e_line,
        "gpu_launches": launches_per_call * (args.steps + passes * n_layers),
        "clocks": clk,
    }
    if not args.no_cpu_baseline:
        import oracle
        threads = oracle.default_threads()
        t0 = time.perf_counter()
        oracle.run_workload(w, n_threads=threads)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": T / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"one call (layer 0: {T} tokens, all {w.h_v} heads), fp64 recurrence, {dt:.1f} s",
            "s_per_48_calls": 48 * dt, "s_per_48_calls_kind": "the one-call time x 48"}
    return line


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--kernel", choices=["tc", "simt"], default="tc")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer timing")
    ap.add_argument("--subset-seqs", type=int, default=0,
                    help="time only the first K sequences of the batch (small profiling case)")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="seconds of untimed steps while the clock sampler warms up")
    ap.add_argument("--tree", action="store_true",
                    help="time the config 3 prefix tree (one launch vs level by level vs full paths)")
    ap.add_argument("--latency", action="store_true",
                    help="per-call latency of configs 0, 1, short two-chunk paths and the config 3 tree")
    ap.add_argument("--gated-rmsnorm", action="store_true",
                    help="time the gated RMSNorm on the 74-prompt batch's output shape")
    ap.add_argument("--input-prep", action="store_true",
                    help="time the GDN input prep (conv + SiLU + split, gates) on the 74-prompt batch")
    ap.add_argument("--long", action="store_true",
                    help="time one 16,384-token prompt: one call and 48 back-to-back calls (48 layers)")
    ap.add_argument("--no-long", action="store_true",
                    help="leave the long-prompt workload out of the default run's line")
    ap.add_argument("--layers", type=int, default=48,
                    help="--long: input sets drawn and timed back to back (48 = every linear-attention "
                         "layer; fewer only for short profiling runs)")
    args = ap.parse_args(argv)
    if args.long:
        run_long_bench(args)
        return
    if args.input_prep:
        run_prep_bench(args)
        return
    if args.gated_rmsnorm:
        run_norm_bench(args)
        return
    if args.latency:
        run_latency_bench(args)
        return
    if args.tree:
        run_tree_bench(args)
        return
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gdn(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    main()

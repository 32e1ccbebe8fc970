"""Benchmark of the SpecPrefill scoring path (token importance + chunk
selection).

Default workload (the headline): the 2B-draft-like prompt, N = 32768 prompt
tokens, 6 attention layers, 8 query / 2 KV heads, head_dim 256, 8 lookahead
queries, fixed keep fraction 0.15, W = 13 pool, 32-token chunks, boost, BOS
and the final chunk forced. `--workload` selects any workload of the scope
table (tiny, draft08b, draft2b, serving, long_fixed, long_mass).

One step = one call of the whole path (sp_specprefill_score) on one batch of
seeded synthetic inputs already resident in HBM. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--paged-block 8,16,...] [--legs a,b,...]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no cross-GPU exchange); the reported value is the tokens all
ranks scored divided by the slowest rank's time.

Timing: the clock sampler starts first (its start-up stays outside every
timed region); each timed region is preceded directly by its own warm-up
calls and a device synchronisation, then a short GPU sleep so that the host
can queue calls ahead of the device, then the start event, the K calls and
the stop event. `host_us_per_call` reports how long the host took to
enqueue one call.

`value` is the single-stream rate (one call after another on one stream).
Legs reported beside it (`--legs`): `pipelined`, the rate with
--pipeline-streams calls in flight on as many streams; `importance_paths`,
the importance phase with the tcgen05 logits kernel and with the CUDA-core
one; `listing_rule`, the same calls under the pages' own selection rule
(reference-compatibility mode); `head_pool`, the pool applied to every
attention row before the max; `paged_kv`, the keys read in place from
block-paged per-layer pools (one entry per --paged-block size); `draft_kv`,
the same scoring of a random-weight draft model's own cache (projected,
QK-normed, rotated keys of the prompt in 16-token blocks and the queries of
its lookahead tokens, synth/draft.py) at the workload's attention shape;
`consumer`, the bandwidth of the sparse-prefill gathers (kept token ids,
kept K and V rows).
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prompt tokens scored+selected/sec at N=32K; HBM GB/s vs GB300 peak"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
ALL_LEGS = ("e2e", "pipelined", "importance", "listing", "head_pool", "paged", "draft", "consumer")
# DRAM bytes (read + write) of one logits-kernel launch per workload, from an
# ncu application-replay capture of this bench's own calls; reported only
# while the kernel sources are the ones that were measured.
TRAFFIC = {"source_sha1": "3a1037bcb5c72f7db03760e08566114be940a9cf",
           "bytes_per_launch": {"draft2b": 202251904}}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="draft2b",
                    choices=["tiny", "draft08b", "draft2b", "serving", "long_fixed", "long_mass"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pipeline-streams", type=int, default=3,
                    help="streams of the pipelined-throughput leg")
    ap.add_argument("--paged-block", default="16",
                    help="comma-separated block sizes of the paged-key leg")
    ap.add_argument("--legs", default=",".join(ALL_LEGS),
                    help="comma-separated legs to run beside the headline (or 'none')")
    ap.add_argument("--copies", type=int, default=0,
                    help="rotating copies of the inputs (0: enough to exceed the L2)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="prompt length of a single-prompt workload (a smaller case of the same "
                         "kernels, e.g. for a profiler capture); 0 keeps the workload's")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


LOGITS_SOURCES = ("sp_logits_tc.cu", "sp_logits_phase.cuh", "sp_ptx.cuh", "sp_device.cuh")


def kernel_sha1():
    """Digest of the sources that define the logits kernel (the recorded
    DRAM traffic is only reported while they are unchanged)."""
    h = hashlib.sha1()
    for name in LOGITS_SOURCES:
        with open(os.path.join(ROOT, "speculative_prefill_token_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def describe(w, n_tokens):
    sel = (f"fixed p={w.keep_p:g}" if w.mode == "fixed" else f"mass {w.mass:g}")
    lens = (f"N={n_tokens}" if w.n_prompts == 1
            else f"{w.n_prompts} prompts, {n_tokens} tokens packed")
    return (f"{w.name}: {lens}, {w.n_layers} attention layers, {w.n_q_heads} query / "
            f"{w.n_kv_heads} KV heads, head_dim {w.head_dim}, {w.n_lookahead} lookahead queries, "
            f"W={w.pool_w}, C={w.chunk}, {sel}"
            + (", normalise" if w.normalize else "")
            + (", boost" if w.boost_first_mult != 1.0 or w.boost_last_mult != 1.0 else "")
            + ", BOS + final chunk forced")


class RawEvents:
    """CUDA events created through the process's CUDA runtime, so that the
    library can record them on its launch stream and we can read the elapsed
    time (torch's Event only times events that torch itself recorded)."""

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.rt = None
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                self.rt = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.rt is None:
            raise RuntimeError("CUDA runtime library not found")
        self.rt.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        self.rt.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p,
                                                 ctypes.c_void_p]
        self.rt.cudaEventDestroy.argtypes = [ctypes.c_void_p]
        self.made = []

    def pair(self):
        a, b = self.ct.c_void_p(), self.ct.c_void_p()
        assert self.rt.cudaEventCreate(self.ct.byref(a)) == 0
        assert self.rt.cudaEventCreate(self.ct.byref(b)) == 0
        self.made += [a, b]
        return _Ev(a.value), _Ev(b.value)

    def elapsed_ms(self, a, b):
        ms = self.ct.c_float()
        rc = self.rt.cudaEventElapsedTime(self.ct.byref(ms), a.cuda_event, b.cuda_event)
        assert rc == 0, f"cudaEventElapsedTime failed ({rc})"
        return float(ms.value)

    def close(self):
        for e in self.made:
            self.rt.cudaEventDestroy(e)
        self.made = []


class _Ev:
    def __init__(self, handle):
        self.cuda_event = handle


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed regions run."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(1.0)  # nvidia-smi's start (NVML initialisation) stays out of the timed regions
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        loaded = [v for v in sm if mx and v >= 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_inputs(name, tokens=0):
    from tests.gpu_helpers import workload_inputs
    if not tokens:
        return workload_inputs(name)
    from synth import get_workload, make_inputs as draw
    w = get_workload(name)
    if w.n_prompts != 1:
        raise SystemExit("--tokens applies to single-prompt workloads")
    w = w.with_(lengths=(int(tokens),))
    return w, draw(w)


def oracle_rate(w, inp, budget_s, max_runs=3):
    """Tokens per second of the float64 oracle as it stands on the full
    workload (repeated while it fits the time budget)."""
    import oracle
    kw = w.selection_kwargs()
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.run(inp.q, inp.k, inp.seq_off, **kw)
        runs += 1
        el = time.perf_counter() - t0
        if el + el / runs > budget_s or runs >= max_runs:
            break
    return runs * inp.n_tokens_total / el, runs, el


def oracle_sample_main(args):
    """Child process of cpu_baseline: the oracle with the thread count the
    parent set in the environment; prints one JSON line."""
    w, inp = make_inputs(args.workload)
    rate, runs, el = oracle_rate(w, inp, budget_s=10.0, max_runs=100)
    print(json.dumps({"value": rate, "runs": runs, "seconds": el}), flush=True)


def single_thread_rate(workload):
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample",
                            "--workload", workload], env=env, capture_output=True, text=True,
                           timeout=300)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as exc:  # reported, not fatal: the all-core figure stands
        return {"error": f"{type(exc).__name__}: {exc}"}


def cpu_baseline(w, inp):
    """The float64 oracle as it stands on the host cores: all cores (BLAS
    threads = host cores, in this process) and one thread (a child process
    with the BLAS thread count set to 1), each on the full workload."""
    rate, runs, el = oracle_rate(w, inp, budget_s=10.0, max_runs=100)
    one = single_thread_rate(w.name)
    return {"value": rate, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"full {w.name} workload (N={inp.n_tokens_total}) x{runs}, numpy float64, "
                      f"BLAS threads = host cores, {el:.1f} s; single-thread: "
                      f"x{one.get('runs')}, {one.get('seconds') or 0:.1f} s",
            "single_thread": {"value": one.get("value"), "unit": UNIT, "cores": 1,
                              "seconds": one.get("seconds"), "error": one.get("error")}}


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, on the same workload and
    config as the GPU arm (every step one full call)."""
    if rank != 0:
        return
    import oracle
    w, inp = make_inputs(args.workload)
    kw = w.selection_kwargs()
    for _ in range(args.warmup):
        oracle.run(inp.q, inp.k, inp.seq_off, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.run(inp.q, inp.k, inp.seq_off, **kw)
    el = time.perf_counter() - t0
    ntot = inp.n_tokens_total
    value = args.steps * ntot / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 Q/K with planted needles)",
            "config": {"workload": describe(w, ntot)},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"full {w.name} workload (N={ntot}) per step, numpy float64, "
                                       "BLAS threads = host cores"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


class Timer:
    """Device timing of K calls on one stream: warm-up calls, a device
    synchronisation, a GPU sleep that lets the host queue calls ahead, then
    events around the K calls."""

    PRIME_CYCLES = 1_000_000  # about 0.5 ms at the GB300's SM clock

    def __init__(self, torch, stream):
        self.torch = torch
        self.stream = stream

    def run(self, fn, steps, warmup, streams=None):
        torch = self.torch
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize()
        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(self.PRIME_CYCLES)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        for s in streams or ():
            s.wait_stream(self.stream)
        h0 = time.perf_counter()
        for i in range(steps):
            fn(i)
        host = time.perf_counter() - h0
        for s in streams or ():
            self.stream.wait_stream(s)
        t1.record(self.stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1), host


def max_over_ranks(values, world, device):
    """The element-wise maximum over the ranks of per-rank timings (ms):
    every rank gets it (one all-reduce; a single rank keeps its own)."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(world, ntot, steps, elapsed_ms):
    """Tokens per second of the whole job: every replica scores ntot tokens
    per step, and the slowest rank's timed region sets the time."""
    return world * ntot * steps / (elapsed_ms / 1e3)


def run_ours(args, rank, world, local):
    import torch
    import speculative_prefill_token_gb300 as sp
    from speculative_prefill_token_gb300 import _build

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    _build.build()
    sp.load()
    legs = set() if args.legs == "none" else set(args.legs.split(","))
    w, inp = make_inputs(args.workload, args.tokens)
    params = sp.SelectionParams(**w.selection_kwargs())
    ntot = inp.n_tokens_total
    q_np = np.ascontiguousarray(inp.q).view(np.int16)
    k_np = np.ascontiguousarray(inp.k).view(np.int16)
    # rotating copies: together larger than the 129 MB L2
    copies = args.copies or max(2, min(8, -(-(768 << 20) // max(k_np.nbytes, 1))))
    qs = [torch.from_numpy(q_np).to(dev) for _ in range(copies)]
    ks = [torch.from_numpy(k_np).to(dev) for _ in range(copies)]
    off = torch.from_numpy(np.asarray(inp.seq_off, dtype=np.int32)).to(dev)
    shape = sp.shape_of(qs[0], ks[0])
    ws = sp.make_workspace(shape, params, dev)
    out = sp.alloc_outputs(qs[0], ks[0], params, intermediates=False)
    stream = torch.cuda.current_stream()
    timer = Timer(torch, stream)
    k_bytes = shape.n_layers * shape.n_kv_heads * ntot * shape.head_dim * 2
    legs_out = {}

    def step(i, ev=None):
        sp.specprefill_score(qs[i % copies], ks[i % copies], off, params, out=out, ws=ws,
                             stream=stream, profile_events=ev)

    with ClockSampler(local) as clk:
        # whole-step timing: K back-to-back calls, no events inside the region
        if world > 1:
            torch.distributed.barrier()
        elapsed_ms, host_s = timer.run(step, args.steps, args.warmup)
        if world > 1:
            torch.distributed.barrier()
        status = sp.device_status(ws)
        n_kept = int(out.n_kept.item())

        # logits-kernel timing (roofline): the same steps again with events
        # recorded on the launch stream immediately around the logits kernel
        raw = RawEvents()
        evs = [raw.pair() for _ in range(args.steps)]
        timer.run(lambda i: step(i, evs[i]), args.steps, args.warmup)
        logits_ms = [raw.elapsed_ms(a, b) for a, b in evs]
        raw.close()

        if "pipelined" in legs and args.pipeline_streams > 1:
            legs_out["pipelined"] = leg_pipelined(sp, torch, args, timer, shape, params, qs, ks, off,
                                                  world, ntot, dev)
        if "importance" in legs:
            legs_out["importance_paths"] = leg_importance(sp, torch, args, timer, shape, params, qs,
                                                          ks, off, ntot, dev)
        if "listing" in legs:
            legs_out["listing_rule"] = leg_variant(
                sp, args, timer, w, shape, qs, ks, off, world, ntot, dev,
                "listing rule, min_tok 128, max_keep 2000", rule="listing", min_tok=128,
                max_keep=2000)
        if "head_pool" in legs:
            legs_out["head_pool"] = leg_variant(
                sp, args, timer, w, shape, qs, ks, off, world, ntot, dev,
                "W=13 pool on every attention row before the max", pool_at="head")
        if "paged" in legs:
            legs_out["paged_kv"] = [leg_paged(sp, torch, args, timer, shape, params, qs, ks, off,
                                              out, n_kept, world, ntot, dev, int(bs))
                                    for bs in args.paged_block.split(",") if bs]
        if "draft" in legs:
            legs_out["draft_kv"] = leg_draft(sp, torch, args, timer, w, params, world, dev)
        if "consumer" in legs:
            legs_out["consumer"] = leg_consumer(sp, torch, args, timer, shape, ks, out, n_kept,
                                                ntot, dev)
    if "e2e" in legs:
        e2e_ms, h2d, d2h = leg_e2e(sp, torch, args, shape, params, q_np, k_np, inp, qs, ks, off, out,
                                   ws, stream, ntot)
    else:
        e2e_ms, h2d, d2h = float("nan"), 0, 0

    # max over ranks of the timed regions
    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], world, dev)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    value = whole_job_rate(world, ntot, args.steps, elapsed_ms)
    peak, peak_kind = measured_peaks()
    avg_logits_s = statistics.mean(logits_ms) / 1e3
    achieved = k_bytes / avg_logits_s / 1e9
    rec = TRAFFIC["bytes_per_launch"].get(args.workload)
    traffic = rec if (rec is not None and TRAFFIC["source_sha1"] == kernel_sha1()) else None
    launches_per_step = sp.kernels_per_call(shape, params)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K with planted needles)",
        "config": {"workload": describe(w, ntot),
                   "l2": f"inputs larger than L2: {copies} rotating copies of the "
                         f"{k_np.nbytes / 1e6:.0f} MB key cache",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "logits_tc_kernel (tcgen05 + TMA)",
                     "algorithmic_bytes_per_launch": k_bytes,
                     "avg_launch_ms": avg_logits_s * 1e3, "peak_kind": f"{peak_kind} hbm_gbs"},
        "hbm_gbs_whole_step": k_bytes / (elapsed_ms / args.steps / 1e3) / 1e9,
        "host_us_per_call": 1e6 * host_s / args.steps,
        "clocks": clk.summary(),
        "e2e": {"value": world * ntot / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "kept_tokens": n_kept, "device_status": status,
    }
    line.update(legs_out)
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def leg_e2e(sp, torch, args, shape, params, q_np, k_np, inp, qs, ks, off, out, ws, stream, ntot):
    """End to end through the public API with host buffers: H2D of the
    step's inputs from pinned memory, the call, D2H of the kept lists."""
    q_host = torch.from_numpy(q_np).pin_memory()
    k_host = torch.from_numpy(k_np).pin_memory()
    off_host = torch.from_numpy(np.asarray(inp.seq_off, dtype=np.int32)).pin_memory()
    res_host = [torch.empty(ntot, dtype=torch.int32).pin_memory() for _ in range(2)]
    koff_host = torch.empty(shape.n_seqs + 1, dtype=torch.int32).pin_memory()
    nk_host = torch.empty(1, dtype=torch.int32).pin_memory()
    qd, kd, od = qs[0], ks[0], off
    e2e_steps = max(1, min(args.e2e_steps, args.steps))

    def e2e_step():
        qd.copy_(q_host, non_blocking=True)
        kd.copy_(k_host, non_blocking=True)
        od.copy_(off_host, non_blocking=True)
        sp.specprefill_score(qd, kd, od, params, out=out, ws=ws, stream=stream)
        res_host[0].copy_(out.kept_idx, non_blocking=True)
        res_host[1].copy_(out.kept_pos, non_blocking=True)
        koff_host.copy_(out.kept_off, non_blocking=True)
        nk_host.copy_(out.n_kept, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    h2d = q_np.nbytes + k_np.nbytes + off_host.numel() * 4
    d2h = 2 * ntot * 4 + koff_host.numel() * 4 + 4
    return e0.elapsed_time(e1) / e2e_steps, h2d, d2h


def leg_pipelined(sp, torch, args, timer, shape, params, qs, ks, off, world, ntot, dev):
    """S calls in flight on S streams, each with its own workspace and
    outputs, as a server scoring a stream of requests would run them; one
    call's latency-bound selection overlaps the next call's key stream."""
    S = args.pipeline_streams
    copies = len(ks)
    p_streams = [torch.cuda.Stream(device=dev) for _ in range(S)]
    p_ws = [sp.make_workspace(shape, params, dev) for _ in range(S)]
    p_out = [sp.alloc_outputs(qs[0], ks[0], params, intermediates=False) for _ in range(S)]

    def p_step(i):
        j = i % S
        sp.specprefill_score(qs[i % copies], ks[i % copies], off, params, out=p_out[j], ws=p_ws[j],
                             stream=p_streams[j])

    p_ms, _ = timer.run(p_step, args.steps, max(args.warmup, S), streams=p_streams)
    p_ok = all(sp.device_status(x) == 0 for x in p_ws)
    return {"streams": S, "value": world * ntot * args.steps / (p_ms / 1e3), "unit": UNIT,
            "ms_per_step": p_ms / args.steps, "device_status_ok": p_ok}


def leg_variant(sp, args, timer, w, shape, qs, ks, off, world, ntot, dev, what, **over):
    """The same calls with other selection settings."""
    v_params = sp.SelectionParams(**dict(w.selection_kwargs(), **over))
    v_ws = sp.make_workspace(shape, v_params, dev)
    v_out = sp.alloc_outputs(qs[0], ks[0], v_params, intermediates=False)
    copies = len(ks)

    def v_step(i):
        sp.specprefill_score(qs[i % copies], ks[i % copies], off, v_params, out=v_out, ws=v_ws,
                             stream=timer.stream)

    v_ms, _ = timer.run(v_step, args.steps, args.warmup)
    v_ms /= args.steps
    return {"what": what, "ms_per_step": v_ms, "value": world * ntot / (v_ms / 1e3), "unit": UNIT,
            "kernels_per_step": sp.kernels_per_call(shape, v_params),
            "kept_tokens": int(v_out.n_kept.item()), "device_status": sp.device_status(v_ws)}


def leg_importance(sp, torch, args, timer, shape, params, qs, ks, off, ntot, dev):
    """The tensor-core choice: token importance (prep, logits and importance
    kernels) with the tcgen05 logits kernel against the CUDA-core (fp32 FMA)
    logits kernel of the same path."""
    imp_buf = torch.empty(ntot, dtype=torch.float32, device=dev)
    imp_ws = sp.make_workspace(shape, params, dev)
    copies = len(ks)

    def imp_ms(simt):
        def f(i):
            sp.attn_importance(qs[i % copies], ks[i % copies], off, params, imp=imp_buf, ws=imp_ws,
                               stream=timer.stream, simt=simt)
        steps = args.steps if not simt else max(3, args.steps // 10)
        return timer.run(f, steps, args.warmup)[0] / steps

    tc, simt = imp_ms(False), imp_ms(True)
    return {"what": "token importance only (prep, logits, importance kernels)",
            "tcgen05_ms": tc, "simt_fp32_ms": simt, "simt_over_tcgen05": simt / tc,
            "device_status": sp.device_status(imp_ws)}


def leg_paged(sp, torch, args, timer, shape, params, qs, ks, off, out, n_kept, world, ntot, dev, bs):
    """Keys read in place from a block-paged draft cache: one pool of bs-token
    blocks per layer, the batch's blocks shuffled over the pool (a copy of
    the same keys per rotation, so the inputs stay larger than L2)."""
    ly, hk, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
    seq = off.cpu().numpy().astype(np.int64)
    lengths = np.diff(seq)
    nblk_b = -(-lengths // bs)
    nblk = int(nblk_b.sum())
    maxb = int(max(1, nblk_b.max()))
    perm = np.random.default_rng(bs).permutation(nblk)
    table_np = np.zeros((len(lengths), maxb), dtype=np.int32)
    # logical block j of prompt b -> pool block perm[first_b + j]
    src_rows = np.zeros(nblk * bs, dtype=np.int64)
    first = 0
    for b, (n, nb) in enumerate(zip(lengths, nblk_b)):
        table_np[b, :nb] = perm[first:first + nb]
        for j in range(int(nb)):
            t = np.minimum(np.arange(j * bs, (j + 1) * bs), max(int(n) - 1, 0))
            src_rows[perm[first + j] * bs:(perm[first + j] + 1) * bs] = seq[b] + t
        first += int(nb)
    table = torch.from_numpy(table_np).to(dev)
    rows = torch.from_numpy(src_rows).to(dev)
    pools = []
    for x in ks:
        kk = x.view(torch.bfloat16).view(ly, ntot, hk, d)
        pools.append([kk[l].index_select(0, rows).view(nblk, bs, hk, d) for l in range(ly)])
    kv_shape = sp.shape_of_kv(qs[0], pools[0], ntot, table)
    kv_ws = sp.make_workspace(kv_shape, params, dev)
    kv_out = sp.alloc_outputs(qs[0], ks[0], params, intermediates=False)
    copies = len(ks)

    def kv_step(i):
        sp.specprefill_score_kv(qs[i % copies], pools[i % copies], off, ntot, params,
                                block_table=table, out=kv_out, ws=kv_ws, stream=timer.stream)

    kv_ms, _ = timer.run(kv_step, args.steps, args.warmup)
    kv_ms /= args.steps
    nk = int(kv_out.n_kept.item())
    res = {"what": f"keys read in place from per-layer pools of {bs}-token blocks (shuffled)",
           "block_size": bs, "ms_per_step": kv_ms, "value": world * ntot / (kv_ms / 1e3),
           "unit": UNIT, "kept_tokens": nk, "device_status": sp.device_status(kv_ws),
           "same_kept_as_dense": bool(nk == n_kept and torch.equal(kv_out.kept_idx[:nk],
                                                                   out.kept_idx[:nk]))}
    del pools
    torch.cuda.empty_cache()
    return res


def leg_draft(sp, torch, args, timer, w, params, world, dev):
    """Keys and lookahead queries of a random-weight draft model with the
    workload's attention shape and prompt lengths (hidden 2048 for 32K-token
    prompts, else 1024), its cache in 16-token blocks shuffled over one pool
    per layer, scored in place; the kept lists are compared with the dense
    call on the same keys."""
    from synth import DraftShape, draft_attention_inputs, page_keys
    from synth.inputs import prompt_lengths
    lengths = prompt_lengths(w)
    t0 = time.perf_counter()
    shape_d = DraftShape(hidden=2048 if int(lengths.sum()) >= 32768 else 1024, n_layers=w.n_layers,
                         n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                         n_lookahead=w.n_lookahead, rotary_dim=w.head_dim // 4, seed=2002)
    q_np, k_np, off_np = draft_attention_inputs(shape_d, lengths)
    pools_np, table_np = page_keys(k_np, off_np, 16, seed=2)
    build_s = time.perf_counter() - t0
    ntot = int(off_np[-1])
    qd = torch.from_numpy(np.ascontiguousarray(q_np).view(np.int16)).to(dev)
    od = torch.from_numpy(off_np).to(dev)
    td = torch.from_numpy(table_np).to(dev)
    copies = max(2, min(4, -(-(768 << 20) // max(k_np.nbytes, 1))))
    pools = [[torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in pools_np]
             for _ in range(copies)]
    kv_shape = sp.shape_of_kv(qd, pools[0], ntot, td)
    kv_ws = sp.make_workspace(kv_shape, params, dev)
    nb = len(lengths)
    kv_out = sp.ScoreOutputs(kept_idx=torch.empty(ntot, dtype=torch.int32, device=dev),
                             kept_pos=torch.empty(ntot, dtype=torch.int32, device=dev),
                             kept_off=torch.empty(nb + 1, dtype=torch.int32, device=dev),
                             n_kept=torch.empty(1, dtype=torch.int32, device=dev))

    def d_step(i):
        sp.specprefill_score_kv(qd, pools[i % copies], od, ntot, params, block_table=td, out=kv_out,
                                ws=kv_ws, stream=timer.stream)

    d_ms, _ = timer.run(d_step, args.steps, args.warmup)
    d_ms /= args.steps
    nk = int(kv_out.n_kept.item())
    kd = torch.from_numpy(np.ascontiguousarray(k_np).view(np.int16)).to(dev)
    flat = sp.specprefill_score(qd, kd, od, params)
    same = bool(int(flat.n_kept.item()) == nk and torch.equal(flat.kept_idx[:nk], kv_out.kept_idx[:nk]))
    res = {"what": f"random-weight draft (hidden {shape_d.hidden}, QK-norm, RoPE on {shape_d.rotary_dim} of "
                   f"{shape_d.head_dim} dims), cache in 16-token blocks scored in place",
           "ms_per_step": d_ms, "value": world * ntot / (d_ms / 1e3), "unit": UNIT, "kept_tokens": nk,
           "device_status": sp.device_status(kv_ws), "same_kept_as_dense": same,
           "fixture_build_s": build_s}
    del pools, kd
    torch.cuda.empty_cache()
    return res


def leg_consumer(sp, torch, args, timer, shape, ks, out, n_kept, ntot, dev):
    """Sparse-prefill consumer: the kept tokens' ids and their K and V rows
    (two draft-cache tensors) gathered on the device from the scoring
    call's kept list."""
    ly, hk, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
    kb = [x.view(torch.bfloat16).view(ly, ntot, hk, d) for x in ks]
    copies = len(kb)
    ids = torch.arange(ntot, dtype=torch.int32, device=dev)
    tok_out = torch.empty(ntot, dtype=torch.int32, device=dev)
    rows_out = [torch.empty_like(kb[0]) for _ in range(2)]

    def c_step(i):
        sp.gather_tokens(ids, out.kept_idx, out.n_kept, out=tok_out, stream=timer.stream)
        for j in range(2):
            sp.gather_rows(kb[(2 * i + j) % copies], out.kept_idx, out.n_kept, out=rows_out[j],
                           stream=timer.stream)

    c_ms, _ = timer.run(c_step, args.steps, args.warmup)
    c_ms /= args.steps
    c_bytes = 2 * 2 * n_kept * ly * hk * d * 2 + n_kept * 12
    ref_rows = kb[0][:, out.kept_idx[:n_kept].long()]
    c_ok = bool(torch.equal(rows_out[0][:, :n_kept], ref_rows))   # every copy holds the same keys
    peak, _ = measured_peaks()
    gbs = c_bytes / (c_ms / 1e3) / 1e9
    return {"what": "kept token ids + kept K and V rows (gather_tokens, 2x gather_rows)",
            "ms_per_step": c_ms, "bytes_per_step": c_bytes, "gbs": gbs, "frac": gbs / peak,
            "kernels_per_step": 3, "rows_match_torch_index": c_ok}


def main():
    args = parse()
    if args.oracle_sample:
        oracle_sample_main(args)
        return
    rank, world, local = dist_info()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()

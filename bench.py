"""Throughput of the selected-token logprob on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl rlk|reference]

One step = one pass of the whole path over one packed batch of the
Qwen3-8B-shaped head (T=4096 tokens = 8 x 512, H=4096, V=151936, bf16, 4
vocabulary shards): the logits GEMM with the fused tile epilogue, then the
tile tree, shard records and final lse/logprob.  Inputs are synthetic and
seeded (see invariant_selected_token_gb300/workloads.py) and resident in HBM
before the timed region; W (1.24 GB) is larger than L2, so no flush is
needed between steps.  Prints one JSON line (rank 0).

With --gpus N > 1 (launched by torchrun) each rank runs its own independent
batch against its own copy of W -- the path shards over tokens with no data
exchange -- and `value` is the tokens of all ranks over the slowest rank's
time (weak scaling).

--impl reference times the fp64 CPU oracle on the host cores instead
(bounded samples of the same batch), on rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, V, T_PACKED, N_SHARDS = 4096, 151936, 4096, 4
METRIC = "selected-logprob tokens/s at H=4096,V=151936 bf16; % of roofline; mismatch=0"
WORKLOAD = "packed training batch T=4096 (8x512), H=4096, V=151936, bf16, 4 vocab shards"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="rlk", choices=["rlk", "reference"])
    p.add_argument("--workload", default="packed",
                   choices=["packed", "decode1", "decode8", "decode64", "decode128", "decode256",
                            "decode512",
                            "logits_fp32", "logits_bf16", "log_softmax_fp32", "backward",
                            "train_step", "grpo",
                            "rmsnorm", "rmsnorm16k", "sweep"],
                   help="packed: the T=4096 training batch (the headline); decodeN: N rows of it "
                        "as a rollout-side decode batch; logits_*: the same batch's logits "
                        "materialised in HBM, reduced by the materialised-logits path; "
                        "log_softmax_fp32: the full log_softmax [T, V] of those logits; "
                        "backward: the deterministic backward of the packed batch; train_step: "
                        "forward + backward of it, the forward saving its fp32 logits for the "
                        "backward (the recomputing pair timed beside it); grpo: the "
                        "long-response GRPO batch (64 sequences, ~221 k rows in 8192-row calls); "
                        "rmsnorm: the strict RMSNorm (residual in and out) that produces the "
                        "packed batch's hidden states (L2 flushed between calls); rmsnorm16k: the "
                        "same on 16384 rows, inputs larger than L2 and no flush; sweep: tokens/s against batch size on the "
                        "8192-token sweep set")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self, t0=None, t1=None):
        """Summary of the samples taken between host times t0 and t1 (all if too few)."""
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        import datetime
        rows = []
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), float(f[4]) if f[4] else 0.0, f[6:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        use = inside if len(inside) >= 2 else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for n, v in zip(names, r[4]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use),
                "power_w_max": max(r[3] for r in use), "samples": len(use),
                "samples_in_timed_region": len(inside), "reasons": sorted(reasons)}


def k1_traffic_record(workload):
    """Per-launch DRAM bytes of the tile-partials kernel from the committed ncu summary of
    this workload, if the loaded library was built from the sources here and the kernel's
    translation unit is the one the counters were taken from (else None)."""
    path = os.path.join(ROOT, "profiles", "tile_partials_%s.md" % workload)
    try:
        import re
        from invariant_selected_token_gb300 import binding
        from invariant_selected_token_gb300 import build as lib_build
        loaded = binding.build_fingerprint().split("rev=")[1].split(";")[0]
        if loaded != "src-" + lib_build.source_digest():
            return None
        rec = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.strip().startswith("- "):
                    k, v = line.strip()[2:].split(":", 1)
                    rec[k.strip()] = v.strip().strip("`")
        if rec.get("kernel_unit_rev", "").split()[0].strip("`") == lib_build.unit_digest("rlk_logits.cu"):
            return int(re.search(r"\d+", rec["dram_bytes_per_launch"]).group(0))
    except Exception:
        pass
    return None


def rank_batch_seed(rank: int) -> int:
    """Seed of a rank's own batch: ranks share W but never a token."""
    return 1234 + 1000 * rank


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time (every rank gets it); identity without a process group."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, tokens_per_rank: int, steps: int, ms_total: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / (ms_total / 1000.0)


def timed_steps(step, K, stream):
    """Run K steps between two events on `stream`, each step also recording events around
    its logits-kernel launch.  Returns (total ms of the K steps, mean ms of the kernel
    launches, how many were timed).  Every kernel interval lies inside the region and the
    intervals do not overlap, so the kernel time can never exceed the step time.  (With no
    event between them, a step's kernels overlap their neighbours' launch and set-up
    through programmatic dependent launch, and the step can be shorter than one kernel
    timed alone; the events here cost every step that overlap.)"""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(K):
        step(*ev[k])
    end.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    return total, statistics.mean(a.elapsed_time(b) for a, b in ev), len(ev)


DECODE_SIZES = (1, 64)
DECODE_STEPS = 200


def decode_record(n, W, hidden, targets, out_lp, out_lse, binding, WL, dev, stream, status,
                  peaks):
    """One decode batch of n rows of the packed batch (the rollout side's call), timed as
    the packed steps are: step rate and logits-kernel time over DECODE_STEPS steps,
    against the HBM roofline (W + the n hidden rows read once).
    Its outputs must equal the packed run's outputs for the same rows bit for bit."""
    import torch
    idx = torch.from_numpy(WL.decode_rows(n)).to(dev)
    h, tg = hidden[idx].contiguous(), targets[idx].contiguous()
    ws = binding.new_workspace(n, V, N_SHARDS, dev)
    lp = torch.empty(n, dtype=torch.float32, device=dev)
    lse = torch.empty(n, dtype=torch.float32, device=dev)

    def step(ev0=None, ev1=None):
        if ev0 is not None:
            ev0.record(stream)
        binding.tile_partials(h, W, tg, None, N_SHARDS, ws, status, stream)
        if ev1 is not None:
            ev1.record(stream)
        binding.tile_merge(tg, None, V, N_SHARDS, lp, lse, ws, status, stream)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    ms_total, k_ms, n_k = timed_steps(step, DECODE_STEPS, stream)
    binding.raise_on_device_status(status)
    step_ms = ms_total / DECODE_STEPS
    check_kernel_within_step(k_ms, step_ms)
    nbytes = float(W.numel() * 2 + h.numel() * 2)
    mism = sum(int((a.view(torch.int32) != b.view(torch.int32)).sum().item())
               for a, b in ((lp, out_lp[idx]), (lse, out_lse[idx])))
    maxd = max(float((a.double() - b.double()).abs().max().item())
               for a, b in ((lp, out_lp[idx]), (lse, out_lse[idx])))
    achieved = nbytes / (k_ms / 1000.0) / 1e9
    return {"T": n, "steps": DECODE_STEPS, "ms_per_step": round(step_ms, 5),
            "tokens_per_s": n / (step_ms / 1000.0), "kernel_ms": round(k_ms, 5),
            "kernel_launches_timed": n_k, "gpu_launches": 2 * DECODE_STEPS, "bound": "hbm",
            "bytes": nbytes,
            "achieved_gbs": round(achieved, 1), "peak_gbs": peaks["hbm_gbs"],
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "step_frac": round(nbytes / (step_ms / 1000.0) / 1e9 / peaks["hbm_gbs"], 4),
            "invariance_vs_packed": {"mismatch_count": mism, "max_abs_diff": maxd}}


def check_kernel_within_step(kernel_ms, step_ms):
    """The logits kernel is one part of a step: its time cannot exceed the step's.  A
    violation means the two were not measured on the same work, so refuse the line."""
    if kernel_ms > step_ms:
        raise SystemExit("bench: logits kernel %.4f ms > step %.4f ms -- inconsistent timing"
                         % (kernel_ms, step_ms))


def cpu_oracle_sample(hidden_bits, W_bits, targets, rows, want_values=False):
    """Time the fp64 oracle on the listed rows; returns (seconds, rows) and, with
    want_values, also its (logprob, lse) for those rows."""
    from oracle import linear_logprob as oracle
    t0 = time.perf_counter()
    lp, lse = oracle.selected_logprob(hidden_bits, W_bits, targets, rows=rows)
    took = time.perf_counter() - t0, (hidden_bits.shape[0] if rows is None else len(rows))
    return took + (lp, lse) if want_values else took


def hardware_fingerprint(dev):
    import torch
    p = torch.cuda.get_device_properties(dev)
    driver = None
    try:
        driver = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                                 "-i", str(dev.index or 0)], capture_output=True, text=True,
                                timeout=10).stdout.strip() or None
    except Exception:
        pass
    return {"device": p.name, "sm_count": p.multi_processor_count,
            "cc": "%d.%d" % (p.major, p.minor), "memory_gb": round(p.total_memory / 1e9, 1),
            "driver": driver, "torch": torch.__version__}


def diff_stats(d):
    import numpy as np
    d = np.asarray(d, dtype=np.float64)
    return {"mean": float(d.mean()), "max": float(d.max()), "p50": float(np.percentile(d, 50)),
            "p90": float(np.percentile(d, 90)), "p99": float(np.percentile(d, 99))}


def host_threads() -> int:
    """Host cores this process may run on (the oracle's BLAS and OpenMP threads use them)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def reference_arm(args, rank, world):
    if rank != 0:
        return 0
    import numpy as np
    from invariant_selected_token_gb300 import workloads as WL
    # the same batch as the GPU arm, generated on the CPU when no GPU is used
    import torch
    if torch.cuda.is_available():
        dev = torch.device("cuda:0")
        W = WL.head_weights(dev)
        pk = WL.packed(W, dev)
        hid_bits = WL.bf16_tensor_bits(pk.hidden)
        tg = pk.targets.cpu().numpy()
    else:  # same shapes and distributions; uniform targets (they do not change the cost)
        dev = torch.device("cpu")
        W = WL.head_weights(dev)
        hid_bits = WL.bf16_tensor_bits(WL.rms_hidden(T_PACKED, H, dev, 1234))
        tg = np.random.default_rng(1234).integers(0, V, T_PACKED).astype(np.int32)
    W_bits = WL.bf16_tensor_bits(W)
    # A bounded sample per step.  Each oracle call first decodes all of W to fp64
    # (~0.7 s on 16 host cores), so rows are taken in batches large enough for the
    # call to be mostly dot products: 64 rows per step at the default 300 steps
    # (~4 minutes), up to 512 for shorter runs.
    K = max(1, args.steps)
    rows_per_step = 64 if K >= 100 else min(512, max(64, 6400 // K))
    rng = np.random.default_rng(4321)
    for _ in range(args.warmup):
        cpu_oracle_sample(hid_bits, W_bits, tg, rng.choice(T_PACKED, 2, replace=False))
    times = []
    for _ in range(args.steps):
        s, n = cpu_oracle_sample(hid_bits, W_bits, tg, rng.choice(T_PACKED, rows_per_step, replace=False))
        times.append(s)
    total = sum(times)
    value = args.steps * rows_per_step / total
    cores = host_threads()
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "impl": "reference",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "T": T_PACKED, "H": H, "V": V, "n_shards": N_SHARDS,
                      "sample": "%d seeded rows of the batch per step" % rows_per_step},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": "%d steps x %d rows of the packed batch, full vocabulary"
                                      % (args.steps, rows_per_step)},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


# FMA-pipe lanes per SM (4 sub-partitions x 32): the unit count of the
# materialised path's arithmetic roofline.
FMA_LANES_PER_SM = 128
# FMA-pipe lane operations per logit that the numeric contract fixes on the
# materialised path: subtract the tile max (1); exp: t = fma (1), n = t -
# shift (1), r in two fmas (2), degree-7 Horner (7), scale multiply (1); the
# tree add (1).  Packed two-lane instructions halve the issue slots, not
# these operations.
FMA_OPS_PER_LOGIT = 14


def materialised_arm(args, rank, world, dev, dist, W, pk, binding, WL):
    """Selected logprob from the packed batch's logits materialised in HBM."""
    import torch
    T = pk.hidden.shape[0]
    L = binding.debug_logits(pk.hidden, W)
    if args.workload == "logits_bf16":
        L = L.to(torch.bfloat16)
    del W
    torch.cuda.empty_cache()
    ws = binding.new_workspace(T, V, N_SHARDS, dev)
    lp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    status = binding.new_status(dev)
    stream = torch.cuda.current_stream(dev)

    full = args.workload == "log_softmax_fp32"
    out_full = torch.empty((T, V), dtype=torch.float32, device=dev) if full else None
    ws_full = binding.new_workspace(T, V, 1, dev) if full else None

    def step():
        if full:
            binding.log_softmax(L, None, out_full, lse, ws_full, status, stream)
        else:
            binding.logits_logprob(L, pk.targets, None, N_SHARDS, lp, lse, ws, status, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    binding.raise_on_device_status(status)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(int(str(dev).split(":")[-1]) if ":" in str(dev) else 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(t0, time.time())
    ms_total = sum(a.elapsed_time(b) for a, b in ev)
    ms_total = max_over_ranks(ms_total, dist, dev)
    call_ms = ms_total / K
    nbytes = float(L.numel() * L.element_size())
    if full:  # the logits are read twice (tile pairs, then the output pass); T x V written
        nbytes = 3.0 * L.numel() * 4
    peaks = load_peaks()
    sm_hz = ((clk or {}).get("sm_max_mhz") or 2070.0) * 1e6
    peak_ops = FMA_LANES_PER_SM * torch.cuda.get_device_properties(dev).multi_processor_count * sm_hz
    ops = FMA_OPS_PER_LOGIT * float(T) * V
    t_alu = ops / peak_ops
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    call_s = call_ms / 1000.0
    common = {"kernel": ("k_mat_tile_partials + k_tile_tree + k_log_softmax_out (whole call)"
                         if full else "k_mat_tile_partials + k_tile_tree (whole call)"),
              "traffic": None,
              "kernel_ms": round(call_ms, 4),
              "algorithmic": {"bytes": nbytes, "fma_ops": ops,
                              "fma_ops_per_logit": FMA_OPS_PER_LOGIT},
              "roofline_ms": {"hbm": round(t_hbm * 1000, 4), "fma_pipe": round(t_alu * 1000, 4)}}
    if t_hbm >= t_alu:
        achieved = nbytes / call_s / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "peak_kind": "copy bandwidth (%s)" % peaks["source"]}
    else:
        achieved = ops / call_s / 1e9
        roofline = {"bound": "alu", "achieved": round(achieved, 1),
                    "peak": round(peak_ops / 1e9, 1), "unit": "Gop/s",
                    "frac": round(achieved / (peak_ops / 1e9), 4),
                    "peak_kind": "FMA-pipe lane operations: 128 lanes/SM x SMs x max SM clock"}
    roofline.update(common)
    if rank == 0:
        out = {"metric": METRIC, "value": weak_scaling_value(world, T, K, ms_total),
               "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
               "ms_per_step": call_ms, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "bf16" if args.workload == "logits_bf16" else "f32",
               "data": "synthetic",
               "config": {"workload": ("full log_softmax [T, V] fp32 of the packed batch's "
                                       "materialised fp32 logits (T=4096, V=151936)") if full else
                                      ("materialised logits of the packed batch (T=4096, "
                                       "V=151936, %s), 4 vocab shards" % args.workload[7:]),
                          "T": T, "V": V, "n_shards": N_SHARDS,
                          "l2": "inputs larger than L2 (logits %.2f GB)" % (nbytes / 1e9)},
               "roofline": roofline,
               "cpu_baseline": None, "e2e": None, "gpu_launches": 2 * K, "clocks": clk,
               "contract": binding.contract_id(), "build": binding.build_fingerprint()}
        print(json.dumps(out))
    return 0


def grpo_arm(args, rank, world, dev, dist, W, binding, WL):
    """The long-response GRPO batch: 8 prompts x 8 samples, prompt rows inactive, response
    rows active, packed back to back and processed in 8192-row calls.  One step = every
    call of the batch; tokens counted are the active (response) rows."""
    import torch
    g = WL.grpo_long(W, dev, seed=1235 + 1000 * rank)
    chunks = g.meta["chunks"]
    N = g.hidden.shape[0]
    n_active = int(g.active.sum().item())
    rows_max = max(r1 - r0 for r0, r1 in chunks)
    ws = binding.new_workspace(rows_max, V, N_SHARDS, dev)
    out_lp = torch.empty(N, dtype=torch.float32, device=dev)
    out_lse = torch.empty(N, dtype=torch.float32, device=dev)
    status = binding.new_status(dev)
    stream = torch.cuda.current_stream(dev)

    def step(k1_events=None):
        for i, (r0, r1) in enumerate(chunks):
            if k1_events is not None:
                k1_events[i][0].record(stream)
            binding.tile_partials(g.hidden[r0:r1], W, g.targets[r0:r1], g.active[r0:r1],
                                  N_SHARDS, ws, status, stream)
            if k1_events is not None:
                k1_events[i][1].record(stream)
            binding.tile_merge(g.targets[r0:r1], g.active[r0:r1], V, N_SHARDS, out_lp[r0:r1],
                               out_lse[r0:r1], ws, status, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    binding.raise_on_device_status(status)
    K = args.steps
    k1_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in chunks] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(int(str(dev).split(":")[-1]) if ":" in str(dev) else 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    start.record(stream)
    for k in range(K):
        step(k1_ev[k])
    end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(t0, time.time())
    binding.raise_on_device_status(status)
    ms_total = max_over_ranks(start.elapsed_time(end), dist, dev)
    k1_ms_step = statistics.mean(sum(a.elapsed_time(b) for a, b in ev) for ev in k1_ev)

    e2e = None
    if not args.no_e2e:
        h_hidden = g.hidden.cpu().pin_memory()
        h_tg = g.targets.cpu().pin_memory()
        h_act = g.active.cpu().pin_memory()
        h_lp = torch.empty(N, dtype=torch.float32).pin_memory()
        h_lse = torch.empty(N, dtype=torch.float32).pin_memory()
        d_hidden = torch.empty_like(g.hidden)
        d_tg = torch.empty_like(g.targets)
        d_act = torch.empty_like(g.active)

        # chunk i+1's inputs cross to the device on a copy stream while chunk i
        # computes; each chunk's call waits for its own copy
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in chunks]
        computed = torch.cuda.Event()

        def e2e_step():
            copy_stream.wait_event(computed)  # the previous step is done with the buffers
            with torch.cuda.stream(copy_stream):
                for i, (r0, r1) in enumerate(chunks):
                    d_hidden[r0:r1].copy_(h_hidden[r0:r1], non_blocking=True)
                    d_tg[r0:r1].copy_(h_tg[r0:r1], non_blocking=True)
                    d_act[r0:r1].copy_(h_act[r0:r1], non_blocking=True)
                    copied[i].record(copy_stream)
            for i, (r0, r1) in enumerate(chunks):
                stream.wait_event(copied[i])
                binding.linear_logprob(d_hidden[r0:r1], W, d_tg[r0:r1], d_act[r0:r1], N_SHARDS,
                                       out_lp[r0:r1], out_lse[r0:r1], ws, status, stream)
            h_lp.copy_(out_lp, non_blocking=True)
            h_lse.copy_(out_lse, non_blocking=True)
            computed.record(stream)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)  # no copy of the timed steps starts before e0
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
        e2e = {"value": weak_scaling_value(world, n_active, K, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": int(N * (H * 2 + 4 + 1)),
               "d2h_bytes_per_step": int(N * 8),
               "copies": "per 8192-row chunk on a second stream, overlapping the previous "
                         "chunk's compute; results read back once per step"}

    peaks = load_peaks()
    flops = 2.0 * N * H * V  # every row of every call goes through the GEMM
    achieved = flops / (k1_ms_step / 1000.0) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": None, "peak_kind": "burst bf16 (%s)" % peaks["source"],
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "kernel": "k_tile_partials", "kernel_ms_per_step": round(k1_ms_step, 4),
                "launches_per_step": len(chunks),
                "algorithmic": {"flops_per_step": flops, "rows_per_step": N,
                                "active_rows_per_step": n_active}}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        act_rows = torch.nonzero(g.active).flatten().cpu().numpy()
        rows = act_rows[WL.permutation(len(act_rows), 4321)[:2048]]
        W_bits = WL.bf16_tensor_bits(W)
        hid_bits = WL.bf16_tensor_bits(g.hidden[torch.from_numpy(rows).to(dev)])
        s_, n_ = cpu_oracle_sample(hid_bits, W_bits, g.targets.cpu().numpy()[rows], None)
        cpu = {"value": n_ / s_, "unit": "tokens/s", "cores": host_threads(), "kind": "oracle",
               "sample": "%d active rows of the batch over the full vocabulary (%.1f s)" % (n_, s_)}
    if rank == 0:
        ms_per_step = ms_total / K
        out = {"metric": METRIC, "value": weak_scaling_value(world, n_active, K, ms_total),
               "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
               "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": "long-response GRPO batch: 8 prompts x 8 samples, prompt "
                                      "U[64,512] rows inactive, response U[256,6912] rows active, "
                                      "%d rows (%d active) in %d calls of <= 8192 rows, H=4096, "
                                      "V=151936, bf16, 4 vocab shards" % (N, n_active, len(chunks)),
                          "rows": N, "active_rows": n_active, "calls_per_step": len(chunks),
                          "tokens_counted": "active rows", "H": H, "V": V, "n_shards": N_SHARDS,
                          "l2": "inputs larger than L2 (W = 1.24 GB, hidden %.2f GB)"
                                % (N * H * 2 / 1e9),
                          "parallelism": "dp%d (independent batches)" % world},
               "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": 2 * len(chunks) * K, "clocks": clk,
               "contract": binding.contract_id(), "build": binding.build_fingerprint()}
        print(json.dumps(out))
    return 0


SWEEP_SIZES = (1, 7, 64, 1024, 8192)


def sweep_arm(args, rank, world, dev, dist, W, binding, WL):
    """Tokens/s against batch size: the 8192-token sweep set cut into consecutive batches
    of T rows (the last one ragged), each batch one rlk_tile_partials + rlk_tile_merge,
    4 shards.  One step = one pass over all 8192 tokens at that T; `value` is the
    T = 8192 point, the curve lists every T."""
    import torch
    sw = WL.sweep_set(W, dev, seed=1236 + 1000 * rank)
    N = sw.hidden.shape[0]
    ws = binding.new_workspace(max(SWEEP_SIZES), V, N_SHARDS, dev)
    out_lp = torch.empty(N, dtype=torch.float32, device=dev)
    out_lse = torch.empty(N, dtype=torch.float32, device=dev)
    status = binding.new_status(dev)
    stream = torch.cuda.current_stream(dev)
    curve = {}
    clk = None
    for T in SWEEP_SIZES:
        batches = [(r0, min(N, r0 + T)) for r0 in range(0, N, T)]

        def step():
            for r0, r1 in batches:
                binding.tile_partials(sw.hidden[r0:r1], W, sw.targets[r0:r1], None, N_SHARDS, ws,
                                      status, stream)
                binding.tile_merge(sw.targets[r0:r1], None, V, N_SHARDS, out_lp[r0:r1],
                                   out_lse[r0:r1], ws, status, stream)

        # a pass over 8192 tokens at T = 1 is 8192 calls: fewer steps for small T
        K = max(1, min(args.steps, 8 if T < 64 else args.steps))
        for _ in range(max(3, args.warmup) if T >= 64 else 1):
            step()
        torch.cuda.synchronize()
        clocks = ClockSampler(int(str(dev).split(":")[-1]) if ":" in str(dev) else 0)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        clocks.start()
        time.sleep(0.3)
        t0 = time.time()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        c = clocks.stop(t0, time.time())
        binding.raise_on_device_status(status)
        ms = max_over_ranks(a.elapsed_time(b), dist, dev)
        curve[str(T)] = {"tokens_per_s": weak_scaling_value(world, N, K, ms),
                         "ms_per_pass": ms / K, "calls_per_pass": len(batches), "passes": K,
                         "sm_mhz": (c or {}).get("sm_mhz")}
        if T == max(SWEEP_SIZES):
            clk, K_top, ms_top = c, K, ms
    if rank == 0:
        out = {"metric": METRIC, "value": curve[str(max(SWEEP_SIZES))]["tokens_per_s"],
               "unit": "tokens/s", "n_gpus": world, "steps": K_top,
               "warmup": max(3, args.warmup), "ms_per_step": ms_top / K_top,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "bf16", "data": "synthetic",
               "config": {"workload": "sweep set: 8192 tokens (packed-batch distributions) in "
                                      "consecutive batches of T rows, H=4096, V=151936, bf16, "
                                      "4 vocab shards; value at T=8192",
                          "sizes": list(SWEEP_SIZES), "H": H, "V": V, "n_shards": N_SHARDS,
                          "l2": "inputs larger than L2 (W = 1.24 GB)",
                          "parallelism": "dp%d (independent batches)" % world},
               "curve": curve, "roofline": None, "cpu_baseline": None, "e2e": None,
               "gpu_launches": 2 * K_top, "clocks": clk,
               "contract": binding.contract_id(), "build": binding.build_fingerprint()}
        print(json.dumps(out))
    return 0


def rmsnorm_arm(args, rank, world, dev, dist, binding, WL):
    """The strict RMSNorm producing the head's hidden states for the packed batch: residual
    add (bf16 residual stream out) and normalisation, T = 4096, H = 4096.  Its four
    [T, H] bf16 tensors (134 MB) are about L2's size, so L2 is flushed (a 512 MB write)
    between timed calls, outside the timed interval.  The write leaves L2 full of dirty
    lines that the call's reads must first write back.  rmsnorm16k: T = 16384 rows, whose
    tensors (537 MB) are larger than L2, with no flush."""
    import torch
    big = args.workload == "rmsnorm16k"
    T = 4 * T_PACKED if big else T_PACKED
    g = torch.Generator(device=dev)
    g.manual_seed(4242 + 1000 * rank)
    x = (torch.randn((T, H), generator=g, device=dev) * 2.0).to(torch.bfloat16)
    res = torch.randn((T, H), generator=g, device=dev).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn((H,), generator=g, device=dev)).to(torch.bfloat16)
    out = torch.empty_like(x)
    res_out = torch.empty_like(x)
    flush = None if big else torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        binding.rmsnorm(x, gamma, 1e-6, res, True, out, res_out, stream)

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(int(str(dev).split(":")[-1]) if ":" in str(dev) else 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    for a, b in ev:
        if flush is not None:
            flush.fill_(1)
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(t0, time.time())
    ms_total = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dist, dev)
    call_ms = ms_total / K
    peaks = load_peaks()
    nbytes = float(4 * T * H * 2 + H * 2)
    achieved = nbytes / (call_ms / 1000.0) / 1e9
    if rank == 0:
        out_line = {"metric": METRIC, "value": weak_scaling_value(world, T, K, ms_total),
                    "unit": "tokens/s", "n_gpus": world, "steps": K,
                    "warmup": max(3, args.warmup), "ms_per_step": call_ms,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "bf16", "data": "synthetic",
                    "config": {"workload": ("strict RMSNorm with residual add, T=16384 rows "
                                            "(4 packed batches), H=4096, bf16 in/out, eps 1e-6")
                                           if big else
                                           ("strict RMSNorm with residual add of the packed batch "
                                            "(T=4096, H=4096, bf16 in/out, eps 1e-6)"),
                               "T": T, "H": H,
                               "l2": ("inputs larger than L2 (4 x %.0f MB), no flush"
                                      % (T * H * 2 / 1e6)) if big else
                                     "flushed between calls (512 MB write outside the timed "
                                     "interval)"},
                    "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                                 "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                                 "peak_kind": "copy bandwidth (%s)" % peaks["source"],
                                 "kernel": "k_rmsnorm", "kernel_ms": round(call_ms, 4),
                                 "algorithmic": {"bytes": nbytes,
                                                 "per_row": "read x, residual; write out, "
                                                            "residual_out (4 x H x 2 B)"}},
                    "cpu_baseline": None, "e2e": None, "gpu_launches": K, "clocks": clk,
                    "contract": binding.contract_id(), "build": binding.build_fingerprint()}
        print(json.dumps(out_line))
    return 0


def backward_arm(args, rank, world, dev, dist, W, pk, binding):
    """grad_hidden and grad_W of sum_t g[t] logprob[t] for the packed batch."""
    import torch
    T = pk.hidden.shape[0]
    _, lse = binding.linear_logprob(pk.hidden, W, pk.targets, None, N_SHARDS)
    g = torch.randn(T, generator=torch.Generator(device=dev).manual_seed(7), device=dev)
    ws = torch.empty(binding.backward_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    dh = torch.empty((T, H), dtype=torch.float32, device=dev)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    status = binding.new_status(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        binding.linear_logprob_backward(pk.hidden, W, pk.targets, g, lse, None, True, True, dh, dW,
                                        ws, status, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    binding.raise_on_device_status(status)
    K = max(1, args.steps // 4)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index or 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    s0.record(stream)
    for _ in range(K):
        step()
    s1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop(t0, time.time())
    ms_total = max_over_ranks(s0.elapsed_time(s1), dist, dev)
    ms = ms_total / K
    flops = 3 * 2.0 * T * H * V  # logits again, grad_hidden, grad_W
    peaks = load_peaks()
    achieved = flops / (ms / 1000.0) / 1e12
    if rank == 0:
        out = {"metric": METRIC.replace("selected-logprob", "selected-logprob backward"),
               "value": weak_scaling_value(world, T, K, ms_total), "unit": "tokens/s",
               "n_gpus": world, "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
               "data": "synthetic",
               "config": {"workload": "backward of the packed batch (T=4096, H=4096, V=151936): "
                                      "grad_hidden and grad_W", "T": T, "H": H, "V": V},
               "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": None,
                            "kernel": "whole backward call (gradient epilogue + 2 GEMMs + split sum)",
                            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)},
               "cpu_baseline": None, "e2e": None, "gpu_launches": 4 * K, "clocks": clk,
               "contract": binding.contract_id(), "build": binding.build_fingerprint()}
        print(json.dumps(out))
    return 0


def train_step_arm(args, rank, world, dev, dist, W, pk, binding):
    """One training step of the packed batch: forward (logprob, lse) and the backward of
    sum_t g[t] logprob[t] (grad_hidden, grad_W).  Timed: the forward that saves its fp32
    logits and the backward that forms G from them; beside it, in the same way, the
    recomputing pair (plain forward, backward that runs the logits GEMM again).  Both give
    the same bits; the line checks it."""
    import torch
    T = pk.hidden.shape[0]
    g = torch.randn(T, generator=torch.Generator(device=dev).manual_seed(7), device=dev)
    ws_f = binding.new_workspace(T, V, N_SHARDS, dev)
    ws_b = torch.empty(binding.backward_workspace_size(T, H, V), dtype=torch.uint8, device=dev)
    logits = torch.empty((T, (V + 3) // 4 * 4), dtype=torch.float32, device=dev)
    dh = torch.empty((T, H), dtype=torch.float32, device=dev)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    dh_r = torch.empty_like(dh)
    dW_r = torch.empty_like(dW)
    status = binding.new_status(dev)
    stream = torch.cuda.current_stream(dev)

    def step_saved():
        _, lse, _ = binding.linear_logprob_save_logits(pk.hidden, W, pk.targets, None, N_SHARDS,
                                                       logits=logits, workspace=ws_f,
                                                       status=status, stream=stream)
        binding.linear_logprob_backward_from_logits(logits, pk.hidden, W, pk.targets, g, lse,
                                                    None, True, True, dh, dW, ws_b, status,
                                                    stream)

    def step_recompute():
        _, lse = binding.linear_logprob(pk.hidden, W, pk.targets, None, N_SHARDS,
                                        workspace=ws_f, status=status, stream=stream)
        binding.linear_logprob_backward(pk.hidden, W, pk.targets, g, lse, None, True, True,
                                        dh_r, dW_r, ws_b, status, stream)

    K = max(1, args.steps // 4)
    peaks = load_peaks()
    out = {}
    for name, step in (("recompute", step_recompute), ("saved", step_saved)):
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        binding.raise_on_device_status(status)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(dev.index or 0)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        clocks.start()
        time.sleep(0.3)
        t0 = time.time()
        s0.record(stream)
        for _ in range(K):
            step()
        s1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop(t0, time.time())
        binding.raise_on_device_status(status)
        out[name] = (max_over_ranks(s0.elapsed_time(s1), dist, dev), clk)
    mismatch = int((dh.view(torch.int32) != dh_r.view(torch.int32)).sum().item() +
                   (dW.view(torch.int32) != dW_r.view(torch.int32)).sum().item())
    ms_total, clk = out["saved"]
    ms = ms_total / K
    flops = 3 * 2.0 * T * H * V  # forward, grad_hidden, grad_W
    achieved = flops / (ms / 1000.0) / 1e12
    if rank == 0:
        line = {"metric": METRIC.replace("selected-logprob", "selected-logprob training step"),
                "value": weak_scaling_value(world, T, K, ms_total), "unit": "tokens/s",
                "n_gpus": world, "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "training step of the packed batch (T=4096, H=4096, "
                                       "V=151936): forward saving fp32 logits + backward from "
                                       "them (grad_hidden, grad_W)", "T": T, "H": H, "V": V,
                           "n_shards": N_SHARDS, "saved_logits_gb": round(logits.numel() * 4 / 1e9, 3),
                           "recompute_ms_per_step": out["recompute"][0] / K,
                           "recompute_clocks": out["recompute"][1],
                           "grad_bits_vs_recompute": {"mismatch_count": mismatch}},
                "roofline": {"bound": "tensor", "achieved": round(achieved, 1),
                             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": round(achieved / peaks["bf16_tflops"], 4), "traffic": None,
                             "kernel": "whole step (logits GEMM with the logits stored, G from "
                                       "the logits, 2 GEMMs, split sum, tile tree)",
                             "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)},
                "cpu_baseline": None, "e2e": None, "gpu_launches": 6 * K, "clocks": clk,
                "contract": binding.contract_id(), "build": binding.build_fingerprint()}
        print(json.dumps(line))
    if mismatch:
        raise SystemExit("saved-logits backward differs from the recomputing one")
    return 0


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import numpy as np
    import torch
    from invariant_selected_token_gb300 import binding, workloads as WL
    from invariant_selected_token_gb300 import build as lib_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        lib_build.build()
    if dist is not None:
        dist.barrier()
    binding.lib()

    if args.workload in ("rmsnorm", "rmsnorm16k"):
        return rmsnorm_arm(args, rank, world, dev, dist, binding, WL)
    W = WL.head_weights(dev)                       # same weights on every rank
    if args.workload == "grpo":
        return grpo_arm(args, rank, world, dev, dist, W, binding, WL)
    if args.workload == "sweep":
        return sweep_arm(args, rank, world, dev, dist, W, binding, WL)
    pk = WL.packed(W, dev, seed=rank_batch_seed(rank))  # each rank its own batch
    if args.workload.startswith("logits_") or args.workload == "log_softmax_fp32":
        return materialised_arm(args, rank, world, dev, dist, W, pk, binding, WL)
    if args.workload == "backward":
        return backward_arm(args, rank, world, dev, dist, W, pk, binding)
    if args.workload == "train_step":
        return train_step_arm(args, rank, world, dev, dist, W, pk, binding)
    if args.workload == "packed":
        hidden, targets = pk.hidden, pk.targets
        workload = WORKLOAD
    else:
        n = int(args.workload[len("decode"):])
        idx = torch.from_numpy(WL.decode_rows(n)).to(dev)
        hidden, targets = pk.hidden[idx].contiguous(), pk.targets[idx].contiguous()
        workload = ("decode batch T=%d (rows of the packed batch), H=4096, V=151936, bf16, "
                    "4 vocab shards" % n)
    T = hidden.shape[0]
    ws = binding.new_workspace(T, V, N_SHARDS, dev)
    out_lp = torch.empty(T, dtype=torch.float32, device=dev)
    out_lse = torch.empty(T, dtype=torch.float32, device=dev)
    status = binding.new_status(dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev0=None, ev1=None):
        if ev0 is not None:
            ev0.record(stream)
        binding.tile_partials(hidden, W, targets, None, N_SHARDS, ws, status, stream)
        if ev1 is not None:
            ev1.record(stream)
        binding.tile_merge(targets, None, V, N_SHARDS, out_lp, out_lse, ws, status, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    binding.raise_on_device_status(status)

    # ---------------- timed region (device-resident inputs)
    # K steps bracketed by two events give the step rate (`value`).  Inside the same
    # region every step also records events around its logits-kernel launch: their
    # average is the kernel's duration for the roofline.  Both numbers come from one
    # pass at one clock, and the kernel intervals are disjoint parts of the region, so
    # the kernel time cannot exceed the step time.
    K = args.steps
    clocks = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_host0 = time.time()
    ms_total, k1_ms, n_k1 = timed_steps(step, K, stream)
    t_host1 = time.time()
    clk = clocks.stop(t_host0, t_host1)
    binding.raise_on_device_status(status)
    check_kernel_within_step(k1_ms, ms_total / K)
    ms_total = max_over_ranks(ms_total, dist, dev)
    ms_per_step = ms_total / K
    value = weak_scaling_value(world, T, K, ms_total)

    # ---------------- end to end through the public call, host buffers
    e2e = None
    if not args.no_e2e:
        # one pinned input buffer (hidden rows, then targets) and one pinned output buffer
        # (logprob, then lse): a single copy each way per step.  Inputs and outputs are
        # double-buffered on the device, uploads and read-backs run on their own
        # streams: step k+1's upload and step k-1's read-back overlap step k.
        hid_bytes = hidden.numel() * 2
        h_in = torch.empty(hid_bytes + T * 4, dtype=torch.uint8).pin_memory()
        h_in[:hid_bytes].view(torch.bfloat16).view(T, H).copy_(hidden.cpu())
        h_in[hid_bytes:].view(torch.int32).copy_(targets.cpu())
        h_out = torch.empty((2, T), dtype=torch.float32).pin_memory()
        d_in = [torch.empty(hid_bytes + T * 4, dtype=torch.uint8, device=dev) for _ in range(2)]
        d_out = [torch.empty((2, T), dtype=torch.float32, device=dev) for _ in range(2)]
        up_stream, down_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        uploaded = [torch.cuda.Event() for _ in range(2)]
        in_free = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]
        for e in in_free + out_free:
            e.record(stream)
        n_e2e = [0]

        def e2e_step():
            b = n_e2e[0] % 2
            n_e2e[0] += 1
            up_stream.wait_event(in_free[b])       # the step two back has read this input
            with torch.cuda.stream(up_stream):
                d_in[b].copy_(h_in, non_blocking=True)
                uploaded[b].record(up_stream)
            stream.wait_event(uploaded[b])
            stream.wait_event(out_free[b])         # this output's previous read-back is done
            binding.linear_logprob(d_in[b][:hid_bytes].view(torch.bfloat16).view(T, H), W,
                                   d_in[b][hid_bytes:].view(torch.int32), None, N_SHARDS,
                                   d_out[b][0], d_out[b][1], ws, status, stream)
            in_free[b].record(stream)
            computed[b].record(stream)
            down_stream.wait_event(computed[b])
            with torch.cuda.stream(down_stream):
                h_out.copy_(d_out[b], non_blocking=True)
                out_free[b].record(down_stream)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up_stream.wait_event(e0)  # no copy of the timed steps starts before e0
        for _ in range(K):
            e2e_step()
        for e in out_free:
            stream.wait_event(e)  # the last read-backs are inside the timed region
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1)
        e_ms = max_over_ranks(e_ms, dist, dev)
        binding.raise_on_device_status(status)
        assert torch.equal(h_out[0], out_lp.cpu()) and torch.equal(h_out[1], out_lse.cpu())  # last step
        e2e = {"value": weak_scaling_value(world, T, K, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h_in.numel()),
               "d2h_bytes_per_step": int(h_out.numel() * 4),
               "copies_per_step": "one host-to-device and one device-to-host (pinned), each on "
                                  "its own stream, overlapping the neighbouring steps' compute"}

    # ---------------- roofline of the dominant kernel (logits GEMM + fused epilogue)
    peaks = load_peaks()
    flops = 2.0 * T * H * V
    nbytes = float(W.numel() * 2 + hidden.numel() * 2)
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    traffic = k1_traffic_record(args.workload)
    if t_tensor >= t_hbm:
        achieved = flops / (k1_ms / 1000.0) / 1e12
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                    "traffic": traffic, "peak_kind": "burst bf16 (%s)" % peaks["source"],
                    "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}
    else:
        achieved = nbytes / (k1_ms / 1000.0) / 1e9
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                    "traffic": traffic, "peak_kind": "copy bandwidth (%s)" % peaks["source"]}
    roofline.update({"kernel": "k_tile_partials", "kernel_ms": round(k1_ms, 4),
                     "kernel_timing": "CUDA events around the kernel's launch in every step of "
                                      "the timed region (%d launches)" % n_k1,
                     "algorithmic": {"flops": flops, "bytes": nbytes}})
    step_roof_ms = max(t_tensor, t_hbm) * 1000.0

    # ---------------- invariance, live: sample rows recomputed as their own small batch
    # (and, for a decode batch, the packed batch they came from) must give the timed
    # run's outputs bit for bit
    rows = WL.permutation(T, 4321)[:min(T, 2048)]
    rows_t = torch.from_numpy(rows).to(dev)
    sub_lp, sub_lse = binding.linear_logprob(hidden[rows_t].contiguous(), W,
                                             targets[rows_t].contiguous(), None, N_SHARDS)
    pairs = [(sub_lp, out_lp[rows_t]), (sub_lse, out_lse[rows_t])]
    layouts = ["%d-row batch of sample rows vs the timed T=%d batch" % (len(rows), T)]
    if args.workload != "packed":
        pk_lp, pk_lse = binding.linear_logprob(pk.hidden, W, pk.targets, None, N_SHARDS)
        pairs += [(out_lp, pk_lp[idx]), (out_lse, pk_lse[idx])]
        layouts.append("decode batch vs the same rows inside the packed T=4096 batch")
    torch.cuda.synchronize()
    mism = sum(int((a.view(torch.int32) != b.view(torch.int32)).sum().item()) for a, b in pairs)
    maxd = max(float((a.double() - b.double()).abs().max().item()) for a, b in pairs)
    invariance = {"mismatch_count": mism, "max_abs_diff": maxd, "compared": layouts}

    # ---------------- decode batches of the packed run's rows (rollout side), timed the
    # same way, bit-compared with the packed run's outputs for those rows
    decode = None
    if args.workload == "packed":
        decode = {}
        for n in DECODE_SIZES:
            decode["T%d" % n] = decode_record(n, W, hidden, targets, out_lp, out_lse, binding, WL,
                                              dev, stream, status, load_peaks())

    # ---------------- CPU baseline: the fp64 oracle on a bounded sample (rank 0, N=1),
    # whose values also give the parity of the timed run's outputs on those rows
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        W_bits = WL.bf16_tensor_bits(W)
        hid_bits = WL.bf16_tensor_bits(hidden[rows_t])
        s_, n_, ref_lp, ref_lse = cpu_oracle_sample(hid_bits, W_bits, targets.cpu().numpy()[rows],
                                                    None, want_values=True)
        cpu = {"value": n_ / s_, "unit": "tokens/s", "cores": host_threads(), "kind": "oracle",
               "sample": "%d rows of the batch over the full vocabulary (%.1f s)" % (n_, s_)}
        got_lp = out_lp[rows_t].double().cpu().numpy()
        got_lse = out_lse[rows_t].double().cpu().numpy()
        d_lp = abs(got_lp - ref_lp)
        d_lse = abs(got_lse - ref_lse) / abs(ref_lse)
        parity = {"rows": int(n_), "logprob_abs_diff": diff_stats(d_lp),
                  "lse_rel_diff_max": float(d_lse.max()),
                  "tolerance": {"logprob_abs": 1e-4, "lse_rel": 2e-5},
                  "within_tolerance": bool(d_lp.max() <= 1e-4 and d_lse.max() <= 2e-5)}

    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
               "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "bf16", "data": "synthetic",
               "config": {"workload": workload, "T": T, "H": H, "V": V, "n_shards": N_SHARDS,
                          "accumulate": "fp32", "l2": "inputs larger than L2 (W = 1.24 GB)",
                          "parallelism": "dp%d (independent batches)" % world,
                          "roofline_step_ms": round(step_roof_ms, 4),
                          "frac_of_step_roofline": round(step_roof_ms / ms_per_step, 4)},
               "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
               "gpu_launches": 2 * K, "clocks": clk,
               "active_tokens_per_step": T, "invariance": invariance, "parity": parity,
               "decode": decode,
               "peak_memory_gb": round(torch.cuda.max_memory_allocated(dev) / 1e9, 3),
               "hardware": hardware_fingerprint(dev),
               "contract": binding.contract_id(), "build": binding.build_fingerprint()}
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

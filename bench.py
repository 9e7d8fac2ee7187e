"""Benchmark: fused two-copy block-diffusion attention, forward + backward.

One step = one forward and one backward pass over one batch of seeded
synthetic bf16 inputs, through the C-ABI library (csbp_attn_fwd then
csbp_attn_bwd; for sharded workloads the forward runs per-shard partials plus
the LSE merge).  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                  [--impl {csbp,reference}] [--no-cpu-baseline]

metric = useful (mask-allowed) TFLOP/s of fwd+bwd: 4*d FLOPs per allowed
(query, key) pair per query head forward, 2.5x that backward.  `value` is
timed with CUDA events on the launch stream with inputs resident in HBM;
`e2e` repeats the step through the same API with host-pinned inputs copied in
and the outputs/gradients copied back inside the timed region.
With N > 1 (torchrun) every rank runs an independent replica of the
workload on its own GPU (no collective on the data path): weak scaling.

Configs: the attention workloads of inputs.WORKLOADS (default long, the
L = 131,072 fine-tune layer; dense14b, sharded, drafter, window1k,
block128 .. block1024, tiny), and the
LM-head cross-entropy workloads of inputs.CE_WORKLOADS (lmhead14b,
lmhead_frozen, lmhead_2k), for which one step is one csbp_vocab_ce call
(loss, dH and dW of every row) and the metric is its TFLOP/s (2 N V Dm per
GEMM: logits, dH and, for a trained head, dW).
"""
from __future__ import annotations

import argparse
import atexit
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "useful TFLOP/s fwd+bwd block-diffusion attention (1 GB300) and % of BF16 peak"
DEFAULT_CONFIG = "long"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="csbp", choices=["csbp", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end leg (auxiliary measurements)")
    ap.add_argument("--L", type=int, default=None,
                    help="override the sequence length (profiling captures of a smaller case)")
    ap.add_argument("--bwd-chunk", type=int, default=0,
                    help="backward query-tile window (csbp_problem.bwd_chunk; 0: none)")
    return ap.parse_args()


# Sources that determine bwd_kernel's machine code; a DRAM-traffic figure
# counts only while their hash matches the one recorded with it.
BWD_KERNEL_SOURCES = ("attn_bwd.cu", "ptx_sm100.cuh", "pair_math.cuh", "mbar_spin.cuh", "csbp_internal.h")


def bwd_kernel_source_hash():
    return source_hash(BWD_KERNEL_SOURCES)


# the CE kernels' device code comes from these two files alone
CE_KERNEL_SOURCES = ("vocab_ce.cu", "ptx_sm100.cuh")


def source_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "block_diffusion_lm_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


TRAFFIC_RECORDS = os.path.join(ROOT, "profiles", "dram_traffic.json")


def recorded_dram_bytes(kernel, workload, sources):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from
    the committed ncu records (profiles/dram_traffic.json), or None if there
    is no record or the kernel's sources changed since it was taken."""
    if not os.path.exists(TRAFFIC_RECORDS):
        return None
    with open(TRAFFIC_RECORDS) as f:
        records = json.load(f).get("records", [])
    want = source_hash(sources)
    for r in records:
        if r.get("kernel") == kernel and r.get("workload") == workload:
            if r.get("kernel_source_sha256") != want:
                return None
            return int(r["dram_bytes_per_launch"])
    return None


def recorded_ce_traffic(workload, kernel):
    """DRAM bytes per launch of one CE GEMM (`logits_gemm`, `dh_gemm`,
    `dw_gemm`), while the CE kernels' sources match the record."""
    return recorded_dram_bytes(f"ce_gemm_kernel/{kernel}", workload, CE_KERNEL_SOURCES)


def recorded_traffic(workload):
    """DRAM bytes per bwd_kernel launch of this workload, while the kernel's
    sources match the record."""
    return recorded_dram_bytes("bwd_kernel", workload, BWD_KERNEL_SOURCES)


# --------------------------------------------------------------- ranks
def max_over_ranks(value, device):
    """The largest of every rank's value (the slowest rank sets the job's
    time); the value itself when not running under torch.distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    x = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(x, op=dist.ReduceOp.MAX)
    return x.item()


def whole_job_tflops(world, flops_per_rank_step, ms_per_step):
    """Useful TFLOP/s of the whole job: every rank does one replica's step in
    ms_per_step (the max over ranks)."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"bf16": p.get("bf16_tflops", 1914.7),
                "bf16_sustained": p.get("bf16_tflops_sustained", 1693.2),
                "hbm": p.get("hbm_gbs", 6783.8), "source": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "source": "fallback"}


# a region shorter than this is a burst for the power controller
SUSTAINED_REGION_S = 2.0


def choose_bf16_peak(pk, clocks, region_s):
    """The bf16 denominator that matches how the timed region ran: the
    sustained (power-capped) peak only when the region lasted seconds and
    the clock record shows the power cap acting; the burst peak otherwise
    (including when no clock record exists).  Returns (peak, name, why)."""
    capped = bool(clocks) and "sw_power_cap" in clocks.get("reasons", [])
    if region_s >= SUSTAINED_REGION_S and capped:
        return (pk["bf16_sustained"], f"bf16_tflops_sustained of {pk['source']}",
                f"timed region {region_s:.1f} s with sw_power_cap active "
                f"in {clocks.get('power_cap_samples', 0)} of {clocks.get('samples', 0)} samples")
    why = (f"timed region {region_s:.2f} s" + (", sw_power_cap never active" if clocks
                                                else ", no clock record"))
    return pk["bf16"], f"bf16_tflops of {pk['source']} (burst)", why


def peak_fractions(tflops, pk):
    return {"of_burst": tflops / pk["bf16"], "of_sustained": tflops / pk["bf16_sustained"]}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    PERIOD_MS = 50

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
            return
        # the sampler loops until told to stop: end it even if the timed
        # region raises and stop() is never reached
        atexit.register(self._end)

    def _end(self):
        """Terminate the sampler (kill it if it lingers); safe to call twice."""
        if self.proc is None or self.proc.poll() is not None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait(timeout=5)

    def stop(self):
        if self.proc is None:
            return None
        self._end()
        atexit.unregister(self._end)
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file if ln.strip()]
        os.unlink(self.file.name)
        return self.summarise(rows)

    @staticmethod
    def summarise(rows):
        """Median SM clock, max clock, sample count, the throttle reasons seen
        and how many samples had the power cap active."""
        sm, mx, reasons, capped = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
                    capped += n == "sw_power_cap"
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons), "power_cap_samples": capped,
                "period_ms": ClockSampler.PERIOD_MS}


# ------------------------------------------------------------ cpu oracle
def cpu_oracle_sample(w, seconds, seed=7):
    """Time the float64 oracle on seeded sampled query rows of the workload
    (forward + analytic backward of each row against its full masked key
    set) until about `seconds` of CPU work; returns useful TFLOP/s and a
    description.  Inputs are drawn on the CPU with the workload's recipe at a
    length capped so the sample stays bounded."""
    import numpy as np
    import torch

    from block_diffusion_lm_gb300.inputs import make_inputs
    from oracle import csbp_oracle as O

    L = w.L
    t = make_inputs(w, "cpu", seed=seed)
    f = {k: (v[0] if v is not None else None) for k, v in t.items()}

    class View:
        def __init__(self, x):
            self.x, self.shape = x, tuple(x.shape)

        def __getitem__(self, idx):
            return self.x[idx].to(torch.float32).numpy()

    fv = {k: (View(v) if v is not None else None) for k, v in f.items()}
    rng = np.random.default_rng(seed)
    streams = [0, 1] if w.has_clean_queries else [1]
    G = w.Hq // w.Hkv
    rows_done = 0
    useful = 0.0
    t0 = time.perf_counter()
    batch_rows = 16
    while time.perf_counter() - t0 < seconds:
        h = int(rng.integers(0, w.Hq))
        samples = [(int(rng.choice(streams)), int(rng.integers(0, L)), h) for _ in range(batch_rows)]
        O.sampled_rows(fv["q_clean"], fv["k_clean"], fv["v_clean"], fv["q_corr"], fv["k_corr"],
                       fv["v_corr"], fv["do_clean"], fv["do_corr"], w.M, w.scale, samples,
                       w.window, w.clean_causal)
        for qs, i, _ in samples:
            useful += 4.0 * w.d * w.keys_of_row(qs, i) * 3.5
        rows_done += batch_rows
    dt = time.perf_counter() - t0
    del G
    value = useful / dt / 1e12
    full = w.useful_fwd_flops() + w.useful_bwd_flops()
    return {"value": value, "unit": "TFLOP/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{rows_done} seeded query rows (fwd + analytic bwd per row against all "
                      f"2L={2 * L} keys, masked), {dt:.1f} s; useful FLOPs counted as in the metric",
            "extrapolated_step_s": full / (value * 1e12)}


# ----------------------------------------------------------- HBM kernels
def hbm_kernels(w, csbp):
    """GB/s of the HBM-bound launches of the timed steps: algorithmic bytes
    per launch (each input read once, each output written once) over the
    average CUDA-event duration of that launch, against the measured copy
    bandwidth."""
    d, rows = w.d, w.batch * w.L
    per_launch = {
        # n partial (O fp32, z fp32) read, O bf16 + z written, per (row, head)
        6: ("lse_merge", w.L * w.Hq * ((w.P + 1) * (4 * d + 4) + 2 * d + 4)),
        # O, dO read; D and the zeroed fp32 dQ row written
        7: ("bwd_pre", rows * w.Hq * (8 * d + 4)),
        # fp32 dQ read, bf16 dQ written
        8: ("dq_convert", rows * w.Hq * 6 * d),
        # fp32 dK and dV read, bf16 written (windowed backward)
        9: ("dkv_convert", 2 * rows * w.Hkv * 6 * d),
    }
    if w.e4m3:  # fp8 inputs: 1 byte read, 2 written per element; the average launch
        n_qs = 2 if w.has_clean_queries else 1
        elems = rows * d * (4 * w.Hkv + 2 * n_qs * w.Hq)
        per_launch[10] = ("e4m3_decode", 3 * elems / (4 + 2 * n_qs))
    peak = peaks()["hbm"]
    out = {}
    for kind, (name, nbytes) in per_launch.items():
        ms, n = csbp.kernel_timing_read_kind(kind)
        if n:
            gbs = nbytes / (ms / n * 1e-3) / 1e9
            out[name] = {"launches": n, "avg_launch_ms": ms / n, "bytes_per_launch": nbytes,
                         "gbs": gbs, "frac_of_measured_hbm": gbs / peak}
    return out or None


# --------------------------------------------------------------- launches
def launches_per_step(w):
    """Kernels this library launches per fwd+bwd step (mirrors csbp_api.cu)."""
    n_qs = 2 if w.has_clean_queries else 1
    fwd = 1 + ((1 + n_qs * w.batch) if w.P > 1 else 0)   # [fill] + fwd + [merges]
    bwd = n_qs + 1 + n_qs                                  # pre per stream + main + convert
    dec = (4 + 2 * n_qs) if w.e4m3 else 0                 # fp8 decodes: K, V x 2, Q and dO
    return fwd + bwd + dec


# ------------------------------------------------------- vocabulary loss
CE_METRIC = ("TFLOP/s streamed LM-head cross-entropy, loss + dH (+ dW for a trained head) "
             "(1 GB300) and % of BF16 peak")
CE_KINDS = {2: "logits_gemm", 3: "row_kernel", 4: "dh_gemm", 5: "dw_gemm"}


def ce_cpu_oracle_sample(w, seconds, seed=7):
    """The float64 oracle on seeded sample rows of the workload for about
    `seconds`: each row's logits over the whole vocabulary, its LSE, loss
    and dH (4 V Dm FLOPs per row; dW needs every row and is not sampled)."""
    import numpy as np
    import torch

    from block_diffusion_lm_gb300.inputs import make_ce_inputs
    from oracle import vocab_ce_oracle as C

    x = make_ce_inputs(w, "cpu")
    W = x["w"].to(torch.float64).numpy()
    H = x["h"]
    t = x["target"].numpy()
    rng = np.random.default_rng(seed)
    rows_done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        rows = rng.choice(w.N, size=8, replace=False)
        C.vocab_ce_rows(H[torch.as_tensor(rows)].to(torch.float64).numpy(), W, t[rows],
                        x["grad_scale"], np.arange(8))
        rows_done += 8
    dt = time.perf_counter() - t0
    value = rows_done * 4.0 * w.V * w.Dm / dt / 1e12
    return {"value": value, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{rows_done} seeded rows (logits over V={w.V}, LSE, loss, dH; "
                      f"4*V*Dm FLOPs each), {dt:.1f} s",
            "extrapolated_step_s": w.flops() / (value * 1e12)}


def bench_ce(args, w, rank, world, local):
    config = {"workload": w.name, "rows": w.N, "d_model": w.Dm, "vocab": w.V,
              "chunk_rows": w.chunk, "head_grad": w.head_grad,
              "parallelism": f"replicas{args.gpus}" if args.gpus > 1 else "single"}
    flops = w.flops()
    if args.impl == "reference":
        if rank != 0:
            return
        for _ in range(args.warmup):
            ce_cpu_oracle_sample(w, 2.0)
        steps = [ce_cpu_oracle_sample(w, max(2.0, args.cpu_seconds / max(args.steps, 1)))
                 for _ in range(args.steps)]
        v = statistics.median(s["value"] for s in steps)
        print(json.dumps({
            "impl": "reference", "metric": CE_METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": flops / (v * 1e12) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": dict(steps[0], value=v),
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    import torch
    import torch.distributed as dist

    from block_diffusion_lm_gb300 import build, csbp
    from block_diffusion_lm_gb300.inputs import make_ce_inputs

    build.build()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    x = make_ce_inputs(w, dev)
    ce = csbp.VocabCrossEntropy(w.N, w.Dm, w.V, w.chunk, w.head_grad, x["grad_scale"],
                                device=dev)
    out = ce.alloc_outputs()
    n_chunks = -(-w.N // (w.chunk if w.chunk > 0 else 8192))
    in_bytes = sum(v.numel() * v.element_size() for v in (x["h"], x["w"], x["target"]))

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            ce(x["h"], x["w"], x["target"], out, stream=stream)
    ce.check(stream)
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    csbp.kernel_timing(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            ce(x["h"], x["w"], x["target"], out, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    csbp.kernel_timing(False)
    ce.check(stream)
    total_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    if world > 1:
        dist.barrier()
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(world, flops, ms_per_step)

    kernels = {}
    for kind, name in CE_KINDS.items():
        ms, n = csbp.kernel_timing_read_kind(kind)
        if n:
            kernels[name] = {"ms_per_step": ms / args.steps, "launches": n,
                             "avg_launch_ms": ms / n}
    gemm_flops = 2.0 * w.N * w.V * w.Dm
    for name in ("logits_gemm", "dh_gemm", "dw_gemm"):
        if name in kernels:
            kernels[name]["tflops"] = gemm_flops / (kernels[name]["ms_per_step"] * 1e-3) / 1e12
    if "row_kernel" in kernels:
        row_bytes = w.N * w.V * 6.0  # fp32 logits in, bf16 g out
        kernels["row_kernel"]["gbs"] = row_bytes / (kernels["row_kernel"]["ms_per_step"] * 1e-3) / 1e9
    top = max((k for k in kernels if k.endswith("gemm")), key=lambda k: kernels[k]["ms_per_step"])
    pk = peaks()
    peak, peak_name, peak_why = choose_bf16_peak(pk, clocks, total_ms * 1e-3)
    top_launch_flops = gemm_flops / n_chunks
    achieved = top_launch_flops / (kernels[top]["avg_launch_ms"] * 1e-3) / 1e12

    # end to end: pinned host inputs up, loss/LSE/dH(/dW) down, every step.
    # Copies run on their own streams with two buffer sets, so step i+1's
    # inputs go up and step i's results come down while step i computes; the
    # region runs from the first upload to the last download.
    host = {k: x[k].cpu().pin_memory() for k in ("h", "w", "target")}
    sets = []
    for k in range(2):
        d_in = {n: torch.empty_like(x[n]) for n in host}
        o = out if k == 0 else ce.alloc_outputs()
        res = [r for r in o if r is not None]
        sets.append((d_in, o, res, [torch.empty(r.shape, dtype=r.dtype, pin_memory=True)
                                    for r in res]))
    out_bytes = sum(r.numel() * r.element_size() for r in sets[0][2])
    e2e_steps = max(3, min(args.steps, 10))
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]
    for e in done + read:
        e.record(stream)

    def run(n, e_start=None, e_end=None):
        for i in range(n):
            k = i % 2
            d_in, o, res, h_out = sets[k]
            with torch.cuda.stream(up):
                up.wait_event(done[k])          # the step that last read these inputs
                if i == 0 and e_start is not None:
                    e_start.record(up)
                for n_, v in host.items():
                    d_in[n_].copy_(v, non_blocking=True)
                in_ready[k].record(up)
            stream.wait_event(in_ready[k])
            stream.wait_event(read[k])          # its outputs were copied down
            ce(d_in["h"], d_in["w"], d_in["target"], o, stream=stream)
            done[k].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done[k])
                for src, dst in zip(res, h_out):
                    dst.copy_(src, non_blocking=True)
                read[k].record(down)
        if e_end is not None:
            with torch.cuda.stream(down):
                e_end.record(down)

    run(2)
    torch.cuda.synchronize(dev)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(e2e_steps, f0, f1)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / e2e_steps, dev)
    e2e = {"value": whole_job_tflops(world, flops, e2e_ms), "unit": "TFLOP/s",
           "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
           "overlap": "copies on separate streams, 2 buffer sets"}

    line = {
        "metric": CE_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(config, l2=f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB resident "
                                  f"vs {L2_BYTES / 2**20:.0f} MiB L2); no flush"),
        "pct_of_bf16_peak": value / world / peak,
        "pct_of_bf16_peak_by_peak": peak_fractions(value / world, pk),
        "kernels": kernels,
        "roofline": {"bound": "tensor", "kernel": f"ce_gemm_kernel ({top})",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "frac_by_peak": peak_fractions(achieved, pk),
                     "peak_source": peak_name, "peak_choice": peak_why,
                     "launch_ms": kernels[top]["avg_launch_ms"],
                     "launches_timed": kernels[top]["launches"],
                     "traffic": recorded_ce_traffic(w.name, top)},
        "e2e": e2e,
        "gpu_launches": n_chunks * (4 if w.head_grad else 3) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = ce_cpu_oracle_sample(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from block_diffusion_lm_gb300.inputs import CE_WORKLOADS, WORKLOADS
    if args.config in CE_WORKLOADS:
        bench_ce(args, CE_WORKLOADS[args.config], rank, world, local)
        return
    if args.config not in WORKLOADS:
        sys.exit(f"unknown --config {args.config!r}; choose one of "
                 f"{', '.join(sorted(WORKLOADS) + sorted(CE_WORKLOADS))}")

    import dataclasses

    from block_diffusion_lm_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.config]
    if args.L is not None:
        w = dataclasses.replace(w, name=f"{w.name}@L={args.L}", L=args.L)
    flops = w.useful_fwd_flops() + w.useful_bwd_flops()
    config = {"workload": w.name, "batch": w.batch, "L": w.L, "M": w.M, "Hq": w.Hq,
              "Hkv": w.Hkv, "d": w.d, "P": w.P, "clean_queries": w.has_clean_queries,
              "parallelism": f"replicas{args.gpus}" if args.gpus > 1 else "single"}
    if w.e4m3:
        config["inputs"] = "fp8 e4m3, per-tensor power-of-two scales, decoded to bf16 each step"
    if args.bwd_chunk:
        config["bwd_chunk"] = args.bwd_chunk

    if args.impl == "reference":
        if rank != 0:
            return
        steps = []
        for _ in range(args.warmup):
            cpu_oracle_sample(w, 2.0)
        for _ in range(args.steps):
            steps.append(cpu_oracle_sample(w, max(2.0, args.cpu_seconds / max(args.steps, 1))))
        v = statistics.median(s["value"] for s in steps)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
                "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": flops / (v * 1e12) * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": config,
                "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": steps[0]["cores"],
                                 "kind": "oracle", "sample": steps[0]["sample"],
                                 "extrapolated_step_s": flops / (v * 1e12)},
                "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import torch.distributed as dist

    from block_diffusion_lm_gb300 import build, csbp
    from block_diffusion_lm_gb300.inputs import make_inputs

    build.build()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)

    codes = None
    if w.e4m3:
        # Q, K, V and dO kept in fp8 E4M3; every step decodes them into the
        # bf16 buffers the attention reads
        from block_diffusion_lm_gb300.inputs import make_inputs_e4m3
        codes, scales = make_inputs_e4m3(w, dev)
        t = {k: (csbp.e4m3_to_bf16(c, scales[k]) if c is not None else None)
             for k, c in codes.items()}

        def decode(src, dst):
            for k, c in src.items():
                if c is not None:
                    csbp.e4m3_to_bf16(c, scales[k], out=dst[k], stream=stream)
    else:
        t = make_inputs(w, dev)
    attn = csbp.BlockDiffusionAttention(w.batch, w.L, w.M, w.Hq, w.Hkv, w.d, P=w.P,
                                        has_clean_queries=w.has_clean_queries, device=dev,
                                        window=w.window, clean_causal=w.clean_causal,
                                        bwd_chunk=args.bwd_chunk)
    out = attn.alloc_outputs()
    grads = attn.alloc_grads()
    src = codes if codes is not None else t
    in_bytes = sum(v.numel() * v.element_size() for v in src.values() if v is not None)

    def step():
        if codes is not None:
            decode(codes, t)
        attn.forward(t, out=out, stream=stream)
        attn.backward(t, out, grads=grads, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    attn.check(stream)

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    csbp.kernel_timing(True)
    start_all = torch.cuda.Event(enable_timing=True)
    end_all = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start_all.record(stream)
        for i in range(args.steps):
            if codes is not None:
                decode(codes, t)
            ev[i][0].record(stream)
            attn.forward(t, out=out, stream=stream)
            ev[i][1].record(stream)
            attn.backward(t, out, grads=grads, stream=stream)
            ev[i][2].record(stream)
        end_all.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    csbp.kernel_timing(False)
    fwd_k_ms, n_fwd_k, bwd_k_ms, n_bwd_k = csbp.kernel_timing_read()
    hbm = hbm_kernels(w, csbp)
    attn.check(stream)
    total_ms = start_all.elapsed_time(end_all)
    fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    bwd_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = max_over_ranks(total_ms, dev)
    if world > 1:
        dist.barrier()
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(world, flops, ms_per_step)

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        if codes is not None:
            e2e = run_e2e(args, w, codes, attn, out, grads, stream, dev, world, flops, in_bytes,
                          prep=lambda d_in: (decode(d_in, t), t)[1])
        else:
            e2e = run_e2e(args, w, t, attn, out, grads, stream, dev, world, flops, in_bytes)

    pk = peaks()
    peak, peak_name, peak_why = choose_bf16_peak(pk, clocks, total_ms * 1e-3)
    bwd_avg = statistics.mean(bwd_ms)
    fwd_avg = statistics.mean(fwd_ms)
    bwd_call_tflops = w.useful_bwd_flops() / (bwd_avg * 1e-3) / 1e12
    bwd_kernel_ms = bwd_k_ms / max(n_bwd_k, 1)      # main kernel alone, CUDA events
    fwd_kernel_ms = fwd_k_ms / max(n_fwd_k, 1)
    achieved = w.useful_bwd_flops() / (bwd_kernel_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(config, l2=f"inputs larger than L2 ({in_bytes / 2**20:.0f} MiB resident "
                                  f"vs {L2_BYTES / 2**20:.0f} MiB L2); no flush"),
        "pct_of_bf16_peak": value / world / peak,
        "pct_of_bf16_peak_by_peak": peak_fractions(value / world, pk),
        "fwd_ms": fwd_avg, "bwd_ms": bwd_avg,
        "fwd_tflops": w.useful_fwd_flops() / (fwd_avg * 1e-3) / 1e12,
        "bwd_tflops": bwd_call_tflops,
        # the same backward time against 2x the forward FLOPs (no S recompute counted)
        "bwd_tflops_strict_2x": 2 * w.useful_fwd_flops() / (bwd_avg * 1e-3) / 1e12,
        "fwd_kernel_ms": fwd_kernel_ms, "bwd_kernel_ms": bwd_kernel_ms,
        "roofline": {"bound": "tensor", "kernel": f"bwd_kernel<{w.d}>",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "frac_by_peak": peak_fractions(achieved, pk),
                     "peak_source": peak_name, "peak_choice": peak_why,
                     "launch_ms": bwd_kernel_ms, "launches_timed": n_bwd_k,
                     "traffic": recorded_traffic(w.name)},
        "hbm_kernels": hbm,
        "e2e": e2e,
        "gpu_launches": launches_per_step(w) * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_e2e(args, w, t, attn, out, grads, stream, dev, world, flops, in_bytes, prep=None):
    """Same steps through the public API from pinned host inputs, with the
    outputs and gradients copied back, all inside the timed region.  Copies
    run on their own streams with two buffer sets, so step i+1's inputs go
    up and step i's results come down while step i computes; the region runs
    from the first input copy to the last result copy.  `prep` turns a step's
    uploaded inputs into the attention's (the fp8 workload decodes them)."""
    import torch
    import torch.distributed as dist

    host_in = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in t.items()}
    sets = []
    for k in range(2):
        o = out if k == 0 else attn.alloc_outputs()
        g = grads if k == 0 else attn.alloc_grads()
        d_in = {n: (torch.empty_like(v) if v is not None else None) for n, v in t.items()}
        res = [x for x in (*o, *g.values()) if x is not None]
        h_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in res]
        sets.append((d_in, o, g, res, h_out))
    out_bytes = sum(x.numel() * x.element_size() for x in sets[0][3])
    # the first upload and the last download are not overlapped: spread
    # them over up to 20 steps (on one GB300 machine: 211 / 193 GB/s host link,
    # and a dense14b step with both copies beside it 18.35 vs 18.11 ms)
    e2e_steps = max(3, min(args.steps, 20))
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_ready = [ev(), ev()]
    done = [ev(), ev()]
    read = [ev(), ev()]
    for e in done + read:
        e.record(stream)

    def run(n, e_start=None, e_end=None):
        for i in range(n):
            k = i % 2
            d_in, o, g, res, h_out = sets[k]
            with torch.cuda.stream(up):
                up.wait_event(done[k])          # the step that last read these inputs
                if i == 0 and e_start is not None:
                    e_start.record(up)
                for name, v in host_in.items():
                    if v is not None:
                        d_in[name].copy_(v, non_blocking=True)
                in_ready[k].record(up)
            stream.wait_event(in_ready[k])
            stream.wait_event(read[k])          # its outputs were copied down
            with torch.cuda.stream(stream):
                x = prep(d_in) if prep is not None else d_in
            attn.forward(x, out=o, stream=stream)
            attn.backward(x, o, grads=g, stream=stream)
            done[k].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done[k])
                for hsrc, hdst in zip(res, h_out):
                    hdst.copy_(hsrc, non_blocking=True)
                read[k].record(down)
        if e_end is not None:
            with torch.cuda.stream(down):
                e_end.record(down)

    run(2)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    run(e2e_steps, e0, e1)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    e2e_value = whole_job_tflops(world, flops, e2e_ms)
    return {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": in_bytes,
            "d2h_bytes_per_step": out_bytes, "overlap": "copies on separate streams, 2 buffer sets"}


if __name__ == "__main__":
    main()

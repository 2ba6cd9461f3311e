"""Benchmark of the fused attention forward on GB300, one JSON line on stdout (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload s4k|s8k|s16k|ragged]
  python bench.py --impl reference ...      # the CPU oracle on the host cores, same metric

A step is one attn_fwd call (the whole hot path: one kernel) on one batch of seeded
synthetic BF16 input already resident in HBM. Between timed steps L2 is flushed by writing a
256 MB buffer; each step is timed by its own CUDA events on the launching stream, so the
flush is outside the measured kernel time. Under torchrun every rank runs the same workload
on its own GPU (independent replicas, no collective on the data path: weak scaling); the
value is all ranks' FLOPs over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "attention fwd TFLOPS (4·B·H·S²·D) at S=4K/8K/16K; % of GB300 BF16 dense peak"
UNIT = "TFLOPS"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_FLUSH_BYTES = 256 << 20

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from an ncu capture,
# keyed by sweep entry; each is valid only for the kernel source it was taken on (hash of the
# kernel's CUDA sources), and is reported as null otherwise.
TRAFFIC: dict[str, tuple[int, str]] = {
    "s4k": (240544768, "a8b815de643e88de"),         # 201,434,368 B read + 39,110,400 B written
    "s16k": (244620288, "a8b815de643e88de"),        # 201,450,752 B read + 43,169,536 B written
    "s4k_causal": (282608128, "a8b815de643e88de"),  # 237,624,064 B read + 44,984,064 B written
    "s8k": (242760192, "a8b815de643e88de"),         # 201,384,192 B read + 41,376,000 B written
    "ragged": (843931392, "a8b815de643e88de"),      # 648,556,544 B read + 195,374,848 B written
    "s8k_causal": (280591616, "a8b815de643e88de"),  # 234,008,832 B read + 46,582,784 B written
    "s16k_causal": (337310208, "a8b815de643e88de"), # 292,638,208 B read + 44,672,000 B written
}

# Dense BF16 tensor rate of one SM: an M128 N128 K16 tcgen05.mma (2*128*128*16 FLOP) every 64
# cycles, measured on this part with isolated MMA chains.
FLOP_PER_CLK_SM = 8192
# The nominal dense (no 2:4 sparsity) BF16 rate of one GB300, PFLOP/s.
NOMINAL_BF16_TFLOPS = 2250.0
KERNEL_SOURCES = ("attn_fwd.cu", "ptx.cuh")


def strip_comments(src: str) -> str:
    """C++ source without its comments (string and character literals kept), whitespace runs
    collapsed: what the compiler sees of the code."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash() -> str:
    """Hash of the kernel's CUDA sources without comments: traffic counters stay valid across
    comment edits and lapse with any change to the code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_attention_forward_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def step_stats(times_ms):
    """mean / median / min / max of per-step kernel times (ms)."""
    return {"mean": round(sum(times_ms) / len(times_ms), 5), "median": round(statistics.median(times_ms), 5),
            "min": round(min(times_ms), 5), "max": round(max(times_ms), 5)}


def roofline(flops, ms, peak, sm_count, sm_mhz, traffic=None):
    """Achieved TFLOP/s per launch against three denominators: the measured cuBLAS BF16 burst
    (`peak`, the headline fraction), the nominal dense BF16 figure, and the SM count x the
    per-SM MMA rate x the SM clock sampled during the run."""
    achieved = flops / (ms * 1e-3) / 1e12
    out = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
           "frac": round(achieved / peak, 4), "traffic": traffic,
           "peak_nominal": NOMINAL_BF16_TFLOPS, "frac_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4)}
    if sm_mhz:
        clk_peak = sm_count * FLOP_PER_CLK_SM * sm_mhz * 1e6 / 1e12
        out["peak_clock"] = round(clk_peak, 1)
        out["frac_clock"] = round(achieved / clk_peak, 4)
    return out


def config_of(w: wl.Workload, world: int, causal: bool = False) -> dict:
    """The workload description both arms print."""
    return {"workload": w.label(), "B": w.B, "H": w.H, "S": w.S, "D": w.D, "causal": causal,
            "scale": w.scale, "inputs": "seeded N(0,1) BF16" + (f", Q and K x{w.qk_gain:g}" if w.qk_gain != 1 else ""),
            "l2": "flushed between timed steps (256 MB write)" + (
                "; inputs larger than L2" if 3 * w.rows * w.D * 2 > 129e6 else ""),
            "parallelism": f"replicas x{world}"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's time: every rank passes its own, every rank gets the maximum."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, ms: float, world: int) -> float:
    """Whole-job TFLOPS: every rank's work over the slowest rank's time (weak scaling)."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def time_oracle(w: wl.Workload, q, k, v, budget_s: float, min_chunks: int = 1, causal: bool = False):
    """Time the oracle on row chunks (all heads) until `budget_s` has elapsed. Returns
    (TFLOPS, seconds, rows_per_head, cores). Causal work is counted as the keys each row sees
    (4*D FLOP per key), which sums to the 2*B*H*S^2*D convention over a whole call."""
    from oracle import attn_ref as ref
    qf, kf, vf = wl.to_f64(q), wl.to_f64(k), wl.to_f64(v)
    chunk = 32
    rows_done = 0
    keys_done = 0
    t0 = time.perf_counter()
    i = 0
    while True:
        r0 = (i * chunk) % w.S
        rows = list(range(r0, min(w.S, r0 + chunk)))
        ref.attention_rows(qf, kf, vf, w.scale, rows, causal=causal)
        rows_done += len(rows)
        keys_done += sum(r + 1 for r in rows) if causal else len(rows) * w.S
        i += 1
        el = time.perf_counter() - t0
        if el >= budget_s and i >= min_chunks:
            break
    flops = 4.0 * w.B * w.H * keys_done * w.D
    return flops / el / 1e12, el, rows_done, os.cpu_count()


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    q, k, v = wl.make_qkv(w)
    warm = max(args.warmup, 3)
    for _ in range(warm):
        time_oracle(w, q, k, v, budget_s=0.0, causal=args.causal)
    rates, secs, rows = [], 0.0, 0
    for _ in range(args.steps):
        r, el, nrows, cores = time_oracle(w, q, k, v, budget_s=args.ref_step_seconds, causal=args.causal)
        rates.append(r)
        secs += el
        rows += nrows
    value = statistics.median(rates)
    sample = (f"{args.steps} steps; each step times the fp64 oracle on >= {args.ref_step_seconds:g} s "
              f"of 32-query-row chunks over all {w.B * w.H} heads ({rows} rows per head in total) "
              f"of {w.label()}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": warm, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": config_of(w, world, args.causal),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_gpu(attn, torch, w, q, k, v, o, lse, steps, warmup, flush, stream, causal=False):
    for _ in range(warmup):
        attn.fwd(q, k, v, w.scale, out=o, lse=lse, causal=causal)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.add_(1)  # write > L2 between timed calls
        starts[i].record(stream)
        attn.fwd(q, k, v, w.scale, out=o, lse=lse, causal=causal)
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def run_gpu(args, w):
    import torch
    import dense_attention_forward_gb300 as attn

    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count

    q, k, v = (t.to(dev) for t in wl.make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), device=dev, dtype=torch.float32)
    flush = torch.zeros(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    warm = max(args.warmup, 3)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timed region
    barrier()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        times = time_gpu(attn, torch, w, q, k, v, o, lse, args.steps, warm, flush, stream, causal=args.causal)
        barrier()
        t_wall = time.perf_counter() - t_wall0
    kern_ms = sum(times) / len(times)
    kern_ms = max_over_ranks(kern_ms, dist, dev)
    flops = w.flops / 2 if args.causal else w.flops  # causal: 2*B*H*S^2*D
    value = job_throughput(flops, kern_ms, world)
    status = attn.device_status(reset=True)
    clocks = clk.summary()

    # ---- end to end: the library's host-to-host call (attn_fwd_host) every step: pinned host
    # q, k, v -> device, the kernel, device -> pinned host o and lse. Steps alternate between
    # two streams, each with its own device and output buffers, so step k+1's copy-in overlaps
    # step k's kernel and copy-out, as a serving loop would run them. Every step still moves
    # all of its inputs in and its outputs out.
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    lh = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
    bufs = [tuple(torch.empty_like(t) for t in (q, k, v, o)) + (torch.empty_like(lse),) for _ in range(2)]
    streams = [torch.cuda.Stream(dev) for _ in range(2)]

    def e2e_step(kstep):
        b = kstep & 1
        attn.fwd_host(qh, kh, vh, w.scale, out=oh[b], lse=lh[b], dev=bufs[b], stream=streams[b],
                      causal=args.causal)

    for kstep in range(4):
        e2e_step(kstep)
    barrier()
    for b in range(2):  # poison the outputs: the timed steps must write them again
        oh[b].fill_(float("nan"))
        lh[b].fill_(float("nan"))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    e0.record(stream)
    for st_ in streams:
        st_.wait_stream(stream)
    for kstep in range(e2e_steps):
        e2e_step(kstep)
    for st_ in streams:
        stream.wait_stream(st_)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = job_throughput(flops, e2e_ms, world)
    h2d = 3 * q.numel() * q.element_size()
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    # The timed end-to-end steps computed what the device-resident steps did, bit for bit, and
    # no bounded wait gave up on the way.
    e2e_status = attn.device_status(reset=True)
    last = (e2e_steps - 1) & 1
    o_dev, lse_dev = o.cpu(), lse.cpu()
    e2e_match = bool(torch.equal(oh[last], o_dev) and torch.equal(lh[last], lse_dev) and
                     torch.equal(oh[last ^ 1], o_dev) and torch.equal(lh[last ^ 1], lse_dev))
    if e2e_status != 0 or not e2e_match:
        raise RuntimeError(f"end-to-end steps: status word {e2e_status:#x}, outputs equal to the "
                           f"device-resident call: {e2e_match}")

    peaks, peaks_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sm_mhz = clocks.get("sm_mhz")

    def traffic_of(name):
        rec = TRAFFIC.get(name)
        return rec[0] if (rec and rec[1] == source_hash()) else None

    # ---- other workloads of the same metric (single GPU, same method, fewer steps)
    sweep = {}
    if not args.no_sweep:
        for name, causal in [(n, False) for n in args.sweep] + [(n, True) for n in args.causal_sweep]:
            if name == w.name and causal == args.causal:
                continue
            ws = wl.ALL[name]
            qs, ks, vs = (t.to(dev) for t in wl.make_qkv(ws))
            os_, ls_ = torch.empty_like(qs), torch.empty((ws.B, ws.H, ws.S), device=dev)
            ts = time_gpu(attn, torch, ws, qs, ks, vs, os_, ls_, args.sweep_steps, 3, flush, stream,
                          causal=causal)
            ms = sum(ts) / len(ts)
            # Causal FLOPs are counted as half the dense ones, 2*B*H*S^2*D.
            sflops = ws.flops / 2 if causal else ws.flops
            key = name + ("_causal" if causal else "")
            sweep[key] = {"workload": ws.label() + (" causal" if causal else ""), "ms": round(ms, 4),
                          "step_ms": step_stats(ts), "tflops": round(sflops / (ms * 1e-3) / 1e12, 1),
                          "tflops_median": round(sflops / (statistics.median(ts) * 1e-3) / 1e12, 1),
                          "roofline": roofline(sflops, ms, peak, sm_count, sm_mhz, traffic_of(key))}
            del qs, ks, vs, os_, ls_
        status |= attn.device_status(reset=True)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    rf = roofline(flops, kern_ms, peak, sm_count, sm_mhz, traffic_of(w.name + ("_causal" if args.causal else "")))
    rf["peak_source"] = f"{peaks_src} bf16_tflops (burst, cuBLAS 8192^3)"
    rf["peak_nominal_source"] = "nominal dense BF16 rate of one GB300 (no 2:4 sparsity)"
    rf["peak_clock_source"] = (f"{sm_count} SMs x {FLOP_PER_CLK_SM} FLOP/clk (one M128 N128 K16 MMA per 64 "
                               "cycles) x median sampled SM clock")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": warm, "ms_per_step": round(kern_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": config_of(w, world, args.causal),
        "step_ms": step_stats(times),
        "value_median": round(job_throughput(flops, statistics.median(times), world), 2),
        "value_best": round(job_throughput(flops, min(times), world), 2),
        "roofline": rf,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "schedule": "attn_fwd_host per step (copy-in, kernel, copy-out), steps alternating over 2 streams with their own buffers",
                "device_status": e2e_status, "outputs_equal_device_call": e2e_match},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
        "device_status": status,
        "sweep": sweep,
    }
    if not args.no_cpu_baseline and world == 1:
        qc, kc, vc = wl.make_qkv(w)
        rate, el, rows, cores = time_oracle(w, qc, kc, vc, budget_s=args.cpu_seconds, causal=args.causal)
        line["cpu_baseline"] = {
            "value": round(rate, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle on {rows} query rows of each of the {w.B * w.H} heads of "
                      f"{w.label()} ({el:.1f} s)"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="s4k", choices=sorted(wl.ALL))
    ap.add_argument("--causal", action="store_true",
                    help="time the causal variant as the step (FLOPs counted as 2*B*H*S^2*D)")
    ap.add_argument("--sweep", nargs="*", default=["s8k", "s16k", "ragged"])
    ap.add_argument("--causal-sweep", nargs="*", default=["s4k", "s8k", "s16k"])
    ap.add_argument("--sweep-steps", type=int, default=100)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=2.0)
    args = ap.parse_args()
    w = wl.ALL[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()

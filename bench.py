"""Benchmark: fused attention forward TFLOP/s on one GB300 (or N replicas).

One step = one fused attention forward over the whole batch of the
benchmark workload (default: B=4, H=32, N=4096, D=128, fp16, no mask -- the
pages' benchmark shape, "FlashAttention under the catlass template",
section "Performance data").  Inputs are seeded synthetic tensors resident
in HBM before the timed region; their 512 MiB working set (Q, K, V, O)
exceeds the 126 MB L2, so no extra flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the float64 CPU
oracle on a bounded sample of the same workload instead.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       [--impl reference]
Multi-GPU: torchrun --nproc-per-node N bench.py --gpus N ...  (independent
replicas, one per GPU: the (b, h) problems are independent, so there is no
data exchange; timing is reduced with a max over ranks).
"""

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

METRIC = "fused attention fwd TFLOP/s and % of GB300 dense FP16 tensor peak"
FALLBACK_PEAK_TFLOPS = 1900.0   # only if the measured-peaks file is absent
FALLBACK_HBM_GBS = 6800.0


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="f16_full_4k")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small cases for profiling)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--also", default="auto",
                    help="comma-separated forward workloads timed after the main one and reported under "
                         "'also' ('auto': the causal and window benchmark shapes when the main workload is "
                         "the default; 'none': skip)")
    ap.add_argument("--also-steps", type=int, default=300)
    return ap.parse_args(argv)


ALSO_DEFAULT = ("f16_causal_4k", "bf16_causal_4k", "bf16_window_16k")


# ------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": FALLBACK_PEAK_TFLOPS, "hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


# Sources the tensor-core forward kernel is compiled from (its own file and
# the headers it includes): a recorded traffic figure holds while they do.
FWD_KERNEL_SOURCES = ("fa_tc.cu", "tc_softmax.cuh", "rope_math.cuh", "tc_common.cuh", "ptx.cuh", "fa_geom.h",
                      "fa_internal.h")


def kernel_source_hash(files=FWD_KERNEL_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_16_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)
        self.mark = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = [r.split(", ") for r in self.lines[self.mark:] if r.count(",") >= 8] or \
               [r.split(", ") for r in self.lines if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ distributed

def dist_setup(args):
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "native" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)  # bind this rank to its GPU before NCCL sees it
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def reduce_max(pg, x, device):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg, device):
    if pg is not None:
        import torch
        pg.barrier(device_ids=[device.index]) if device.type == "cuda" else pg.barrier()


# ---------------------------------------------------------- reference arm

def cpu_oracle_sample(w, q, k, v, budget_s, rows=None):
    """Time the oracle, as it stands, on (b, h) heads of the workload until
    `budget_s` seconds pass; returns (TFLOP/s, description, cores)."""
    import numpy as np
    from oracle import attention_three_pass
    from attention_forward_16_gb300.flops import visible_keys_per_row
    qd, kd, vd = (t.float().numpy() for t in (q, k, v))
    per_row = visible_keys_per_row(w.N, w.mask, w.win_l, w.win_r)
    rot = oracle_rotation(w)
    done_flops, heads, t_total = 0, 0, 0.0
    r = rows or w.N
    while t_total < budget_s and heads < w.B * w.H:
        b, h = divmod(heads, w.H)
        r0 = (heads * 977) % max(1, w.N - r + 1) if rows else 0
        t0 = time.perf_counter()
        attention_three_pass(rot(qd[b:b + 1, h:h + 1, r0:r0 + r], r0), rot(kd[b:b + 1, h:h + 1], 0),
                             vd[b:b + 1, h:h + 1], w.scale, w.mask, w.win_l, w.win_r, q_offset=r0)
        t_total += time.perf_counter() - t0
        done_flops += 4 * w.D * int(per_row[r0:r0 + r].sum())
        heads += 1
    desc = f"{heads} of {w.B * w.H} heads" + (f", {r} query rows each" if rows else ", all rows") + \
        f" of {w.name}, float64 numpy" + (", rotary embedding of the head's Q rows and K" if w.rope else "") + \
        f", {t_total:.1f} s"
    return done_flops / t_total / 1e12, desc, blas_threads()


def oracle_rotation(w):
    """x, pos0 -> the oracle's rotary embedding of x (identity without rope)."""
    if not w.rope:
        return lambda x, pos0: x
    from oracle import STYLE_HALF, STYLE_INTERLEAVED, apply_rope, rope_tables
    cos, sin = rope_tables(w.N, w.D, w.rope_base)
    style = STYLE_HALF if w.rope == "half" else STYLE_INTERLEAVED
    return lambda x, pos0: apply_rope(x, cos, sin, style, pos0)


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count()


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    from attention_forward_16_gb300.inputs import make_workload
    q, k, v = make_workload(w)
    import numpy as np
    from oracle import attention_three_pass
    from attention_forward_16_gb300.flops import visible_keys_per_row
    per_row = visible_keys_per_row(w.N, w.mask, w.win_l, w.win_r)
    qd, kd, vd = (t.float().numpy() for t in (q, k, v))
    rows = 64
    rot = oracle_rotation(w)

    def step(i):
        b, h = divmod(i % (w.B * w.H), w.H)
        r0 = (i * 977) % (w.N - rows + 1)
        attention_three_pass(rot(qd[b:b + 1, h:h + 1, r0:r0 + rows], r0), rot(kd[b:b + 1, h:h + 1], 0),
                             vd[b:b + 1, h:h + 1], w.scale, w.mask, w.win_l, w.win_r, q_offset=r0)
        return 4 * w.D * int(per_row[r0:r0 + rows].sum())

    for i in range(args.warmup):
        step(i)
    flops_total = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops_total += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = flops_total / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "dtype_in": w.dtype,
                   "mask": w.mask, "window": [w.win_l, w.win_r], "rope": w.rope or None,
                   "step": f"{rows} query rows of one head"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"{rows} query rows x full keys of one (b, h) per step, float64 numpy"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- native arm

def time_forward_workload(w, args, device, pg, rank, local, peak):
    """Time the fused forward alone on workload ``w`` (inputs resident in HBM,
    larger than L2): ``args.also_steps`` launches after ``args.warmup``, each
    bracketed by CUDA events on the launching stream, with the SM clocks
    sampled meanwhile.  Returns a dict for the bench line's ``also`` key."""
    import torch
    import attention_forward_16_gb300 as fa
    from attention_forward_16_gb300.flops import attention_flops
    from attention_forward_16_gb300.inputs import make_workload

    q, k, v = (t.to(device) for t in make_workload(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    window = (w.win_l, w.win_r) if w.mask == fa.FA_MASK_WINDOW else None
    causal = w.mask == fa.FA_MASK_CAUSAL
    stream = torch.cuda.current_stream(device)

    def step():
        fa.attention_fwd(q, k, v, scale=w.scale, causal=causal, window=window, out=o, lse=lse)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError(f"kernel reported a timeout during warm-up of {w.name}")
    clocks = ClockSampler(local).start() if rank == 0 else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.also_steps)]
    barrier(pg, device)
    torch.cuda.synchronize()
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    barrier(pg, device)
    clk = clocks.stop() if clocks else None
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError(f"kernel reported a timeout while timing {w.name}")
    ms = reduce_max(pg, sum(a.elapsed_time(b) for a, b in ev) / len(ev), device)
    flops = attention_flops(w.B, w.H, w.N, w.D, w.mask, w.win_l, w.win_r)
    tf = flops / (ms / 1e3) / 1e12
    del q, k, v, o, lse
    return {"B": w.B, "H": w.H, "N": w.N, "D": w.D, "dtype": w.dtype, "mask": w.mask,
            "window": [w.win_l, w.win_r], "input_scale": w.input_scale, "steps": args.also_steps,
            "avg_launch_ms": ms, "algorithmic_flops_per_launch": flops, "TFLOP/s": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "traffic": recorded_traffic(w.name),
                         "kernel": "fa_fwd_tc_kernel<%d,%s>" % (w.D, w.dtype)},
            "clocks": clk}


def run_native(args, w, world, rank, local, pg):
    import torch
    import attention_forward_16_gb300 as fa
    from attention_forward_16_gb300.build import build
    from attention_forward_16_gb300.flops import algorithmic_bytes, attention_flops, rope_bytes
    from attention_forward_16_gb300.inputs import make_workload

    build()
    fa.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    q, k, v = make_workload(w)
    dq, dk, dv = q.to(device), k.to(device), v.to(device)
    do = torch.empty_like(dq)
    dl = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    window = (w.win_l, w.win_r) if w.mask == fa.FA_MASK_WINDOW else None
    causal = w.mask == fa.FA_MASK_CAUSAL
    stream = torch.cuda.current_stream(device)
    rope = bool(w.rope)
    if rope:
        # the cos/sin table is an input the caller owns, built once
        cos, sin = fa.rope_tables(w.N, w.D, w.rope_base, device=device)
        rq, rk = torch.empty_like(dq), torch.empty_like(dk)

    # With the rotary embedding, K goes through the rotation pass and Q is
    # rotated inside the attention kernel as its tiles arrive (fa_fwd_rope).
    def rotate(sq, sk, oq, ok_, s_=None):
        fa.apply_rope(None, sk, cos, sin, style=w.rope, k_out=ok_, stream=s_)

    def attend(aq, ak, av, ao, al, s_=None):
        fa.attention_fwd(aq, ak, av, scale=w.scale, causal=causal, window=window, out=ao, lse=al, stream=s_,
                         **({"rope": (cos, sin), "rope_style": w.rope} if rope else {}))

    def step():
        if rope:
            rotate(dq, dk, rq, rk)
            attend(dq, rk, dv, do, dl)
        else:
            attend(dq, dk, dv, do, dl)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError("kernel reported a timeout during warm-up")

    clocks = ClockSampler(local).start() if rank == 0 else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps if rope else 0)]
    barrier(pg, device)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        # the attention launch is bracketed alone (the roofline's kernel); the
        # rotation, when the workload has one, gets its own pair of events
        if rope:
            rev[i][0].record(stream)
            rotate(dq, dk, rq, rk)
            rev[i][1].record(stream)
            ev[i][0].record(stream)
            attend(dq, rk, dv, do, dl)
            ev[i][1].record(stream)
        else:
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(pg, device)
    clk = clocks.stop() if clocks else None
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError("kernel reported a timeout during the timed steps")
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    launch_sorted = sorted(launch_ms)
    launch_stats = {"median_ms": launch_sorted[len(launch_sorted) // 2], "min_ms": launch_sorted[0],
                    "max_ms": launch_sorted[-1]}
    total_ms = reduce_max(pg, total_ms, device)
    avg_launch_ms = reduce_max(pg, sum(launch_ms) / len(launch_ms), device)
    rope_ms = reduce_max(pg, sum(a.elapsed_time(b) for a, b in rev) / len(rev), device) if rope else None

    flops_step = attention_flops(w.B, w.H, w.N, w.D, w.mask, w.win_l, w.win_r)
    value = flops_step * args.steps * world / (total_ms / 1e3) / 1e12

    # ------------------------------------------------ end to end (host buffers)
    # Every step copies its inputs from pinned host memory, runs the fused
    # forward and copies O and LSE back.  Steps alternate between two streams
    # and two device buffer sets, so one step's copies overlap the previous
    # step's kernel (separate copy engines serve each direction).
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    streams = [torch.cuda.Stream(device), torch.cuda.Stream(device)]
    bufs = [(dq, dk, dv, do, dl)] + [tuple(torch.empty_like(t) for t in (dq, dk, dv, do, dl))]
    rbufs = [(rq, rk), (torch.empty_like(dq), torch.empty_like(dk))] if rope else None
    houts = [(torch.empty(do.shape, dtype=do.dtype, pin_memory=True),
              torch.empty(dl.shape, dtype=dl.dtype, pin_memory=True)) for _ in range(2)]

    def e2e_step(i):
        s_ = streams[i % 2]
        bq, bk, bv, bo, bl = bufs[i % 2]
        ho, hl = houts[i % 2]
        with torch.cuda.stream(s_):
            bq.copy_(hq, non_blocking=True)
            bk.copy_(hk, non_blocking=True)
            bv.copy_(hv, non_blocking=True)
            if rope:
                xq, xk = rbufs[i % 2]
                rotate(bq, bk, xq, xk, s_)
                attend(bq, xk, bv, bo, bl, s_)
            else:
                attend(bq, bk, bv, bo, bl, s_)
            ho.copy_(bo, non_blocking=True)
            hl.copy_(bl, non_blocking=True)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(pg, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s_ in streams:
        s_.wait_stream(stream)
    for i in range(args.e2e_steps):
        e2e_step(i)
    for s_ in streams:
        stream.wait_stream(s_)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(pg, e0.elapsed_time(e1), device)
    e2e_value = flops_step * args.e2e_steps * world / (e2e_ms / 1e3) / 1e12
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = houts[0][0].numel() * houts[0][0].element_size() + houts[0][1].numel() * houts[0][1].element_size()
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError("kernel reported a timeout during the end-to-end steps")

    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK_TFLOPS))
    also = {}
    if args.also == "auto":
        names = ALSO_DEFAULT if args.workload == "f16_full_4k" and args.batch is None else ()
    elif args.also == "none":
        names = ()
    else:
        names = tuple(n for n in args.also.split(",") if n)
    if names:
        from attention_forward_16_gb300.inputs import WORKLOADS
        for n in names:
            also[n] = time_forward_workload(WORKLOADS[n], args, device, pg, rank, local, peak)
            torch.cuda.empty_cache()

    if rank != 0:
        return 0
    achieved = flops_step / (avg_launch_ms / 1e3) / 1e12
    traffic = recorded_traffic(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "mask": w.mask,
                   "window": [w.win_l, w.win_r], "scale": w.scale, "global_batch": w.B * world,
                   "seq_len": w.N, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "working set (Q,K,V,O = %d MiB) exceeds L2; no flush" % (
                       algorithmic_bytes(w.B, w.H, w.N, w.D, w.dtype) >> 20),
                   "pct_of_peak": round(100.0 * value / world / peak, 2), "peak_tflops": peak,
                   "peak_source": f"{peak_src} bf16 burst (fp16 dense rate is the same)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "fa_fwd_tc_kernel<%d,%s>" % (w.D, w.dtype),
                     "algorithmic_flops_per_launch": flops_step,
                     "avg_launch_ms": avg_launch_ms, "launch_ms": launch_stats, "peak_source": peak_src},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps, "ms_per_step": e2e_ms / args.e2e_steps,
                "how": "attention_fwd on host inputs: pinned H2D copy, " +
                       ("rotary embedding of K (Q is rotated inside the attention kernel), " if rope else "") +
                       "fused forward, D2H of O and LSE every step; "
                       "steps alternate over two streams so copies overlap the previous step's kernel"},
        "gpu_launches": args.steps * (2 if rope else 1),
        "gpu_launches_also": sum(a["steps"] for a in also.values()),
    }
    if rope:
        hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
        rb = rope_bytes(w)
        line["config"]["rope"] = {"style": w.rope, "base": w.rope_base}
        line["rope_kernel"] = {
            "kernel": "fa_rope_kernel<%s,%s> (K only; Q is rotated in fa_fwd_tc_kernel)" % (w.dtype, w.rope),
            "avg_launch_ms": rope_ms,
            "share_of_step": rope_ms / (total_ms / args.steps),
            "roofline": {"bound": "hbm", "achieved": rb / (rope_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": rb / (rope_ms / 1e3) / 1e9 / hbm, "algorithmic_bytes_per_launch": rb,
                         "peak_source": peak_src}}
    if also:
        line["also"] = also
    if world == 1 and not args.no_cpu_baseline:
        tf, desc, cores = cpu_oracle_sample(w, q, k, v, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)
    return 0


def decode_kernel_name(rows, n_splits, dtype="bf16"):
    """The decode kernels a call runs: one query row per (b, K/V head) takes the
    split kernel; two to sixteen 16-bit rows the tensor-core (mma.sync) kernel;
    fp32 rows the lane-group rows kernel (up to four) or the 16-row split
    kernel; a combine pass follows when the cache is split."""
    if rows == 1:
        main = "fa_decode_split_kernel"
    elif dtype in ("f16", "bf16"):
        main = "fa_decode_mma_kernel"
    else:
        main = "fa_decode_rows_kernel" if rows <= 4 else "fa_decode_split_kernel"
    return main + (" + fa_decode_combine_kernel" if n_splits > 1 else "")


def run_decode(args, w, world, rank, local, pg):
    """Decode against a K/V cache: HBM-bound, reported as achieved GB/s of the
    compulsory traffic (cache read once, Q read, O and LSE written)."""
    import torch
    import attention_forward_16_gb300 as fa
    from attention_forward_16_gb300.build import build
    from attention_forward_16_gb300.inputs import make_decode

    build()
    fa.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    q, k, v = make_decode(w)
    if w.page_size:
        from attention_forward_16_gb300.inputs import make_paged
        k, v, table = make_paged(w, k, v)
        dtab = table.to(device)
        dlens = torch.full((w.B,), w.Nk, dtype=torch.int32, device=device)
    dq, dk, dv = q.to(device), k.to(device), v.to(device)
    do = torch.empty_like(dq)
    dl = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=device)
    Hkv = w.Hkv or w.H
    ns, wb = fa.fa_decode_plan_gqa(w.B, w.H, Hkv, w.Nq, w.Nk, w.D, 0)
    ws = torch.empty(max(wb, 1), dtype=torch.uint8, device=device)
    window = (w.win_l, w.win_r) if w.mask == fa.FA_MASK_WINDOW else None
    stream = torch.cuda.current_stream(device)

    def step():
        if w.page_size:
            fa.attention_decode_paged(dq, dk, dv, dtab, dlens, max_seq_len=w.Nk, scale=w.scale,
                                      causal=w.mask == fa.FA_MASK_CAUSAL, window=window, out=do, lse=dl,
                                      workspace=ws if wb > 0 else None)
        else:
            fa.attention_decode(dq, dk, dv, scale=w.scale, causal=w.mask == fa.FA_MASK_CAUSAL, window=window,
                                out=do, lse=dl, workspace=ws if wb > 0 else None)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local).start() if rank == 0 else None
    barrier(pg, device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(pg, device)
    clk = clocks.stop() if clocks else None
    ms = reduce_max(pg, t0.elapsed_time(t1), device) / args.steps
    e = {"f16": 2, "bf16": 2, "f32": 4}[w.dtype]
    nbytes = w.B * Hkv * 2 * w.Nk * w.D * e + w.B * w.H * (2 * w.Nq * w.D * e + w.Nq * 4)
    if rank != 0:
        return 0
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    gbs = nbytes / (ms / 1e3) / 1e9
    line = {
        "metric": "attention decode HBM GB/s (split-K, K/V cache read once)", "value": gbs * world, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": Hkv, "Nq": w.Nq, "Nk": w.Nk, "D": w.D,
                   "page_size": w.page_size or None,
                   "mask": w.mask,
                   "n_splits": ns, "workspace_bytes": wb,
                   "l2": "K/V cache (%d MiB) exceeds L2; no flush" % (2 * w.B * Hkv * w.Nk * w.D * e >> 20)},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": None, "kernel": decode_kernel_name(w.H // Hkv * w.Nq, ns, w.dtype),
                     "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": ms, "peak_source": src},
        "clocks": clk, "gpu_launches": args.steps * (2 if ns > 1 else 1),
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- backward

METRIC_BWD = "fused attention bwd TFLOP/s (5-product count) and % of GB300 dense FP16 tensor peak"


def make_upstream(w):
    """The upstream gradient dO of a backward workload: drawn like Q, seed + 1."""
    from attention_forward_16_gb300.inputs import make_qkv
    return make_qkv(w.B, w.H, w.N, w.D, w.dtype, seed=w.seed + 1, input_scale=w.input_scale, n_k=1)[0]


def oracle_bwd_sample(w, q, k, v, do, r0, rows):
    """The oracle's backward for `rows` query rows of one head (their dQ and
    their contributions to dK, dV); returns the 5-product flops it covers."""
    from oracle import attention_backward
    from attention_forward_16_gb300.flops import visible_keys_per_row
    attention_backward(q[:, :, r0:r0 + rows], k, v, do[:, :, r0:r0 + rows], w.scale, w.mask, w.win_l, w.win_r,
                       q_offset=r0)
    per_row = visible_keys_per_row(w.N, w.mask, w.win_l, w.win_r)
    return 10 * w.D * int(per_row[r0:r0 + rows].sum())


def run_backward(args, w, world, rank, local, pg):
    """Backward pass: one fa_bwd call (pre-pass, dK/dV kernel, dQ kernel) per
    step for fixed Q, K, V, O, LSE and dO resident in HBM."""
    import torch
    import attention_forward_16_gb300 as fa
    from attention_forward_16_gb300.build import build
    from attention_forward_16_gb300.flops import attention_flops
    from attention_forward_16_gb300.inputs import make_workload

    build()
    fa.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    q, k, v = make_workload(w)
    do_h = make_upstream(w)
    dq_, dk_, dv_, ddo = (t.to(device) for t in (q, k, v, do_h))
    window = (w.win_l, w.win_r) if w.mask == fa.FA_MASK_WINDOW else None
    causal = w.mask == fa.FA_MASK_CAUSAL
    stream = torch.cuda.current_stream(device)
    o, lse = fa.attention_fwd(dq_, dk_, dv_, scale=w.scale, causal=causal, window=window)
    gq, gk, gv = torch.empty_like(dq_), torch.empty_like(dk_), torch.empty_like(dv_)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8, device=device)

    def step(aq=dq_, ak=dk_, av=dv_, ao=o, al=lse, ado=ddo, s_=None):
        fa.attention_bwd(aq, ak, av, ao, al, ado, scale=w.scale, causal=causal, window=window, dq=gq, dk=gk,
                         dv=gv, workspace=ws, stream=s_)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError("kernel reported a timeout during warm-up")
    clocks = ClockSampler(local).start() if rank == 0 else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(pg, device)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(pg, device)
    clk = clocks.stop() if clocks else None
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError("kernel reported a timeout during the timed steps")
    total_ms = reduce_max(pg, t0.elapsed_time(t1), device)
    call_ms = reduce_max(pg, sum(a.elapsed_time(b) for a, b in ev) / args.steps, device)
    flops_step = 2.5 * attention_flops(w.B, w.H, w.N, w.D, w.mask, w.win_l, w.win_r)
    value = flops_step * args.steps * world / (total_ms / 1e3) / 1e12

    # end to end: inputs from pinned host memory, gradients back, every step
    hin = [t.pin_memory() for t in (q, k, v, o.cpu(), lse.cpu(), do_h)]
    bins = [torch.empty_like(t, device=device) for t in hin]
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (gq, gk, gv)]

    def e2e_step():
        for dst, src in zip(bins, hin):
            dst.copy_(src, non_blocking=True)
        step(*bins[:3], bins[3], bins[4], bins[5])
        for dst, src in zip(hout, (gq, gk, gv)):
            dst.copy_(src, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier(pg, device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(pg, e0.elapsed_time(e1), device)
    if fa.fa_device_status(stream.cuda_stream) != 0:
        raise RuntimeError("kernel reported a timeout during the end-to-end steps")
    if rank != 0:
        return 0
    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK_TFLOPS))
    achieved = flops_step / (call_ms / 1e3) / 1e12
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "mask": w.mask,
                   "window": [w.win_l, w.win_r], "scale": w.scale, "pass": "backward",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "working set (Q, K, V, O, dO and the three gradients) exceeds L2; no flush",
                   "flops": "5 products (S, dP, dV, dK, dQ) of 2 N_visible D each; the kernels execute 7 "
                            "(the dQ kernel recomputes S and dP)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "fa_bwd call: fa_bwd_pre_kernel + fa_bwd_dkdv_kernel + fa_bwd_dq_kernel",
                     "algorithmic_flops_per_launch": flops_step, "avg_launch_ms": call_ms,
                     "peak_source": peak_src},
        "clocks": clk,
        "e2e": {"value": flops_step * args.e2e_steps * world / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout),
                "steps": args.e2e_steps, "ms_per_step": e2e_ms / args.e2e_steps,
                "how": "attention_bwd on host Q, K, V, O, LSE, dO: pinned H2D, backward, D2H of dQ, dK, dV"},
        "gpu_launches": 3 * args.steps,
    }
    if world == 1 and not args.no_cpu_baseline:
        qd, kd, vd, dd = (t.float().numpy() for t in (q, k, v, do_h))
        done, t_total, n = 0, 0.0, 0
        while t_total < args.cpu_seconds and n < w.B * w.H:
            b, h = divmod(n, w.H)
            r0 = (n * 977) % (w.N - 64 + 1)
            t_s = time.perf_counter()
            done += oracle_bwd_sample(w, qd[b:b + 1, h:h + 1], kd[b:b + 1, h:h + 1], vd[b:b + 1, h:h + 1],
                                      dd[b:b + 1, h:h + 1], r0, 64)
            t_total += time.perf_counter() - t_s
            n += 1
        line["cpu_baseline"] = {"value": done / t_total / 1e12, "unit": "TFLOP/s", "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": f"{n} heads x 64 query rows (their dQ and dK, dV contributions) of "
                                          f"{w.name}, float64 numpy, {t_total:.1f} s"}
    print(json.dumps(line), flush=True)
    return 0


def run_reference_bwd(args, w, world, rank):
    if rank != 0:
        return 0
    from attention_forward_16_gb300.inputs import make_workload
    q, k, v = make_workload(w)
    qd, kd, vd, dd = (t.float().numpy() for t in (q, k, v, make_upstream(w)))
    rows = 64

    def step(i):
        b, h = divmod(i % (w.B * w.H), w.H)
        r0 = (i * 977) % (w.N - rows + 1)
        return oracle_bwd_sample(w, qd[b:b + 1, h:h + 1], kd[b:b + 1, h:h + 1], vd[b:b + 1, h:h + 1],
                                 dd[b:b + 1, h:h + 1], r0, rows)

    for i in range(args.warmup):
        step(i)
    flops_total = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops_total += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = flops_total / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "dtype_in": w.dtype,
                   "mask": w.mask, "window": [w.win_l, w.win_r], "pass": "backward",
                   "step": f"{rows} query rows of one head"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"{rows} query rows x full keys of one (b, h) per step, float64 numpy"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0}), flush=True)
    return 0


def run_reference_decode(args, w, world, rank):
    """The float64 oracle on the host cores for a decode workload: each step is
    the plain definition for one (b, K/V head) group of queries against its
    whole cache (gathered through the block table when the cache is paged),
    reported as GB/s of that group's compulsory bytes."""
    if rank != 0:
        return 0
    from attention_forward_16_gb300.inputs import make_decode
    from oracle import attention_grouped
    q, k, v = make_decode(w)
    Hkv = w.Hkv or w.H
    G = w.H // Hkv
    e = 4 if w.dtype == "f32" else 2
    qd, kd, vd = (t.float().numpy() for t in (q, k, v))
    sample = "one (b, K/V head) group of queries x its whole cache per step, float64 numpy"
    if w.page_size:
        from attention_forward_16_gb300.inputs import make_paged
        from oracle.paged import gather_pages
        kp, vp, tp = make_paged(w, k, v)
        kc, vc, table = kp.float().numpy(), vp.float().numpy(), tp.numpy()
        sample += ", gathered page by page through the block table"

    def step(i):
        b, hk = i % w.B, (i // w.B) % Hkv
        if w.page_size:
            ks = gather_pages(kc, table[b], w.Nk, w.page_size)[:, hk][None, None]   # [1, 1, Nk, D]
            vs = gather_pages(vc, table[b], w.Nk, w.page_size)[:, hk][None, None]
        else:
            ks, vs = kd[b:b + 1, hk:hk + 1], vd[b:b + 1, hk:hk + 1]
        attention_grouped(qd[b:b + 1, hk * G:(hk + 1) * G], ks, vs, w.scale, w.mask, w.win_l, w.win_r,
                          q_offset=w.Nk - w.Nq)
        return 2 * w.Nk * w.D * e + 2 * G * w.Nq * w.D * e + G * w.Nq * 4

    for i in range(args.warmup):
        step(i)
    nbytes = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        nbytes += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": "attention decode HBM GB/s (split-K, K/V cache read once)", "value": value,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "H_kv": Hkv, "Nq": w.Nq, "Nk": w.Nk, "D": w.D,
                   "page_size": w.page_size or None, "mask": w.mask, "step": "one (b, K/V head) group"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": blas_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    from attention_forward_16_gb300.inputs import DECODE_WORKLOADS, WORKLOADS
    if args.workload in DECODE_WORKLOADS:
        world, rank, local, pg = dist_setup(args)
        try:
            if args.impl == "reference":
                return run_reference_decode(args, DECODE_WORKLOADS[args.workload], world, rank)
            return run_decode(args, DECODE_WORKLOADS[args.workload], world, rank, local, pg)
        finally:
            if pg is not None:
                pg.destroy_process_group()
    w = WORKLOADS[args.workload]
    if args.batch is not None:
        import dataclasses
        w = dataclasses.replace(w, B=args.batch, name=f"{w.name}_b{args.batch}")
    world, rank, local, pg = dist_setup(args)
    try:
        if args.impl == "reference":
            return (run_reference_bwd if w.backward else run_reference)(args, w, world, rank)
        return (run_backward if w.backward else run_native)(args, w, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

"""Throughput of the GPT-2 training step on one B300: tokens/s and bf16 MFU.

One step = zero_grad + n_accum x (forward + backward) + AdamW (norm, clip,
update, bf16 refresh) over synthetic Zipf(1.1) tokens, exactly the step the
C-ABI library runs.  Inputs are resident in HBM before the timed region; the
activations (GBs) are far larger than the 126 MB L2, so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 124M|350M|1558M]
    python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Under torchrun (N > 1) every rank trains its own replica, with no collective
(the data-parallel gradient exchange, dp.DataParallel, is not timed here); the
timed region is bracketed by barriers and the slowest rank's time is used.
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

METRIC = "training tokens/sec and bf16 MFU per step at 1 B300 (GPT-2 124M / 1558M)"

WORKLOADS = {
    # name: L, H, C, V, T, B (micro-batch), n_accum, AdamW hyper-parameters
    "124M": dict(L=12, H=12, C=768, V=50257, T=1024, B=16, accum=8,
                 hp=dict(lr=6e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)),
    "350M": dict(L=24, H=16, C=1024, V=50257, T=1024, B=8, accum=1,
                 hp=dict(lr=3e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)),
    "1558M": dict(L=48, H=25, C=1600, V=50257, T=1024, B=16, accum=32,
                  hp=dict(lr=6e-4, b1=0.9, b2=0.95, eps=1e-8, wd=0.1, clip=1.0)),
}
DESCR = {
    "124M": "GPT-2 124M throughput: L=12 H=12 C=768 V=50257 (padded 50304) T=1024, "
            "micro-batch B=16 x 8 accumulated = 131072 tokens/step, bf16-mixed, AdamW",
    "350M": "GPT-2 350M: L=24 H=16 C=1024 V=50257 (padded 50304) T=1024 B=8 = 8192 "
            "tokens/step, bf16-mixed, AdamW",
    "1558M": "GPT-2 1558M: L=48 H=25 C=1600 V=50257 (padded 50304) T=1024, micro-batch "
             "B=16 x 32 accumulated = 524288 tokens/step, bf16-mixed, AdamW",
}
# oracle samples: same architecture, a short sequence, one full step (forward,
# backward, AdamW).  The reference arm times one per timed step (so that a run
# of many steps stays within minutes); the cpu_baseline of the GPU run times
# one longer sample (about ten seconds of CPU work on the 124M architecture).
CPU_SAMPLE = dict(B=1, T=32)
CPU_BASELINE_SAMPLE = dict(B=1, T=256)


def n_params(L, C, V, T):
    Vp = ((V + 127) // 128) * 128
    return Vp * C + T * C + L * (12 * C * C + 13 * C) + 2 * C


def flops_per_token(w):
    """model flops: 6N + 6 L C T (causal attention counted once), with N the
    padded parameter count -- the definition behind the pages' MFU figures"""
    return 6 * n_params(w["L"], w["C"], w["V"], w["T"]) + 6 * w["L"] * w["C"] * w["T"]


def kernel_sources_hash():
    """sha256 over the CUDA sources (file names and contents, sorted)"""
    import hashlib
    d = os.path.join(ROOT, "scratch_gpt_step_train_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()


def load_traffic(workload):
    """DRAM bytes per launch of each kernel class, from the committed ncu
    summary; None when the kernels changed after the counters were taken."""
    p = os.path.join(ROOT, "profiles", f"dram_traffic_gpt2_{workload}.txt")
    if not os.path.exists(p):
        return None
    out, sha = {}, None
    for line in open(p):
        line = line.strip()
        if line.startswith("# kernel_sources_sha256"):
            sha = line.split()[-1]
        elif line and not line.startswith("#"):
            name, val = line.split()[:2]
            out[name] = float(val)
    if sha != kernel_sources_hash():
        return None
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, \
        "fallback"


# --------------------------------------------------------------------------- CPU
def cpu_oracle_step_rate(w, sample, steps=1, warmup=0):
    """Time the oracle (fp64 build, all host cores) on `sample` tokens of the
    workload's architecture: forward + backward + AdamW per step.  Runs in a
    fresh interpreter so no CUDA context is shared with it."""
    code = f"""
import json, os, sys, time
sys.path.insert(0, {ROOT!r})
from oracle.pyoracle import Model
from scratch_gpt_step_train_b300 import inputs
w = {json.dumps({k: w[k] for k in ('L', 'H', 'C', 'V')})}
B, T = {sample['B']}, {sample['T']}
m = Model(w['L'], w['H'], w['C'], w['V'], T, B, seed=1)
st = inputs.ZipfStream(2, B, T, w['V'])
hp = {json.dumps(w['hp'])}
times = []
for i in range({steps + warmup}):
    tok, tgt = st.next()
    t0 = time.perf_counter()
    m.zero_grad(); m.forward(tok, tgt); m.backward()
    m.adamw_step(hp['lr'], hp['b1'], hp['b2'], hp['eps'], hp['wd'], hp['clip'])
    times.append(time.perf_counter() - t0)
print(json.dumps(dict(times=times[{warmup}:])))
"""
    cores = os.cpu_count() or 1
    env = dict(os.environ, OMP_NUM_THREADS=str(cores))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle run failed: " + r.stderr[-2000:])
    times = json.loads(r.stdout.strip().splitlines()[-1])["times"]
    tok = sample["B"] * sample["T"]
    return tok * len(times) / sum(times), cores, times


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------- GPU
def run_gpu(args, w, rank, world):
    import numpy as np
    import torch
    from scratch_gpt_step_train_b300 import inputs
    from scratch_gpt_step_train_b300.gpt2 import BF16, GPT2

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    B, T, accum = w["B"], w["T"], args.accum or w["accum"]
    hp = w["hp"]
    with torch.cuda.stream(stream):
        model = GPT2(w["L"], w["H"], w["C"], w["V"], T, B, seed=1, mode=BF16, stream=stream)
    # synthetic Zipf(1.1) tokens, resident on the device before timing
    zs = inputs.ZipfStream(2 + rank, B, T, w["V"])
    nbuf = accum
    host = [zs.next() for _ in range(nbuf)]
    dtok = [torch.from_numpy(a).to(f"cuda:{dev}") for a, _ in host]
    dtgt = [torch.from_numpy(b).to(f"cuda:{dev}") for _, b in host]
    torch.cuda.synchronize()

    def step():
        model.zero_grad()
        for i in range(accum):
            model.forward(dtok[i], dtgt[i])
            model.backward()
        return model.adamw_step(**hp)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # calibration pass: which kernel class dominates (events on every class)
    model.prof_enable(None)
    step()
    model.prof_enable([])
    prof = model.prof_read()
    dom = max(prof, key=lambda k: prof[k][0])
    model.prof_reset()
    for _ in range(max(0, args.warmup - 1)):
        step()
    torch.cuda.synchronize()

    # timed region: events around the dominant class only
    model.prof_enable([dom])
    clocks = ClockSampler(dev)
    barrier()
    torch.cuda.synchronize()
    launches0 = model.launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    losses = []
    # an NVTX range marks the timed steps for profilers (a no-op otherwise)
    torch.cuda.nvtx.range_push("timed_steps")
    for _ in range(args.steps):
        step()
    torch.cuda.nvtx.range_pop()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    launches = model.launch_count() - launches0
    model.prof_enable([])
    dprof = model.prof_read()[dom]
    final_loss = model.get_loss()

    # end to end through the public host-buffer call: pinned host tokens
    # copied every micro-step, the loss read back every step
    ptok = [torch.from_numpy(a).pin_memory() for a, _ in host]
    ptgt = [torch.from_numpy(b).pin_memory() for _, b in host]
    htok = [p.numpy() for p in ptok]
    htgt = [p.numpy() for p in ptgt]
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        model.zero_grad()
        for i in range(accum):
            model.forward(htok[i], htgt[i])
            model.backward()
        model.adamw_step(**hp)
        losses.append(model.get_loss())
    torch.cuda.synchronize()
    barrier()
    e2e_s = time.perf_counter() - t0
    return dict(ms=ms, launches=launches, dom=dom, dprof=dprof, clocks=clk, e2e_s=e2e_s,
                e2e_steps=e2e_steps, final_loss=final_loss, accum=accum,
                h2d=accum * 2 * B * T * 4, d2h=24, prof=prof)


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="124M", choices=sorted(WORKLOADS))
    ap.add_argument("--accum", type=int, default=0, help="override micro-batches per step")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = WORKLOADS[args.workload]
    peaks, peak_kind = load_peaks()
    fpt = flops_per_token(w)

    if args.impl == "reference":
        # the CPU oracle as the reference arm; rank 0 alone
        if rank != 0:
            return
        rate, cores, times = cpu_oracle_step_rate(w, CPU_SAMPLE, steps=args.steps,
                                                  warmup=args.warmup)
        sample = (f"{args.workload} architecture, B={CPU_SAMPLE['B']} T={CPU_SAMPLE['T']}, one "
                  f"full step (forward, backward, AdamW) per timed step, fp64 oracle")
        line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s",
                "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": DESCR[args.workload], "sample": sample},
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cores,
                                 "kind": "oracle", "sample": sample, "cpu": cpu_model()},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, cores, times = cpu_oracle_step_rate(w, CPU_BASELINE_SAMPLE, steps=1, warmup=0)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{args.workload} architecture, B={CPU_BASELINE_SAMPLE['B']} "
                         f"T={CPU_BASELINE_SAMPLE['T']}, one full step (forward, backward, AdamW), "
                         f"fp64 oracle, {statistics.mean(times):.1f} s",
               "cpu": cpu_model()}

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    r = run_gpu(args, w, rank, world)
    ms = max_over_ranks(r["ms"], world)
    e2e_s = max_over_ranks(r["e2e_s"], world)
    accum = r["accum"]
    tok_step = w["B"] * w["T"] * accum
    value = world * tok_step * args.steps / (ms / 1e3)
    e2e_value = world * tok_step * r["e2e_steps"] / e2e_s
    peak_tf = peaks.get("bf16_tflops", 1800.0)
    peak_sus = peaks.get("bf16_tflops_sustained", 1400.0)
    mfu = value / world * fpt / (peak_tf * 1e12)

    dom, (dms, dn, dfl, dby) = r["dom"], r["dprof"]
    traffic = load_traffic(args.workload)
    traffic = traffic.get(dom) if traffic else None
    if dfl > 0:
        achieved = dfl / dn / (dms / dn / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved,
                "peak": peak_sus, "unit": "TFLOP/s", "frac": achieved / peak_sus,
                "traffic": traffic, "algorithmic_bytes": dby / dn,
                "peak_kind": f"bf16 sustained ({peak_kind})",
                "launches": dn, "avg_launch_ms": dms / dn}
    else:
        achieved = dby / dn / (dms / dn / 1e3) / 1e9
        hbm = peaks.get("hbm_gbs", 6400.0)
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                "peak_kind": f"hbm copy ({peak_kind})", "launches": dn,
                "avg_launch_ms": dms / dn}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": DESCR[args.workload] if args.accum == 0 or args.accum == w["accum"]
                   else DESCR[args.workload] + f" (accumulation overridden to {accum})",
                   "tokens_per_step": tok_step * world, "seq_len": w["T"],
                   "micro_batch": w["B"], "grad_accum": accum,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "working set (activations) far larger than L2; no flush"},
        "bf16_mfu": {"value": mfu, "flops_per_token": fpt,
                     "peak_tflops": peak_tf, "peak_kind": f"bf16 burst ({peak_kind})",
                     "mfu_vs_sustained": value / world * fpt / (peak_sus * 1e12)},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_steps"]},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "final_loss": r["final_loss"],
        "kernel_ms_calibration_step": {k: round(v[0], 3) for k, v in r["prof"].items() if v[1]},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

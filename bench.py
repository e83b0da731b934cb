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
CPU_SAMPLE_1558M = dict(B=1, T=128)


def n_params(L, C, V, T):
    Vp = ((V + 127) // 128) * 128
    return Vp * C + T * C + L * (12 * C * C + 13 * C) + 2 * C


def flops_per_token(w):
    """model flops: 6N + 6 L C T (causal attention counted once), with N the
    padded parameter count -- the definition behind the pages' MFU figures"""
    return 6 * n_params(w["L"], w["C"], w["V"], w["T"]) + 6 * w["L"] * w["C"] * w["T"]


# the sources of the kernels whose DRAM traffic profiles/dram_traffic_*.txt
# records (the products and attention), with the headers they include
TRAFFIC_SOURCES = ("gemm_tc_kernel.cuh", "gemm_tc.h", "tc_ptx.cuh", "common.cuh", "kernels.h",
                   "k_attn_tc.cu")


def kernel_sources_hash():
    """sha256 over the sources of the product and attention kernels (file
    names and contents, sorted)"""
    import hashlib
    d = os.path.join(ROOT, "scratch_gpt_step_train_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f in TRAFFIC_SOURCES or f.startswith("k_gemm_tc"):
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
def cpu_oracle_step_rate(w, sample, steps=1, warmup=0, threads=None):
    """Time the oracle (fp64 build) on `sample` tokens of the workload's
    architecture: forward + backward + AdamW per step, with `threads` OpenMP
    threads (default: all host cores).  Runs in a fresh interpreter so no
    CUDA context is shared with it.  Returns (tokens/s, threads, step times)."""
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
    cores = threads or os.cpu_count() or 1
    env = dict(os.environ, OMP_NUM_THREADS=str(cores))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle run failed: " + r.stderr[-2000:])
    times = json.loads(r.stdout.strip().splitlines()[-1])["times"]
    tok = sample["B"] * sample["T"]
    return tok * len(times) / sum(times), cores, times


def oracle_bytes(w, sample):
    """host memory the fp64 oracle holds for this architecture and sample:
    params, grads, m, v and the activations it keeps for the backward"""
    L, H, C, V, T, B = w["L"], w["H"], w["C"], w["V"], sample["T"], sample["B"]
    Vp = ((V + 127) // 128) * 128
    n = n_params(L, C, V, T)
    act = L * (17 * B * T * C + B * H * T * T) + 3 * B * T * Vp + 16 * B * T * C
    return 8 * (4 * n + act)


def mem_available():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def cpu_baselines():
    """The oracle, as it stands, on bounded samples of the workloads: the
    124M architecture at all host cores and at one thread, and the 1558M
    architecture at all cores (skipped, with the reason, when the host has
    not the memory for it)."""
    runs = []
    for wl, sample, threads in (("124M", CPU_BASELINE_SAMPLE, None),
                                ("124M", CPU_SAMPLE, 1),
                                ("1558M", CPU_SAMPLE_1558M, None)):
        w = WORKLOADS[wl]
        need, have = oracle_bytes(w, sample), mem_available()
        desc = (f"{wl} architecture, B={sample['B']} T={sample['T']}, one full step "
                f"(forward, backward, AdamW), fp64 oracle")
        if have is not None and need * 1.25 > have:
            runs.append({"sample": desc, "skipped": f"needs {need / 2**30:.0f} GiB of host "
                         f"memory, {have / 2**30:.0f} GiB available"})
            continue
        rate, cores, times = cpu_oracle_step_rate(w, sample, steps=1, warmup=0, threads=threads)
        runs.append({"value": rate, "unit": "tokens/s", "cores": cores,
                     "sample": f"{desc}, {statistics.mean(times):.1f} s"})
    head = runs[0]
    return {"value": head["value"], "unit": "tokens/s", "cores": head["cores"], "kind": "oracle",
            "sample": head["sample"], "cpu": cpu_model(), "runs": runs}


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
def run_gpu(w, rank, world, steps, warmup, accum, rl_steps):
    """Train the workload's model on this rank's GPU and time it.

    1. warm-up steps (untimed);
    2. the timed region: `steps` whole steps between CUDA events on the
       handle's stream, no per-kernel instrumentation, clocks sampled;
    3. a roofline pass (not part of the value): one step with events around
       every kernel class picks the dominant class, then `rl_steps` steps with
       events around that class alone give its average launch duration;
    4. end to end through the public host-buffer call, the same number of
       steps as the timed region: pinned host tokens copied every micro-step,
       the loss read back every step (with the update's norm, clip state and
       error word: 20 bytes), timed on the host clock."""
    import torch
    from scratch_gpt_step_train_b300 import inputs
    from scratch_gpt_step_train_b300.gpt2 import BF16, GPT2

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    B, T = w["B"], w["T"]
    hp = w["hp"]
    with torch.cuda.stream(stream):
        model = GPT2(w["L"], w["H"], w["C"], w["V"], T, B, seed=1, mode=BF16, stream=stream)
    # synthetic Zipf(1.1) tokens, resident on the device before timing
    zs = inputs.ZipfStream(2 + rank, B, T, w["V"])
    host = [zs.next() for _ in range(accum)]
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

    model.prof_enable([])
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()

    # timed region
    clocks = ClockSampler(dev)
    barrier()
    torch.cuda.synchronize()
    launches0 = model.launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    # an NVTX range marks the timed steps for profilers (a no-op otherwise)
    torch.cuda.nvtx.range_push("timed_steps")
    for _ in range(steps):
        step()
    torch.cuda.nvtx.range_pop()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    launches = model.launch_count() - launches0
    final_loss = model.get_loss()

    # roofline pass
    model.prof_reset()
    model.prof_enable(None)
    step()
    torch.cuda.synchronize()
    prof = model.prof_read()
    dom = max(prof, key=lambda k: prof[k][0])
    model.prof_reset()
    model.prof_enable([dom])
    for _ in range(rl_steps):
        step()
    torch.cuda.synchronize()
    model.prof_enable([])
    dprof = model.prof_read()[dom]

    # memory-bound classes: in-step GB/s (from the all-class step above)
    # against a copy of the same bytes (half read, half written) measured now
    mem = {}
    for k, (cms, cn, cfl, cby) in prof.items():
        if cn and cfl == 0 and cby > 0 and cms > 0:
            mem[k] = {"bytes_per_launch": cby / cn, "gbs": cby / cn / (cms / cn / 1e3) / 1e9,
                      "launches": cn}
    for k, v in mem.items():
        v["copy_gbs_same_bytes"] = copy_rate(int(v["bytes_per_launch"]), stream)

    # end to end
    ptok = [torch.from_numpy(a).pin_memory() for a, _ in host]
    ptgt = [torch.from_numpy(b).pin_memory() for _, b in host]
    htok = [p.numpy() for p in ptok]
    htgt = [p.numpy() for p in ptgt]
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        model.zero_grad()
        for i in range(accum):
            model.forward(htok[i], htgt[i])
            model.backward()
        model.adamw_step(**hp)
        model.get_loss()
    torch.cuda.synchronize()
    barrier()
    e2e_s = time.perf_counter() - t0
    model.close()
    del model
    torch.cuda.empty_cache()
    return dict(ms=ms, launches=launches, dom=dom, dprof=dprof, clocks=clk, e2e_s=e2e_s,
                final_loss=final_loss, h2d=accum * 2 * B * T * 4, d2h=20, prof=prof, mem=mem)


def copy_rate(nbytes, stream, reps=7):
    """GB/s of torch's device copy moving nbytes in all (nbytes/2 read,
    nbytes/2 written), median of `reps`, on the bench's stream: the ceiling a
    memory-bound kernel of that size meets, ramp and tail included"""
    import torch
    n = max(16, nbytes // 2)
    src = torch.empty(n, dtype=torch.uint8, device="cuda")
    dst = torch.empty_like(src)
    ts = []
    with torch.cuda.stream(stream):
        for _ in range(reps + 2):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src)
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
    return 2 * n / (statistics.median(ts[2:]) / 1e3) / 1e9


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
    ap.add_argument("--rl-steps", type=int, default=3,
                    help="steps of the roofline pass (events around the dominant class)")
    ap.add_argument("--secondary", default="1558M:3,350M:30",
                    help="workloads timed after the first, NAME[:STEPS] separated by commas "
                         "(1-GPU runs; '' for none): the first is reported as `secondary`, "
                         "the others as `secondary_NAME`")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = WORKLOADS[args.workload]
    peaks, peak_kind = load_peaks()

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
        cpu = cpu_baselines()

    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    line = workload_line(args.workload, w, args.steps, args.warmup, args.accum, args.rl_steps,
                         rank, world, peaks, peak_kind)
    if world == 1:
        first = True
        for name, steps in parse_secondary(args.secondary):
            if name == args.workload:
                continue
            sec = workload_line(name, WORKLOADS[name], steps, 3, 0, 1, rank, world, peaks,
                                peak_kind)
            line["secondary" if first else "secondary_" + name] = {k: sec[k] for k in (
                "value", "unit", "ms_per_step", "steps", "warmup", "config", "bf16_mfu",
                "roofline", "e2e", "gpu_launches", "clocks", "final_loss", "memory_bound")}
            first = False
    if rank != 0:
        return
    line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def parse_secondary(spec):
    """'1558M:3,350M:30' -> [('1558M', 3), ('350M', 30)]; a name without a
    step count gets 3 timed steps"""
    out = []
    for item in filter(None, (x.strip() for x in (spec or "").split(","))):
        name, _, steps = item.partition(":")
        if name not in WORKLOADS:
            raise SystemExit(f"unknown workload {name!r} in --secondary")
        out.append((name, int(steps) if steps else 3))
    return out


def workload_line(name, w, steps, warmup, accum_override, rl_steps, rank, world, peaks,
                  peak_kind):
    accum = accum_override or w["accum"]
    fpt = flops_per_token(w)
    r = run_gpu(w, rank, world, steps, warmup, accum, rl_steps)
    ms = max_over_ranks(r["ms"], world)
    e2e_s = max_over_ranks(r["e2e_s"], world)
    tok_step = w["B"] * w["T"] * accum
    value = world * tok_step * steps / (ms / 1e3)
    e2e_value = world * tok_step * steps / e2e_s
    peak_tf = peaks.get("bf16_tflops", 1800.0)
    peak_sus = peaks.get("bf16_tflops_sustained", 1400.0)
    mfu = value / world * fpt / (peak_tf * 1e12)

    dom, (dms, dn, dfl, dby) = r["dom"], r["dprof"]
    traffic = load_traffic(name)
    traffic = traffic.get(dom) if traffic else None
    if dfl > 0:
        achieved = dfl / dn / (dms / dn / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved,
                "peak": peak_sus, "unit": "TFLOP/s", "frac": achieved / peak_sus,
                "traffic": traffic, "algorithmic_bytes": dby / dn,
                "peak_kind": f"bf16 sustained ({peak_kind})",
                "launches": dn, "avg_launch_ms": dms / dn,
                "frac_of_burst": achieved / peak_tf}
    else:
        achieved = dby / dn / (dms / dn / 1e3) / 1e9
        hbm = peaks.get("hbm_gbs", 6400.0)
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                "peak_kind": f"hbm copy ({peak_kind})", "launches": dn,
                "avg_launch_ms": dms / dn}
    descr = DESCR[name] if accum == w["accum"] else \
        DESCR[name] + f" (accumulation overridden to {accum})"
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": descr, "tokens_per_step": tok_step * world, "seq_len": w["T"],
                   "micro_batch": w["B"], "grad_accum": accum,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "working set (activations) far larger than L2; no flush"},
        "bf16_mfu": {"value": mfu, "flops_per_token": fpt,
                     "peak_tflops": peak_tf, "peak_kind": f"bf16 burst ({peak_kind})",
                     "mfu_vs_sustained": value / world * fpt / (peak_sus * 1e12)},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "steps": steps},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "final_loss": r["final_loss"],
        "kernel_ms_calibration_step": {k: round(v[0], 3) for k, v in r["prof"].items() if v[1]},
        "memory_bound": {k: {"gbs": round(v["gbs"], 1),
                             "mb_per_launch": round(v["bytes_per_launch"] / 1e6, 2),
                             "copy_gbs_same_bytes": round(v["copy_gbs_same_bytes"], 1),
                             "frac_of_peak": round(v["gbs"] / peaks.get("hbm_gbs", 6400.0), 3),
                             "frac_of_copy": round(v["gbs"] / v["copy_gbs_same_bytes"], 3)}
                         for k, v in r["mem"].items()},
    }


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput of causal GQA attention forward + backward (RoPE on Q/K) on GB300.

One step = ne_attn_fwd + ne_attn_bwd over one batch of the 116M-model
attention shape (B=16, T=512, Hq=12, Hkv=4, D=64; synthetic N(0,1) bf16
inputs, seeded).  The metric is algorithmic TFLOP/s: 14 * B * Hq * D *
T(T+1)/2 matmul flops per fwd+bwd (QK^T and PV forward; recomputed QK^T,
dP, dV, dK, dQ backward), over the device time of the step.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

--workload times another of the workload shapes the same way (the long-context
stress workload in split precision with fp32 o, the mode its parity needs).

With N > 1 (launched by torchrun, one process per GPU) every rank runs its
own replica of the workload (the attention has no exchange step) and the
value is the total over ranks divided by the slowest rank's time.
--impl reference times the fp64 CPU oracle on the host cores instead.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from causal_gqa_attention_flashattention_gb300 import inputs  # noqa: E402

METRIC = "causal GQA attn fwd+bwd TFLOP/s on 1 GB300 (% of bf16 tensor peak)"
UNIT = "TFLOP/s"
WORKLOAD = "gpu_116m_model"
NUM_SETS = 4  # rotating input/output sets so consecutive steps do not hit a warm L2


def algo_flops(B, T, Hq, D):
    pairs = T * (T + 1) / 2.0
    return dict(fwd=4.0 * B * Hq * D * pairs, bwd=10.0 * B * Hq * D * pairs, total=14.0 * B * Hq * D * pairs)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(bf16_tflops=float(p["bf16_tflops"]), bf16_tflops_sustained=float(p["bf16_tflops_sustained"]),
                    hbm_gbs=float(p["hbm_gbs"]), source="measured")
    except Exception:
        return dict(bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, hbm_gbs=6800.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        finally:
            os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        loaded = [x for x in sm if mx and x >= 0.5 * max(mx)] or sm
        return dict(sm_mhz=statistics.median(loaded) if loaded else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=reasons, samples=len(rows))


def slowest_over_ranks(ms, world, device):
    """The slowest rank's time: every rank passes its own, all get the maximum
    (the step's wall time when ranks run side by side)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_rank_step, ms_per_step):
    """Throughput of the whole job: every rank runs its own replica of the
    step, so the work is world x the per-rank work, over the slowest rank's time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def traffic_record(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel source as it stands now (hash match); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec:
        return None
    src = os.path.join(ROOT, "causal_gqa_attention_flashattention_gb300", "csrc", rec["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if h != rec.get("source_sha256_16"):
        return None
    return rec


def cpu_oracle_sample(budget_s, shape, x, workload=WORKLOAD):
    """Times the fp64 oracle (fwd + bwd) on whole (batch, kv-head) groups of the
    workload until about budget_s seconds of CPU work have been done."""
    import oracle
    B, T, Hq, Hkv, D = shape
    order = [(b, g) for b in range(B) for g in range(Hkv)]
    t0 = time.perf_counter()
    oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], inputs.ROPE_BASE, groups=order[:1])
    one = time.perf_counter() - t0
    n = max(1, min(len(order), int(budget_s / max(one, 1e-3))))
    groups = order[:n]
    t0 = time.perf_counter()
    oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], inputs.ROPE_BASE, groups=groups)
    dt = time.perf_counter() - t0
    G = Hq // Hkv
    fl = algo_flops(1, T, G, D)["total"] * n
    return dict(value=fl / dt / 1e12, unit=UNIT, cores=oracle.num_threads(), kind="oracle",
                sample="%d of %d (batch, kv-head) groups of %s (fp64 fwd+bwd, %.1f s)" % (n, len(order), workload, dt),
                seconds=dt)


def run_reference(args, world, rank):
    """The fp64 CPU oracle on this host's cores, same metric and workload."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    shape = tuple(inputs.WORKLOADS[WORKLOAD][:5])
    B, T, Hq, Hkv, D = shape
    x = inputs.make_workload_inputs(WORKLOAD)
    G = Hq // Hkv
    order = [(b, g) for b in range(B) for g in range(Hkv)]
    # size each step so the whole run stays within about two minutes
    t0 = time.perf_counter()
    oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], inputs.ROPE_BASE, groups=order[:1])
    one = time.perf_counter() - t0
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    n = max(1, min(len(order), int(per_step_budget / max(one, 1e-3))))
    for i in range(args.warmup):
        oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], inputs.ROPE_BASE, groups=order[:n])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], inputs.ROPE_BASE, groups=order[:n])
    dt = time.perf_counter() - t0
    fl = algo_flops(1, T, G, D)["total"] * n
    value = fl * args.steps / dt / 1e12
    sample = "%d of %d (batch, kv-head) groups of %s per step (fp64 fwd+bwd)" % (n, len(order), WORKLOAD)
    line = dict(impl="reference", metric=METRIC, value=value, unit=UNIT, n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, ms_per_step=dt * 1e3 / args.steps, higher_is_better=True, scaling="weak",
                vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload=WORKLOAD, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, rope_base=inputs.ROPE_BASE),
                cpu_baseline=dict(value=value, unit=UNIT, cores=oracle.num_threads(), kind="oracle", sample=sample),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    from causal_gqa_attention_flashattention_gb300 import binding

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    workload = args.workload
    shape = tuple(inputs.WORKLOADS[workload][:5])
    B, T, Hq, Hkv, D = shape
    fl = algo_flops(B, T, Hq, D)
    x = inputs.make_workload_inputs(workload)
    base = inputs.ROPE_BASE
    grad_dtype = torch.float32
    # the stress workload's logits reach ~1.7e4: it runs in split precision with an fp32 o
    precise = workload == "long_context_stress"
    o_dtype = torch.float32 if precise else torch.bfloat16

    def host_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16)

    hq, hk, hv, hdo = (host_bf16(x[n + "_bits"]) for n in ("q", "k", "v", "dout"))
    sets = []
    for _ in range(NUM_SETS):
        q, k, v, do = (t.to(dev) for t in (hq, hk, hv, hdo))
        sets.append(dict(q=q, k=k, v=v, do=do, o=torch.empty(q.shape, dtype=o_dtype, device=dev),
                         lse=torch.empty(((2 if precise else 1) * B, Hq, T), dtype=torch.float32, device=dev),
                         dq=torch.empty(q.shape, dtype=grad_dtype, device=dev),
                         dk=torch.empty(k.shape, dtype=grad_dtype, device=dev),
                         dv=torch.empty(k.shape, dtype=grad_dtype, device=dev),
                         ws=binding.alloc_workspace(B, T, Hq, Hkv, D, precise=precise, device=dev)))
    set_bytes = sum(t.numel() * t.element_size() for t in sets[0].values())
    torch.cuda.synchronize(dev)
    # a side stream: CUDA graphs are captured on a non-default stream
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)

    def step(i):
        s = sets[i % NUM_SETS]
        # the forward's workspace (rotated q, k) is the first part of the backward's
        binding.attn_fwd(s["q"], s["k"], s["v"], base, o=s["o"], lse=s["lse"], workspace=s["ws"], o_dtype=o_dtype,
                         precise=precise, stream=stream)
        binding.attn_bwd(s["q"], s["k"], s["v"], s["o"], s["lse"], s["do"], base, grad_dtype=grad_dtype,
                         dq=s["dq"], dk=s["dk"], dv=s["dv"], workspace=s["ws"], qk_rotated=not precise,
                         precise=precise, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for i in range(args.warmup):
        step(i)
    binding.check_status(stream)
    torch.cuda.synchronize(dev)

    # The timed region replays CUDA graphs of whole steps, so the GPU never waits
    # for the host between kernels.  One graph holds NUM_SETS steps (one per
    # buffer set); a one-step graph per set covers a remainder of K.  A separate
    # graph of the same steps carries the library's per-kernel timing events
    # (event nodes between the kernels); it runs after the timed region.
    n_kinds = len(binding.KERNEL_KINDS)
    binding.profile_start(n_kinds * NUM_SETS + 4)
    g_prof = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_prof, stream=stream):
        for i in range(NUM_SETS):
            step(i)
    prof_cap = binding.profile_stop_deferred()
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        for i in range(NUM_SETS):
            step(i)
    g_one = []
    for i in range(NUM_SETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(i)
        g_one.append(g)
    for _ in range(2):
        g_all.replay()
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)

    # Clocks: the sampler runs while the same graph replays for --clock-seconds seconds
    # before the timed region and again after it, so that the samples (every 50 ms)
    # see the load the timed steps run under; the timed region itself is exactly
    # the K steps between the two events.
    g_all.replay()
    torch.cuda.synchronize(dev)
    t_rep = time.perf_counter()
    g_all.replay()
    torch.cuda.synchronize(dev)
    load_reps = int(args.clock_seconds / max(time.perf_counter() - t_rep, 1e-5))
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(load_reps):
        g_all.replay()
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    full, rest = divmod(args.steps, NUM_SETS)
    e0.record(stream)
    for _ in range(full):
        g_all.replay()
    for i in range(rest):
        g_one[i].replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    for _ in range(load_reps):
        g_all.replay()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if clk is not None:
        clk["how"] = "sampled every 50 ms over %.1f s of the same graph replaying around the timed region" % (
            2 * args.clock_seconds)
    binding.check_status(stream)
    # per-kernel device time: the profiled graph (NUM_SETS steps), warm, then read once
    for _ in range(3):
        g_prof.replay()
    torch.cuda.synchronize(dev)
    prof = binding.profile_read(prof_cap)
    ms_total = e0.elapsed_time(e1)
    barrier()
    ms_step = slowest_over_ranks(ms_total, world, dev) / args.steps
    value = whole_job_tflops(world, fl["total"], ms_step)

    # end to end through the public API: pinned host inputs in, results out, every step
    e2e_steps = max(3, min(args.steps, 200))
    pin = [t.pin_memory() for t in (hq, hk, hv, hdo)]
    s0 = sets[0]
    outs = dict(o=torch.empty(s0["o"].shape, dtype=s0["o"].dtype).pin_memory(),
                lse=torch.empty(s0["lse"].shape, dtype=torch.float32).pin_memory(),
                dq=torch.empty(s0["dq"].shape, dtype=grad_dtype).pin_memory(),
                dk=torch.empty(s0["dk"].shape, dtype=grad_dtype).pin_memory(),
                dv=torch.empty(s0["dv"].shape, dtype=grad_dtype).pin_memory())

    # the public pipelined call: inputs go up on one stream, the kernels run on a
    # second, results come down on a third, three device buffer sets rotate; the
    # timed region opens before the first copy up and closes after the last copy down
    pipe = binding.HostStepPipeline(B, T, Hq, Hkv, D, base, depth=3, grad_dtype=grad_dtype, device=dev,
                                    precise=precise)
    for i in range(3):
        pipe.submit(*pin, outs)
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    barrier()
    e0.record(pipe.up)
    for i in range(e2e_steps):
        pipe.submit(*pin, outs)
    e1.record(pipe.down)
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    e2e_ms = slowest_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    h2d = sum(t.numel() * t.element_size() for t in pin)
    d2h = sum(t.numel() * t.element_size() for t in outs.values())

    if rank != 0:
        return 0
    peaks = load_peaks()
    # dominant kernel of the step
    prof = {k: v for k, v in prof.items() if v[1] > 0}
    launches_per_step = sum(v[1] for v in prof.values()) // NUM_SETS
    dom = max(prof, key=lambda k: prof[k][0])
    ms_dom, n_dom = prof[dom]
    per_launch_ms = ms_dom / max(1, n_dom)
    pairs = T * (T + 1) / 2.0
    if dom in ("fwd", "bwd_dkdv"):
        work = (4.0 if dom == "fwd" else 10.0) * B * Hq * D * pairs
        achieved = work / (per_launch_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = dict(bound="tensor", achieved=achieved, peak=peak, unit="TFLOP/s", frac=achieved / peak)
    else:
        work = None
        roof = dict(bound="hbm", achieved=None, peak=peaks["hbm_gbs"], unit="GB/s", frac=None)
    kernel_names = dict(fwd="k_attn_fwd" if precise else "k_attn_fwd4", fwd_rope="k_rope_qk", bwd_prep="k_bwd_prep",
                        bwd_dkdv="k_bwd_dkdv" if precise else "k_bwd_dkdv3", bwd_dq="k_bwd_dq")
    tr = traffic_record(kernel_names.get(dom, dom))
    roof.update(kernel=dom, traffic=(tr["dram_bytes_per_launch"] if tr else None),
                peak_source="%s bf16 burst" % peaks["source"] if roof["bound"] == "tensor" else
                "%s hbm" % peaks["source"], per_launch_us=per_launch_ms * 1e3,
                kernels={k: dict(us_per_launch=v[0] / v[1] * 1e3, launches=v[1])
                         for k, v in prof.items() if v[1]})
    # the streaming kernels against the measured copy rate: algorithmic bytes per
    # launch (each tensor read or written once) over the launch's event time
    Tp = -(-T // 128) * 128
    oe = 4 if precise else 2
    stream_bytes = dict(
        fwd_rope=(2 * B * T * (Hq + Hkv) * D * 2) * (2 if precise else 1),  # q, k in; rotated fp16 (hi, lo) out
        bwd_prep=B * T * Hq * D * (oe + 2) + B * Hq * T * 4 * (2 if precise else 1)   # o, dO, lse in
        + B * Hq * Tp * 4 * (3 if precise else 2) + B * Hq * Tp * D * 4,             # Delta, lse2 out; dQacc zeroed
        bwd_dq=B * Hq * Tp * D * 4 + B * T * Hq * D * 4)                             # dQacc in, fp32 dq out
    streaming = {}
    for k, nbytes in stream_bytes.items():
        if k in prof and prof[k][1]:
            us = prof[k][0] / prof[k][1] * 1e3
            gbs = nbytes / (us * 1e-6) / 1e9
            streaming[k] = dict(kernel=kernel_names[k], algorithmic_bytes=nbytes, us_per_launch=us, achieved_gbs=gbs,
                                peak_gbs=peaks["hbm_gbs"], frac=gbs / peaks["hbm_gbs"])
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample(args.cpu_seconds, shape, x, workload)
        cpu.pop("seconds", None)
    line = dict(metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps, warmup=args.warmup,
                ms_per_step=ms_step, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
                data="synthetic",
                config=dict(workload=workload, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, rope_base=base,
                            gflop_per_step=fl["total"] / 1e9,
                            precision=("split precision (NE_ATTN_PRECISE_QK): fp16 hi + lo rotated q/k, bf16 hi + lo "
                                       "P, fp32 accumulate, fp32 o and dq/dk/dv") if precise else
                            "fp16 rotated q/k, bf16 P/V/dO, fp32 accumulate, bf16 o, fp32 dq/dk/dv",
                            l2="%d rotating buffer sets of %.0f MB (%.0f MB > L2)" % (
                                NUM_SETS, set_bytes / 1e6, NUM_SETS * set_bytes / 1e6),
                            parallelism="replicas" if world > 1 else "single GPU",
                            launch="CUDA graph replay of %d-step graphs (%d library kernels per step)" % (
                                NUM_SETS, launches_per_step)),
                pct_of_bf16_peak=100.0 * value / world / peaks["bf16_tflops"],
                roofline=roof, prepass=streaming.get("bwd_prep"), streaming=streaming, cpu_baseline=cpu,
                e2e=dict(value=whole_job_tflops(world, fl["total"], e2e_ms), unit=UNIT, h2d_bytes_per_step=h2d,
                         d2h_bytes_per_step=d2h, ms_per_step=e2e_ms,
                         how="binding.HostStepPipeline: pinned host inputs up, forward + backward, every output "
                             "(o, lse, dq, dk, dv) down, each step; copies overlap other steps' kernels"),
                gpu_launches=launches_per_step * args.steps,
                clocks=clk)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# Decode with a KV cache (one new token per sequence): B, Tkv, Tq, Hq, Hkv, D.
DECODE_WORKLOADS = {
    "decode_116m_ctx512": (16, 512, 1, 12, 4, 64),    # the 116M model at its full context
    "decode_116m_ctx8192": (16, 8192, 1, 12, 4, 64),  # the same heads over an 8192-position cache
}


def run_decode(args):
    """One JSON line per decode workload: KV-cache bytes read per second.

    The caches (rotated fp16 keys, bf16 values) are filled through the public
    append call from seeded N(0,1) data; enough cache sets rotate through the
    timed graph that their total exceeds L2 twice over.  The timed region
    replays a CUDA graph of decode calls (query packing, then the split sweep with its merge).
    """
    import torch
    from causal_gqa_attention_flashattention_gb300 import binding
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    for name, (B, Tkv, Tq, Hq, Hkv, D) in DECODE_WORKLOADS.items():
        if args.decode_workload and name != args.decode_workload:
            continue
        cache_bytes = B * Tkv * Hkv * D * (2 + 2)
        nsets = max(2, min(64, -(-2 * 129 * 2 ** 20 // cache_bytes)))
        g = torch.Generator(device=dev).manual_seed(5)
        sets = []
        for _ in range(nsets):
            kc, vc = binding.kv_cache(B, Tkv, Hkv, D, dev)
            k = torch.randn((B, Tkv, Hkv, D), device=dev, generator=g).bfloat16()
            v = torch.randn((B, Tkv, Hkv, D), device=dev, generator=g).bfloat16()
            binding.kv_append(k, v, kc, vc, 0)
            q = torch.randn((B, Tq, Hq, D), device=dev, generator=g).bfloat16()
            sets.append(dict(q=q, kc=kc, vc=vc, o=torch.empty_like(q),
                             lse=torch.empty((B, Hq, Tq), dtype=torch.float32, device=dev)))
        ws = torch.empty(binding.decode_workspace_size(B, Tq, Tkv, Hq, Hkv, D), dtype=torch.uint8, device=dev)

        def call(s):
            binding.attn_decode(s["q"], s["kc"], s["vc"], Tkv, o=s["o"], lse=s["lse"], workspace=ws, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                for s in sets:
                    call(s)
        binding.check_status(stream)
        binding.profile_start(3 * nsets + 4)
        g_prof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_prof, stream=stream):
            for s in sets:
                call(s)
        prof_cap = binding.profile_stop_deferred()
        g_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all, stream=stream):
            for s in sets:
                call(s)
        reps = max(1, args.steps // nsets)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # graphs replay on the current stream, events time that stream
            g_all.replay()
            torch.cuda.synchronize(dev)
            clocks = ClockSampler(0)
            clocks.start()
            e0.record(stream)
            for _ in range(reps):
                g_all.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            clk = clocks.stop()
            binding.check_status(stream)
            for _ in range(3):
                g_prof.replay()
        torch.cuda.synchronize(dev)
        prof = binding.profile_read(prof_cap)
        ms_call = e0.elapsed_time(e1) / (reps * nsets)
        ms_sweep = prof["decode"][0] / max(1, prof["decode"][1])
        dec_tr = traffic_record("k_decode")
        achieved = cache_bytes / (ms_sweep * 1e-3) / 1e9
        line = dict(metric="decode: KV-cache bytes read per second (one decode step, all sequences)",
                    value=cache_bytes / (ms_call * 1e-3) / 1e9, unit="GB/s", n_gpus=1, steps=reps * nsets,
                    warmup=args.warmup, ms_per_step=ms_call, higher_is_better=True, scaling="weak",
                    vs_baseline=None, dtype="fp16 keys, bf16 values, fp32 accumulate", data="synthetic",
                    config=dict(workload=name, B=B, Tkv=Tkv, Tq=Tq, Hq=Hq, Hkv=Hkv, D=D, cache_sets=nsets,
                                l2="%d rotating cache sets of %.1f MB" % (nsets, cache_bytes / 1e6),
                                launch="CUDA graph replay (2 library kernels per decode call)"),
                    tokens_per_s=B * Tq / (ms_call * 1e-3),
                    roofline=dict(bound="hbm", achieved=achieved, peak=peaks["hbm_gbs"], unit="GB/s",
                                  frac=achieved / peaks["hbm_gbs"], kernel="decode",
                                  # the committed capture is of the 8192-position workload
                                  traffic=(dec_tr["dram_bytes_per_launch"]
                                           if dec_tr and name == "decode_116m_ctx8192" else None),
                                  peak_source="%s hbm" % peaks["source"], per_launch_us=ms_sweep * 1e3,
                                  kernels={k: dict(us_per_launch=v[0] / v[1] * 1e3, launches=v[1])
                                           for k, v in prof.items() if v[1]}),
                    clocks=clk)
        print(json.dumps(line), flush=True)
    return 0


def run_prologue(args):
    """One JSON line for the step in front of attention: RMSNorm + the fused
    Q/K/V projection at the 116M model's width (ne_attn_qkv_rmsnorm writing
    v and the rotated q, k into the attention workspace, as a block runs it).

    Metric: projection TFLOP/s (2 * B*T * C * N per call).  Seeded inputs
    (x ~ N(0,1), norm weight ~ 1 + 0.1 N(0,1), projection ~ N(0,1)/sqrt(C))
    rotate through enough sets that their total exceeds L2; the timed region
    replays a CUDA graph of calls.
    """
    import numpy as np
    import torch
    import oracle
    from causal_gqa_attention_flashattention_gb300 import binding
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    name = "gpu_116m_model"
    B, T, C, Hq, Hkv, D = inputs.PROLOGUE_WORKLOADS[name]
    M, N = B * T, (Hq + 2 * Hkv) * D
    flops = 2.0 * M * C * N
    x = inputs.make_prologue_inputs(B, T, C, Hq, Hkv, D, seed=21)

    def dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    ws_bytes = binding.qkv_workspace_size(B, T, C, Hq, Hkv, D, rotated=True)
    set_bytes = 2 * (M * C + C + N * C) + ws_bytes + 2 * M * Hkv * D + 4 * M
    nsets = max(2, min(16, -(-2 * 129 * 2 ** 20 // set_bytes)))
    sets = []
    for i in range(nsets):
        sets.append(dict(x=dev_bf16(x["x_bits"]), w=dev_bf16(x["norm_w_bits"]), W=dev_bf16(x["w_qkv_bits"]),
                         v=torch.empty((B, T, Hkv, D), dtype=torch.bfloat16, device=dev),
                         rstd=torch.empty((B, T), dtype=torch.float32, device=dev),
                         ws=torch.empty(ws_bytes, dtype=torch.uint8, device=dev)))

    def call(st):
        binding.qkv_rmsnorm(st["x"], st["w"], st["W"], Hq, Hkv, D, rotated=True, write_qk=False, v=st["v"],
                            rstd=st["rstd"], workspace=st["ws"], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for st in sets:
                call(st)
    binding.check_status(stream)
    binding.profile_start(2 * nsets + 4)
    g_prof = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_prof, stream=stream):
        for st in sets:
            call(st)
    prof_cap = binding.profile_stop_deferred()
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        for st in sets:
            call(st)
    reps = max(1, args.steps // nsets)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g_all.replay()
        torch.cuda.synchronize(dev)
        clocks = ClockSampler(0)
        clocks.start()
        e0.record(stream)
        for _ in range(reps):
            g_all.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        binding.check_status(stream)
        for _ in range(3):
            g_prof.replay()
    torch.cuda.synchronize(dev)
    prof = binding.profile_read(prof_cap)
    ms_call = e0.elapsed_time(e1) / (reps * nsets)
    ms_gemm = prof["qkv"][0] / max(1, prof["qkv"][1])
    achieved = flops / (ms_gemm * 1e-3) / 1e12
    tr = traffic_record("k_qkv_gemm")
    cpu = None
    if not args.no_cpu_baseline:
        # the whole workload, repeated until about two seconds of CPU work are done
        xs = x["x"].reshape(M, 1, C)
        reps, t0 = 0, time.perf_counter()
        while reps == 0 or time.perf_counter() - t0 < 2.0:
            oracle.qkv_rmsnorm(xs, x["norm_w"], x["w_qkv"], Hq, Hkv, D)
            reps += 1
        dt = time.perf_counter() - t0
        cpu = dict(value=2.0 * reps * M * C * N / dt / 1e12, unit="TFLOP/s", cores=os.cpu_count(), kind="oracle",
                   sample="%d x all %d rows (fp64 numpy RMSNorm + projection, %.1f s)" % (reps, M, dt))
    line = dict(metric="RMSNorm + fused Q/K/V projection with the rotary epilogue: projection TFLOP/s",
                value=flops / (ms_call * 1e-3) / 1e12, unit="TFLOP/s", n_gpus=1, steps=reps * nsets,
                warmup=args.warmup, ms_per_step=ms_call, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="bf16 operands, fp32 accumulate", data="synthetic",
                config=dict(workload=name, B=B, T=T, C=C, Hq=Hq, Hkv=Hkv, D=D, N=N, input_sets=nsets,
                            l2="%d rotating input/output sets of %.1f MB" % (nsets, set_bytes / 1e6),
                            outputs="v (bf16) and the rotated q, k (fp16) in the attention workspace",
                            launch="CUDA graph replay (2 library kernels per call)"),
                tokens_per_s=M / (ms_call * 1e-3),
                roofline=dict(bound="tensor", achieved=achieved, peak=peaks["bf16_tflops"], unit="TFLOP/s",
                              frac=achieved / peaks["bf16_tflops"], kernel="qkv",
                              traffic=(tr["dram_bytes_per_launch"] if tr else None),
                              peak_source="%s bf16 (burst)" % peaks["source"], per_launch_us=ms_gemm * 1e3,
                              kernels={k: dict(us_per_launch=v[0] / v[1] * 1e3, launches=v[1])
                                       for k, v in prof.items() if v[1]}),
                cpu_baseline=cpu, gpu_launches=2 * reps * nsets, clocks=clk)
    print(json.dumps(line), flush=True)
    return 0


def run_fp8(args):
    """One JSON line for the FP8 forward (NE_ATTN_FP8, an inference variant) on
    the 116M model's attention shape: forward TFLOP/s with e4m3 rotated q, k.
    The default (fp16 q, k) forward is timed the same way beside it.  Input
    sets rotate so that their total exceeds L2; graph replay as in the main line.
    """
    import torch
    from causal_gqa_attention_flashattention_gb300 import binding
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    B, T, Hq, Hkv, D = inputs.WORKLOADS[WORKLOAD][:5]
    flops = algo_flops(B, T, Hq, D)["fwd"]
    set_bytes = 2 * B * T * (2 * Hq + 2 * Hkv) * D + B * T * (Hq + Hkv) * D
    nsets = max(2, min(16, -(-2 * 129 * 2 ** 20 // set_bytes)))
    g = torch.Generator(device=dev).manual_seed(9)
    sets = []
    for _ in range(nsets):
        q = torch.randn((B, T, Hq, D), device=dev, generator=g).bfloat16()
        k = torch.randn((B, T, Hkv, D), device=dev, generator=g).bfloat16()
        v = torch.randn((B, T, Hkv, D), device=dev, generator=g).bfloat16()
        sets.append(dict(q=q, k=k, v=v, o=torch.empty_like(q),
                         lse=torch.empty((B, Hq, T), dtype=torch.float32, device=dev),
                         ws8=torch.empty(binding.fwd_workspace_size(B, T, Hq, Hkv, D, fp8=True), dtype=torch.uint8,
                                         device=dev),
                         ws=torch.empty(binding.fwd_workspace_size(B, T, Hq, Hkv, D), dtype=torch.uint8, device=dev)))

    def timed(fp8):
        def call(st):
            binding.attn_fwd(st["q"], st["k"], st["v"], o=st["o"], lse=st["lse"], fp8=fp8,
                             workspace=st["ws8"] if fp8 else st["ws"], stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                for st in sets:
                    call(st)
        binding.check_status(stream)
        binding.profile_start(4 * nsets + 4)
        g_prof = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_prof, stream=stream):
            for st in sets:
                call(st)
        cap = binding.profile_stop_deferred()
        g_all = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_all, stream=stream):
            for st in sets:
                call(st)
        reps = max(1, args.steps // nsets)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g_all.replay()
            torch.cuda.synchronize(dev)
            clocks = ClockSampler(0)
            clocks.start()
            e0.record(stream)
            for _ in range(reps):
                g_all.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            clk = clocks.stop()
            binding.check_status(stream)
            for _ in range(3):
                g_prof.replay()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / (reps * nsets), binding.profile_read(cap), reps * nsets, clk

    ms8, prof8, n8, clk = timed(True)
    ms16, prof16, _, _ = timed(False)
    ms_attn = prof8["fwd"][0] / max(1, prof8["fwd"][1])
    achieved = flops / (ms_attn * 1e-3) / 1e12
    line = dict(metric="FP8 forward: causal GQA attention TFLOP/s, e4m3 rotated q and k (inference variant)",
                value=flops / (ms8 * 1e-3) / 1e12, unit="TFLOP/s", n_gpus=1, steps=n8, warmup=args.warmup,
                ms_per_step=ms8, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="e4m3 q/k, bf16 v and P, fp32 accumulate", data="synthetic",
                config=dict(workload=WORKLOAD, B=B, T=T, Hq=Hq, Hkv=Hkv, D=D, input_sets=nsets,
                            l2="%d rotating input sets of %.1f MB" % (nsets, set_bytes / 1e6),
                            launch="CUDA graph replay (max pass, quantising pass, attention kernel)"),
                default_forward=dict(ms_per_step=ms16, value=flops / (ms16 * 1e-3) / 1e12, unit="TFLOP/s",
                                     kernels={k: dict(us_per_launch=v[0] / v[1] * 1e3, launches=v[1])
                                              for k, v in prof16.items() if v[1]}),
                roofline=dict(bound="tensor", achieved=achieved, peak=peaks["bf16_tflops"], unit="TFLOP/s",
                              frac=achieved / peaks["bf16_tflops"], kernel="fwd",
                              traffic=(lambda tr: tr["dram_bytes_per_launch"] if tr else None)(
                                  traffic_record("k_attn_fwd4_fp8")),
                              peak_source="%s bf16 (burst); S runs at the 8-bit rate, P V at bf16"
                              % peaks["source"], per_launch_us=ms_attn * 1e3,
                              kernels={k: dict(us_per_launch=v[0] / v[1] * 1e3, launches=v[1])
                                       for k, v in prof8.items() if v[1]}),
                gpu_launches=3 * n8, clocks=clk)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", action="store_true",
                    help="measure decode with a KV cache (one JSON line per decode workload) instead")
    ap.add_argument("--decode-workload", default=None, choices=sorted(DECODE_WORKLOADS),
                    help="with --decode: only this workload")
    ap.add_argument("--prologue", action="store_true",
                    help="measure RMSNorm + the fused Q/K/V projection (one JSON line) instead")
    ap.add_argument("--fp8", action="store_true",
                    help="measure the FP8 forward (one JSON line) instead")
    ap.add_argument("--clock-seconds", type=float, default=0.4,
                    help="seconds of graph replays before and after the timed region while clocks are sampled")
    ap.add_argument("--workload", default=WORKLOAD, choices=list(inputs.WORKLOAD_ORDER),
                    help="the training step's workload shape (default: the 116M model's)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.decode:
        return run_decode(args)
    if args.prologue:
        return run_prologue(args)
    if args.fp8:
        return run_fp8(args)
    world, rank, local = dist_init()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())

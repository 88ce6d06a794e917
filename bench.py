#!/usr/bin/env python
"""Benchmark of the Gemma-4 26B-A4B sparse MoE feed-forward block on GB300.

One step = one forward of the whole block (router, top-k, permutation, gate_up and down grouped
GEMMs, combine with the post-norms) over one batch of synthetic tokens, through the C ABI.

  python bench.py [--gpus N --steps K --warmup W] [--workload decode64|prefill4096|moe8|layer --T T]
  python bench.py --impl reference ...      (the oracle, timed on the host cores)

Default workload: the full dual-path layer at decode batch T=64, uniform routing, which gives the
line's `value`. The metric is quoted at T=64 and at T=4096, so the default run also measures, in
the same process and under the same rules, the full layer at prefill T=4096 with Zipf(1.1)-skewed
routing, and adds it to the same line as the `prefill4096` object (tokens/s, step time, layer and
dominant-kernel rooflines, kernel breakdown, end-to-end figure, clocks). Multi-GPU runs (torchrun,
one rank per GPU) are weak scaling: each rank runs its own replica of the layer on its own tokens;
there is no data-path collective. Prints one JSON line (rank 0).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-FFN tokens/s at T=64 & T=4096; % of HBM or bf16 TC roofline"
UNIT = "tokens/s"
H, E, K, I, D = 2816, 128, 8, 704, 2112

# Algorithmic bytes per unit: one expert's gate_up and down slices, the shared MLP's matrices and
# the router matrix, each read once per forward.
GATE_UP_BYTES_PER_EXPERT = 2 * I * H * 2        # 7,929,856
DOWN_BYTES_PER_EXPERT = H * I * 2               # 3,964,928
DENSE_GATE_UP_BYTES = 2 * D * H * 2             # 23,789,568
DENSE_DOWN_BYTES = H * D * 2                    # 11,894,784
ROUTER_BYTES = E * H * 4                        # 1,441,792
FLOPS_PER_TOKEN_EXPERTS = K * 2 * (2 * I * H + H * I)   # 95,158,272
FLOPS_PER_TOKEN_DENSE = 2 * (2 * D * H + H * D)         # 35,684,352

# Nominal GB300 peaks, for context beside the measured ones: the ~8 TB/s HBM3e figure decode is
# quoted against, and the dense bf16 tensor rate.
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0


def layer_roofline(layer_bytes, layer_flops, step_s, hbm_gbs, bf16_tflops, experts_hit, layers):
    """The whole layer's roofline time max(bytes / HBM, FLOPs / bf16 peak) and the fraction of it a
    measured per-layer step reaches: `frac` against the measured peaks passed in, `frac_nominal`
    against the nominal ones."""
    t_hbm, t_tc = layer_bytes / (hbm_gbs * 1e9), layer_flops / (bf16_tflops * 1e12)
    t_roof = max(t_hbm, t_tc)
    t_nom = max(layer_bytes / (NOMINAL_HBM_GBS * 1e9), layer_flops / (NOMINAL_BF16_TFLOPS * 1e12))
    return {"bytes": layer_bytes, "flops": layer_flops, "roofline_us": t_roof * 1e6, "step_us": step_s * 1e6,
            "frac": t_roof / step_s, "bound": "hbm" if t_hbm >= t_tc else "tensor",
            "roofline_nominal_us": t_nom * 1e6, "frac_nominal": t_nom / step_s,
            "nominal_peaks": {"hbm_gbs": NOMINAL_HBM_GBS, "bf16_tflops": NOMINAL_BF16_TFLOPS},
            "experts_hit": experts_hit, "layers_per_step": layers}


WORKLOADS = {
    "decode64": dict(full=True, T=64, skew=False,
                     desc="Gemma-4 26B-A4B full dual-path FFN layer, decode batch T=64, uniform routing"),
    "prefill4096": dict(full=True, T=4096, skew=True,
                        desc="Gemma-4 26B-A4B full dual-path FFN layer, prefill T=4096, Zipf(1.1)-scaled router rows"),
    "decode64_int8": dict(full=True, T=64, skew=False, int8=True,
                          desc="Gemma-4 26B-A4B full dual-path FFN layer, decode batch T=64, uniform routing, "
                               "int8 per-channel experts"),
    "decode64_fp4": dict(full=True, T=64, skew=False, fp4=True,
                         desc="Gemma-4 26B-A4B full dual-path FFN layer, decode batch T=64, uniform routing, "
                              "MXFP4 experts"),
    "moe8": dict(full=False, T=8, skew=False, desc="Gemma-4 26B-A4B MoE block only (router + experts), T=8"),
    "layer": dict(full=True, T=None, skew=False, desc="Gemma-4 26B-A4B full dual-path FFN layer, uniform routing"),
    "stack30": dict(full=True, T=256, skew=False, layers=30,
                    desc="Gemma-4 26B-A4B 30-layer stack of full dual-path FFN layers (attention omitted), "
                         "decode T=256, fresh weights per layer, activations carried layer to layer"),
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="decode64")
    p.add_argument("--T", type=int, default=None, help="tokens per step for --workload layer")
    p.add_argument("--seed", type=int, default=1234)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true",
                   help="default workload only: skip the T=4096 prefill leg of the line")
    p.add_argument("--no-configs", action="store_true",
                   help="default workload only: skip the other configurations (experts-only T=8, the T sweep, "
                        "the 30-layer stack) measured after the two legs of the line")
    p.add_argument("--ep", action="store_true",
                   help="expert parallel: each rank runs its contiguous share of the 128 experts on the same "
                        "tokens, then the partial expert sums are all-reduced (NCCL) before the post norms")
    return p.parse_args(argv)


def workload_of(args):
    w = dict(WORKLOADS[args.workload])
    if w["T"] is None:
        if not args.T:
            raise SystemExit("--workload layer needs --T")
        w["T"] = args.T
        w["desc"] = w["desc"] + ", T=%d" % args.T
    return w


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def job_throughput(tokens_per_rank: int, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * steps * world / max_seconds


# ------------------------------------------------------------------ clocks during the timed region

class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    CLOCK_PERIOD_MS = 50
    SUSTAIN_S = 0.6

    def __init__(self, uuid=None, period_ms=CLOCK_PERIOD_MS):
        self.uuid = uuid
        self.period_ms = period_ms
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)
        return self

    def rows_between(self, t0, t1):
        return [r for (t, r) in self.rows
                if t0 <= t <= t1 and len(r) >= 10 and (self.uuid is None or self.uuid in r[1])]

    def summary(self, t0, t1, s0=None, s1=None):
        """Clocks during the timed region [t0, t1]. If no sample fell inside it (a region shorter
        than the sampling period), the samples of the sustained run of the same step [s0, s1] that
        followed it, and `window` says which."""
        timed = self.rows_between(t0, t1)
        if timed:
            use, window = timed, "timed region"
        elif s0 is not None:
            use = self.rows_between(s0, s1)
            window = ("no sample inside the %.1f ms timed region (sampling period %d ms); these are the samples "
                      "of the same step run for %.1f s right after it" % ((t1 - t0) * 1e3, self.period_ms, s1 - s0))
        else:
            use, window = [], "no sample inside the timed region"
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "in_timed_region": False,
                    "window": window}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in use if num(r[2]) is not None]
        mx = [num(r[3]) for r in use if num(r[3]) is not None]
        reasons = set()
        names = {6: "hw_slowdown", 7: "hw_thermal_slowdown", 8: "sw_thermal_slowdown", 9: "sw_power_cap"}
        for r in use:
            for i, n in names.items():
                if r[i].lower().startswith("active"):
                    reasons.add(n)
        pw = [num(r[4]) for r in use if num(r[4]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(use), "in_timed_region": bool(timed), "window": window,
                "power_w_max": max(pw) if pw else None}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get("%s/%s" % (kernel, workload))
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return rec.get("dram_bytes_per_launch") if h.hexdigest() == rec.get("sources_sha256") else None


# ------------------------------------------------------------------ the CPU arms (oracle)

def oracle_tokens_per_s(wl, w_host, x_bits, n_tokens, min_seconds=10.0, max_passes=400):
    """Times the oracle on the host cores over the first n_tokens of one step's batch (host copies
    of the tensors the GPU arm used), repeating the pass until about min_seconds of CPU work."""
    import oracle
    x = x_bits[:n_tokens]
    dims = oracle.gemma_dims(wl["full"])
    passes, total = 0, 0.0
    while passes < 3 or (total < min_seconds and passes < max_passes):
        t0 = time.perf_counter()
        oracle.forward(dims, x, w_host, want=("out",))
        total += time.perf_counter() - t0
        passes += 1
    return n_tokens * passes / total, oracle.max_threads(), total, passes


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from mixture_experts_ffn_router_gb300 import synth
    T = wl["T"]
    n = min(T, 64)
    w = synth.host_arrays(synth.make_weights(seed=args.seed, device="cpu", full_layer=wl["full"], skew=wl["skew"]))
    if wl.get("int8"):
        for name, cols in (("gate_up", H), ("down", I)):
            q, sc = oracle.quantize_int8(w.pop(name).reshape(-1, cols))
            w[name + "_q"], w[name + "_scale"] = q, sc
    if wl.get("fp4"):
        for name, cols in (("gate_up", H), ("down", I)):
            c4, s4 = oracle.quantize_mxfp4(w.pop(name).reshape(-1, cols))
            w[name + "_f4"], w[name + "_f4s"] = c4, s4
    x = synth.bf16_bits(synth.make_x(T, seed=args.seed, device="cpu"))[:n]
    dims = oracle.gemma_dims(wl["full"])
    for _ in range(max(args.warmup, 0)):
        oracle.forward(dims, x, w, want=("out",))
    steps = max(1, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.forward(dims, x, w, want=("out",))
    dt = time.perf_counter() - t0
    value = n * steps / dt
    sample = "first %d of the %d tokens of one step, %d steps" % (n, T, steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 (router f32)", "data": "synthetic",
        "config": config_of(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ the GPU arm

def config_of(wl, world):
    """The `config` object of a JSON line, the same for the GPU arm and the reference arm."""
    return {"workload": wl["desc"], "T": wl["T"], "tokens_per_gpu": wl["T"], "hidden": H, "experts": E, "top_k": K,
            "moe_inter": I, "dense_inter": D if wl["full"] else 0,
            "expert_weights": ("int8, per-row fp32 scale" if wl.get("int8") else
                               "MXFP4 (E2M1, E8M0 scale per 32 weights)" if wl.get("fp4") else "bf16"),
            "layers": wl.get("layers", 1),
            "l2": "inputs larger than L2: every step reads the routed experts' weights (11.9 MB per expert hit, "
                  "1.52 GB for all 128) and the shared MLP's 35.7 MB, against a 126 MB L2",
            "parallelism": "replicas (dp%d, no collective)" % world}


def measure(args, wl, weights, x, dev, world, rank, with_cpu, clocks, label):
    """Times one workload: untimed breakdown pass, exactly args.steps timed steps (CUDA events on the
    launching stream, barrier + synchronize on both sides), the end-to-end leg with host buffers,
    and the clocks seen while that workload ran. Returns the numbers of one JSON line."""
    import numpy as np
    import torch
    from mixture_experts_ffn_router_gb300 import binding as B
    from mixture_experts_ffn_router_gb300 import synth

    T = wl["T"]
    L = wl.get("layers", 1)
    mode = B.MOE_FFN_FULL_LAYER if wl["full"] else B.MOE_FFN_MOE_ONLY
    local = dev.index
    bufs = [torch.empty_like(x), torch.empty_like(x)]
    ctxs = [B.MoeFFN(mode, T, device=local)]
    for _ in range(1, L):
        ctxs.append(B.MoeFFN(mode, T, device=local, workspace=ctxs[0].workspace))
    m = ctxs[0]
    wss = [B.weights_struct(w) for w in weights]
    stream = torch.cuda.current_stream(dev)
    s = stream.cuda_stream
    out = bufs[(L - 1) % 2]

    def step(x_in=None, sync_each=None, x_out=None):
        src = x if x_in is None else x_in
        for l in range(L):
            dst = x_out if (x_out is not None and l == L - 1) else bufs[l % 2]
            rc = B.moe_ffn_forward(ctxs[l].ctx, src.data_ptr(), T, wss[l], dst.data_ptr(), s)
            if rc != B.MOE_FFN_OK:
                raise B.MoeFFNError("moe_ffn_forward", rc)
            if sync_each is not None:
                sync_each(l)
            src = dst

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    rc, word = m.status()
    if rc != B.MOE_FFN_OK:
        raise RuntimeError("%s: device status 0x%x after warm-up" % (label, word))
    hits = []

    def count_hits(l):
        torch.cuda.synchronize()
        c = B.view_tensor(ctxs[l].views().counts, (E,), torch.int32).cpu().numpy()
        hits.append(int((c > 0).sum()))

    step(sync_each=count_hits)
    experts_hit = float(np.mean(hits))

    # Breakdown pass (untimed): events around every kernel slot of each forward, to rank the
    # kernels (a slot a forward of this size leaves empty records its two events back to back).
    nslots = len(B.KERNEL_NAMES)
    n_b = max(1, min(50, args.steps))

    def event_pairs(n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:  # torch creates the CUDA event on first record
            a.record(stream)
            b.record(stream)
        return ev

    # Events go on the last layer's context (every layer runs the same kernels).
    mk = ctxs[-1]
    bd = [event_pairs(nslots) for _ in range(n_b)]
    torch.cuda.synchronize()
    for i in range(n_b):
        for k in range(nslots):
            B.moe_ffn_set_kernel_events(mk.ctx, k, bd[i][k][0].cuda_event, bd[i][k][1].cuda_event)
        step()
    torch.cuda.synchronize()
    for k in range(nslots):
        B.moe_ffn_set_kernel_events(mk.ctx, k, None, None)
    # Slots a forward of this size leaves empty are not reported.
    used = B.moe_ffn_kernel_slots(m.ctx, T)
    nk = len(used)
    kernel_us = {B.slot_name(k, T): float(np.mean([bd[i][k][0].elapsed_time(bd[i][k][1]) for i in range(n_b)]) * 1e3)
                 for k in used}
    gemms = {"gate_up_gemm": B.KERNEL_NAMES.index("gate_up_gemm"), "down_gemm": B.KERNEL_NAMES.index("down_gemm")}
    dom = max(gemms, key=lambda n: kernel_us[n])
    dom_k = gemms[dom]

    # Timed region: exactly K steps; events around the dominant kernel only, on its stream, in one
    # step of every DOM_EVERY (and always the first). An event recorded between two kernels stops
    # the later one from launching early beside the earlier one (programmatic dependent launch),
    # so bracketing the kernel in every step slowed the timed steps by about 2% at decode.
    DOM_EVERY = 8
    timed_dom = [i for i in range(args.steps) if i % DOM_EVERY == 0]
    ev = event_pairs(len(timed_dom))
    torch.cuda.synchronize()
    time.sleep(0.15)  # let the clock sampler see the GPU idle-to-busy edge on its own samples
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        if i % DOM_EVERY == 0:
            ea, eb = ev[i // DOM_EVERY]
            B.moe_ffn_set_kernel_events(mk.ctx, dom_k, ea.cuda_event, eb.cuda_event)
        elif i % DOM_EVERY == 1:
            B.moe_ffn_set_kernel_events(mk.ctx, dom_k, None, None)
        step()
    t_stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world, dev)
    B.moe_ffn_set_kernel_events(mk.ctx, dom_k, None, None)
    rc, word = m.status()
    if rc != B.MOE_FFN_OK:
        raise RuntimeError("%s: device status 0x%x after the timed steps" % (label, word))
    # The sampler's period is CLOCK_PERIOD_MS; a timed region shorter than that holds no sample of
    # its own. The same step then runs, untimed, for SUSTAIN_S right after the timed region, and
    # the clocks of that window are reported instead, marked as such.
    sus0 = sus1 = None
    if clocks is not None and (wall1 - wall0) * 1e3 < 4 * ClockSampler.CLOCK_PERIOD_MS:
        sus0 = time.time()
        while time.time() - sus0 < ClockSampler.SUSTAIN_S:
            for _ in range(8):
                step()
            torch.cuda.synchronize()
        sus1 = time.time()

    ms = t_start.elapsed_time(t_stop)
    ms_max = max_over_ranks(ms, world, dev)
    value = job_throughput(T, args.steps, world, ms_max / 1e3)
    dom_us = float(np.mean([a.elapsed_time(b) for a, b in ev]) * 1e3)

    # ---- roofline of the dominant kernel and of the whole layer
    hbm, tc_burst, tc_sus, peak_src = measured_peaks()
    S = T * K
    full = wl["full"]
    # int8 experts: one byte per weight plus a 4-byte scale per row; MXFP4: half a byte per weight
    # plus a 1-byte scale per 32 weights.
    if wl.get("int8"):
        gu_pe, dn_pe = 2 * I * H + 2 * I * 4, H * I + H * 4
    elif wl.get("fp4"):
        gu_pe, dn_pe = 2 * I * H // 2 + 2 * I * H // 32, H * I // 2 + H * I // 32
    else:
        gu_pe, dn_pe = GATE_UP_BYTES_PER_EXPERT, DOWN_BYTES_PER_EXPERT
    gu_bytes = experts_hit * gu_pe + (DENSE_GATE_UP_BYTES if full else 0) \
        + T * H * 2 * (2 if full else 1) + S * I * 2 + (T * D * 2 if full else 0)
    gu_flops = 2 * S * 2 * I * H + (2 * T * 2 * D * H if full else 0)
    dn_bytes = experts_hit * dn_pe + (DENSE_DOWN_BYTES if full else 0) \
        + S * I * 2 + (T * D * 2 if full else 0) + S * H * 2 + (T * H * 4 if full else 0)
    dn_flops = 2 * S * H * I + (2 * T * H * D if full else 0)
    per_kernel = {"gate_up_gemm": (gu_bytes, gu_flops), "down_gemm": (dn_bytes, dn_flops)}
    kb, kf = per_kernel[dom]
    dur_s = dom_us / 1e6
    if kb / (hbm * 1e9) >= kf / (tc_burst * 1e12):
        roof = {"bound": "hbm", "achieved": kb / dur_s / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": kf / dur_s / 1e12, "peak": tc_burst, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic_record(dom, label if label != "layer" else "layer_T%d" % T)
    roof["kernel"] = dom
    roof["kernel_us"] = dom_us
    roof["algorithmic_bytes"] = kb
    roof["algorithmic_flops"] = kf
    roof["peak_source"] = peak_src
    roof["launch_timing"] = "CUDA events around the kernel in %d of the %d timed steps (one in %d)" % (
        len(ev), args.steps, DOM_EVERY)
    layer_bytes = experts_hit * (gu_pe + dn_pe) + ROUTER_BYTES + T * H * 2 * 2 \
        + ((DENSE_GATE_UP_BYTES + DENSE_DOWN_BYTES) if full else 0)
    layer_flops = T * (FLOPS_PER_TOKEN_EXPERTS + (FLOPS_PER_TOKEN_DENSE if full else 0))
    step_s = ms / args.steps / 1e3 / L  # per layer
    layer = layer_roofline(layer_bytes, layer_flops, step_s, hbm, tc_burst, experts_hit, L)

    # ---- end to end through the public API with host buffers. Every step copies its whole input
    # from pinned host memory and its whole output back. As in a serving loop, the copies run on two
    # copy streams with double-buffered device input and output: step i+1's input and step i-1's
    # output cross while step i computes. The timed region spans the first input copy to the last
    # output copy.
    x_host = x.cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()
    e_steps = max(1, min(args.steps, 500))
    x_dev = [torch.empty_like(x), torch.empty_like(x)]
    o_dev = [torch.empty_like(x), torch.empty_like(x)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    eev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "fwd", "out")}

    def e2e_steps(n):
        for i in range(n):
            j = i % 2
            if i >= 2:
                h2d.wait_event(eev["fwd"][j])      # step i-2 has finished reading x_dev[j]
            with torch.cuda.stream(h2d):
                x_dev[j].copy_(x_host, non_blocking=True)
            eev["in"][j].record(h2d)
            stream.wait_event(eev["in"][j])
            if i >= 2:
                stream.wait_event(eev["out"][j])   # step i-2's output has left o_dev[j]
            step(x_in=x_dev[j], x_out=o_dev[j])
            eev["fwd"][j].record(stream)
            d2h.wait_event(eev["fwd"][j])
            with torch.cuda.stream(d2h):
                out_host.copy_(o_dev[j], non_blocking=True)
            eev["out"][j].record(d2h)
        for j in range(2):
            stream.wait_event(eev["out"][j])

    e2e_steps(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    e0.record(stream)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    e2e_steps(e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e = {"value": job_throughput(T, e_steps, world, e_ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": x.numel() * 2, "d2h_bytes_per_step": out.numel() * 2, "steps": e_steps,
           "copies": "two copy streams, double-buffered device input and output"}
    torch.testing.assert_close(out_host, o_dev[(e_steps - 1) % 2].cpu(), rtol=0, atol=0)

    cpu = None
    if with_cpu:
        n = min(T, 64)
        tps, cores, secs, passes = oracle_tokens_per_s(wl, synth.host_arrays(weights[0]), synth.bf16_bits(x), n)
        cpu = {"value": tps / L, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "first %d tokens of the step's batch through layer 0, %d passes, %.1f s of oracle time%s"
                         % (n, passes, secs, "; the stack rate is that layer rate / %d" % L if L > 1 else "")}

    clk = clocks.summary(wall0, wall1, sus0, sus1) if clocks is not None else None
    for c in ctxs:
        c.close()
    return {"value": value, "ms_per_step": ms_max / args.steps, "roofline": roof, "layer_roofline": layer,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": nk * L * args.steps, "clocks": clk,
            "kernels_us": kernel_us,
            "kernels_us_note": "untimed breakdown pass, %d steps, events around every kernel" % n_b}


def ep_exchange(part, dense, world, dist=None):
    """The exchange step of the expert-parallel layer ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to
    AWS Inferentia2", section "The traceable trick": row-parallel down, then an all-reduce): the
    ranks' fp32 partial expert sums are added in place (all-reduce, sum), and the shared MLP's
    output, which rank 0 computes, is sent to every rank (broadcast). Both happen before
    post_feedforward_layernorm_2, which is not linear."""
    if world > 1:
        if dist is None:
            import torch.distributed as dist
        dist.all_reduce(part, op=dist.ReduceOp.SUM)
        dist.broadcast(dense, src=0)


def ep_rank_step(rank, world, shard, exchange, finish, n_experts=E):
    """One expert-parallel layer step of one rank: its experts (expert_range) and, on rank 0, the
    shared MLP; the exchange; the rest of the block. shard(begin, end, with_dense) -> (part, dense
    buffer); exchange(part, dense); finish(part, dense) -> output."""
    from mixture_experts_ffn_router_gb300.binding import expert_range
    b, e = expert_range(rank, world, n_experts)
    part, dense = shard(b, e, rank == 0)
    exchange(part, dense)
    return finish(part, dense)


def run_ep(args, wl):
    import torch
    from mixture_experts_ffn_router_gb300 import binding as B
    from mixture_experts_ffn_router_gb300 import synth

    rank, world = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T = wl["T"]
    if not wl["full"] or wl.get("layers", 1) != 1 or wl.get("int8") or wl.get("fp4"):
        raise SystemExit("--ep runs the full layer with bf16 experts, one layer")
    # Every rank draws the same layer and tokens (the same seeds): the router and the top-8 choice
    # are replicated, the experts split.
    w = synth.make_weights(seed=args.seed, device=dev, full_layer=True, skew=wl["skew"])
    x = synth.make_x(T, seed=args.seed, device=dev)
    m = B.MoeFFN(B.MOE_FFN_FULL_LAYER, T, device=local)
    ws = B.weights_struct(w)
    s = torch.cuda.current_stream(dev).cuda_stream
    part = torch.empty((T, H), dtype=torch.float32, device=dev)
    dense = torch.zeros((T, H), dtype=torch.float32, device=dev)
    out = torch.empty_like(x)
    import torch.distributed as dist

    def shard(b, e, with_dense):
        rc = B.moe_ffn_forward_shard(m.ctx, x.data_ptr(), T, ws, b, e, with_dense, part.data_ptr(),
                                     dense.data_ptr() if with_dense else 0, s)
        if rc != B.MOE_FFN_OK:
            raise B.MoeFFNError("moe_ffn_forward_shard", rc)
        return part, dense

    def finish(p_, d_):
        rc = B.moe_ffn_finish_shards(m.ctx, x.data_ptr(), T, ws, p_.data_ptr(), d_.data_ptr(), out.data_ptr(), s)
        if rc != B.MOE_FFN_OK:
            raise B.MoeFFNError("moe_ffn_finish_shards", rc)
        return out

    def step():
        return ep_rank_step(rank, world, shard, lambda p_, d_: ep_exchange(p_, d_, world, dist), finish)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(args.steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    barrier(world, dev)
    rc, word = m.status()
    if rc != B.MOE_FFN_OK:
        raise RuntimeError("device status 0x%x after the timed steps" % word)
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    if rank == 0:
        cfg = config_of(wl, world)
        cfg["parallelism"] = "expert parallel over %d ranks (experts split, tokens and router replicated; " \
                             "all-reduce of the partial expert sums, broadcast of the shared-MLP output)" % world
        line = {"metric": METRIC, "value": T * args.steps / (ms / 1e3), "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": cfg, "impl": "ours-expert-parallel",
                "gpu_launches": args.steps * (B.moe_ffn_kernels_per_forward(m.ctx, T) + 1)}
        print(json.dumps(line), flush=True)
    m.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


SWEEP_T = (1, 16, 256, 1024, 4096, 16384)


def compact_result(res, wl, args):
    """The figures of one measured configuration, for the line's `configs` object."""
    lr, rf, ck = res["layer_roofline"], res["roofline"], res["clocks"] or {}
    return {"workload": wl["desc"], "T": wl["T"], "value": res["value"], "unit": UNIT,
            "ms_per_step": res["ms_per_step"], "steps": args.steps, "warmup": max(args.warmup, 3),
            "layer_roofline": {k: lr[k] for k in ("frac", "bound", "roofline_us", "step_us", "experts_hit")},
            "roofline": {k: rf[k] for k in ("kernel", "bound", "achieved", "peak", "unit", "frac", "traffic")},
            "e2e": res["e2e"]["value"], "gpu_launches": res["gpu_launches"],
            "clocks": {k: ck.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "in_timed_region")},
            "kernels_us": res["kernels_us"]}


def run_configs(args, layer_weights, dev, world, rank, clocks):
    import torch
    from mixture_experts_ffn_router_gb300 import synth

    out = {}
    wl = dict(WORKLOADS["moe8"])
    w_moe = synth.make_weights(seed=args.seed, layer=0, device=dev, full_layer=False, skew=False)
    x = synth.make_x(wl["T"], seed=args.seed, device=dev)
    out["moe8"] = compact_result(measure(args, wl, [w_moe], x, dev, world, rank, False, clocks, "moe8"), wl, args)
    del w_moe
    sweep = {"T=64": "the line's value (decode64)"}
    for T in SWEEP_T:
        wl = workload_of(argparse.Namespace(workload="layer", T=T))
        x = synth.make_x(T, seed=args.seed, device=dev)
        sweep["T=%d" % T] = compact_result(measure(args, wl, [layer_weights], x, dev, world, rank, False, clocks,
                                                   "layer"), wl, args)
    out["sweep"] = sweep
    wl = dict(WORKLOADS["stack30"])
    ws = [synth.make_weights(seed=args.seed, layer=l, device=dev, full_layer=True, skew=False)
          for l in range(wl["layers"])]
    x = synth.make_x(wl["T"], seed=args.seed, device=dev)
    res = measure(args, wl, ws, x, dev, world, rank, False, clocks, "stack30")
    out["stack30"] = {**compact_result(res, wl, args), "layers": wl["layers"],
                      "note": "value is end-to-end tokens/s through all 30 layers; layer_roofline is per layer"}
    del ws
    torch.cuda.empty_cache()
    return out


def run_ours(args, wl):
    import torch
    from mixture_experts_ffn_router_gb300 import synth

    rank, world = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T = wl["T"]
    L = wl.get("layers", 1)
    weights = [synth.make_weights(seed=args.seed, layer=l, device=dev, full_layer=wl["full"], skew=wl["skew"])
               for l in range(L)]
    if wl.get("int8") or wl.get("fp4"):
        from mixture_experts_ffn_router_gb300 import binding as B
        # int8 or MXFP4 experts, made on the device; the bf16 experts are then dropped.
        q = B.quantize_experts_int8 if wl.get("int8") else B.quantize_experts_mxfp4
        weights = [q(w) for w in weights]
        torch.cuda.synchronize()
        for w in weights:
            del w["gate_up"], w["down"]
    x = synth.make_x(T, seed=args.seed, device=dev)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid=uuid).start()
    time.sleep(0.3)
    res = measure(args, wl, weights, x, dev, world, rank, rank == 0 and world == 1 and not args.no_cpu_baseline,
                  clocks, args.workload)

    # The metric is quoted at decode T=64 and at prefill T=4096: the default run measures both in
    # this process. The prefill leg runs the same layer's weights with the skewed router rows
    # (Zipf(1.1) row scales, the same draw the prefill4096 workload makes) on 4096 tokens.
    prefill = None
    if args.workload == "decode64" and not args.no_prefill:
        wl_p = workload_of(argparse.Namespace(workload="prefill4096", T=None))
        w_p = dict(weights[0])
        w_p["router_w"] = synth.make_router_w(seed=args.seed, layer=0, device=dev, skew=True)
        x_p = synth.make_x(wl_p["T"], seed=args.seed, device=dev)
        prefill = measure(args, wl_p, [w_p], x_p, dev, world, rank, False, clocks, "prefill4096")
        prefill = {"metric": METRIC, "unit": UNIT, "steps": args.steps, "warmup": max(args.warmup, 3),
                   "config": config_of(wl_p, world), **prefill}
        del prefill["cpu_baseline"]
    # The block's other configurations, measured in the same process under the same rules, so that
    # every configuration the metric is reported on has a number from this run: the experts-only
    # block at T=8, the full layer swept over T with uniform routing (T=64 is the line's value),
    # and the 30-layer stack at T=256.
    configs = None
    if args.workload == "decode64" and not args.no_configs:
        configs = run_configs(args, weights[0], dev, world, rank, clocks)
    time.sleep(0.25)
    clocks.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(wl, world),
            "roofline": res["roofline"], "layer_roofline": res["layer_roofline"], "cpu_baseline": res["cpu_baseline"],
            "e2e": res["e2e"], "gpu_launches": res["gpu_launches"] + (prefill["gpu_launches"] if prefill else 0),
            "gpu_launches_note": "both timed regions (decode and prefill legs)" if prefill else "the timed region",
            "clocks": res["clocks"], "kernels_us": res["kernels_us"], "kernels_us_note": res["kernels_us_note"],
        }
        if prefill is not None:
            line["prefill4096"] = prefill
        if configs is not None:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    wl = workload_of(args)
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.ep:
        return run_ep(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())

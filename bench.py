"""Benchmark: conv2d training step (forward + backward) on one GB300 per rank.

Workload: the `large` layer - N=256, 56x56x256 NHWC bf16 -> 256 channels,
3x3 stride 1 pad 1, training batch norm (eps 1e-5, momentum 0.1), ReLU,
seeded synthetic inputs (X ~ N(0,1), Kaiming-normal weights, dY ~ N(0,1e-2)).
A step = conv2d_fwd_train + conv2d_bwd (dx, dw, dbias, dgamma, dbeta) through
the C ABI. Throughput = 3 x 2*N*OH*OW*OC*KH*KW*IC FLOPs (full-tap
convention) / step time. Every operand (411 MB per activation tensor) is
larger than the 129 MB L2, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (plain fp64 loops, all host cores) on a
bounded sample of the same workload. Under torchrun each rank runs its own
replica (no collective on the data path) and rank 0 prints one JSON line.
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

METRIC = "conv2d fwd+bwd TFLOP/s (and % of dense TC peak) per layer on 1 GB300"
WORKLOAD = "large"
NOMINAL_BF16_TFLOPS = 2250.0

# DRAM bytes (read + write) per launch of the GEMM kernels on the 256-image layer, from the ncu capture
# summarised in profiles/large_step_kernels.md (96-image case, scaled by 256/96). Reset to None whenever
# a GEMM kernel changes and re-capture.
NCU_TRAFFIC_BYTES = {"fprop_gemm": 715e6, "dgrad_gemm": 706e6, "wgrad_gemm": 822e6}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sust=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


def _workload_desc(spec):
    return ("large: N=%d %dx%dx%d -> %d, %dx%d stride %d pad %d, batch norm + ReLU, bf16 operands, fp32 accumulate"
            % (spec.N, spec.H, spec.W, spec.IC, spec.OC, spec.KH, spec.KW, spec.stride, spec.pad))


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None
        self.windows = []

    def start(self):
        """Start sampling every 20 ms; called well before the timed regions (nvidia-smi takes a moment)."""
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None

    def mark(self, t0, t1):
        """Wall-clock bounds of a timed region; only samples inside one are kept."""
        self.windows.append((t0, t1))

    def stop(self):
        import datetime
        if self.p is None:
            return None
        time.sleep(0.1)
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except Exception:
            self.p.kill()
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(f[2]), float(f[3])
            except ValueError:
                continue
            if self.windows and not any(a - 0.02 <= ts <= b + 0.02 for a, b in self.windows):
                continue
            sm.append(clk)
            mx = cmax
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * (mx or 1)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def run_gpu(args, rank, world, local_rank):
    import torch

    from conv2d_layer_gb300 import abi
    from conv2d_layer_gb300.layer import Conv2dLayer
    from conv2d_layer_gb300.workloads import WORKLOADS, make_inputs

    from dataclasses import replace

    torch.cuda.set_device(local_rank)
    spec = WORKLOADS[WORKLOAD].layers[0]
    if args.images:
        spec = replace(spec, N=args.images)
    inp = make_inputs(WORKLOAD, n_images=args.images or None)
    li = inp["layers"][0]
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta, li.running_mean, li.running_var)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    stream = torch.cuda.current_stream()
    flops = spec.flops_step()

    def step():
        L.fwd_train(x)
        L.bwd(x, dy)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    rc, site = abi.conv2d_device_status()
    if rc != abi.OK:
        raise RuntimeError("device status %d site %d" % (rc, site))

    # launches per step, counted from the library's own launch records
    abi.conv2d_prof_enable(True)
    abi.conv2d_prof_read()
    step()
    per_step = len(abi.conv2d_prof_read())
    abi.conv2d_prof_enable(False)

    def timed(n, instrumented):
        # n steps between two events on the launching stream; with `instrumented` the library also
        # brackets every launch with its own CUDA events (per-kernel durations), which costs a little
        if instrumented:
            abi.conv2d_prof_enable(True)
            abi.conv2d_prof_read()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if instrumented:
            # the GPU idles in a ~2 ms sleep kernel before the first event while the host runs ahead, so
            # that the per-launch events bracket back-to-back kernels
            with torch.cuda.stream(stream):
                torch.cuda._sleep(4_000_000)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        recs = []
        if instrumented:
            abi.conv2d_prof_enable(False)
            recs = abi.conv2d_prof_read(8192)
        return e0.elapsed_time(e1) / n, recs

    clocks = Clocks(local_rank)
    clocks.start()
    time.sleep(0.3)  # let the sampler start
    w0 = time.time()
    ms, _ = timed(args.steps, False)                   # the headline: no per-launch instrumentation
    w1 = time.time()
    ms_instr, recs = timed(args.steps, True)           # per-kernel durations over a second timed region
    w2 = time.time()
    clocks.mark(w0, w1)
    clocks.mark(w1, w2)
    ck = clocks.stop()
    rc, site = abi.conv2d_device_status()
    if rc != abi.OK:
        raise RuntimeError("device status %d site %d" % (rc, site))

    kern = {}
    for name, t in recs:
        k = kern.setdefault(name, [0, 0.0])
        k[0] += 1
        k[1] += t

    # end to end through the public API with host buffers: every step copies its X and dY in from pinned
    # host memory and its parameter gradients (dW, dbias, dgamma, dbeta) out. The copies of step k+1 run
    # on a second stream while step k computes (two device input buffers), as a training loop would;
    # every step's copies are inside the timed region.
    xh = inp["x"].pin_memory()
    dyh = inp["dy"].pin_memory()
    outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (L.dw, L.db, L.dgamma, L.dbeta)]
    h2d = xh.numel() * xh.element_size() + dyh.numel() * dyh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs)
    xs = [x, torch.empty_like(x)]
    dys = [dy, torch.empty_like(dy)]
    copy_stream = torch.cuda.Stream()

    def e2e_run(n):
        copied = [torch.cuda.Event() for _ in range(n)]
        done = [torch.cuda.Event() for _ in range(n)]
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        copy_stream.wait_stream(stream)
        for k in range(n):
            b = k % 2
            with torch.cuda.stream(copy_stream):
                if k >= 2:
                    copy_stream.wait_event(done[k - 2])  # buffer b is free once step k-2 is done
                xs[b].copy_(xh, non_blocking=True)
                dys[b].copy_(dyh, non_blocking=True)
                copied[k].record(copy_stream)
            stream.wait_event(copied[k])
            L.fwd_train(xs[b])
            L.bwd(xs[b], dys[b])
            for o, t in zip(outs, (L.dw, L.db, L.dgamma, L.dbeta)):
                o.copy_(t, non_blocking=True)
            done[k].record(stream)
        f1.record(stream)
        torch.cuda.synchronize()
        return f0.elapsed_time(f1) / n

    e2e_run(2)
    n_e2e = max(3, min(args.steps, 10))
    barrier()
    e2e_ms = e2e_run(n_e2e)

    return dict(ms=ms, ms_instr=ms_instr, e2e_ms=e2e_ms, flops=flops, spec=spec, kern=kern, per_step=per_step,
                clocks=ck, h2d=h2d, d2h=d2h, n_e2e=n_e2e)


# Per-launch algorithmic bytes of the bandwidth-bound kernels, in units of one [n_pix][OC] tensor of the
# layer's element type: apply reads pre_act and writes y; the backward reduce reads pre_act and dY; d_conv
# reads both and writes d_conv.
HBM_TENSORS = {"bn_apply": 2, "ln_apply": 2, "gn_apply": 2, "gn_stats": 1, "bn_bwd_reduce": 2, "ln_bwd_reduce": 2,
               "bn_bwd_dconv": 3, "ln_bwd_dconv": 3, "act_bwd_dconv": 3}

PER_CONFIG = (
    # (label, workload, overrides of every layer spec)
    ("tiny", "tiny", {}),
    ("rl", "rl", {}),
    ("bn", "bn", {}),
    ("mixed", "mixed", {}),
    ("large", "large", {}),
    ("bn+layernorm", "bn", {"norm": 2}),
    ("large+layernorm", "large", {"norm": 2}),
    ("large+groupnorm32", "large", {"norm": 3, "groups": 32}),
)


# Images of each per-config workload the oracle runs for its CPU baseline (a bounded sample, a few
# seconds in all on the host cores).
CPU_SAMPLE_IMAGES = {"tiny": 2, "rl": 8, "bn": 4, "mixed": 1, "large": 1}


def cpu_baseline_config(name, over, n_img):
    """The oracle, as it stands, on a bounded sample of one per-config workload: n_img images through
    fwd_train + bwd of every layer (a stack feeds each layer's output to the next and its dX back as the
    previous layer's dY). Returns the cpu_baseline object of that entry."""
    from dataclasses import replace

    import oracle
    from conv2d_layer_gb300.workloads import BF16, WORKLOADS, make_inputs

    specs = [replace(sp, N=n_img, **over) for sp in WORKLOADS[name].layers]
    inp = make_inputs(name, layers=specs)
    f64 = lambda t: t.double().numpy()  # noqa: E731
    ols = [oracle.Layer(sp.N, sp.H, sp.W, sp.IC, sp.OC, sp.KH, sp.KW, sp.stride, sp.pad, norm=sp.norm, act=sp.act,
                        eps=sp.eps, momentum=sp.momentum, store="bf16" if sp.dtype == BF16 else "f32",
                        groups=sp.groups) for sp in specs]
    params = [(f64(li.w), f64(li.b), f64(li.gamma), f64(li.beta)) for li in inp["layers"]]
    x0, dy = f64(inp["x"]), f64(inp["dy"])
    t0 = time.perf_counter()
    acts, fw = [x0], []
    for OL, (w, b, gm, bt) in zip(ols, params):
        f = oracle.fwd_train(OL, acts[-1], w, b, gm, bt)
        fw.append(f)
        acts.append(f["y"])
    g = dy
    for OL, (w, b, gm, bt), f, a in zip(reversed(ols), reversed(params), reversed(fw), reversed(acts[:-1])):
        g = oracle.bwd(OL, a, w, f["ypre"], g, gm, bt, f["mean"], f["inv_std"])["dx"]
    dt = time.perf_counter() - t0
    flops = sum(sp.flops_step() for sp in specs)
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d image(s) of this workload, one fwd_train + bwd step (%.3f GFLOP fp64, %.2f s)"
                      % (n_img, flops / 1e9, dt)}


def per_config_cpu():
    """CPU baselines of every per-config entry (run before any GPU work)."""
    return {label: cpu_baseline_config(name, over, CPU_SAMPLE_IMAGES[name]) for label, name, over in PER_CONFIG}


def tf32_peak():
    """Dense TF32 tensor throughput of this GPU: a cuBLAS fp32 matmul of 8192^3 with TF32 allowed
    (torch.matmul), best of 10 CUDA-event timings. The fp32 layers run 3xTF32, whose bound is a third of
    it. Measured in the run, outside every timed region."""
    import torch

    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        n = 8192
        a = torch.randn(n, n, device="cuda")
        b = torch.randn(n, n, device="cuda")
        c = torch.empty(n, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = 1e30
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def layer_bytes(sp):
    """Algorithmic HBM bytes of one training step of a layer (each tensor moved once per pass that needs
    it): the three GEMMs read and write their operands (fprop X, W, pre_act; dgrad d_conv, W, dX; wgrad
    d_conv, X, dW in fp32); with a norm, apply 2|Y|, backward reduce 2|Y|, d_conv 3|Y|; without, the
    activation is in the fprop epilogue (one more |Y| write) and d_conv 3|Y|."""
    es = 2 if sp.dtype == 1 else 4
    x = sp.N * sp.H * sp.W * sp.IC * es
    y = sp.n_pix * sp.OC * es
    w = sp.OC * sp.KH * sp.KW * sp.IC * es
    gemm = (x + w + y) + (y + w + x) + (y + x + sp.OC * sp.KH * sp.KW * sp.IC * 4)
    return gemm + (7 * y if sp.norm != 0 else 4 * y)


def per_config_timing(peaks, steps=10, warmup=3):
    """fwd_train + bwd of every workload (the mixed stack as its two chained layers) and of the BN-layer and
    large shapes with layer and group norm: step time through the ABI calls, the same step replayed from a
    CUDA graph (no host launch work), TFLOP/s, and per-kernel times from one extra profiled step, with the
    HBM fraction of the bandwidth-bound kernels."""
    import torch

    from conv2d_layer_gb300 import abi

    out = {}
    for label, name, over in PER_CONFIG:
        specs, step, release = config_step(name, over)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        # the same step captured once in a CUDA graph and replayed: no host launch work per step
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(steps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_graph = e0.elapsed_time(e1) / steps
        del graph
        abi.conv2d_prof_enable(True)
        # the launches of each ABI call of the step (a stack's layers launch different kernels: the layer of
        # every launch below comes from these counts)
        owner = []
        for li, call in step.calls():
            abi.conv2d_prof_read()
            call()
            torch.cuda.synchronize()
            owner += [li] * len(abi.conv2d_prof_read(4096))
        abi.conv2d_prof_read()
        # the GPU idles in a ~2 ms sleep kernel while the host queues the whole step, so that the per-launch
        # events bracket back-to-back kernels (not the host's launch work between short kernels)
        torch.cuda._sleep(4_000_000)
        step()
        torch.cuda.synchronize()
        abi.conv2d_prof_enable(False)
        recs = abi.conv2d_prof_read(4096)
        kern = {}
        for kname, t in recs:
            kern[kname] = kern.get(kname, 0.0) + t
        fl = sum(s.flops_step() for s in specs)
        # algorithmic bytes of each bandwidth-bound launch from its own layer's output tensor, summed with
        # the times over the launches of the same kernel
        hb, ht = {}, {}
        if len(owner) == len(recs):
            for (kname, t), li in zip(recs, owner):
                if kname in HBM_TENSORS:
                    sp = specs[li]
                    hb[kname] = hb.get(kname, 0.0) + HBM_TENSORS[kname] * sp.n_pix * sp.OC * (2 if sp.dtype == 1 else 4)
                    ht[kname] = ht.get(kname, 0.0) + t
        hbm = {k: round(hb[k] / (ht[k] * 1e-3) / 1e9 / peaks["hbm"], 3) for k in hb}
        bf = specs[0].dtype == 1
        # the tensor-core bound of the contractions: bf16 burst, or a third of the measured TF32 rate for
        # 3xTF32; GEMM kernels (the column-form dgrad's GEMM is a launch named fprop_gemm)
        gemm_ms = sum(t for k, t in kern.items() if k.endswith("_gemm"))
        peak = peaks["bf16"] if bf else (peaks["tf32"] / 3 if peaks.get("tf32") else None)
        ach = fl / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
        floor_ms = sum(layer_bytes(sp) for sp in specs) / (peaks["hbm"] * 1e9) * 1e3
        roof = {"bound": "tensor", "kind": "bf16 burst" if bf else "3xTF32: measured TF32 burst / 3",
                "gemm_ms": round(gemm_ms, 4), "achieved": round(ach, 1) if ach else None, "unit": "TFLOP/s",
                "peak": round(peak, 1) if peak else None,
                "frac": round(ach / peak, 4) if (ach and peak) else None,
                "memory_floor_ms": round(floor_ms, 4), "step_frac_of_memory_floor": round(floor_ms / ms, 4)}
        out[label] = {"ms_per_step": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 2),
                      "ms_per_step_graph": round(ms_graph, 4),
                      "dtype": "bf16" if bf else "fp32 (3xTF32)", "layers": len(specs),
                      "kernels_ms": {k: round(t, 4) for k, t in kern.items()}, "hbm_frac_of_measured": hbm,
                      "roofline": roof}
        release()
        torch.cuda.empty_cache()
    abi.check(abi.conv2d_device_status()[0], "device status")
    return out


def config_step(name, over):
    """Layers, inputs and the fwd_train + bwd step of one workload (every layer spec updated by `over`; a
    stack chains its layers forward and backward). Returns (specs, step, release)."""
    from dataclasses import replace

    from conv2d_layer_gb300.layer import Conv2dLayer
    from conv2d_layer_gb300.workloads import WORKLOADS, make_inputs

    specs = [replace(s, **over) for s in WORKLOADS[name].layers]
    inp = make_inputs(name, layers=specs)
    state = {"layers": [Conv2dLayer(s, li.w, li.b, li.gamma, li.beta, li.running_mean, li.running_var)
                        for s, li in zip(specs, inp["layers"])],
             "x": inp["x"].cuda(), "dy": inp["dy"].cuda()}

    def calls():
        """The step's ABI calls in order, as (layer index, call): every layer's fwd_train, then every
        layer's bwd from the last layer back."""
        layers = state["layers"]
        acts = [state["x"]]
        g = [state["dy"]]
        seq = []
        for i, L in enumerate(layers):
            seq.append((i, lambda i=i, L=L: acts.append(L.fwd_train(acts[i]))))
        for i in reversed(range(len(layers))):
            def b(i=i):
                g[0] = layers[i].bwd(acts[i], g[0])
            seq.append((i, b))
        return seq

    def step():
        for _, call in calls():
            call()

    step.calls = calls
    return specs, step, state.clear


def profile_workload(label, steps, warmup):
    """Training steps of one per-config entry and nothing else: a short program for profiler captures
    of the smaller workloads. Prints the step time (CUDA events), not the benchmark line."""
    import torch

    from conv2d_layer_gb300 import abi

    entry = {lab: (name, over) for lab, name, over in PER_CONFIG}[label]
    _, step, release = config_step(*entry)
    for _ in range(max(warmup, 1)):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    abi.check(abi.conv2d_device_status()[0], "device status")
    print(json.dumps({"profile_workload": label, "steps": steps, "ms_per_step": round(e0.elapsed_time(e1) / steps, 4)}),
          flush=True)
    release()


def gemm_roofline(spec, kern, steps, peaks):
    """Per-kernel figures; the dominant kernel (largest total time) becomes the roofline entry."""
    gemm_flops = 2.0 * spec.n_pix * spec.OC * spec.KH * spec.KW * spec.IC
    y_bytes = spec.n_pix * spec.OC * 2
    # algorithmic bytes per launch of the bandwidth-bound kernels (bf16 tensors)
    bytes_per = {"bn_stats": y_bytes, "bn_apply": 2 * y_bytes, "bn_bwd_reduce": 2 * y_bytes,
                 "bn_bwd_dconv": 3 * y_bytes, "act_bwd_dconv": 3 * y_bytes}
    out = {}
    for name, (n, tot) in kern.items():
        avg = tot / max(n, 1)
        e = {"launches": n, "avg_ms": round(avg, 4), "share": 0.0}
        if name in ("fprop_gemm", "dgrad_gemm", "wgrad_gemm"):
            a = gemm_flops / (avg * 1e-3) / 1e12
            e.update(bound="tensor", achieved=round(a, 1), unit="TFLOP/s", frac=round(a / peaks["bf16"], 4))
        elif name in bytes_per:
            a = bytes_per[name] / (avg * 1e-3) / 1e9
            e.update(bound="hbm", achieved=round(a, 1), unit="GB/s", frac=round(a / peaks["hbm"], 4))
        out[name] = e
    total = sum(t for _, t in kern.values()) or 1.0
    for name, (n, tot) in kern.items():
        out[name]["share"] = round(tot / total, 4)
    return out


def run_reference(args, rank):
    """The CPU oracle, as it stands, on a bounded sample of the workload (a few images)."""
    import numpy as np

    import oracle
    from conv2d_layer_gb300.workloads import WORKLOADS, make_inputs

    n_img = args.ref_images
    spec = WORKLOADS[WORKLOAD].layers[0]
    inp = make_inputs(WORKLOAD, n_images=n_img)
    li = inp["layers"][0]
    f64 = lambda t: t.double().numpy()  # noqa: E731
    OL = oracle.Layer(n_img, spec.H, spec.W, spec.IC, spec.OC, spec.KH, spec.KW, spec.stride, spec.pad,
                      norm=spec.norm, act=spec.act, eps=spec.eps, momentum=spec.momentum, store="bf16")
    x, w, dy = f64(inp["x"]), f64(li.w), f64(inp["dy"])
    b, gm, bt = f64(li.b), f64(li.gamma), f64(li.beta)
    flops = 3.0 * 2.0 * n_img * spec.OH * spec.OW * spec.OC * spec.KH * spec.KW * spec.IC

    def step():
        f = oracle.fwd_train(OL, x, w, b, gm, bt)
        oracle.bwd(OL, x, w, f["ypre"], dy, gm, bt, f["mean"], f["inv_std"])

    for _ in range(args.warmup if args.ref_warmup else 0):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = flops / dt / 1e12
    cores = oracle.num_threads()
    sample = "%d image(s) of the large workload per step (%.1f GFLOP fp64)" % (n_img, flops / 1e9)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_desc(spec), "sample_images": n_img, "flops_per_step": flops},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(n_img=1):
    import oracle
    from conv2d_layer_gb300.workloads import WORKLOADS, make_inputs

    spec = WORKLOADS[WORKLOAD].layers[0]
    inp = make_inputs(WORKLOAD, n_images=n_img)
    li = inp["layers"][0]
    f64 = lambda t: t.double().numpy()  # noqa: E731
    OL = oracle.Layer(n_img, spec.H, spec.W, spec.IC, spec.OC, spec.KH, spec.KW, spec.stride, spec.pad,
                      norm=spec.norm, act=spec.act, eps=spec.eps, momentum=spec.momentum, store="bf16")
    x, w, dy = f64(inp["x"]), f64(li.w), f64(inp["dy"])
    t0 = time.perf_counter()
    f = oracle.fwd_train(OL, x, w, f64(li.b), f64(li.gamma), f64(li.beta))
    oracle.bwd(OL, x, w, f["ypre"], dy, f64(li.gamma), f64(li.beta), f["mean"], f["inv_std"])
    dt = time.perf_counter() - t0
    flops = 3.0 * 2.0 * n_img * spec.OH * spec.OW * spec.OC * spec.KH * spec.KW * spec.IC
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "%d image(s) of the large workload, one fwd_train + bwd step (%.1f GFLOP fp64, %.1f s)"
                      % (n_img, flops / 1e9, dt)}


def max_over_ranks(vals, device):
    """Each value's maximum over the ranks of the default process group: the slowest rank sets the step
    time of the job."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tflops(world, flops_per_gpu, ms):
    """Whole-job TFLOP/s: the work of every replica over the (slowest rank's) step time."""
    return world * flops_per_gpu / (ms * 1e-3) / 1e12


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-images", type=int, default=1)
    ap.add_argument("--ref-warmup", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--images", type=int, default=0,
                    help="run the large layer with this many images instead of 256 (small profiling cases)")
    ap.add_argument("--profile-workload", default="", choices=[""] + [c[0] for c in PER_CONFIG],
                    help="only run --steps training steps of this per-config entry (profiler captures)")
    args = ap.parse_args()

    if args.profile_workload:
        profile_workload(args.profile_workload, args.steps, args.warmup)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            args.steps = min(args.steps, 3)
            run_reference(args, rank)
        return

    # the CPU baseline runs before any GPU work (rank 0, single GPU only)
    cpu = None
    cpu_cfg = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.ref_images)
        if not args.no_per_config and not args.images:
            cpu_cfg = per_config_cpu()

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    r = run_gpu(args, rank, world, local_rank)
    ms, e2e_ms = r["ms"], r["e2e_ms"]
    per_cfg = None
    tf32 = None
    if rank == 0 and world == 1 and not args.no_per_config and not args.images:
        tf32 = tf32_peak()
        per_cfg = per_config_timing(dict(_peaks(), tf32=tf32))
        for label, c in (cpu_cfg or {}).items():
            per_cfg[label]["cpu_baseline"] = c
    if world > 1:
        ms, e2e_ms = max_over_ranks([ms, e2e_ms], "cuda")
    if rank != 0:
        return
    spec = r["spec"]
    peaks = _peaks()
    value = job_tflops(world, r["flops"], ms)
    kern = gemm_roofline(spec, r["kern"], args.steps, peaks)
    gemms = {k: v for k, v in kern.items() if k.endswith("_gemm")}
    dom = max(gemms, key=lambda k: gemms[k]["avg_ms"] * gemms[k]["launches"])
    d = kern[dom]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded X~N(0,1), Kaiming-normal W, dY~N(0,1e-2), random init",
        "config": {"workload": _workload_desc(spec), "global_batch": spec.N * world,
                   "flops_per_step_per_gpu": r["flops"], "flop_convention": "3 GEMMs x 2*n_pix*OC*KH*KW*IC (full tap)",
                   "l2": "no flush: every operand (411 MB) is larger than the 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_dense_tc_peak": {"of_measured_burst": round(value / world / peaks["bf16"], 4),
                              "of_measured_sustained": round(value / world / peaks["bf16_sust"], 4),
                              "of_nominal_2250": round(value / world / NOMINAL_BF16_TFLOPS, 4),
                              "peaks": peaks["src"]},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": d["achieved"], "peak": peaks["bf16"],
                     "unit": "TFLOP/s", "frac": d["frac"],
                     "traffic": (NCU_TRAFFIC_BYTES or {}).get(dom) if spec.N == 256 else None,
                     "peak_kind": "bf16 burst (%s): the kernel is timed with CUDA events inside a region of "
                                  "about 50 ms, not a seconds-long loop" % peaks["src"]},
        "kernels": kern,
        "kernels_timing": {"ms_per_step_instrumented": round(r["ms_instr"], 4),
                           "what": "per-launch CUDA events over a second timed region of the same steps"},
        "gpu_launches": r["per_step"] * args.steps,
        "e2e": {"value": round(job_tflops(world, r["flops"], e2e_ms), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": round(e2e_ms, 4),
                "what": "every step: pinned host X, dY copied in, dW, dbias, dgamma, dbeta copied out, same ABI "
                        "calls; the copies of step k+1 overlap step k (second stream, two input buffers)"},
        "clocks": r["clocks"],
        "per_config": per_cfg,
        "tf32_peak": ({"burst_tflops": round(tf32, 1), "how": "cuBLAS fp32 matmul 8192^3 with TF32 allowed "
                       "(torch.matmul), best of 10, measured in this run"} if tf32 else None),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

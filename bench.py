"""Benchmark of the nested-bit quantized linear layer on one GB300 (or N replicas).

Workload: the Qwen-4B-like MLP triplet (gate and up 9728x2560, down 2560x9728),
2-bit base + 7-bit residual with 128-column fp16 scales, synthetic
N(0, 0.02^2) weights with 0.5% Student-t(4) outliers, bf16 N(0,1)
activations.  Weights are quantised and packed on the device by the library
itself.  `--copies` distinct quantised copies of the triplet (a stack of
layers) are resident in HBM so each pass streams far more than the 129 MB L2.

One step = one speculative check over the stack: a draft pass at T = 1
(rotate in, base-only GEMV, rotate out for every linear), then a verify pass
at T = 16 (rotate in, base + residual GEMM, rotate out).  `value` is the
effective HBM bandwidth of the step: the algorithmic bytes of every linear
(M*K*(2.125 [+ b + 0.125])/8 weight bytes + 2*T*K input + 4*T*M output bytes)
divided by the step time.  The verify GEMM alone is timed as well (at T = 16
and T = 1) and carries the roofline figure.

`--impl reference` times the CPU oracle (numpy fp64) on the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify GEMM effective HBM GB/s and µs/layer at T=16 (vs T=1), % of 8 TB/s roofline"
WORKLOAD = "mlp_triplet_4b"
BITS = 7
T_VERIFY, T_DRAFT = 16, 1
SWEEP_T = (1, 4, 8, 16, 32, 64)
PREFILL_T = (128, 256)
# DRAM bytes per linear of the roofline kernel, from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum of a grouped gate+up verify launch at T=16, divided by its two
# linears).  Valid only for the kernel source it was taken on: reported as null otherwise.
NCU_TRAFFIC = {"src": "nested_bit_quantized_gb300/csrc/nest_gemm.cu",
               "sha256": "c5dbe9c81dfdf5262491e54484328e5ac759a9f27a0f16d45e236c909c77002f",
               "bytes_per_linear": (59.046400e6 + 0.015872e6) / 2}


def ncu_traffic():
    import hashlib
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), NCU_TRAFFIC["src"])
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return NCU_TRAFFIC["bytes_per_linear"] if digest == NCU_TRAFFIC["sha256"] else None


def bits_per_weight(bits):
    """Algorithmic weight bits per weight.  bits: 0 = 2-bit base alone (draft), 6/7/8 = base +
    b-bit residual (verify), 40 = W4 base alone (draft), 48 = W4 base + 4-bit refinement (verify)."""
    if bits == 40:
        return 4.125
    if bits == 48:
        return 8.125
    return 2.125 + ((bits + 0.125) if bits else 0.0)


def lin_bytes(M, K, T, bits):
    return M * K * bits_per_weight(bits) / 8.0 + 2.0 * T * K + 4.0 * T * M


def weight_bytes(M, K, bits):
    return M * K * (2.125 + ((bits + 0.125) if bits else 0.0)) / 8.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense fp16 tensor peak in TFLOP/s: the measured bf16 burst figure (fp16 and bf16 have
    the same nominal dense rate), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------

_ORACLE_LAYERS = {}


def _oracle_layer(lin):
    """The oracle's quantised layer, computed once per linear (offline work, not timed)."""
    if lin.name not in _ORACLE_LAYERS:
        from nested_bit_quantized_gb300 import synth
        from oracle import nest_oracle as O
        W = synth.weights(lin.M, lin.K, lin.w_seed, lin.outliers)
        s_o, s_i = synth.sign_pair(lin.M, lin.K, lin.sign_seed)
        _ORACLE_LAYERS[lin.name] = (O.quantize_layer(W, s_o, s_i, BITS), s_o, s_i)
    return _ORACLE_LAYERS[lin.name]


def oracle_sample(n_linears=3, seconds_cap=25.0):
    """Times the oracle's draft (T=1) and verify (T=16) forward passes on the
    workload's linears (offline quantisation excluded, done once per linear).
    Returns bytes, seconds, what."""
    from nested_bit_quantized_gb300 import synth
    from oracle import nest_oracle as O
    wl = synth.WORKLOADS[WORKLOAD]
    tot_b, tot_s, done = 0.0, 0.0, []
    for lin in wl.linears[:n_linears]:
        q, s_o, s_i = _oracle_layer(lin)
        for T, verify in ((T_DRAFT, False), (T_VERIFY, True)):
            _, x = synth.activations(T, lin.K, wl.x_seed)
            t0 = time.perf_counter()
            O.forward(q, s_o, s_i, x, verify)
            tot_s += time.perf_counter() - t0
            tot_b += lin_bytes(lin.M, lin.K, T, BITS if verify else 0)
        done.append(lin.name)
        if tot_s > seconds_cap:
            break
    what = (f"oracle draft T={T_DRAFT} + verify T={T_VERIFY} forward of {'/'.join(done)} "
            f"(one copy, quantisation untimed)")
    return tot_b, tot_s, what


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def max_over_ranks(value, dist, device):
    """The largest value over the ranks of the process group (the slowest rank's time),
    or value itself without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    if rank != 0:
        return
    tot_b = tot_s = 0.0
    what = ""
    for i in range(args.warmup + args.steps):
        b, s, what = oracle_sample(n_linears=1)
        if i >= args.warmup:
            tot_b += b
            tot_s += s
    value = tot_b / tot_s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "bits": BITS, "T_verify": T_VERIFY, "T_draft": T_DRAFT,
                       "sample": what},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle", "sample": what},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args, rank, world):
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import build as nb
    from nested_bit_quantized_gb300 import nest, synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    nb.build()
    nest.load()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    wl = synth.WORKLOADS[WORKLOAD]
    C = args.copies
    w4w8 = args.codec == "w4w8"
    DC, VC = (40, 48) if w4w8 else (0, BITS)      # byte accounting of the draft and verify passes
    # quantise and pack C copies of the triplet on the device
    layers = []
    work = None
    for c in range(C):
        trip = []
        for lin in wl.linears:
            seed = lin.w_seed + 1000 * c + 100_000 * rank
            W = synth.weights_device(lin.M, lin.K, seed, lin.outliers, dev)
            s_o, s_i = synth.sign_pair(lin.M, lin.K, lin.sign_seed + 2 * c)
            if work is None or work.numel() < lin.M * lin.K:
                work = torch.empty(lin.M * lin.K, dtype=torch.float64, device=dev)
            so, si = torch.from_numpy(s_o).to(dev), torch.from_numpy(s_i).to(dev)
            if w4w8:
                q = nest.quantize_w4w8(W, so, si, work=work[:lin.M * lin.K].view(lin.M, lin.K))
                trip.append(nest.pack_w4w8(q["q4"], q["s4"], q["qr"], so, si))
            else:
                q = nest.quantize(W, so, si, BITS, work=work[:lin.M * lin.K].view(lin.M, lin.K))
                trip.append(nest.pack(q["base_codes"], q["base_scales"], q["resid_codes"], q["resid_scales"], BITS,
                                      so, si))
            del W, q
        layers.append(trip)
    del work
    torch.cuda.synchronize()

    # activations (bf16), one per (input width, T); gate and up read the same input, as in an MLP
    xs = {}
    for T in (T_DRAFT, T_VERIFY):
        for K in sorted({l.K for l in wl.linears}):
            b, _ = synth.activations(T, K, wl.x_seed + K + T)
            xs[(K, T)] = torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    maxM = max(l.M for l in wl.linears)
    # launch groups: linears that read the same input share one grouped launch
    groups = [[0, 1], [2]]                        # (gate, up), (down)
    scratch = torch.zeros(max(nest.linear_group_scratch_bytes([layers[0][k] for k in grp], T)
                              for grp in groups for T in (T_DRAFT, T_VERIFY)), dtype=torch.uint8, device=dev)
    ys = {(k, T): torch.empty((T, wl.linears[k].M), dtype=torch.float32, device=dev)
          for k in range(3) for T in (T_DRAFT, T_VERIFY)}
    xops = {(k, T): nest.new_xop(wl.linears[k].K, T, dev) for k in range(3) for T in (T_DRAFT, T_VERIFY)}
    zbuf = {(k, T): torch.zeros((T, wl.linears[k].M), dtype=torch.float32, device=dev)  # accumulated into
            for k in range(3) for T in (T_DRAFT, T_VERIFY)}

    def run_pass(T, verify):
        for trip in layers:
            for grp in groups:
                nest.linear_group([trip[k] for k in grp], [xs[(trip[k].K, T)] for k in grp], verify,
                                  ys=[ys[(k, T)] for k in grp], scratch=scratch)

    def step():
        run_pass(T_DRAFT, False)                  # draft pass through the stack
        run_pass(T_VERIFY, True)                  # verify pass through the stack

    def gemm_only(T, verify):
        for trip in layers:
            for grp in groups:
                nest.gemm_group([trip[k] for k in grp], [xops[(k, T)] for k in grp], T, verify,
                                zs=[zbuf[(k, T)] for k in grp])

    # operands for the GEMM-only regions
    for k, l in enumerate(layers[0]):
        for T in (T_DRAFT, T_VERIFY):
            nest.rotate(xs[(l.K, T)], l.sign_in, 0, x_op=xops[(k, T)])

    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    with torch.cuda.stream(stream):
        for name, fn in (("step", step), ("v16", lambda: gemm_only(T_VERIFY, True)),
                         ("v1", lambda: gemm_only(T_DRAFT, True)), ("d1", lambda: gemm_only(T_DRAFT, False))):
            fn()                                  # first launches configure the kernels
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs[name] = g
    torch.cuda.synchronize()
    nest.error_check()

    def timed(g, reps, warm):
        for _ in range(warm):
            g.replay()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s.record(stream)
            for _ in range(reps):
                g.replay()
            e.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(s.elapsed_time(e), dist, dev)

    n_lin = 3 * C
    step_bytes = sum(lin_bytes(L.M, L.K, T_DRAFT, DC) + lin_bytes(L.M, L.K, T_VERIFY, VC)
                     for trip in layers for L in trip)
    with ClockSampler(local) as clk:
        ms = timed(graphs["step"], args.steps, args.warmup)
    clocks = clk.summary()
    ms_step = ms / args.steps
    value = world * step_bytes / (ms_step * 1e-3) / 1e9

    sub = {}
    for name, T, bits in (("v16", T_VERIFY, VC), ("v1", T_DRAFT, VC), ("d1", T_DRAFT, DC)):
        reps = max(3, args.steps)
        tms = timed(graphs[name], reps, max(3, args.warmup)) / reps
        per = tms * 1e3 / n_lin                   # us per linear (all three linears move equal bytes)
        n_launch = len(groups) * C
        by = sum(lin_bytes(L.M, L.K, T, bits) for L in layers[0]) / 3
        sub[name] = {"us_per_gemm": per, "GBps": by / (per * 1e-6) / 1e9, "bytes_per_gemm": by,
                     "launches": n_launch}
    hbm, src = peaks()

    # GEMM-only sweep over T (draft and verify), same copies and launch groups
    sweep = []
    if not args.no_sweep:
        for T in SWEEP_T:
            sx = {k: nest.new_xop(l.K, T, dev) for k, l in enumerate(layers[0])}
            sz = {k: torch.zeros((T, l.M), dtype=torch.float32, device=dev) for k, l in enumerate(layers[0])}
            for k, l in enumerate(layers[0]):
                b, _ = synth.activations(T, l.K, wl.x_seed + 7 * T + k)
                nest.rotate(torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16), l.sign_in, 0,
                            x_op=sx[k])
            rec = {"T": T}
            for verify in (False, True):
                def fn():
                    for trip in layers:
                        for grp in groups:
                            nest.gemm_group([trip[k] for k in grp], [sx[k] for k in grp], T, verify,
                                            zs=[sz[k] for k in grp])
                with torch.cuda.stream(stream):
                    fn()
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        fn()
                reps = 20
                per = timed(g, reps, 3) / reps * 1e3 / n_lin
                by = sum(lin_bytes(L.M, L.K, T, VC if verify else DC) for L in layers[0]) / 3
                key = "verify" if verify else "draft"
                rec[key + "_us"] = per
                rec[key + "_GBps"] = by / (per * 1e-6) / 1e9
                del g
            sweep.append(rec)
        nest.error_check()

    # prefill-size verify (T = 128, 256): a dense contraction on tcgen05, measured as TFLOP/s
    prefill = []
    if not args.no_sweep:
        tpk, tsrc = tensor_peak()
        for T in PREFILL_T:
            sx = {k: nest.new_xop(l.K, T, dev) for k, l in enumerate(layers[0])}
            sz = {k: torch.zeros((T, l.M), dtype=torch.float32, device=dev) for k, l in enumerate(layers[0])}
            for k, l in enumerate(layers[0]):
                b, _ = synth.activations(T, l.K, wl.x_seed + 7 * T + k)
                nest.rotate(torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16), l.sign_in, 0,
                            x_op=sx[k])

            def fn():
                for trip in layers:
                    for grp in groups:
                        nest.gemm_group([trip[k] for k in grp], [sx[k] for k in grp], T, True,
                                        zs=[sz[k] for k in grp])
            with torch.cuda.stream(stream):
                fn()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    fn()
            reps = 10
            per = timed(g, reps, 3) / reps * 1e3 / n_lin
            flops = sum(2.0 * L.M * L.K * T for L in layers[0]) / 3
            by = sum(lin_bytes(L.M, L.K, T, VC) for L in layers[0]) / 3
            tf = flops / (per * 1e-6) / 1e12
            prefill.append({"T": T, "verify_us": per, "GBps": by / (per * 1e-6) / 1e9, "TFLOPs": tf,
                            "frac_of_tensor_peak": tf / tpk, "tensor_peak": tpk, "peak_source": tsrc})
            del g
        nest.error_check()

    # end to end through the public API: pinned host inputs in, the last verify output back
    host_x = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in xs.items()}
    for k in xs:
        host_x[k].copy_(xs[k].cpu())
    host_y = torch.empty(ys[(2, T_VERIFY)].shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host_x.values())
    d2h = host_y.numel() * 4

    def e2e_once():
        with torch.cuda.stream(stream):
            for k in xs:
                xs[k].copy_(host_x[k], non_blocking=True)
            graphs["step"].replay()
            host_y.copy_(ys[(2, T_VERIFY)], non_blocking=True)

    for _ in range(args.warmup):
        e2e_once()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(args.steps):
        e2e_once()
    e.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s.elapsed_time(e) / args.steps, dist, dev)
    nest.error_check()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b, sec, what = oracle_sample()
        cpu = {"value": b / sec / 1e9, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle", "sample": what}

    if rank == 0:
        v16, v1, d1 = sub["v16"], sub["v1"], sub["d1"]
        ach = v16["GBps"]
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": ("mlp_triplet_4b: gate/up 9728x2560, down 2560x9728, "
                                    + ("BitNest W4 base + 4-bit refinement (W8 target), g128 fp16 scales"
                                       if w4w8 else "2-bit base + 7-bit residual, g128 fp16 scales")
                                    + "; draft T=1 then verify T=16 per step"),
                       "copies": C,
                       "resident_weight_GB": C * sum(l.M * l.K * bits_per_weight(VC) / 8 for l in wl.linears) / 1e9,
                       "l2": f"inputs larger than L2: {C} distinct quantised triplet copies per pass",
                       "accumulate": "f32", "parallelism": f"replicas x{world}",
                       "launch_groups": "gate+up in one grouped launch (same input), down alone"},
            "verify_T16": {"us_per_gemm": v16["us_per_gemm"], "GBps": v16["GBps"],
                           "frac_of_8TBps": v16["GBps"] / 8000.0},
            "verify_T1": {"us_per_gemm": v1["us_per_gemm"], "GBps": v1["GBps"]},
            "t16_over_t1": v16["us_per_gemm"] / v1["us_per_gemm"],
            "draft_T1": {"us_per_gemm": d1["us_per_gemm"], "GBps": d1["GBps"]},
            "roofline": {"bound": "hbm",
                         "kernel": f"k_nest_gemm<{VC},16> (verify, T=16; gate+up grouped, down alone)",
                         "achieved": ach,
                         "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "peak_source": src,
                         "traffic": None if w4w8 else ncu_traffic(), "traffic_unit": "DRAM bytes per linear (ncu)",
                         "algorithmic_bytes_per_linear": v16["bytes_per_gemm"]},
            "sweep": sweep,
            "prefill": prefill,
            "cpu_baseline": cpu,
            "e2e": {"value": world * step_bytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * 3 * len(groups) * C * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# chained 31B-class layers: one layer (draft T=1, verify T=64) or the 60-layer spec cycle
# ----------------------------------------------------------------------------

def run_stack(args):
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import build as nb
    from nested_bit_quantized_gb300 import chain, nest, synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    nb.build()
    nest.load()
    cycle = args.workload == "stack_31b"
    n_layers = args.layers if args.layers else (60 if cycle else 1)
    stack = synth.stack_31b(n_layers)
    bits = 8
    work = torch.empty(max(l.M * l.K for l in stack[0]), dtype=torch.float64, device=dev)
    lin = []
    for layer in stack:
        d = {}
        for l in layer:
            W = synth.weights_device(l.M, l.K, l.w_seed, l.outliers, dev)
            s_o, s_i = synth.sign_pair(l.M, l.K, l.sign_seed)
            so, si = torch.from_numpy(s_o).to(dev), torch.from_numpy(s_i).to(dev)
            q = nest.quantize(W, so, si, bits, work=work[:l.M * l.K].view(l.M, l.K))
            d[l.name.split(".")[-1]] = nest.pack(q["base_codes"], q["base_scales"], q["resid_codes"], q["resid_scales"],
                                                 bits, so, si)
            del W, q
        lin.append(d)
    del work
    torch.cuda.synchronize()
    T_d, T_v = (1, 16) if cycle else (1, 64)
    hidden = stack[0][0].K
    xs = {}
    for T in (T_d, T_v):
        b, _ = synth.activations(T, hidden, 31 + T)
        xs[T] = torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    bufs = {T: [chain.LayerBuffers(d, T, dev) for d in lin] for T in (T_d, T_v)}

    def run_pass(T, verify):
        chain.layer_input(lin[0], xs[T], bufs[T][0])
        for i in range(n_layers):
            nxt = i + 1 < n_layers
            chain.layer_forward(lin[i], bufs[T][i], verify, lin[i + 1] if nxt else None,
                                bufs[T][i + 1] if nxt else None)

    gamma = 8 if cycle else 1
    def step():
        for _ in range(gamma):
            run_pass(T_d, False)
        run_pass(T_v, True)

    stream = torch.cuda.Stream(device=dev)
    graphs = {}
    with torch.cuda.stream(stream):
        for name, fn in (("step", step), ("draft", lambda: run_pass(T_d, False)), ("verify", lambda: run_pass(T_v, True))):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs[name] = g
    torch.cuda.synchronize()
    nest.error_check()

    def timed(g, reps, warm):
        for _ in range(warm):
            g.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s.record(stream)
            for _ in range(reps):
                g.replay()
            e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    def lbytes(T, verify):
        return sum(lin_bytes(l.M, l.K, T, bits if verify else 0) for layer in stack for l in layer)

    with ClockSampler(dev.index) as clk:
        ms = timed(graphs["step"], args.steps, args.warmup)
    ms_d = timed(graphs["draft"], max(3, args.steps), args.warmup)
    ms_v = timed(graphs["verify"], max(3, args.steps), args.warmup)
    nest.error_check()
    step_bytes = gamma * lbytes(T_d, False) + lbytes(T_v, True)
    hbm, src = peaks()
    line = {
        "metric": METRIC, "value": step_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": {"workload": (f"31B-class stack, {n_layers} chained layers (q 8192x5376, k/v 4096x5376, o 5376x8192, "
                                f"gate/up 21504x5376, down 5376x21504), 2-bit base + 8-bit residual; step = "
                                f"{gamma} draft pass(es) at T={T_d} + 1 verify pass at T={T_v}"),
                   "resident_weight_GB": sum(weight_bytes(l.M, l.K, bits) for layer in stack for l in layer) / 1e9,
                   "l2": "inputs larger than L2 (every linear streams 0.1-0.4 GB)", "accumulate": "f32"},
        "draft_pass": {"T": T_d, "ms": ms_d, "us_per_layer": 1e3 * ms_d / n_layers,
                       "GBps": lbytes(T_d, False) / (ms_d * 1e-3) / 1e9},
        "verify_pass": {"T": T_v, "ms": ms_v, "us_per_layer": 1e3 * ms_v / n_layers,
                        "GBps": lbytes(T_v, True) / (ms_v * 1e-3) / 1e9,
                        "frac_of_measured_hbm": lbytes(T_v, True) / (ms_v * 1e-3) / 1e9 / hbm},
        "ideal_ms_at_measured_hbm": step_bytes / (hbm * 1e9) * 1e3,
        "gpu_launches": (gamma + 1) * 13 * n_layers * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# nested KV4/KV8 cache: decode attention at a 31B-class head configuration
# ----------------------------------------------------------------------------

def run_kv(args):
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import build as nb
    from nested_bit_quantized_gb300 import nest

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    nb.build()
    nest.load()
    Hq, Hkv, d = 64, 32, 128                      # q 8192 = 64 x 128, k/v 4096 = 32 x 128
    L = args.context
    copies = 2                                    # two layers' caches, alternating (>= L2 for KV4 at 32K)
    g = torch.Generator(device=dev).manual_seed(7)
    caches = []
    for c in range(copies):
        kc, vc = nest.KVCache(Hkv, L, dev), nest.KVCache(Hkv, L, dev)
        for s0 in range(0, L, 4096):
            n = min(4096, L - s0)
            nest.kv_write(kc, torch.randn((n, Hkv, d), generator=g, device=dev), s0)
            nest.kv_write(vc, torch.randn((n, Hkv, d), generator=g, device=dev), s0)
        caches.append((kc, vc))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    hbm, _ = peaks()
    recs = []
    cases = (("draft KV4", 1, 4, 0), ("draft KV4 + Recent-1024", 1, 4, 1024),
             ("verify KV8", 16, 8, 0), ("draft KV8", 1, 8, 0))
    if args.kv_case is not None:
        cases = (cases[args.kv_case],)
    for name, T, view, rn in cases:
        q = torch.randn((T, Hq, d), generator=g, device=dev).to(torch.bfloat16)
        out = torch.empty((T, Hq, d), dtype=torch.float32, device=dev)
        work = torch.empty(int(nest.load().nest_kv_attention_work_bytes(T, Hq, Hkv, L)) // 4 + 1,
                           dtype=torch.float32, device=dev)

        def fn():
            for kc, vc in caches:
                nest.kv_attention(q, kc, vc, L, view, rn, out=out, work=work)
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                fn()
        for _ in range(3):
            gr.replay()
        torch.cuda.synchronize()
        reps = max(10, args.steps)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s.record(stream)
            for _ in range(reps):
                gr.replay()
            e.record(stream)
        torch.cuda.synchronize()
        us = s.elapsed_time(e) * 1e3 / reps / copies
        hi = min(rn, L) if view == 4 else L
        per_pos = (64 + 2) * 2 if view == 4 else (128 + 2) * 2        # K and V rows read per position
        by = Hkv * ((L - hi) * per_pos + hi * (128 + 2) * 2) + T * Hq * d * (2 + 4)
        recs.append({"case": name, "T": T, "us_per_layer": us, "GBps": by / (us * 1e-6) / 1e9,
                     "frac_of_measured_hbm": by / (us * 1e-6) / 1e9 / hbm, "bytes": by})
        del gr
    nest.error_check()
    line = {"metric": "nested KV-cache decode attention, effective HBM GB/s per layer", "value": recs[0]["GBps"],
            "unit": "GB/s", "n_gpus": 1, "higher_is_better": True, "dtype": "f32 (4-bit planes)",
            "data": "synthetic",
            "config": {"workload": f"KV4/KV8 nested cache, Hq={Hq}, Hkv={Hkv}, d={d}, context {L}, "
                                   f"{copies} layers' caches alternating"},
            "cases": recs}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nest", choices=["nest", "reference"])
    ap.add_argument("--copies", type=int, default=12)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the GEMM-only sweep over T")
    ap.add_argument("--codec", default="l2", choices=["l2", "w4w8"],
                    help="weight codec of the default workload: l2 (2-bit base + 7-bit residual, the metric's) "
                         "or w4w8 (BitNest W4 base + 4-bit refinement)")
    ap.add_argument("--context", type=int, default=32768, help="context length of --workload kv_31b")
    ap.add_argument("--kv-case", type=int, default=None, choices=[0, 1, 2, 3],
                    help="--workload kv_31b: one case only (0 KV4 draft, 1 KV4 + Recent-1024, 2 KV8 verify "
                         "T=16, 3 KV8 draft)")
    ap.add_argument("--workload", default=WORKLOAD, choices=[WORKLOAD, "decoder_31b", "stack_31b", "kv_31b"],
                    help="mlp_triplet_4b (default, the metric's workload), one chained 31B-class layer, "
                         "or the 60-layer 31B-class speculative cycle")
    ap.add_argument("--layers", type=int, default=0, help="layers of the 31B-class stack (default 1 or 60)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload == "kv_31b":
        run_kv(args)
    elif args.workload != WORKLOAD:
        run_stack(args)
    else:
        run_gpu(args, rank, world if "RANK" in os.environ else 1)


if __name__ == "__main__":
    main()

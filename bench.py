"""Benchmark of the nested-bit quantized linear layer on one GB300 (or N replicas).

Default workload (``single_4096``): one linear of M = K = 4096 with a 2-bit base
and an 8-bit residual, 128-column fp16 scales, synthetic N(0, 0.02^2) weights
with 1% of the input columns scaled by 8, bf16 N(0,1) activations.  Weights are
quantised and packed on the device by the library itself.  ``--copies``
distinct quantised copies are resident in HBM (at least 4x the 129 MB L2), so
every pass streams its weights from HBM.

A timed step is one verify pass at T = 16 over the copies: the verify GEMM of
every copy in one grouped launch (the copies are independent linears; their
units are concatenated and streamed by resident CTAs).  ``value`` is the
effective HBM bandwidth of that GEMM: algorithmic bytes
M*K*(2.125 + b + 0.125)/8 + 2*T*K + 4*T*M per linear, divided by the time per
linear.  The same line reports the verify at T = 1 (t16/t1), the draft GEMV, one
launch per linear instead of one grouped launch, a sweep over T, the whole
linear (rotation in, GEMM, rotation out) draft + verify step, an end-to-end
verify pass through the C entry point with pinned host buffers, and extra
workloads: the Gemma-12B-like layer at b = 6/7/8 (T = 16), the Qwen-4B-like MLP
triplet (b = 7), the 60-layer 31B-class speculative cycle, and the CPU oracle's
timings.

``--impl reference`` times the CPU oracle (numpy fp64) on the same workload and
metric.  Other ``--workload`` values print the line of one extra workload alone.
"""
from __future__ import annotations

import argparse
import json
import math
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
WORKLOAD = "single_4096"
BITS = 8
T_VERIFY, T_DRAFT = 16, 1
SWEEP_T = (1, 4, 8, 16, 32, 64)
LINEAR_GROUP = 32          # whole linears per nest_linear_group call (the library takes up to 64)
PREFILL_T = (128, 256)
NOMINAL_HBM_GBS = 8000.0
# DRAM bytes per linear of the roofline kernel from one ncu capture of a grouped verify launch
# (dram__bytes_read.sum + dram__bytes_write.sum divided by the linears of the launch).  Valid
# only for the kernel source it was taken on: reported as null once that source changes.
NCU_TRAFFIC = {"src": "nested_bit_quantized_gb300/csrc/nest_gemm.cu",
               "sha256": "0197d71816886f6c163bbd26f1a9c65afef789bd75b70222a2282b4f43f94896",
               "bytes_per_linear": (698800128 + 7088896) / 32,
               "what": "ncu DRAM read/write counters of one grouped k_nest_gemm<8,16> launch over 32 copies of "
                       "the 4096x4096 linear at T=16 (the third of four): 698.80 MB read + 7.09 MB written"}


def ncu_traffic():
    import hashlib
    if not NCU_TRAFFIC["sha256"]:
        return None
    path = os.path.join(ROOT, NCU_TRAFFIC["src"])
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
    return M * K * bits_per_weight(bits) / 8.0


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
    """nvidia-smi samples of SM clock and throttle reasons while a timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.05)                      # first sample before the region starts
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        num = lambda v: v.replace(".", "").isdigit()
        sm = [float(r[0]) for r in self.rows if num(r[0])]
        mx = [float(r[1]) for r in self.rows if num(r[1])]
        pw = [float(r[2]) for r in self.rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(self.rows)}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def max_over_ranks(value, dist, device):
    """The largest value over the ranks of the process group (the slowest rank's time),
    or value itself without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------

def _oracle_case(M, K, bits, T, verify, seed, real_weights=None):
    """One timed oracle forward: x' = H_i S_i x, the dense W_v (dequantised base, + residual
    for the verify), z = x' W_v^T, y = S_o H_o z.  The layer's codes are the oracle's own
    quantisation of ``real_weights`` when given, else seeded random codes in the stored
    ranges (the forward does the same work whatever the code values).  Returns seconds."""
    import numpy as np
    from nested_bit_quantized_gb300 import synth
    from oracle import nest_oracle as O
    s_o, s_i = synth.sign_pair(M, K, seed)
    if real_weights is not None:
        layer = O.quantize_layer(real_weights, s_o, s_i, bits)
    else:
        bc, bs, rc, rs = synth.uniform_codes(M, K, bits, seed)
        layer = {"base_codes": bc, "base_scales": bs.view(np.float16), "resid_codes": rc,
                 "resid_scales": rs.view(np.float16)}
    _, x = synth.activations(T, K, seed + 7)
    t0 = time.perf_counter()
    O.forward(layer, s_o, s_i, x, verify)
    return time.perf_counter() - t0


def oracle_sample_main(spec):
    """Runs in a fresh process (``--oracle-sample``): times the oracle on the cases of
    ``spec`` and prints one JSON line.  spec: {"cases": [[name, M, K, bits, T, verify], ...],
    "cap_s": seconds}."""
    out, spent = [], 0.0
    for name, M, K, bits, T, verify, rows in spec["cases"]:
        if spent > spec.get("cap_s", 60.0):
            out.append({"case": name, "skipped": "time cap"})
            continue
        s = _oracle_case(rows, K, bits, T, bool(verify), 11)
        spent += s
        s_full = s * M / rows                     # the forward's work is linear in the rows
        by = lin_bytes(M, K, T, bits if verify else 0)
        rec = {"case": name, "M": M, "K": K, "bits": bits, "T": T, "verify": bool(verify),
               "seconds": s_full, "GBps": by / s_full / 1e9}
        if rows != M:
            rec["sampled_rows"] = rows
        out.append(rec)
    print(json.dumps({"threads": os.environ.get("OMP_NUM_THREADS", "all"), "cases": out}), flush=True)


def run_oracle_subprocess(cases, threads, cap_s):
    env = dict(os.environ)
    if threads:
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[k] = str(threads)
    spec = json.dumps({"cases": cases, "cap_s": cap_s})
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", spec], env=env,
                           capture_output=True, text=True, timeout=cap_s * 3 + 120)
        for line in r.stdout.splitlines()[::-1]:
            if line.startswith("{"):
                return json.loads(line)
        return {"error": (r.stderr or "no output")[-300:]}
    except Exception as e:                        # a baseline that cannot run is reported, not fatal
        return {"error": str(e)[-300:]}


def cpu_baseline_section():
    """The oracle timed per linear on the host cores (a per-workload sample): the
    single linear (T = 1 draft, T = 1 and 16 verify), the MLP triplet, the Gemma-12B-like
    layer and one 31B-class layer (T = 1 draft, T = 16 verify), all threads; the single
    linear again on one thread; the 60-layer cycle extrapolated from the 31B-class layer."""
    from nested_bit_quantized_gb300 import synth
    cases = [["single_4096 draft T=1", 4096, 4096, 8, 1, 0, 4096],
             ["single_4096 verify T=1", 4096, 4096, 8, 1, 1, 4096],
             ["single_4096 verify T=16", 4096, 4096, 8, 16, 1, 4096]]
    for l in synth.WORKLOADS["mlp_triplet_4b"].linears:
        cases.append([f"mlp_triplet_4b {l.name} verify T=16", l.M, l.K, 7, 16, 1, l.M])
    for l in synth.WORKLOADS["decoder_12b"].linears:    # a quarter of the rows, scaled
        cases.append([f"decoder_12b {l.name} verify T=16 (b=8; the oracle's work is the same at b=6/7)",
                      l.M, l.K, 8, 16, 1, l.M // 4])
    for l in synth.WORKLOADS["decoder_31b"].linears:    # an eighth of the rows, scaled
        cases.append([f"decoder_31b {l.name} draft T=1", l.M, l.K, 8, 1, 0, l.M // 8])
        cases.append([f"decoder_31b {l.name} verify T=16", l.M, l.K, 8, 16, 1, l.M // 8])
    allt = run_oracle_subprocess(cases, None, 90.0)
    one = run_oracle_subprocess(cases[:3], 1, 30.0)
    res = {"cores": cpu_cores(), "cpu_model": cpu_model(), "all_threads": allt, "single_thread": one,
           "codes": "seeded random codes in the stored ranges (the forward's work does not depend on them)",
           "sampling": "decoder_12b linears timed on M/4 rows and decoder_31b on M/8 rows, scaled to M (the "
                       "forward's work is linear in the rows); the others at full size"}
    try:
        d31 = {c["case"]: c["seconds"] for c in allt["cases"] if "seconds" in c and c["case"].startswith("decoder_31b")}
        draft = sum(v for k, v in d31.items() if "draft" in k)
        verify = sum(v for k, v in d31.items() if "verify" in k)
        if len(d31) == 14:
            res["stack_31b_cycle_extrapolated"] = {
                "seconds": 60 * (8 * draft + verify), "how": "EXTRAPOLATED: 60 layers x (8 draft passes at T=1 + "
                "1 verify pass at T=16) from one 31B-class layer's seven linears, not measured"}
    except Exception:
        pass
    return res


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the default workload's linear (its own quantisation
    of the same synthetic weights, untimed), one verify forward at T = 16 per step."""
    if rank != 0:
        return
    from nested_bit_quantized_gb300 import synth
    lin = synth.WORKLOADS[WORKLOAD].linears[0]
    W = synth.weights(lin.M, lin.K, lin.w_seed, lin.outliers)
    import numpy as np
    from oracle import nest_oracle as O
    s_o, s_i = synth.sign_pair(lin.M, lin.K, lin.sign_seed)
    layer = O.quantize_layer(W, s_o, s_i, BITS)
    _, x = synth.activations(T_VERIFY, lin.K, synth.WORKLOADS[WORKLOAD].x_seed)
    secs = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        O.forward(layer, s_o, s_i, x, True)
        if i >= args.warmup:
            secs.append(time.perf_counter() - t0)
    sec = sum(secs) / len(secs)
    by = lin_bytes(lin.M, lin.K, T_VERIFY, BITS)
    value = by / sec / 1e9
    what = (f"oracle verify forward (numpy fp64) of one {lin.M}x{lin.K} b={BITS} linear at T={T_VERIFY} per step, "
            f"quantisation untimed; threads as numpy uses them")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "bits": BITS, "T": T_VERIFY, "sample": what},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(), "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": what},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# The pages' own figures for this path, with their hardware (context, not a target): the CPU
# residual kernel of the 2-bit-base post (feedman.me/posts/wZBTJ, Results, "CPU residual kernel").
PAGES_CONTEXT = {"cpu_residual_kernel_ms_per_pass": {"T=1": 108, "T=4": 127, "T=8": 116, "T=16": 125, "T=32": 204},
                 "working_set_GB": 4.29, "ram_GBps": "33-38",
                 "hardware": "AMD Ryzen 9 9950X, 16 threads, DDR5 (int8 residual tiles, AVX-512)",
                 "note": "no page reports a GPU timing of the split; context only"}

WORKLOAD_DESC = ("single_4096: one linear 4096x4096, 2-bit base + 8-bit residual, g128 fp16 scales, "
                 "N(0,0.02^2) weights with 1% columns x8, bf16 N(0,1) activations")


# ----------------------------------------------------------------------------
# GPU helpers
# ----------------------------------------------------------------------------

class nvtx_range:
    """An NVTX range named after a timed region (lets a profiler keep to that region's
    launches); a no-op where NVTX is unavailable."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        try:
            import torch
            torch.cuda.nvtx.range_push(self.name)
            self.on = True
        except Exception:
            self.on = False
        return self

    def __exit__(self, *a):
        if self.on:
            import torch
            torch.cuda.nvtx.range_pop()


class Timer:
    """CUDA-graph capture and timing on one stream: warm-up replays, then events around the
    timed replays with a barrier and synchronise on both sides, the clocks sampled during
    the timed region, the max over ranks."""

    def __init__(self, stream, dev, dist, gpu_index):
        self.stream, self.dev, self.dist, self.gpu = stream, dev, dist, gpu_index
        self.clocks = {}

    def graph(self, fn):
        import torch
        with torch.cuda.stream(self.stream):
            fn()                                  # the first launches configure the kernels
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
        torch.cuda.synchronize()
        return g

    def time(self, name, g, reps, warm=3, min_s=0.0):
        """ms per replay.  With min_s, reps grows until the region lasts about min_s seconds."""
        import torch
        for _ in range(warm):
            g.replay()
        torch.cuda.synchronize()
        if min_s > 0.0:
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(self.stream)
            with torch.cuda.stream(self.stream):
                g.replay()
            e.record(self.stream)
            torch.cuda.synchronize()
            est = max(s.elapsed_time(e) * 1e-3, 1e-6)
            reps = max(reps, min(int(min_s / est) + 1, 100000))
        if self.dist is not None:
            self.dist.barrier()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(self.gpu) as clk, nvtx_range(name):
            with torch.cuda.stream(self.stream):
                s.record(self.stream)
                for _ in range(reps):
                    g.replay()
                e.record(self.stream)
            torch.cuda.synchronize()
        self.clocks[name] = clk.summary()
        return max_over_ranks(s.elapsed_time(e) / reps, self.dist, self.dev)


def build_layers(linears, bits, copies, dev, seed_offset=0):
    """Quantise and pack `copies` distinct copies of `linears` on the device: a list (one
    entry per copy) of lists of nest.Layer."""
    import torch
    from nested_bit_quantized_gb300 import nest, synth
    out, work = [], None
    for c in range(copies):
        row = []
        for lin in linears:
            seed = lin.w_seed + 1000 * c + seed_offset
            W = synth.weights_device(lin.M, lin.K, seed, lin.outliers, dev)
            s_o, s_i = synth.sign_pair(lin.M, lin.K, lin.sign_seed + 2 * c)
            if work is None or work.numel() < lin.M * lin.K:
                work = torch.empty(lin.M * lin.K, dtype=torch.float64, device=dev)
            so, si = torch.from_numpy(s_o).to(dev), torch.from_numpy(s_i).to(dev)
            q = nest.quantize(W, so, si, bits, work=work[:lin.M * lin.K].view(lin.M, lin.K))
            row.append(nest.pack(q["base_codes"], q["base_scales"], q["resid_codes"], q["resid_scales"], bits, so, si))
            del W, q
        out.append(row)
    del work
    torch.cuda.synchronize()
    return out


def xop_for(layer, T, seed, dev):
    """Rotated fp16 operand of seeded bf16 activations for `layer` at T tokens."""
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import nest, synth
    b, _ = synth.activations(T, layer.K, seed)
    x = torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    xo = nest.new_xop(layer.K, T, dev)
    nest.rotate(x, layer.sign_in, 0, x_op=xo)
    return xo


def grouped(layers, xops, zs, T, verify, max_group=64):
    """Grouped GEMM launches over a flat list of layers (at most max_group per launch)."""
    from nested_bit_quantized_gb300 import nest
    for i in range(0, len(layers), max_group):
        nest.gemm_group(layers[i:i + max_group], xops[i:i + max_group], T, verify, zs=zs[i:i + max_group])


# ----------------------------------------------------------------------------
# default line: the single 4096 x 4096 linear
# ----------------------------------------------------------------------------

def single_section(args, dev, timer, world):
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import nest, synth

    wl = synth.WORKLOADS[WORKLOAD]
    lin = wl.linears[0]
    M, K = lin.M, lin.K
    rank = int(os.environ.get("RANK", "0"))
    C = args.copies
    copies = build_layers(wl.linears, BITS, C, dev, seed_offset=100_000 * rank)
    layers = [row[0] for row in copies]
    xops = {T: xop_for(layers[0], T, wl.x_seed + T, dev) for T in set(SWEEP_T) | set(PREFILL_T)}
    zs = {T: [torch.zeros((T, M), dtype=torch.float32, device=dev) for _ in range(C)] for T in set(SWEEP_T) | set(PREFILL_T)}

    def gfn(T, verify):
        return lambda: grouped(layers, [xops[T]] * C, zs[T], T, verify)

    def per_launch_fn(T, verify):
        def fn():
            for L, z in zip(layers, zs[T]):
                nest.gemm(L, xops[T], T, verify, z=z)
        return fn

    hbm, src = peaks()
    by = lambda T, verify: lin_bytes(M, K, T, BITS if verify else 0)
    rec = lambda ms, T, verify: {"us_per_layer": ms * 1e3 / C, "GBps": by(T, verify) / (ms * 1e-3 / C) / 1e9,
                                 "frac_of_measured_hbm": by(T, verify) / (ms * 1e-3 / C) / 1e9 / hbm,
                                 "frac_of_8TBps": by(T, verify) / (ms * 1e-3 / C) / 1e9 / NOMINAL_HBM_GBS}

    # the timed steps: one verify pass at T = 16 over the copies, one grouped launch
    g_main = timer.graph(gfn(T_VERIFY, True))
    ms_main = timer.time("main", g_main, args.steps, args.warmup)
    ms_sustained = timer.time("sustained", g_main, args.steps, 3, min_s=1.0)
    out = {"main_ms": ms_main, "verify_T16": rec(ms_main, T_VERIFY, True),
           "sustained": dict(rec(ms_sustained, T_VERIFY, True), clocks=timer.clocks["sustained"])}
    del g_main
    g = timer.graph(gfn(T_DRAFT, True))
    out["verify_T1"] = rec(timer.time("verify_T1", g, 20, min_s=0.3), T_DRAFT, True)
    g = timer.graph(gfn(T_DRAFT, False))
    out["draft_T1"] = rec(timer.time("draft_T1", g, 20, min_s=0.3), T_DRAFT, False)
    out["t16_over_t1"] = out["verify_T16"]["us_per_layer"] / out["verify_T1"]["us_per_layer"]
    # one launch per linear (a CUDA graph of C launches)
    pl = {}
    for name, T, verify in (("verify_T16", T_VERIFY, True), ("verify_T1", T_DRAFT, True), ("draft_T1", T_DRAFT, False)):
        g = timer.graph(per_launch_fn(T, verify))
        pl[name] = rec(timer.time("per_launch_" + name, g, 20, min_s=0.3), T, verify)
    pl["t16_over_t1"] = pl["verify_T16"]["us_per_layer"] / pl["verify_T1"]["us_per_layer"]
    out["per_launch"] = pl
    # sweep over T (grouped GEMM launches)
    sweep = []
    if not args.no_sweep:
        for T in SWEEP_T:
            r = {"T": T}
            for verify in (False, True):
                g = timer.graph(gfn(T, verify))
                ms = timer.time(f"sweep_{'verify' if verify else 'draft'}_T{T}", g, 20, min_s=0.2)
                key = "verify" if verify else "draft"
                r[key + "_us"] = ms * 1e3 / C
                r[key + "_GBps"] = by(T, verify) / (ms * 1e-3 / C) / 1e9
                r[key + "_frac_of_measured_hbm"] = r[key + "_GBps"] / hbm
                r[key + "_frac_of_8TBps"] = r[key + "_GBps"] / NOMINAL_HBM_GBS
            sweep.append(r)
        tpk, tsrc = tensor_peak()
        pre = []
        for T in PREFILL_T:
            g = timer.graph(gfn(T, True))
            ms = timer.time(f"prefill_T{T}", g, 10, min_s=0.2)
            tf = 2.0 * M * K * T / (ms * 1e-3 / C) / 1e12
            pre.append({"T": T, "verify_us": ms * 1e3 / C, "TFLOPs": tf, "frac_of_tensor_peak": tf / tpk,
                        "tensor_peak": tpk, "peak_source": tsrc})
        out["prefill"] = pre
    out["sweep"] = sweep
    nest.error_check()

    # the whole linear (rotation in, GEMM, rotation out): draft T = 1 then verify T = 16, per copy,
    # the copies' whole linears, LINEAR_GROUP per nest_linear_group call (one call for 32 copies)
    xs = {}
    for T in (T_DRAFT, T_VERIFY):
        b, _ = synth.activations(T, K, wl.x_seed + 100 + T)
        xs[T] = torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    ys = {T: [torch.empty((T, M), dtype=torch.float32, device=dev) for _ in range(C)] for T in (T_DRAFT, T_VERIFY)}
    LG = min(C, LINEAR_GROUP)
    calls = (C + LG - 1) // LG
    scratch = torch.empty(max(nest.linear_group_scratch_bytes(layers[:LG], T) for T in (T_DRAFT, T_VERIFY)),
                          dtype=torch.uint8, device=dev)

    def layer_pass(T, verify, xlist=None):
        for i in range(0, C, LG):
            n = min(LG, C - i)
            nest.linear_group(layers[i:i + n], xlist[i:i + n] if xlist else [xs[T]] * n, verify,
                              ys=ys[T][i:i + n], scratch=scratch)

    g = timer.graph(lambda: (layer_pass(T_DRAFT, False), layer_pass(T_VERIFY, True)))
    ms = timer.time("layer_step", g, 20, min_s=0.3)
    step_bytes = C * (by(T_DRAFT, False) + by(T_VERIFY, True))
    out["layer_step"] = {"ms": ms, "GBps": step_bytes / (ms * 1e-3) / 1e9, "launches": 2 * 3 * calls,
                         "what": "per copy: rotation in, draft GEMV, rotation out at T=1, then rotation in, "
                                 f"verify GEMM, rotation out at T=16 (nest_linear_group over {LG} copies)"}
    del g
    nest.error_check()

    # end to end through the C entry point: every step copies its inputs in from pinned host
    # memory, runs one nest_linear_group call over the copies (verify, T = 16) and copies every
    # output back, all inside the timed region; no graph.  With --e2e-buffers 2 consecutive steps
    # alternate over two streams, each with its own device and host buffers, so one step's copies
    # overlap the neighbouring step's kernels (copy engines and SMs at once), as a serving loop
    # that uploads the next batch while the current one runs would.
    hx = torch.empty((C, T_VERIFY, K), dtype=torch.bfloat16, pin_memory=True)
    for c in range(C):
        b, _ = synth.activations(T_VERIFY, K, wl.x_seed + 500 + c)
        hx[c].copy_(torch.from_numpy(b.view(np.int16)).view(torch.bfloat16))
    stream = timer.stream
    nb = 2 if args.e2e_buffers == 2 else 1
    streams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(nb - 1)]
    bufs = []
    for _ in range(nb):
        xin = torch.empty((C, T_VERIFY, K), dtype=torch.bfloat16, device=dev)
        yout = torch.empty((C, T_VERIFY, M), dtype=torch.float32, device=dev)
        hy = torch.empty((C, T_VERIFY, M), dtype=torch.float32, pin_memory=True)
        sc = torch.empty(nest.linear_group_scratch_bytes(layers[:LG], T_VERIFY), dtype=torch.uint8, device=dev)
        bufs.append((xin, yout, hy, [xin[c] for c in range(C)], [yout[c] for c in range(C)], sc))

    def e2e_once(step):
        xin, yout, hy, xl, yl, sc = bufs[step % nb]
        with torch.cuda.stream(streams[step % nb]):
            xin.copy_(hx, non_blocking=True)
            for i in range(0, C, LG):
                n = min(LG, C - i)
                nest.linear_group(layers[i:i + n], xl[i:i + n], True, ys=yl[i:i + n], scratch=sc)
            hy.copy_(yout, non_blocking=True)

    for i in range(max(3, args.warmup)):
        e2e_once(i)
    torch.cuda.synchronize()
    if timer.dist is not None:
        timer.dist.barrier()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(timer.gpu) as clk, nvtx_range("e2e"):
        s.record(stream)
        for st in streams[1:]:
            st.wait_stream(stream)              # nothing of the timed steps starts before s
        for i in range(args.steps):
            e2e_once(i)
        for st in streams[1:]:
            stream.wait_stream(st)              # ... or ends after e
        e.record(stream)
        torch.cuda.synchronize()
    timer.clocks["e2e"] = clk.summary()
    e2e_ms = max_over_ranks(s.elapsed_time(e) / args.steps, timer.dist, dev)
    ok = all(bool(torch.isfinite(b[2]).all().item()) for b in bufs)
    out["e2e"] = {"value": world * C * by(T_VERIFY, True) / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                  "ms_per_step": e2e_ms, "h2d_bytes_per_step": C * T_VERIFY * K * 2,
                  "d2h_bytes_per_step": C * T_VERIFY * M * 4, "outputs_finite": ok, "buffers": nb,
                  "what": f"per step: the {C} pinned bf16 input blocks copied in (one copy), {calls} "
                          f"nest_linear_group call(s) (rotation in, verify GEMM, rotation out; ctypes into the C "
                          f"entry point), all {C} fp32 outputs copied back to pinned host memory (one copy); "
                          f"no CUDA graph" + ("; consecutive steps alternate over two streams with their own "
                                              "buffers, so one step's copies overlap the next step's kernels"
                                              if nb == 2 else "")}
    nest.error_check()
    out["copies"] = C
    out["bytes_per_linear_verify_T16"] = by(T_VERIFY, True)
    del copies, layers
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------
# Gemma-12B-like decoder layer, residual 6/7/8 bits, T = 16 (GEMM only)
# ----------------------------------------------------------------------------

def decoder12_section(args, dev, timer, copies=2):
    import torch
    from nested_bit_quantized_gb300 import synth
    wl = synth.WORKLOADS["decoder_12b"]
    lins = wl.linears
    hbm, _ = peaks()
    T = T_VERIFY
    res = {"workload": "decoder_12b: q 4096x3840, k/v 2048x3840, o 3840x4096, gate/up 15360x3840, down 3840x15360; "
                       f"T={T}; {copies} distinct layers; GEMM only",
           "by_bits": {}}
    for bits in (6, 7, 8):
        layers = build_layers(lins, bits, copies, dev)
        xo = {l.K: xop_for(layers[0][i], T, wl.x_seed + l.K, dev) for i, l in enumerate(lins)}
        zs = [[torch.zeros((T, l.M), dtype=torch.float32, device=dev) for l in lins] for _ in range(copies)]
        groups = [(0, 1, 2), (3,), (4, 5), (6,)]           # q/k/v, o, gate/up, down: one launch each
        lb = sum(lin_bytes(l.M, l.K, T, bits) for l in lins)

        def layer_launches():
            for c in range(copies):
                for grp in groups:
                    grouped([layers[c][k] for k in grp], [xo[lins[k].K] for k in grp], [zs[c][k] for k in grp], T, True)

        def all_in_one():
            flat = [L for row in layers for L in row]
            grouped(flat, [xo[L.K] for L in flat], [z for row in zs for z in row], T, True)

        g = timer.graph(layer_launches)
        ms = timer.time(f"decoder_12b_b{bits}", g, 20, min_s=0.3) / copies
        g2 = timer.graph(all_in_one)
        ms2 = timer.time(f"decoder_12b_b{bits}_one_launch", g2, 20, min_s=0.3) / copies
        res["by_bits"][str(bits)] = {
            "bpw": bits_per_weight(bits), "bytes_per_layer": lb,
            "four_launches": {"us_per_layer": ms * 1e3, "GBps": lb / (ms * 1e-3) / 1e9,
                              "frac_of_measured_hbm": lb / (ms * 1e-3) / 1e9 / hbm,
                              "frac_of_8TBps": lb / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS},
            "one_launch": {"us_per_layer": ms2 * 1e3, "GBps": lb / (ms2 * 1e-3) / 1e9,
                           "frac_of_measured_hbm": lb / (ms2 * 1e-3) / 1e9 / hbm,
                           "frac_of_8TBps": lb / (ms2 * 1e-3) / 1e9 / NOMINAL_HBM_GBS}}
        del g, g2, layers, zs
        torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------
# Qwen-4B-like MLP triplet, b = 7: the step (draft T=1 + verify T=16, rotations included) and a sweep
# ----------------------------------------------------------------------------

def triplet_section(args, dev, timer, copies=12, codec="l2"):
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import nest, synth
    wl = synth.WORKLOADS["mlp_triplet_4b"]
    w4w8 = codec == "w4w8"
    bits = 7
    DC, VC = (40, 48) if w4w8 else (0, bits)
    layers, work = [], None
    for c in range(copies):
        trip = []
        for lin in wl.linears:
            W = synth.weights_device(lin.M, lin.K, lin.w_seed + 1000 * c, lin.outliers, dev)
            s_o, s_i = synth.sign_pair(lin.M, lin.K, lin.sign_seed + 2 * c)
            if work is None or work.numel() < lin.M * lin.K:
                work = torch.empty(lin.M * lin.K, dtype=torch.float64, device=dev)
            so, si = torch.from_numpy(s_o).to(dev), torch.from_numpy(s_i).to(dev)
            if w4w8:
                q = nest.quantize_w4w8(W, so, si, work=work[:lin.M * lin.K].view(lin.M, lin.K))
                trip.append(nest.pack_w4w8(q["q4"], q["s4"], q["qr"], so, si))
            else:
                q = nest.quantize(W, so, si, bits, work=work[:lin.M * lin.K].view(lin.M, lin.K))
                trip.append(nest.pack(q["base_codes"], q["base_scales"], q["resid_codes"], q["resid_scales"], bits,
                                      so, si))
            del W, q
        layers.append(trip)
    del work
    xs = {}
    for T in (T_DRAFT, T_VERIFY):
        for K in sorted({l.K for l in wl.linears}):
            b, _ = synth.activations(T, K, wl.x_seed + K + T)
            xs[(K, T)] = torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    groups = [[0, 1], [2]]                        # (gate, up) read the same input; down alone
    scratch = torch.zeros(max(nest.linear_group_scratch_bytes([layers[0][k] for k in grp], T)
                              for grp in groups for T in (T_DRAFT, T_VERIFY)), dtype=torch.uint8, device=dev)
    ys = {(k, T): torch.empty((T, wl.linears[k].M), dtype=torch.float32, device=dev)
          for k in range(3) for T in (T_DRAFT, T_VERIFY)}

    def run_pass(T, verify):
        for trip in layers:
            for grp in groups:
                nest.linear_group([trip[k] for k in grp], [xs[(trip[k].K, T)] for k in grp], verify,
                                  ys=[ys[(k, T)] for k in grp], scratch=scratch)

    g = timer.graph(lambda: (run_pass(T_DRAFT, False), run_pass(T_VERIFY, True)))
    ms = timer.time(f"triplet_step_{codec}", g, 20, min_s=0.3)
    step_bytes = sum(lin_bytes(L.M, L.K, T_DRAFT, DC) + lin_bytes(L.M, L.K, T_VERIFY, VC)
                     for trip in layers for L in trip)
    hbm, _ = peaks()
    res = {"workload": ("mlp_triplet_4b: gate/up 9728x2560, down 2560x9728, "
                        + ("BitNest W4 base + 4-bit refinement" if w4w8 else "2-bit base + 7-bit residual")
                        + f"; {copies} copies"),
           "step": {"ms": ms, "GBps": step_bytes / (ms * 1e-3) / 1e9,
                    "what": "draft pass T=1 then verify pass T=16, each linear rotation in, GEMM, rotation out; "
                            "gate+up grouped, down alone"}}
    del g
    sweep = []
    n_lin = 3 * copies
    flat = [L for trip in layers for L in trip]
    for T in (1, 4, 8, 16, 32, 64):
        xo = {K: nest.new_xop(K, T, dev) for K in {l.K for l in wl.linears}}
        for k, l in enumerate(layers[0]):
            b, _ = synth.activations(T, l.K, wl.x_seed + 7 * T + k)
            nest.rotate(torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16), l.sign_in, 0, x_op=xo[l.K])
        zz = [torch.zeros((T, L.M), dtype=torch.float32, device=dev) for L in flat]
        r = {"T": T}
        for verify in (False, True):
            def fn():
                for i in range(copies):
                    for grp in groups:
                        ks = [3 * i + k for k in grp]
                        nest.gemm_group([flat[k] for k in ks], [xo[flat[k].K] for k in ks], T, verify,
                                        zs=[zz[k] for k in ks])
            gg = timer.graph(fn)
            per = timer.time(f"triplet_{codec}_{'v' if verify else 'd'}{T}", gg, 20, min_s=0.2) * 1e3 / n_lin
            b_ = sum(lin_bytes(L.M, L.K, T, VC if verify else DC) for L in layers[0]) / 3
            key = "verify" if verify else "draft"
            r[key + "_us"] = per
            r[key + "_GBps"] = b_ / (per * 1e-6) / 1e9
            if verify:
                r["verify_frac_of_measured_hbm"] = r[key + "_GBps"] / hbm
            del gg
        sweep.append(r)
    res["sweep_gemm_only"] = sweep
    # the same GEMMs with the copies' independent linears of one shape in one launch: all gate
    # and up linears (24), then all down linears (12)
    by_shape = [[L for trip in layers for L in trip[:2]], [trip[2] for trip in layers]]
    grouped_rates = {}
    for T, verify in ((1, False), (16, True)):
        xo = {K: nest.new_xop(K, T, dev) for K in {l.K for l in wl.linears}}
        for k, l in enumerate(layers[0]):
            b, _ = synth.activations(T, l.K, wl.x_seed + 11 * T + k)
            nest.rotate(torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16), l.sign_in, 0, x_op=xo[l.K])
        zz = [[torch.zeros((T, L.M), dtype=torch.float32, device=dev) for L in grp] for grp in by_shape]

        def fn_grouped():
            for grp, zg in zip(by_shape, zz):
                grouped(grp, [xo[L.K] for L in grp], zg, T, verify)
        gg = timer.graph(fn_grouped)
        per = timer.time(f"triplet_{codec}_grouped_{'v' if verify else 'd'}{T}", gg, 20, min_s=0.2) * 1e3 / n_lin
        b_ = sum(lin_bytes(L.M, L.K, T, VC if verify else DC) for L in layers[0]) / 3
        grouped_rates[f"{'verify' if verify else 'draft'}_T{T}"] = {
            "us_per_linear": per, "GBps": b_ / (per * 1e-6) / 1e9, "frac_of_measured_hbm": b_ / (per * 1e-6) / 1e9 / hbm}
        del gg
    res["grouped_gemm_only"] = dict(grouped_rates, what="the 24 gate/up linears of the 12 copies in one launch, "
                                                         "then the 12 down linears in one")
    nest.error_check()
    del layers, flat
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------
# chained 31B-class layers: one layer (draft T=1, verify T=64) or the 60-layer speculative cycle
# ----------------------------------------------------------------------------

def stack_section(args, dev, timer, cycle=True, n_layers=60):
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import chain, nest, synth
    stack = synth.stack_31b(n_layers)
    bits = 8
    t0 = time.time()
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
    prep_s = time.time() - t0
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

    tag = "stack_31b" if cycle else "decoder_31b"
    g = timer.graph(step)
    ms = timer.time(tag + "_cycle", g, max(3, min(args.steps, 10)), 3)
    del g
    g = timer.graph(lambda: run_pass(T_d, False))
    ms_d = timer.time(tag + "_draft_pass", g, 5, 3, min_s=0.2)
    del g
    g = timer.graph(lambda: run_pass(T_v, True))
    ms_v = timer.time(tag + "_verify_pass", g, 5, 3, min_s=0.2)
    del g
    nest.error_check()

    def lbytes(T, verify):
        return sum(lin_bytes(l.M, l.K, T, bits if verify else 0) for layer in stack for l in layer)

    step_bytes = gamma * lbytes(T_d, False) + lbytes(T_v, True)
    hbm, _ = peaks()
    res = {"workload": (f"31B-class stack, {n_layers} chained layers (q 8192x5376, k/v 4096x5376, o 5376x8192, "
                        f"gate/up 21504x5376, down 5376x21504), 2-bit base + 8-bit residual; step = "
                        f"{gamma} draft pass(es) at T={T_d} + 1 verify pass at T={T_v}"),
           "resident_weight_GB": sum(weight_bytes(l.M, l.K, bits) for layer in stack for l in layer) / 1e9,
           "cycle_ms": ms, "cycle_GBps": step_bytes / (ms * 1e-3) / 1e9,
           "ideal_ms_at_measured_hbm": step_bytes / (hbm * 1e9) * 1e3,
           "draft_pass": {"T": T_d, "ms": ms_d, "us_per_layer": 1e3 * ms_d / n_layers,
                          "GBps": lbytes(T_d, False) / (ms_d * 1e-3) / 1e9},
           "verify_pass": {"T": T_v, "ms": ms_v, "us_per_layer": 1e3 * ms_v / n_layers,
                           "GBps": lbytes(T_v, True) / (ms_v * 1e-3) / 1e9,
                           "frac_of_measured_hbm": lbytes(T_v, True) / (ms_v * 1e-3) / 1e9 / hbm},
           # per layer: four grouped GEMMs and two launches per glue (the k and v output
           # rotations ride in the q glue's first launch)
           "launches_per_cycle": (gamma + 1) * (1 + 12 * n_layers), "prep_seconds": prep_s}
    res["cycle_over_ideal"] = ms / res["ideal_ms_at_measured_hbm"]
    del bufs, lin
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------
# nested KV4/KV8 cache: decode attention at a 31B-class head configuration
# ----------------------------------------------------------------------------

def kv_section(args, dev, timer):
    import torch
    from nested_bit_quantized_gb300 import nest
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
        gr = timer.graph(fn)
        us = timer.time("kv_" + name, gr, max(10, args.steps), min_s=0.2) * 1e3 / copies
        hi = min(rn, L) if view == 4 else L
        per_pos = (64 + 2) * 2 if view == 4 else (128 + 2) * 2        # K and V rows read per position
        by = Hkv * ((L - hi) * per_pos + hi * (128 + 2) * 2) + T * Hq * d * (2 + 4)
        recs.append({"case": name, "T": T, "us_per_layer": us, "GBps": by / (us * 1e-6) / 1e9,
                     "frac_of_measured_hbm": by / (us * 1e-6) / 1e9 / hbm, "bytes": by})
        del gr
    nest.error_check()
    return {"workload": f"KV4/KV8 nested cache, Hq={Hq}, Hkv={Hkv}, d={d}, context {L}, {copies} layers' caches "
                        f"alternating", "cases": recs}


# ----------------------------------------------------------------------------
# the 4096 x 4096 linear split over the ranks by output rows (one all-gather of z per linear)
# ----------------------------------------------------------------------------

def shard_rows_section(args, dev, timer, world, rank):
    """Every rank holds its whole-tile row shard of each copy (views of the packed buffers),
    rotates the replicated input, runs the verify GEMM on its rows, and the ranks all-gather
    the rotated-basis blocks (NCCL) before the reorder and the output rotation, which every
    rank runs.  Total work is fixed as ranks are added (strong scaling); the value counts
    the whole job's algorithmic bytes."""
    import numpy as np
    import torch
    from nested_bit_quantized_gb300 import nest, shard, synth

    wl = synth.WORKLOADS[WORKLOAD]
    lin = wl.linears[0]
    C = args.copies
    copies = build_layers(wl.linears, BITS, C, dev)
    lins = [shard.RowShardedLinear(row[0], world, rank, group=None) for row in copies]
    b, _ = synth.activations(T_VERIFY, lin.K, wl.x_seed + 900)
    x = torch.from_numpy(b.view(np.int16)).to(dev).view(torch.bfloat16)
    ys = [torch.empty((T_VERIFY, lin.M), dtype=torch.float32, device=dev) for _ in range(C)]

    def step():
        for L, y in zip(lins, ys):
            L.forward(x, True, y=y)

    if world == 1:                            # no collective: the step is captured in a CUDA graph
        g = timer.graph(step)
        ms = timer.time("shard_rows", g, args.steps, args.warmup)
        how = "CUDA graph"
    else:                                     # the all-gathers run eagerly on the current stream
        for _ in range(max(3, args.warmup)):
            step()
        torch.cuda.synchronize()
        timer.dist.barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()
        with ClockSampler(timer.gpu) as clk, nvtx_range("shard_rows"):
            s.record(cur)
            for _ in range(args.steps):
                step()
            e.record(cur)
            torch.cuda.synchronize()
        timer.clocks["shard_rows"] = clk.summary()
        ms = max_over_ranks(s.elapsed_time(e) / args.steps, timer.dist, dev)
        how = "eager launches"
    nest.error_check()
    by = C * lin_bytes(lin.M, lin.K, T_VERIFY, BITS)
    plan = shard.RowPlan(lin.M, world)
    return {"workload": f"{WORKLOAD_DESC}; each of {world} ranks holds its {plan.count(rank)}-row shard "
                        f"(tiles of 128 rows) of {C} copies; per linear: rotation in, verify GEMM on the "
                        f"rank's rows, one all-gather of z, reorder, rotation out ({how})",
            "ms_per_step": ms, "GBps": by / (ms * 1e-3) / 1e9, "us_per_linear": 1e3 * ms / C,
            "rows_per_rank": plan.Mp, "bytes_per_step": by}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args, rank, world):
    import torch
    from nested_bit_quantized_gb300 import build as nb
    from nested_bit_quantized_gb300 import nest

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    nb.build()
    nest.load()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(device=dev)
    timer = Timer(stream, dev, dist, local)
    wall0 = time.time()
    hbm, src = peaks()

    if args.workload != WORKLOAD:
        if args.workload == "kv_31b":
            sec = kv_section(args, dev, timer)
            value, unit, metric = sec["cases"][0]["GBps"], "GB/s", "nested KV-cache decode attention, effective HBM GB/s per layer"
        elif args.workload == "decoder_12b":
            sec = decoder12_section(args, dev, timer)
            value, unit, metric = sec["by_bits"]["8"]["four_launches"]["GBps"], "GB/s", METRIC
        elif args.workload == "single_4096_rows":
            sec = shard_rows_section(args, dev, timer, world, rank)
            value, unit, metric = sec["GBps"], "GB/s", ("whole linear (rotation, verify GEMM on row shards, all-gather, "
                                                        "output rotation) at T=16, effective HBM GB/s of the job")
        elif args.workload == "mlp_triplet_4b":
            sec = triplet_section(args, dev, timer, copies=args.copies_triplet, codec=args.codec)
            value, unit, metric = sec["step"]["GBps"], "GB/s", "draft T=1 + verify T=16 step, effective HBM GB/s"
        else:
            cyc = args.workload == "stack_31b"
            sec = stack_section(args, dev, timer, cycle=cyc, n_layers=args.layers if args.layers else (60 if cyc else 1))
            value, unit, metric = sec["cycle_GBps"], "GB/s", "speculative cycle (draft passes + verify pass), effective HBM GB/s"
        if rank == 0:
            scaling = "strong" if args.workload == "single_4096_rows" else "weak"
            par = f"rows x{world}" if args.workload == "single_4096_rows" else f"replicas x{world}"
            line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "higher_is_better": True,
                    "scaling": scaling, "dtype": "f16", "data": "synthetic",
                    "config": {"workload": args.workload, "parallelism": par}, "section": sec,
                    "clocks_by_region": timer.clocks, "wall_s": time.time() - wall0}
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return

    main = single_section(args, dev, timer, world)
    extras = {}
    if world == 1 and not args.quick:
        for name, fn in (("decoder_12b", lambda: decoder12_section(args, dev, timer)),
                         ("decoder_31b", lambda: stack_section(args, dev, timer, cycle=False, n_layers=1)),
                         ("mlp_triplet_4b", lambda: triplet_section(args, dev, timer, copies=args.copies_triplet)),
                         ("stack_31b", lambda: stack_section(args, dev, timer, cycle=True, n_layers=60))):
            if name == "stack_31b" and args.no_stack:
                continue
            t0 = time.time()
            try:
                extras[name] = fn()
            except Exception as e:                # an extra workload that fails is reported, not fatal
                extras[name] = {"error": repr(e)[-400:]}
            extras[name]["wall_s"] = time.time() - t0
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_section()
        try:
            c1 = next(c for c in cpu["all_threads"]["cases"] if c["case"] == "single_4096 verify T=16")
            cpu = dict(value=c1["GBps"], unit="GB/s", cores=cpu["cores"], kind="oracle",
                       sample="oracle verify forward of one 4096x4096 b=8 linear at T=16 (numpy fp64, all threads); "
                              "per-config table in per_config", **{"per_config": cpu})
        except Exception:
            cpu = {"value": None, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle", "per_config": cpu}

    if rank == 0:
        v16 = main["verify_T16"]
        ms_step = main["main_ms"]
        C = main["copies"]
        line = {
            "metric": METRIC, "value": world * v16["GBps"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": WORKLOAD_DESC, "T": T_VERIFY, "bits": BITS, "copies": C,
                       "step": f"one verify GEMM pass at T={T_VERIFY} over {C} distinct copies, one grouped launch",
                       "resident_weight_GB": C * weight_bytes(4096, 4096, BITS) / 1e9,
                       "l2": f"inputs larger than L2: {C} distinct quantised copies "
                             f"({C * weight_bytes(4096, 4096, BITS) / 1e6:.0f} MB) streamed per step",
                       "accumulate": "f32", "parallelism": f"replicas x{world}"},
            "us_per_layer_T16": v16["us_per_layer"], "us_per_layer_T1": main["verify_T1"]["us_per_layer"],
            "t16_over_t1": main["t16_over_t1"],
            "verify_T16": v16, "verify_T1": main["verify_T1"], "draft_T1": main["draft_T1"],
            "per_launch": main["per_launch"], "sustained": main["sustained"],
            "roofline": {"bound": "hbm", "kernel": f"k_nest_gemm<{BITS},16> (verify, T=16, grouped over {C} linears)",
                         "achieved": v16["GBps"], "peak": hbm, "unit": "GB/s", "frac": v16["GBps"] / hbm,
                         "peak_source": src, "frac_of_8TBps": v16["GBps"] / NOMINAL_HBM_GBS,
                         "traffic": (ncu_traffic() * C) if ncu_traffic() else None,
                         "traffic_unit": f"DRAM bytes per launch of {C} linears (ncu)",
                         "traffic_per_linear": ncu_traffic(),
                         "algorithmic_bytes_per_launch": C * main["bytes_per_linear_verify_T16"],
                         "algorithmic_bytes_per_linear": main["bytes_per_linear_verify_T16"]},
            "sweep": main["sweep"], "prefill": main.get("prefill", []),
            "pages_context": PAGES_CONTEXT,
            "layer_step": main["layer_step"],
            "extras": extras,
            "cpu_baseline": cpu,
            "e2e": main["e2e"],
            "gpu_launches": args.steps * ((C + 63) // 64),
            "clocks": timer.clocks.get("sustained"),
            "clocks_main": timer.clocks.get("main"),
            "clocks_by_region": timer.clocks,
            "wall_s": time.time() - wall0,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    if len(sys.argv) >= 3 and sys.argv[1] == "--oracle-sample":
        oracle_sample_main(json.loads(sys.argv[2]))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nest", choices=["nest", "reference"])
    ap.add_argument("--copies", type=int, default=32, help="distinct copies of the 4096x4096 linear (>= 4x L2)")
    ap.add_argument("--copies-triplet", type=int, default=12)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-buffers", type=int, default=2, choices=[1, 2],
                    help="end-to-end leg: 2 = consecutive steps alternate over two streams and buffer sets")
    ap.add_argument("--no-sweep", action="store_true", help="skip the GEMM-only sweep over T")
    ap.add_argument("--no-stack", action="store_true", help="skip the 60-layer 31B-class cycle in the default line")
    ap.add_argument("--quick", action="store_true", help="default workload only, no extra workloads")
    ap.add_argument("--codec", default="l2", choices=["l2", "w4w8"],
                    help="--workload mlp_triplet_4b: l2 (2-bit base + 7-bit residual) or w4w8 (BitNest W4/W8)")
    ap.add_argument("--context", type=int, default=32768, help="context length of --workload kv_31b")
    ap.add_argument("--kv-case", type=int, default=None, choices=[0, 1, 2, 3],
                    help="--workload kv_31b: one case only (0 KV4 draft, 1 KV4 + Recent-1024, 2 KV8 verify "
                         "T=16, 3 KV8 draft)")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=[WORKLOAD, "single_4096_rows", "decoder_12b", "mlp_triplet_4b", "decoder_31b", "stack_31b",
                             "kv_31b"],
                    help="single_4096 (default, the metric's workload) or one extra workload alone")
    ap.add_argument("--layers", type=int, default=0, help="layers of the 31B-class stack (default 1 or 60)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus))) if "RANK" in os.environ else 1
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world)


if __name__ == "__main__":
    main()

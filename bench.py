"""Benchmark of the GB300 MoE feed-forward layer.

One step = one pass of the whole layer on one batch: router logits, routing,
dispatch, grouped gate/up (SwiGLU) and down GEMMs, shared expert, combine,
and the full backward (moe_backward).  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2] [--fwd-only]
  python bench.py --impl reference ...   (the CPU oracle, timed on host cores)

Timing: W untimed warm-up steps, then K steps between a barrier and a
device synchronise; each step is bracketed by CUDA events on the launch
stream, and a 256 MB buffer is written before each step (outside its events)
to flush the 129 MB L2.  Multi-GPU (torchrun): independent replicas, no
data-path collective; time = max over ranks; value = all ranks' tokens / time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s fwd & fwd+bwd; grouped-GEMM % of GB300 bf16 tensor peak"
WORKLOAD_NAMES = {
    1: "tiny MoE layer: T=256, d=64, 4 routed top-2 + 1 shared, SwiGLU 128",
    2: "KochiLLM-shaped MoE layer: T=32768, d=1536, 4 routed top-2 + 1 shared, SwiGLU 3072",
    3: "Qwen3-MoE-shaped packed layer: T=65536 (60293 real + PAD tail), d=512, 8 experts "
       "top-2, hidden 768",
    4: "DeepSeekMoE-style layer: T=16384, d=2048, 64 routed top-6 + 2 shared, hidden 1408, "
       "Zipf(1.1) selection bias",
    5: "training-step layer: T=32768, d=1024, 128 experts top-8, hidden 768",
}


def workload_shape(args):
    from mixture_experts_ffn_02_gb300 import synth
    s = synth.shape(args.config)
    if args.tokens:
        T = args.tokens
        T_real = None if s.T_real is None else round(s.T_real * T / s.T)
        s = synth.scaled(s, T=T, T_real=T_real)
    return s


def peaks():
    """(bf16 TFLOP/s burst, bf16 TFLOP/s sustained, HBM GB/s, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                d["hbm_gbs"], "measured")
    return 1900.0, 1700.0, 6800.0, "fallback"


def gemm_flops(s):
    """Algorithmic FLOPs (2 per multiply-add) per step, real tokens only."""
    Tr = s.T_real if s.T_real is not None else s.T
    routed = 2 * Tr * s.k * s.d * s.H * 3     # gate, up, down
    shared = 2 * Tr * s.d * s.Hs_total * 3
    return routed, shared


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
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
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def launches_per_step(s, fwd_only):
    """Kernels of this library launched per step (by router path and shared expert)."""
    small = s.E in (4, 8, 16) and s.d * s.E * 4 + (s.d // 8) * 16 <= 96 * 1024
    tc = not small and s.E % 32 == 0
    shared = s.Hs_total > 0
    # small E: the streamed fused router behind its zeroing kernel (2 launches;
    # MOE_ROUTER_STREAM=0 selects the one-kernel register form); otherwise the
    # logits kernel and the route kernel
    router_route = (1 if os.environ.get("MOE_ROUTER_STREAM") == "0" else 2) if small else 2
    router_bwd = 5 if tc else (2 if small else 3)
    fwd = router_route + 3 + 1 + 1 + (2 if shared else 1)     # shared: combine in its down GEMM
    bwd = 1 + 1 + 1 + 2 + (4 if shared else 1) + router_bwd   # shared: dx sum in its dx GEMM
    return fwd if fwd_only else fwd + bwd


def aggregate_ranks(ms_local, tokens_per_step, steps, world, dist=None, device="cpu"):
    """Whole-job throughput of independent replicas: the timed region's
    length is the maximum over ranks; value = tokens of all ranks / that time.
    Returns (ms_max, tokens_per_second)."""
    import torch
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    if dist is not None and world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, tokens_per_step * steps * world / (ms_max / 1e3)


def run_ours(args):
    import torch
    import torch.distributed as dist

    from mixture_experts_ffn_02_gb300 import binding, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    s = workload_shape(args)
    training = not args.fwd_only
    inp = synth.make_inputs(s, seed=rank, with_grad=True)
    lay = binding.Layer.create(s, training=training, device=f"cuda:{local}")
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    dY = dev["dY"]
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=f"cuda:{local}")

    kev = {n: [] for n in ("router_route", "permute", "gate_up", "combine")}
    if s.Hs_total:
        del kev["combine"]

    def timed(name, fn):
        if name not in kev:
            fn()
            return
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        kev[name].append((a, b))

    def step(record):
        # with a shared expert the combine runs in its down GEMM (shared_combine)
        lay.step(dY if training else None, timed if record else None)

    for _ in range(args.warmup):
        flush.zero_()
        step(False)
    torch.cuda.synchronize()
    if lay.status() != 0:
        raise RuntimeError(f"device status {lay.status()} after warm-up")

    clocks = Clocks(local)
    ev = []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for _ in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(True)
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    status = lay.status()
    if status != 0:
        raise RuntimeError(f"device status {status} in the timed region")
    ms = sum(a.elapsed_time(b) for a, b in ev)
    k_ms = {n: sum(a.elapsed_time(b) for a, b in v) / len(v) for n, v in kev.items()}
    gu_ms = k_ms["gate_up"]
    ms_max, value = aggregate_ranks(ms, s.T, args.steps, world,
                                    dist if world > 1 else None, f"cuda:{local}")
    ms_per_step = ms_max / args.steps

    # fwd-only rate of the same layer (reported beside the fwd+bwd headline)
    fwd_rate = None
    if training:
        fe = []
        for _ in range(max(3, args.steps // 2)):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            lay.forward()
            b.record(stream)
            fe.append((a, b))
        torch.cuda.synchronize()
        fms = statistics.median(a.elapsed_time(b) for a, b in fe)
        fwd_rate = s.T / (fms / 1e3)

    # inference forward (nothing saved for a backward), with the rows copied
    # into x_perm and, as a memory-saving variant, gathered by the gate/up
    # GEMM from x (no x_perm)
    def infer_rate(gather):
        li = binding.Layer.create(s, training=False, gather=gather, device=f"cuda:{local}")
        li.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                      dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
        for _ in range(3):
            li.forward()
        ev_i = []
        for _ in range(max(3, args.steps // 4)):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            li.forward()
            b.record(stream)
            ev_i.append((a, b))
        torch.cuda.synchronize()
        if li.status() != 0:
            raise RuntimeError(f"device status {li.status()} in the inference forward")
        return s.T / (statistics.median(a.elapsed_time(b) for a, b in ev_i) / 1e3)
    fwd_infer_rate = fwd_infer_gather_rate = None
    if not args.no_inference:
        fwd_infer_rate = infer_rate(False)
        fwd_infer_gather_rate = infer_rate(True)

    # inference forward with MXFP8 routed experts (weights quantised once,
    # outside the timed region, as they are between weight updates)
    def mx_run():
        if s.d % 128 or s.H % 128:
            return None
        lm = binding.Layer.create(s, training=False, device=f"cuda:{local}")
        lm.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                      dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
        lm.mx_alloc()
        qa = torch.cuda.Event(enable_timing=True)
        qb = torch.cuda.Event(enable_timing=True)
        qa.record(stream)
        lm.mx_quantize_weights()
        qb.record(stream)
        for _ in range(3):
            lm.mx_forward()
        n = max(3, args.steps // 4)
        ev_f, ev_g, ev_d = [], [], []
        for _ in range(n):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            lm.mx_forward()
            b.record(stream)
            ev_f.append((a, b))
        for _ in range(n):         # the same steps one call at a time, GEMMs timed
            flush.zero_()
            lm.router_route()
            lm.mx_permute()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
            lm.mx_gate_up()
            e[1].record(stream)
            lm.mx_down()
            e[2].record(stream)
            lm.shared_combine()
            ev_g.append((e[0], e[1]))
            ev_d.append((e[1], e[2]))
        torch.cuda.synchronize()
        if lm.status() != 0:
            raise RuntimeError(f"device status {lm.status()} in the MX forward")
        med = lambda v: statistics.median(a.elapsed_time(b) for a, b in v)
        return med(ev_f), med(ev_g), med(ev_d), qa.elapsed_time(qb)
    mx = None if args.no_inference else mx_run()

    # the MXFP8 training step (routed experts' forward and data-gradient
    # products on block-scaled MMAs; weight gradients and shared expert in
    # bf16), weights quantised once outside the timed region
    def mx_train_run():
        if s.d % 256 or s.H % 128:
            return None
        lt = binding.Layer.create(s, training=True, device=f"cuda:{local}")
        lt.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                      dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
        lt.mx_alloc()
        lt.mx_quantize_weights()
        for _ in range(3):
            lt.mx_step(dev["dY"])
        ev_t = []
        for _ in range(max(3, args.steps // 4)):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            lt.mx_step(dev["dY"])
            b.record(stream)
            ev_t.append((a, b))
        torch.cuda.synchronize()
        if lt.status() != 0:
            raise RuntimeError(f"device status {lt.status()} in the MX training step")
        ms_t = statistics.median(a.elapsed_time(b) for a, b in ev_t)
        del lt
        torch.cuda.empty_cache()
        return ms_t
    mx_train_ms = None if (args.no_inference or not training) else mx_train_run()
    f8_measured = None if mx is None else fp8_gemm_peak(local)

    e2e = run_e2e(args, s, inp, lay, training, local)

    bf16_burst, bf16_sustained, hbm_peak, peak_src = peaks()
    # the burst figure for a kernel timed in a short region; the sustained
    # (power-capped) one only when the timed steps ran back to back for
    # seconds, as the sustained figure was measured
    timed_s = ms / 1e3
    if timed_s >= 2.0:
        bf16_peak = bf16_sustained
        peak_label = f"{peak_src} sustained bf16 (timed region {timed_s:.2f} s >= 2 s)"
    else:
        bf16_peak = bf16_burst
        peak_label = f"{peak_src} burst bf16 (timed region {timed_s:.2f} s < 2 s)"
    routed, shared = gemm_flops(s)
    gu_flops = routed * 2 / 3                                  # gate + up of the routed experts
    gu_tflops = gu_flops / (gu_ms / 1e3) / 1e12
    layer_flops = (routed + shared) * (3 if training else 1)
    layer_tflops = layer_flops / (ms_per_step / 1e3) / 1e12
    traffic = load_traffic(args.config)

    mx_out = None
    if mx is not None:
        if f8_measured is not None:
            f8_peak = f8_measured
            f8_src = "measured here: cuBLASLt e4m3 GEMM 8192^3 (torch._scaled_mm), best of 10"
        else:
            f8_peak = 2 * bf16_sustained     # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25)
            f8_src = f"{peak_src} sustained bf16 x 2 (nominal fp8/bf16 ratio)"
        mx_f_ms, mx_g_ms, mx_d_ms, mx_q_ms = mx
        g_tf = gu_flops / (mx_g_ms / 1e3) / 1e12
        d_tf = routed / 3 / (mx_d_ms / 1e3) / 1e12
        mx_out = {
            "fwd_tokens_per_s": round(s.T / (mx_f_ms / 1e3), 1),
            "dtype": "e4m3 x e4m3 (UE8M0 per-32 scales), fp32 accumulate",
            "peak_tflops": round(f8_peak, 1),
            "peak_source": f8_src,
            "fp8_nominal_2x_sustained_bf16_tflops": round(2 * bf16_sustained, 1),
            "gate_up": {"avg_launch_ms": round(mx_g_ms, 4), "achieved_tflops": round(g_tf, 1),
                        "frac": round(g_tf / f8_peak, 4)},
            "down": {"avg_launch_ms": round(mx_d_ms, 4), "achieved_tflops": round(d_tf, 1),
                     "frac": round(d_tf / f8_peak, 4)},
            "weight_quantise_ms": round(mx_q_ms, 4),
        }

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": WORKLOAD_NAMES[args.config] + (" fwd" if args.fwd_only
                                                              else " fwd+bwd"),
                   "config_id": args.config, "T": s.T, "T_real": s.T_real, "d": s.d, "E": s.E, "k": s.k,
                   "H": s.H, "n_shared": s.n_shared, "H_shared": s.H_shared,
                   "parallelism": f"replicas x{world}",
                   "l2": "256 MB buffer written before each step, outside its events"},
        "fwd_tokens_per_s": None if fwd_rate is None else round(fwd_rate, 1),
        "fwd_inference_tokens_per_s": (None if fwd_infer_rate is None
                                       else round(fwd_infer_rate, 1)),
        "fwd_inference_gathered_tokens_per_s": (None if fwd_infer_gather_rate is None
                                                else round(fwd_infer_gather_rate, 1)),
        "fwd_inference_mxfp8": mx_out,
        "train_mxfp8": None if mx_train_ms is None else {
            "fwd_bwd_tokens_per_s": round(s.T / (mx_train_ms / 1e3), 1),
            "ms_per_step": round(mx_train_ms, 4),
            "vs_bf16_step": round(ms_per_step / mx_train_ms, 4),
            "what": "routed experts' forward and data-gradient GEMMs on e4m3 (UE8M0 per-32 "
                    "scales); weight gradients, shared expert and router in bf16/fp32",
            "timing": "median of steps, each bracketed by events after a 256 MB L2 flush"},
        "layer_tflops": round(layer_tflops, 1),
        "layer_frac_of_burst_peak": round(layer_tflops / bf16_burst, 4),
        "layer_frac_of_sustained_peak": round(layer_tflops / bf16_sustained, 4),
        "roofline": {"kernel": "grouped gate/up GEMM + SwiGLU (tcgen05)", "bound": "tensor",
                     "achieved": round(gu_tflops, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": round(gu_tflops / bf16_peak, 4),
                     "peak_source": peak_label,
                     "frac_of_burst_peak": round(gu_tflops / bf16_burst, 4),
                     "frac_of_sustained_peak": round(gu_tflops / bf16_sustained, 4),
                     "algorithmic_flops_per_launch": gu_flops,
                     "avg_launch_ms": round(gu_ms, 4), "traffic": traffic},
        "hbm_kernels": hbm_kernels(s, k_ms, hbm_peak),
        "gpu_launches": launches_per_step(s, args.fwd_only) * args.steps,
        "e2e": e2e,
        "clocks": clk,
    }
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(args, s)
    print(json.dumps(out), flush=True)


def fp8_gemm_peak(local):
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput of the vendor library on
    this GPU (torch._scaled_mm, per-tensor scales, 8192^3, best of 10), in
    TFLOP/s: the denominator of the MXFP8 kernels' fractions.  None if the
    library call is not available."""
    import torch
    try:
        n = 8192
        dev = f"cuda:{local}"
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = float("inf")
        for _ in range(10):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        return 2.0 * n ** 3 / (best / 1e3) / 1e12
    except Exception:
        return None


def hbm_bytes(s):
    """Algorithmic bytes of the memory-bound forward calls, each byte of the
    tensors they must read or write counted once, in the layouts the library
    stores (out_perm bf16, s_out fp32; PAD rows of the segments are not
    counted)."""
    T, Tr, d, E, k = s.T, (s.T_real if s.T_real is not None else s.T), s.d, s.E, s.k
    M = Tr * k
    valid = T if s.T_real is not None else 0
    bias = 4 * E if s.zipf_bias > 0 else 0
    return {
        # x and W_r in; logits, topk_idx and gates out; valid mask and bias in
        "router_route": T * d * 2 + d * E * 4 + T * E * 4 + T * k * 8 + valid + bias,
        # x rows in, x_perm rows out, topk_idx in, perm + inv out
        "permute": Tr * d * 2 + M * d * 2 + T * k * 4 + M * 4 + T * k * 4,
        # out_perm (bf16) + s_out (fp32) in, inv + gates in, y out
        "combine": M * d * 2 + (Tr * d * 4 if s.Hs_total else 0) + T * k * 8 + T * d * 2,
    }


def hbm_kernels(s, k_ms, hbm_peak):
    out = {}
    for name, nbytes in hbm_bytes(s).items():
        if name not in k_ms:
            continue
        ms = k_ms[name]
        gbs = nbytes / (ms / 1e3) / 1e9
        out[name] = {"avg_launch_ms": round(ms, 4), "algorithmic_bytes": nbytes,
                     "achieved_gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / hbm_peak, 4)}
    return out


def load_traffic(cfg):
    """DRAM bytes per launch of the gate/up kernel from the committed ncu
    summary for this workload, or None if there is none or if the GEMM source
    changed since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", f"gate_up_traffic_cfg{cfg}.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        h = hashlib.sha256()
        for f in ("moe_gemm.cu", "moe_common.cuh"):
            h.update(open(os.path.join(ROOT, "mixture_experts_ffn_02_gb300", "csrc", f),
                          "rb").read())
        if h.hexdigest() != d.get("source_sha256"):
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


def run_e2e(args, s, inp, lay, training, local):
    """The same layer step through moe_forward/moe_backward with host
    buffers, driven the way a training loop would: every step copies its
    inputs x and dY in from pinned host memory and its results y, aux and dx
    back out, all inside the timed region.  Uploads run on one stream and
    downloads on another (the two directions use separate copy engines),
    ordered by events: x, dY, y and dx are double-buffered, so the next
    step's uploads overlap this step's compute and this step's downloads
    overlap the next step's."""
    import torch
    hx = inp["x"].pin_memory()
    hdy = inp["dY"].pin_memory()
    hy = torch.empty_like(inp["x"]).pin_memory()
    hdx = torch.empty_like(inp["x"]).pin_memory()
    haux = torch.empty(4, dtype=torch.float32).pin_memory()
    main = torch.cuda.current_stream()
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()
    xbuf = [lay.bufs["x"], torch.empty_like(lay.bufs["x"])]
    dybuf = [torch.empty_like(lay.bufs["x"]), torch.empty_like(lay.bufs["x"])]
    dxbuf = [lay.grads["dx"], torch.empty_like(lay.bufs["x"])] if training else [None, None]
    ybuf = [lay.bufs["y"], torch.empty_like(lay.bufs["y"])]
    ev = lambda: torch.cuda.Event()            # noqa: E731
    in_ready, step_done, dx_out, y_out = [None, None], [None, None], [None, None], [None, None]

    def upload(i):
        j = i % 2
        if step_done[j] is not None:
            up.wait_event(step_done[j])        # step i-2 no longer reads these buffers
        with torch.cuda.stream(up):
            xbuf[j].copy_(hx, non_blocking=True)
            if training:
                dybuf[j].copy_(hdy, non_blocking=True)
        in_ready[j] = ev()
        in_ready[j].record(up)

    def step(i):
        j = i % 2
        main.wait_event(in_ready[j])
        if dx_out[j] is not None:
            main.wait_event(dx_out[j])         # step i-2's dx download is done
        if y_out[j] is not None:
            main.wait_event(y_out[j])          # step i-2's y download is done
        lay.bufs["x"] = xbuf[j]
        lay.bufs["y"] = ybuf[j]
        if training:
            lay.grads["dx"] = dxbuf[j]
        lay.forward()
        haux.copy_(lay.bufs["aux"], non_blocking=True)   # 16 bytes, ordered on main
        y_ready = ev()
        y_ready.record(main)
        down.wait_event(y_ready)
        with torch.cuda.stream(down):
            hy.copy_(ybuf[j], non_blocking=True)
        y_out[j] = ev()
        y_out[j].record(down)
        if training:
            lay.backward(dybuf[j])
        step_done[j] = ev()
        step_done[j].record(main)
        upload(i + 2)                          # the step after next reuses these buffers
        if training:
            down.wait_event(step_done[j])
            with torch.cuda.stream(down):
                hdx.copy_(dxbuf[j], non_blocking=True)
            dx_out[j] = ev()
            dx_out[j].record(down)

    i = 0
    upload(0)
    upload(1)
    for _ in range(2):
        step(i)
        i += 1
    main.wait_stream(up)
    main.wait_stream(down)
    torch.cuda.synchronize()
    n = max(3, args.steps // 2)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(main)
    for _ in range(n):
        step(i)
        i += 1
    main.wait_stream(up)                       # every copy issued in the timed steps is done
    main.wait_stream(down)
    b.record(main)
    b.synchronize()
    lay.bufs["x"] = xbuf[0]
    lay.bufs["y"] = ybuf[0]
    if training:
        lay.grads["dx"] = dxbuf[0]
    ms = a.elapsed_time(b) / n
    nb = s.T * s.d * 2
    return {"value": round(s.T / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": nb * (2 if training else 1),
            "d2h_bytes_per_step": nb * (2 if training else 1) + 16,
            "ms_per_step": round(ms, 4)}


_SAMPLE_INPUTS = {}


def oracle_sample(s, n_tok, training):
    """Time the CPU oracle on the first n_tok tokens of the workload (the
    seeded inputs are drawn once per sample size, outside the timing)."""
    from mixture_experts_ffn_02_gb300 import synth
    from oracle import moe_oracle as O
    key = (s.name, s.T, n_tok)
    if key not in _SAMPLE_INPUTS:
        _SAMPLE_INPUTS.clear()
        sub = synth.scaled(s, T=n_tok, T_real=None if s.T_real is None
                           else min(n_tok, s.T_real))
        _SAMPLE_INPUTS[key] = synth.make_inputs(sub, seed=0, with_grad=True)
    inp = _SAMPLE_INPUTS[key]
    t0 = time.perf_counter()
    fwd = O.forward(inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
                    inp["Ws_down"], k=s.k, bias=inp["bias"], valid=inp["valid"],
                    norm_topk=bool(s.norm_topk))
    if training:
        O.backward(inp["x"], inp["Wr"], inp["W_gu"], inp["W_down"], inp["Ws_gu"],
                   inp["Ws_down"], fwd, inp["dY"], norm_topk=bool(s.norm_topk),
                   aux_coef=s.aux_coef)
    return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def oracle_sample_tokens(s, training, target_s=3.0):
    """Tokens per oracle sample: doubled from 512 until one sample takes at
    least target_s (so the oracle's fixed per-call cost -- widening the
    weights to fp64 -- is amortised as it is on a full batch).  Returns
    (tokens, seconds of the last sample)."""
    n = min(512, s.T)
    dt = oracle_sample(s, n, training)
    while dt < target_s and n < s.T:
        n = min(s.T, n * 2)
        dt = oracle_sample(s, n, training)
    return n, dt


def host_desc():
    return {"nproc": os.cpu_count(), "cpu_model": cpu_model()}


def cpu_baseline(args, s, repeats=3):
    """The oracle as it stands on the host cores: the same sample size as
    the reference arm (oracle_sample_tokens), timed `repeats` times (about
    10-20 s of CPU work in all)."""
    training = not args.fwd_only
    n, _ = oracle_sample_tokens(s, training)
    t = sum(oracle_sample(s, n, training) for _ in range(repeats))
    return {"value": round(n * repeats / t, 2), "unit": "tokens/s", "cores": blas_threads(),
            "kind": "oracle", **host_desc(),
            "sample": f"first {n} of {s.T} tokens, same shapes, numpy fp64 "
                      f"{'fwd+bwd' if training else 'fwd'}; {repeats} runs, {t:.1f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = workload_shape(args)
    training = not args.fwd_only
    # the cpu_baseline leg's sample size (about 3 s per pass), so both report
    # one rate -- smaller when the step count would make the run longer than
    # about 150 s of oracle work (a sample ends at most twice its target)
    n, _ = oracle_sample_tokens(s, training,
                                target_s=min(3.0, 75.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(s, n, training)
    dt = sum(oracle_sample(s, n, training) for _ in range(args.steps))
    v = n * args.steps / dt
    sample = f"first {n} of {s.T} tokens per step, same shapes, numpy fp64"
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD_NAMES[args.config] + (" fwd" if args.fwd_only
                                                                  else " fwd+bwd"),
                      "config_id": args.config, "sample": sample},
           "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": blas_threads(),
                            "kind": "oracle", **host_desc(), "sample": sample},
           "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_mx_train_only(args):
    """The MXFP8 training step alone on one GPU: weights quantised once, W
    untimed steps, then K steps each bracketed by events after an L2 flush.
    Prints one line with the median step time and its tokens/s."""
    import statistics

    import torch

    from mixture_experts_ffn_02_gb300 import binding, synth
    s = workload_shape(args)
    inp = synth.make_inputs(s, seed=0, with_grad=True)
    lay = binding.Layer.create(s, training=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    lay.set_inputs(dev["x"], dev["Wr"], dev["W_gu"], dev["W_down"], dev["Ws_gu"],
                   dev["Ws_down"], bias=dev["bias"], valid=dev["valid"])
    lay.mx_alloc()
    lay.mx_quantize_weights()
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        flush.zero_()
        lay.mx_step(dev["dY"])
    ev = []
    for _ in range(args.steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        lay.mx_step(dev["dY"])
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    if lay.status() != 0:
        raise RuntimeError(f"device status {lay.status()} in the MX training step")
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    print(json.dumps({"mx_train_step": WORKLOAD_NAMES[args.config], "T": s.T,
                      "steps": args.steps, "ms_per_step_median": round(ms, 4),
                      "tokens_per_s": round(s.T / (ms / 1e3), 1)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--tokens", type=int, default=None,
                    help="smaller token count of the same layer (profiling cases)")
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-inference", action="store_true",
                    help="skip the inference-forward rates (e.g. for a launch list of the step)")
    ap.add_argument("--mx-train-only", action="store_true",
                    help="time only the MXFP8 training step (for launch lists and profiles); "
                         "prints its own line, not the benchmark's")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.mx_train_only:
        run_mx_train_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Benchmark of the NVFP4 sparse-MoE FFN layer on one B300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode_b1|decode_b64|stack|prefill]
                    [--impl ours|reference] [--no-cpu-baseline]

Default workload (decode_b1): batch-1 decode through one Flint-shaped MoE layer
(d_model 2048, 256 routed experts top-6 + 1 shared, d_ff 512, NVFP4 weights
quantised from N(0, 0.02), fp32 router 2048x256), one fresh bf16 token per
step.  Sixteen independently seeded copies of the layer (7.3 GB, far above the
126 MB L2) are used round-robin, so every step's weights come from HBM.

A step is one whole pass of the layer (router, top-6, bucketing, experts,
combine) over one token; steps are serialised, as in real decode.  K steps are
captured in one CUDA graph and timed with CUDA events on the launching stream,
bracketed by a barrier and a device synchronise.  Rank 0 prints one JSON line.

``--impl reference`` times the CPU oracle (the only reference this method
has) on a bounded sample of the same workload and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

EXPERT_BYTES = 3 * 2048 * 512 // 2 + 3 * 2048 * 512 // 16      # 1,769,472 B per Flint expert
ROUTER_BYTES = 2048 * 256 * 4


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def _build_layers(lib, torch, synth, n_copies, max_tokens, bias=None, seed0=0):
    s = synth.FLINT
    E = s.n_experts
    ctxs = []
    for i in range(n_copies):
        wg, wu, wd = synth.expert_weights(s, synth.layer_seed(seed0 + i), device="cuda")
        router = synth.router_weight(s, synth.router_seed(seed0 + i), device="cuda")
        weights = {"router": router, "router_bias": None if bias is None else bias.cuda()}
        keep = []
        for name, w in (("gate", wg), ("up", wu), ("down", wd)):
            c, sc, ts = lib.quantize(w)
            keep.append((c, sc, ts))
            weights[name] = dict(codes=c[:E], scales=sc[:E], tensor_scale=ts[:E])
            weights["shared_" + name] = dict(codes=c[E:], scales=sc[E:], tensor_scale=ts[E:])
        torch.cuda.synchronize()
        cfg = dict(d_model=s.d_model, n_experts=E, top_k=s.top_k, d_ff=s.d_ff, n_shared=s.n_shared,
                   d_ff_shared=s.d_ff, max_tokens=max_tokens, weight_format=0)
        ctxs.append(lib.moe_init(cfg, weights, device=torch.cuda.current_device()))
        del wg, wu, wd, keep, weights
        torch.cuda.empty_cache()
    return ctxs


def run_ours(args):
    import torch
    import nvfp4_expert_ffn_gemv_b300 as lib
    import synth

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    s = synth.FLINT
    K, W = args.steps, args.warmup
    T = 64 if args.workload == "decode_b64" else 1
    n_copies = int(os.environ.get("MOE_BENCH_COPIES", "16"))
    bias = synth.zipf_bias(s, seed=4242) if T == 64 else None
    ctxs = _build_layers(lib, torch, synth, n_copies, max_tokens=T, bias=bias, seed0=100 * rank)
    stream = torch.cuda.Stream()
    n_tok = (K + W) * T
    xb, _ = synth.tokens(s, n_tok, seed=synth.token_seed(rank), device="cuda")
    x = xb.view(K + W, T, s.d_model)
    y = torch.empty_like(x)

    def step(i, profile=None):
        if profile is not None:
            lib.moe_set_profile_events(ctxs[i % n_copies], *profile)
        lib.moe_forward_decode(ctxs[i % n_copies], x[i], T, y[i], 0, stream)
        if profile is not None:
            lib.moe_set_profile_events(ctxs[i % n_copies], None, None)

    with torch.cuda.stream(stream):
        for i in range(K, K + W):                # warm-up on inputs the timed steps never use
            step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(K):
            step(i)
    # per-kernel timing graph: events around the expert kernels of every step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:                               # events are created lazily at their first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=stream):
        for i in range(K):
            step(i, profile=ev[i])
    for st in ctxs:
        assert lib.moe_get_device_status(st) == 0

    def timed(graph):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):          # replay() launches on the current stream
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return a.elapsed_time(b)

    with torch.cuda.stream(stream):
        for _ in range(2):
            g.replay()                            # graph warm-up
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = timed(g)
        with torch.cuda.stream(stream):
            gp.replay()
        torch.cuda.synchronize()
        kern_ms = sorted(a.elapsed_time(b) for a, b in ev)
    if world > 1:
        t = torch.tensor([ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # end to end: host (pinned) token in, host result out, every step
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    xd = torch.empty((T, s.d_model), dtype=torch.bfloat16, device="cuda")
    yd = torch.empty_like(xd)
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=stream):
        for i in range(K):
            xd.copy_(xh[i], non_blocking=True)
            lib.moe_forward_decode(ctxs[i % n_copies], xd, T, yd, 0, stream)
            yh[i].copy_(yd, non_blocking=True)
    with torch.cuda.stream(stream):
        ge.replay()
    torch.cuda.synchronize()
    e2e_ms = timed(ge)
    if world > 1:
        t = torch.tensor([e2e_ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())

    launches = K * lib.moe_kernels_per_forward(ctxs[0], T, 0)
    for c in ctxs:
        lib.moe_destroy(c)
    if rank != 0:
        return
    tok = world * K * T
    value = tok / (ms / 1e3)
    kmed = kern_ms[len(kern_ms) // 2]
    kavg = sum(kern_ms) / len(kern_ms)
    peak, peak_kind = _peaks()
    if T == 1:
        alg_bytes = 7 * EXPERT_BYTES
    else:
        alg_bytes = None
    achieved = alg_bytes / (kavg / 1e3) / 1e9 if alg_bytes else None
    line = {
        "metric": "MoE decode tok/s (batch-%d, one Flint-shaped NVFP4 MoE layer)" % T,
        "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (nvfp4 weights, bf16 activations)", "data": "synthetic",
        "config": {"workload": args.workload, "d_model": 2048, "n_experts": 256, "top_k": 6, "n_shared": 1,
                   "d_ff": 512, "tokens_per_step": T, "layer_copies": n_copies,
                   "l2": "16 rotating layer copies (7.3 GB > 126 MB L2); no weight re-read from L2",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "expert_kernels_us": {"avg": round(kavg * 1e3, 3), "median": round(kmed * 1e3, 3)},
        "roofline": {"kernel": "expert kernels (gate/up+SwiGLU, down)", "bound": "hbm",
                     "achieved": round(achieved, 1) if achieved else None, "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4) if achieved else None,
                     "peak_kind": peak_kind, "algorithmic_bytes_per_launch": alg_bytes, "traffic": None},
        "e2e": {"value": round(tok / (e2e_ms / 1e3), 1), "unit": "tok/s",
                "h2d_bytes_per_step": T * s.d_model * 2, "d2h_bytes_per_step": T * s.d_model * 2},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, T, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
def _blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        return max([i.get("num_threads", 1) for i in info] or [1])
    except Exception:
        return 1


def cpu_baseline(workload: str, T: int, budget_s: float = 15.0):
    """Time the oracle as it stands on a bounded sample of the decode workload:
    tokens one at a time (T = 1) or one batch of T, weights of the chosen experts
    quantised by the oracle beforehand (untimed, as moe_init is)."""
    import numpy as np
    import synth
    from oracle import moe as omoe

    s = synth.FLINT
    router = synth.router_weight(s, synth.router_seed(0)).numpy()
    bias = synth.zipf_bias(s, seed=4242).numpy() if T > 1 else None
    n_steps = 8 if T == 1 else 1
    xb, x = synth.tokens(s, n_steps * T, seed=synth.token_seed(0))
    x = x.double().numpy().reshape(n_steps, T, s.d_model)
    cache = {}

    def weights_for(experts):
        for e in experts:
            if e not in cache:
                wg, wu, wd = synth.expert_weights_one(s, synth.layer_seed(0), int(e))
                lw = omoe.quantize_layer(wg.numpy()[None], wu.numpy()[None], wd.numpy()[None],
                                         np.zeros((s.d_model, 1), np.float32))
                cache[e] = (lw.gate, lw.up, lw.down)
        n = s.n_all
        tens = []
        for m in range(3):
            c = np.zeros((n,) + cache[experts[0]][m].codes.shape[1:], np.uint8)
            sc = np.zeros((n,) + cache[experts[0]][m].scales.shape[1:], np.uint8)
            ts = np.zeros((n,), np.float32)
            for e in experts:
                t = cache[e][m]
                c[e], sc[e], ts[e] = t.codes[0], t.scales[0], t.ts[0]
            tens.append(omoe.NVFP4Tensor(c, sc, ts))
        return omoe.LayerWeights(router=router, bias=bias, gate=tens[0], up=tens[1], down=tens[2])

    layers = []
    for i in range(n_steps):
        idx = omoe.top_k(omoe.router_logits(x[i], router, bias), s.top_k)
        layers.append(weights_for(sorted(set(idx.ravel().tolist()) | {s.n_experts})))
    t0 = time.perf_counter()
    done = 0
    for i in range(n_steps):
        omoe.moe_layer(layers[i], x[i], s.top_k, s.n_shared)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done * T / dt, 3), "unit": "tok/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"{done} decode step(s) of {T} token(s) through one Flint-shaped layer "
                      f"(numpy fp64 oracle, experts dequantised per step), {dt:.1f} s"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    T = 64 if args.workload == "decode_b64" else 1
    cb = cpu_baseline(args.workload, T, budget_s=args.cpu_budget)
    line = {"impl": "reference", "metric": "MoE decode tok/s (batch-%d, one Flint-shaped NVFP4 MoE layer)" % T,
            "value": cb["value"], "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "d_model": 2048, "n_experts": 256, "top_k": 6, "n_shared": 1,
                       "d_ff": 512, "tokens_per_step": T},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode_b1", choices=["decode_b1", "decode_b64"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

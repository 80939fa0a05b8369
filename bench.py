"""Benchmark of the NVFP4 sparse-MoE FFN layer on one B300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--workload decode_b1|decode_b64|stack|prefill|prefill_32k|lm_head|dense_ffn]
                    [--impl ours|reference]
                    [--no-cpu-baseline]

Workloads (Flint-shaped layer: d_model 2048, 256 routed experts top-6 + 1
shared, d_ff 512, NVFP4 weights quantised from N(0, 0.02), fp32 router 2048x256):

  decode_b1  (default) batch-1 decode, one fresh bf16 token per step through one
             layer.  Sixteen independently seeded copies of the layer (7.3 GB,
             far above the 126 MB L2) are used round-robin, so every step's
             weights come from HBM.
  decode_b64 64 tokens per step, router skewed by a Zipf(1.1) per-expert bias
             (~200 distinct experts per step); 16 layer copies as above.
  stack      47 distinct MoE layers (~21 GB of NVFP4 experts) with the residual
             add between them, one fresh token per step: a step is one token
             through all 47 layers.
  prefill    4096 tokens through one layer per step with the block-scaled FP4
             tensor-core GEMMs; 16 layer copies.
  lm_head    one token through the 4-bit output layer (151,936 x 2048 NVFP4,
             two rotating copies, 350 MB): fp32 logits.
  dense_ffn  one token through a dense 2048 x 18,432 NVFP4 SwiGLU layer (four
             rotating copies, 255 MB), residual added.

A step is one whole pass of the path (router, top-6, bucketing, experts,
combine) over one batch; steps are serialised as in real decode.  A chunk of
steps is captured in one CUDA graph and replayed until K steps have run, timed
with CUDA events on the launching stream, bracketed by a barrier and a device
synchronise.  Rank 0 prints one JSON line.

``--impl reference`` times the C++ CPU oracle (the only reference this method
has) on a bounded sample of the same workload, on all host cores, and prints
the same line with "impl": "reference".
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

D_MODEL, N_EXP, TOP_K, D_FF, N_SHARED = 2048, 256, 6, 512, 1
EXPERT_BYTES = 3 * D_MODEL * D_FF // 2 + 3 * D_MODEL * D_FF // 16   # 1,769,472 B per expert
ROUTER_BYTES = D_MODEL * N_EXP * 4
N_LAYERS_STACK = 47
FLOP_PER_TOKEN = (TOP_K + N_SHARED) * 3 * 2 * D_MODEL * D_FF        # expert FLOPs per token
FP4_OVER_BF16 = 13.5 / 2.25                                          # nominal dense ratio
HBM_NOMINAL_GBS = 8000.0                                             # the ~8 TB/s the targets are quoted against

WORKLOADS = {
    "decode_b1": dict(T=1, layers=16, steps=50000, chunk=1000, e2e_depth=8,
                      metric="MoE decode tok/s (batch-1, one Flint-shaped NVFP4 MoE layer)"),
    "decode_b64": dict(T=64, layers=16, steps=2000, chunk=100, e2e_depth=8,
                       metric="MoE decode tok/s (batch-64 Zipf-skewed, one Flint-shaped NVFP4 MoE layer)"),
    "stack": dict(T=1, layers=N_LAYERS_STACK, steps=512, chunk=1,
                  metric="MoE decode tok/s (batch-1, 47-layer Flint MoE stack, attention omitted)"),
    "prefill": dict(T=4096, layers=16, steps=40, chunk=4,
                    metric="MoE prefill tok/s (4096 tokens, one Flint-shaped NVFP4 MoE layer)"),
    "prefill_32k": dict(T=32768, layers=4, steps=8, chunk=2,
                        metric="MoE prefill tok/s (32768 tokens, one Flint-shaped NVFP4 MoE layer)"),
    "lm_head": dict(T=1, layers=2, steps=2000, chunk=200, e2e_depth=8,
                    metric="lm_head decode tok/s (batch-1, 151936 x 2048 NVFP4 output layer)"),
    "dense_ffn": dict(T=1, layers=4, steps=4000, chunk=400, e2e_depth=8,
                      metric="dense FFN decode tok/s (batch-1, 2048 x 18432 NVFP4 SwiGLU layer)"),
}
DENSE_WORKLOADS = ("lm_head", "dense_ffn")


#: CUDA sources whose kernels each workload's roofline covers (every header they include)
TRAFFIC_SOURCES = {
    "decode_b1": ("decode_b1.cu", "mma_frag.cuh", "sm100.cuh", "internal.h", "common.cuh"),
    "stack": ("decode_b1.cu", "mma_frag.cuh", "sm100.cuh", "internal.h", "common.cuh"),
    "decode_b64": ("decode_mma.cu", "mma_frag.cuh", "internal.h", "common.cuh"),
    "prefill": ("prefill.cu", "sm100.cuh", "internal.h", "common.cuh"),
    "prefill_32k": ("prefill.cu", "sm100.cuh", "internal.h", "common.cuh"),
    "lm_head": ("dense_gemv.cu", "mma_frag.cuh", "sm100.cuh", "internal.h", "common.cuh"),
    "dense_ffn": ("dense_gemv.cu", "mma_frag.cuh", "sm100.cuh", "internal.h", "common.cuh"),
}


def _sources_digest(names):
    """sha256 over the named files of the package's csrc directory, in the given order."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "nvfp4_expert_ffn_gemv_b300", "csrc")
    for n in names:
        h.update(n.encode())
        with open(os.path.join(d, n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic(workload):
    """DRAM bytes per launch from profiles/traffic.txt, or None once the workload's kernel
    sources differ from the ones the counters were taken on."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as fh:
            lines = [ln.strip() for ln in fh if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    for ln in lines:
        toks = ln.split()
        if toks[0] != workload:
            continue
        kv = dict(t.split("=", 1) for t in toks[1:] if "=" in t)
        if workload not in TRAFFIC_SOURCES or kv.get("sha256") != _sources_digest(TRAFFIC_SOURCES[workload]):
            return None
        return int(kv["traffic_bytes"]) if "traffic_bytes" in kv else None
    return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)   # let the sampler start before the timed region
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


def max_over_ranks(value: float, device: str = "cuda") -> float:
    """The largest of every rank's value (the whole job ends with its slowest rank);
    the value itself when the job has one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def build_layers(lib, torch, synth, n_layers, max_tokens, bias=None, seed0=0):
    """n independently seeded Flint-shaped layers, quantised on the device by the library."""
    s = synth.FLINT
    E = s.n_experts
    ctxs = []
    for i in range(n_layers):
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


def e2e_graph(torch, chunk, xh, yh, xd, yd, step, stream, depth=1):
    """One CUDA graph of `chunk` end-to-end steps.  Every step has its own host-to-device copy of
    its input (pinned xh[i] -> device) and its own device-to-host copy of its result (device ->
    pinned yh[i]), on two side streams.  The steps run in blocks of `depth`: a block's input copies
    are issued together once their buffers are free (the forwards of two blocks back have read
    them), and the block's first forward waits for them and for the result copies of two blocks
    back (whose buffers it rewrites).  Inside a block no other edge enters the forward stream, so
    consecutive steps keep their programmatic (PDL) overlap: a cross-stream wait in front of a
    forward costs it that overlap, while the result copies, which only leave the stream, do not.
    xd / yd hold 2 * depth device buffers each."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    nb = 2 * depth
    assert len(xd) >= nb and len(yd) >= nb
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        fwd_done, out_done = {}, {}               # block -> its last forward / its result copies
        for j0 in range(0, chunk, depth):
            j = j0 // depth
            steps = range(j0, min(chunk, j0 + depth))
            with torch.cuda.stream(s_in):
                if j - 2 in fwd_done:
                    s_in.wait_event(fwd_done[j - 2])
                for i in steps:
                    xd[i % nb].copy_(xh[i], non_blocking=True)
                in_ready = torch.cuda.Event()
                in_ready.record(s_in)
            stream.wait_event(in_ready)
            if j - 2 in out_done:
                stream.wait_event(out_done[j - 2])
            for i in steps:
                step(i, xd[i % nb], yd[i % nb])
                done = torch.cuda.Event()
                done.record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done)
                    yh[i].copy_(yd[i % nb], non_blocking=True)
            fwd_done[j] = done
            with torch.cuda.stream(s_out):
                out_done[j] = torch.cuda.Event()
                out_done[j].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
    return g


def run_ours(args):
    import torch
    import nvfp4_expert_ffn_gemv_b300 as lib
    import synth

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    wl = WORKLOADS[args.workload]
    s = synth.FLINT
    T, n_layers = wl["T"], args.layers or wl["layers"]
    K, W = args.steps or wl["steps"], args.warmup
    chunk = min(wl["chunk"], K)
    replays = (K + chunk - 1) // chunk
    K = replays * chunk
    stack = args.workload == "stack"
    prefill = args.workload.startswith("prefill")
    bias = synth.zipf_bias(s, seed=4242) if args.workload == "decode_b64" else None
    ctxs = build_layers(lib, torch, synth, n_layers, max_tokens=T, bias=bias, seed0=100 * rank)
    stream = torch.cuda.Stream()
    forward = lib.moe_forward_prefill if prefill else lib.moe_forward_decode
    n_inputs = chunk + W                      # distinct token sets (chunk for the graph + warm-up)
    xb, _ = synth.tokens(s, n_inputs * T, seed=synth.token_seed(rank), device="cuda")
    x = xb.view(n_inputs, T, s.d_model)
    y = torch.empty_like(x)
    bufs = [torch.empty((T, s.d_model), dtype=torch.bfloat16, device="cuda") for _ in range(2)]

    def step(i, profile=None):
        """One step: one layer (single-layer workloads) or all layers with the residual (stack)."""
        if not stack:
            c = ctxs[i % n_layers]
            if profile is not None:
                lib.moe_set_profile_events(c, *profile)
            forward(c, x[i], T, y[i], 0, stream)
            if profile is not None:
                lib.moe_set_profile_events(c, None, None)
            return
        cur = x[i]
        for l, c in enumerate(ctxs):
            out = y[i] if l == n_layers - 1 else bufs[l % 2]
            if profile is not None and l == 0:
                lib.moe_set_profile_events(c, profile[0], None)
            if profile is not None and l == n_layers - 1:
                lib.moe_set_profile_events(c, None, profile[1])
            forward(c, cur, T, out, 1, stream)
            if profile is not None and l in (0, n_layers - 1):
                lib.moe_set_profile_events(c, None, None)
            cur = out

    with torch.cuda.stream(stream):
        for i in range(chunk, chunk + W):          # warm-up on inputs the timed steps never use
            step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(chunk):
            step(i)
    # per-kernel timing graph: events around the expert kernels of every step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(chunk)]
    for a, b in ev:                               # events are created lazily at their first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=stream):
        for i in range(chunk):
            step(i, profile=ev[i])
    for c in ctxs:
        assert lib.moe_get_device_status(c) == 0

    def timed(graph, n):
        """Device time of n back-to-back replays.  One untimed replay is queued first, so the
        host's submission of the start event and of the timed replays overlaps device work
        and the region between the events holds device time only, at any step count."""
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):          # replay() launches on the current stream
            graph.replay()
            a.record(stream)
            for _ in range(n):
                graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return a.elapsed_time(b)

    with torch.cuda.stream(stream):
        g.replay()                                # graph warm-up
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = timed(g, replays)
    with torch.cuda.stream(stream):
        gp.replay()
    torch.cuda.synchronize()
    kern_ms = sorted(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms)

    # end to end: pinned host tokens in, host result out, every step (double-buffered)
    xh = x[:chunk].cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    depth = min(wl.get("e2e_depth", 1), chunk)
    xd = [torch.empty((T, s.d_model), dtype=torch.bfloat16, device="cuda") for _ in range(2 * depth)]
    yd = [torch.empty_like(xd[0]) for _ in range(2 * depth)]

    def e2e_step(i, xdb, ydb):
        if stack:
            cur = xdb
            for l, c in enumerate(ctxs):
                out = ydb if l == n_layers - 1 else bufs[l % 2]
                forward(c, cur, T, out, 1, stream)
                cur = out
        else:
            forward(ctxs[i % n_layers], xdb, T, ydb, 0, stream)

    ge = e2e_graph(torch, chunk, xh, yh, xd, yd, e2e_step, stream, depth)
    with torch.cuda.stream(stream):
        ge.replay()
    torch.cuda.synchronize()
    e2e_ms = timed(ge, replays)
    e2e_ms = max_over_ranks(e2e_ms)
    if not prefill:
        # the decode kernels are deterministic: the host results equal the device-resident run's,
        # bit for bit (compared as bit patterns, so NaN outputs match too)
        if not torch.equal(yh.view(torch.int16), y[:chunk].cpu().view(torch.int16)):
            raise RuntimeError("end-to-end results differ from the device-resident run")

    # algorithmic bytes of a batched-decode step: every distinct chosen expert once, plus the shared one
    # expert load of the timed inputs (routing only, outside the timed region): distinct experts
    # per step (the algorithmic bytes of a batched-decode step) and the max/mean tokens per expert
    distinct_mean, distinct_bytes, load = 0.0, 0, None
    if args.workload == "decode_b64" or prefill:
        idx = torch.empty((T, s.top_k), dtype=torch.int32, device="cuda")
        cnt = torch.empty((s.n_experts,), dtype=torch.int32, device="cuda")
        distinct, ratios, maxes = [], [], []
        for i in range(min(chunk, 8)):
            lib.moe_route(ctxs[i % n_layers], x[i], T, idx, None, cnt)
            c = cnt.float()
            used = c[c > 0]
            distinct.append(int(used.numel()))
            ratios.append(float(c.max() / c.mean()))
            maxes.append(int(c.max()))
        distinct_mean = sum(distinct) / len(distinct)
        distinct_bytes = (distinct_mean + s.n_shared) * EXPERT_BYTES
        load = {"distinct_experts": round(distinct_mean, 2), "max_tokens_per_expert": max(maxes),
                "mean_tokens_per_expert": round(T * s.top_k / s.n_experts, 2),
                "max_over_mean": round(sum(ratios) / len(ratios), 3)}
    per_fwd = lib.moe_kernels_per_forward(ctxs[0], T, int(prefill))
    launches = K * per_fwd * (n_layers if stack else 1)
    for c in ctxs:
        lib.moe_destroy(c)
    if rank != 0:
        return
    tok = world * K * T
    value = tok / (ms / 1e3)
    kavg = sum(kern_ms) / len(kern_ms)
    kmed = kern_ms[len(kern_ms) // 2]
    hbm_peak, bf16_peak, bf16_sust, peak_kind = _peaks()
    traffic = _traffic(args.workload) if n_layers == wl["layers"] or args.workload != "stack" else None
    line = {
        "metric": wl["metric"], "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms / K, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 accumulate (nvfp4 weights, bf16 activations)"
        if not prefill else "nvfp4 x nvfp4 -> f32 (tcgen05 block-scaled)", "data": "synthetic",
        "config": {"workload": args.workload if n_layers == wl["layers"] else f"{args.workload} ({n_layers} layers)",
                   "d_model": D_MODEL, "n_experts": N_EXP, "top_k": TOP_K,
                   "n_shared": N_SHARED, "d_ff": D_FF, "tokens_per_step": T, "layers": n_layers,
                   **({"activations": "residual stream without normalisation: it overflows fp32 at layer 25, "
                                      "later layers see NaN and route to experts 0-5 (7 experts streamed per "
                                      "layer either way)"} if stack else {}),
                   "l2": ("47 distinct layers, ~21 GB of weights" if stack else
                          f"{n_layers} rotating layer copies ({n_layers * 0.455:.1f} GB of NVFP4 experts, far above "
                          "the 126 MB L2): no weight is re-read from L2 between steps"),
                   "parallelism": "independent replicas" if world > 1 else "single GPU"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    kus = {"avg": round(kavg * 1e3, 3), "median": round(kmed * 1e3, 3)}
    if args.workload in ("decode_b1", "stack"):
        # The timed graph holds nothing but these PDL chains, so its per-step time is the
        # chain's steady-state duration; events around each chain (launch_us) cut the PDL
        # overlap between consecutive tokens and are reported only for reference.
        chain_ms = ms / K
    if args.workload == "decode_b1":
        alg = 7 * EXPERT_BYTES + ROUTER_BYTES     # 7 experts' NVFP4 weights + the fp32 router
        ach = alg / chain_ms / 1e6
        line["roofline"] = {"kernel": "router -> experts (gate/up + SwiGLU) -> down/combine PDL chain, per token",
                            "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                            "frac": round(ach / hbm_peak, 4), "peak_kind": peak_kind + " copy bandwidth",
                            "frac_of_nominal_8tbs": round(ach / HBM_NOMINAL_GBS, 4),
                            "algorithmic_bytes_per_launch": alg, "traffic": traffic,
                            "launch_us": round(chain_ms * 1e3, 3), "launch_us_isolated": kus}
        line["expert_weight_gbs"] = round(7 * EXPERT_BYTES * K / (ms / 1e3) / 1e9, 1)
        line["expert_weight_frac_of_nominal_8tbs"] = round(line["expert_weight_gbs"] / HBM_NOMINAL_GBS, 4)
    elif args.workload == "stack":
        alg = n_layers * (7 * EXPERT_BYTES + ROUTER_BYTES)
        ach = alg / chain_ms / 1e6
        line["roofline"] = {"kernel": f"whole {n_layers}-layer token step (router, experts, down/combine per layer)",
                            "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                            "frac": round(ach / hbm_peak, 4), "peak_kind": peak_kind + " copy bandwidth",
                            "frac_of_nominal_8tbs": round(ach / HBM_NOMINAL_GBS, 4),
                            "algorithmic_bytes_per_launch": alg, "traffic": traffic,
                            "launch_us": round(chain_ms * 1e3, 3), "launch_us_isolated": kus}
        line["expert_weight_gbs"] = round(n_layers * 7 * EXPERT_BYTES * K / (ms / 1e3) / 1e9, 1)
        line["expert_weight_frac_of_nominal_8tbs"] = round(line["expert_weight_gbs"] / HBM_NOMINAL_GBS, 4)
    elif prefill:
        flop = FLOP_PER_TOKEN * T
        tf = flop / (kavg / 1e3) / 1e12
        fp4_peak = bf16_peak * FP4_OVER_BF16      # burst figure: the GEMMs run in a short graph
        wbytes = (N_EXP + N_SHARED) * EXPERT_BYTES
        line["roofline"] = {"kernel": "prefill expert kernels (quantise + scatter x, x scale atoms, gate/up GEMM, down GEMM)",
                            "bound": "hbm", "achieved": round(wbytes / (kavg / 1e3) / 1e9, 1), "peak": hbm_peak,
                            "unit": "GB/s", "frac": round(wbytes / (kavg / 1e3) / 1e9 / hbm_peak, 4),
                            "peak_kind": peak_kind + " copy bandwidth",
                            "frac_of_nominal_8tbs": round(wbytes / (kavg / 1e3) / 1e9 / HBM_NOMINAL_GBS, 4),
                            "algorithmic_bytes_per_launch": wbytes, "traffic": traffic, "launch_us": kus,
                            "tensor": {"achieved_tflops": round(tf, 1), "peak_tflops": round(fp4_peak, 1),
                                       "frac": round(tf / fp4_peak, 4),
                                       "peak_kind": "measured burst bf16 x nominal fp4/bf16 ratio 6"}}
        line["prefill_tflops"] = round(FLOP_PER_TOKEN * T * K / (ms / 1e3) / 1e12, 1)
    else:
        alg = distinct_bytes
        ach = alg / (kavg / 1e3) / 1e9
        line["roofline"] = {"kernel": "batched-decode expert kernels (x prescale, gate/up + SwiGLU, down), per step",
                            "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                            "frac": round(ach / hbm_peak, 4), "peak_kind": peak_kind + " copy bandwidth",
                            "frac_of_nominal_8tbs": round(ach / HBM_NOMINAL_GBS, 4),
                            "algorithmic_bytes_per_launch": int(alg), "traffic": traffic, "launch_us": kus,
                            "distinct_experts_per_step": round(distinct_mean, 2)}
        line["expert_weight_gbs"] = round(alg * K / (ms / 1e3) / 1e9, 1)
    if load is not None:
        line["expert_load"] = load
    line["e2e"] = {"value": round(tok / (e2e_ms / 1e3), 1), "unit": "tok/s",
                   "h2d_bytes_per_step": T * D_MODEL * 2, "d2h_bytes_per_step": T * D_MODEL * 2,
                   "input_copies_ahead": depth}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


def run_dense(args):
    """lm_head / dense FFN at batch 1: one streaming NVFP4 GEMV pass (two for the FFN) per step."""
    import torch
    import nvfp4_expert_ffn_gemv_b300 as lib
    import synth

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    wl = WORKLOADS[args.workload]
    head = args.workload == "lm_head"
    d, V, F = D_MODEL, synth.FLINT_VOCAB, synth.FLINT_DENSE_FF
    T, n_copies = wl["T"], args.layers or wl["layers"]
    K, W = args.steps or wl["steps"], args.warmup
    chunk = min(wl["chunk"], K)
    replays = (K + chunk - 1) // chunk
    K = replays * chunk
    ctxs = []
    for i in range(n_copies):
        if head:
            w = synth.head_weight(V, d, synth.head_seed() + 100 * rank + i, device="cuda")
            c, sc, ts = lib.quantize(w)
            del w
            ctxs.append(lib.moe_head_init(V, d, dict(codes=c, scales=sc, tensor_scale=ts), T))
        else:
            mats = []
            for w in synth.dense_ffn_weights(d, F, synth.dense_seed(i) + 100 * rank, device="cuda"):
                c, sc, ts = lib.quantize(w)
                mats.append(dict(codes=c, scales=sc, tensor_scale=ts))
            ctxs.append(lib.moe_ffn_init(d, F, *mats, T))
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    stream = torch.cuda.Stream()
    n_inputs = chunk + W
    xb, _ = synth.tokens(synth.FLINT, n_inputs * T, seed=synth.token_seed(rank), device="cuda")
    x = xb.view(n_inputs, T, d)
    out = (torch.empty((n_inputs, T, V), dtype=torch.float32, device="cuda") if head
           else torch.empty_like(x))

    def step(i, xi=None, oi=None):
        c = ctxs[i % n_copies]
        xi = x[i] if xi is None else xi
        oi = out[i] if oi is None else oi
        if head:
            lib.moe_head_forward(c, xi, T, oi, stream)
        else:
            lib.moe_ffn_forward(c, xi, T, oi, 1, stream)

    with torch.cuda.stream(stream):
        for i in range(chunk, chunk + W):
            step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(chunk):
            step(i)
    # external events: recorded inside the capture as event-record nodes that can be timed
    ev = [(torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
          for _ in range(chunk)]
    for a, b in ev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    gp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gp, stream=stream):
        for i in range(chunk):
            ev[i][0].record(stream)
            step(i)
            ev[i][1].record(stream)
    for c in ctxs:
        assert lib.moe_dense_get_device_status(c) == 0

    def timed(graph, n):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            graph.replay()                     # untimed: device busy while the timed replays are queued
            a.record(stream)
            for _ in range(n):
                graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        return a.elapsed_time(b)

    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = timed(g, replays)
    with torch.cuda.stream(stream):
        gp.replay()
    torch.cuda.synchronize()
    kern_ms = sorted(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms)
    # end to end: pinned host token in, host result out, every step (double-buffered)
    xh = x[:chunk].cpu().pin_memory()
    oh = torch.empty((chunk,) + tuple(out.shape[1:]), dtype=out.dtype).pin_memory()
    depth = min(wl.get("e2e_depth", 1), chunk)
    xd = [torch.empty_like(x[0]) for _ in range(2 * depth)]
    od = [torch.empty_like(out[0]) for _ in range(2 * depth)]
    ge = e2e_graph(torch, chunk, xh, oh, xd, od, step, stream, depth)
    with torch.cuda.stream(stream):
        ge.replay()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(timed(ge, replays))
    per_fwd = lib.moe_dense_kernels_per_forward(ctxs[0], T)
    for c in ctxs:
        lib.moe_dense_destroy(c)
    if rank != 0:
        return
    hbm_peak, _, _, peak_kind = _peaks()
    tok = world * K * T
    step_ms = ms / K
    alg = V * d * 9 // 16 if head else 3 * d * F * 9 // 16
    ach = alg / step_ms / 1e6
    kus = {"avg": round(sum(kern_ms) / len(kern_ms) * 1e3, 3), "median": round(kern_ms[len(kern_ms) // 2] * 1e3, 3)}
    line = {
        "metric": wl["metric"], "value": round(tok / (ms / 1e3), 1), "unit": "tok/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(step_ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 accumulate (nvfp4 weights, bf16 activations)", "data": "synthetic",
        "config": {"workload": args.workload, "d_model": d, ("vocab" if head else "d_ff"): V if head else F,
                   "tokens_per_step": T, "copies": n_copies,
                   "l2": f"{n_copies} rotating weight copies ({n_copies * alg / 1e6:.0f} MB, above the 126 MB L2)",
                   "parallelism": "independent replicas" if world > 1 else "single GPU"},
        "gpu_launches": K * per_fwd,
        "clocks": clk.summary(),
        "roofline": {"kernel": "streaming NVFP4 GEMV (lm_head)" if head else
                     "dense FFN: gate/up GEMV + SwiGLU, down GEMV, slice reduction",
                     "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(ach / hbm_peak, 4), "peak_kind": peak_kind + " copy bandwidth",
                     "frac_of_nominal_8tbs": round(ach / HBM_NOMINAL_GBS, 4),
                     "algorithmic_bytes_per_launch": alg, "traffic": _traffic(args.workload),
                     "launch_us": round(step_ms * 1e3, 3), "launch_us_isolated": kus},
        "e2e": {"value": round(tok / (e2e_ms / 1e3), 1), "unit": "tok/s", "h2d_bytes_per_step": T * d * 2,
                "d2h_bytes_per_step": T * (V * 4 if head else d * 2), "input_copies_ahead": depth},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------
def _dense_oracle_sample(workload: str):
    """Oracle weights of one lm_head / dense layer and one token (quantised beforehand, untimed)."""
    import synth
    from oracle import cpp
    d = D_MODEL
    _, x = synth.tokens(synth.FLINT, 1, seed=synth.token_seed(0))
    x = x.numpy()
    if workload == "lm_head":
        m = cpp.quantize(synth.head_weight(synth.FLINT_VOCAB, d, synth.head_seed()).numpy())
        return (lambda nt: cpp.gemv(*m, x, nthreads=nt)), "one token through the 151936 x 2048 output layer"
    mats = [cpp.quantize(w.numpy()) for w in synth.dense_ffn_weights(d, synth.FLINT_DENSE_FF, synth.dense_seed(0))]
    return (lambda nt: cpp.dense_ffn(*mats, x, nthreads=nt)), "one token through a 2048 x 18432 dense SwiGLU layer"


def _oracle_sample(workload: str):
    """The bounded sample the CPU oracle runs: (layer, token batches, prefill flag, what).

    Weights of the experts the sample's tokens choose (plus the shared expert)
    are drawn and quantised by the oracle beforehand, untimed, as moe_init is."""
    import numpy as np
    import synth
    from oracle import cpp

    s = synth.FLINT
    T = {"decode_b1": 1, "stack": 1, "decode_b64": 64, "prefill": 256, "prefill_32k": 256}[workload]
    n_steps = 4 if T == 1 else 1
    router = synth.router_weight(s, synth.router_seed(0)).numpy()
    bias = synth.zipf_bias(s, seed=4242).numpy() if workload == "decode_b64" else None
    _, x = synth.tokens(s, n_steps * T, seed=synth.token_seed(0))
    x = x.numpy().reshape(n_steps, T, s.d_model)
    chosen = set()
    for i in range(n_steps):
        chosen |= set(cpp.route(x[i], router, bias, s.top_k).idx.ravel().tolist())
    sel = sorted(chosen) + list(range(s.n_experts, s.n_all))
    n, f, d = s.n_all, s.d_ff, s.d_model
    wg = np.zeros((n, f, d), np.float32)
    wu = np.zeros((n, f, d), np.float32)
    wd = np.zeros((n, d, f), np.float32)
    for e in sel:
        g_, u_, d_ = synth.expert_weights_one(s, synth.layer_seed(0), int(e))
        wg[e], wu[e], wd[e] = g_.numpy(), u_.numpy(), d_.numpy()
    layer = cpp.quantize_layer(wg, wu, wd, router, bias, k=s.top_k, S=s.n_shared, experts=sel)
    what = {"decode_b1": "single-token decode steps through one layer",
            "stack": "single-token decode steps through one layer, divided by 47 layers",
            "decode_b64": "one 64-token Zipf-skewed decode batch through one layer",
            "prefill": "a 256-token prefill-mode batch through one layer",
            "prefill_32k": "a 256-token prefill-mode batch through one layer"}[workload]
    return layer, x, workload.startswith("prefill"), what


def _time_oracle(layer, x, prefill, nthreads, budget_s):
    from oracle import cpp
    t0 = time.perf_counter()
    done = 0
    while True:   # the sample's steps, repeated until about budget_s of CPU work
        cpp.moe_layer(layer, x[done % len(x)], prefill=prefill, nthreads=nthreads)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return done, time.perf_counter() - t0


def cpu_baseline(workload: str, budget_s: float = 10.0):
    """Time the C++ oracle as it stands, on a bounded sample of the workload, on all of
    the host's cores (its std::thread pool) and on one thread."""
    cores = os.cpu_count() or 1
    if workload in DENSE_WORKLOADS:
        fn, what = _dense_oracle_sample(workload)
        res = []
        for nt, budget in ((cores, budget_s), (1, budget_s / 2)):
            t0, done = time.perf_counter(), 0
            while True:
                fn(nt)
                done += 1
                if time.perf_counter() - t0 > budget:
                    break
            res.append((done, time.perf_counter() - t0))
        (done, dt), (done1, dt1) = res
        return {"value": round(done / dt, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
                "single_thread_value": round(done1 / dt1, 4),
                "sample": f"{done} x 1 token: {what} (C++ oracle, weights dequantised each call), {dt:.2f} s on "
                          f"{cores} threads; {done1} in {dt1:.2f} s on one thread"}
    layer, x, prefill, what = _oracle_sample(workload)
    T = x.shape[1]
    done, dt = _time_oracle(layer, x, prefill, cores, budget_s)
    done1, dt1 = _time_oracle(layer, x, prefill, 1, budget_s / 2)
    div = N_LAYERS_STACK if workload == "stack" else 1
    value = done * T / dt / div
    value1 = done1 * T / dt1 / div
    return {"value": round(value, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
            "single_thread_value": round(value1, 4),
            "sample": f"{done} x {T} token(s) ({len(x)} distinct step(s) repeated): {what} (C++ oracle: fp32 values, "
                      f"fp64 accumulation, chosen experts dequantised each step), {dt:.2f} s timed on {cores} "
                      f"threads; {done1} repeats in {dt1:.2f} s on one thread"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    wl = WORKLOADS[args.workload]
    cb = cpu_baseline(args.workload, budget_s=args.cpu_budget)
    line = {"impl": "reference", "metric": wl["metric"], "value": cb["value"], "unit": "tok/s", "n_gpus": world,
            "steps": args.steps or wl["steps"], "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (f64 accumulation)", "data": "synthetic",
            "config": {"workload": args.workload, "d_model": D_MODEL, "n_experts": N_EXP, "top_k": TOP_K,
                       "n_shared": N_SHARED, "d_ff": D_FF, "tokens_per_step": wl["T"], "layers": wl["layers"]},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: per workload)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode_b1", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0,
                    help="layer copies (default: per workload; smaller only for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in DENSE_WORKLOADS:
        run_dense(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

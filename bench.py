"""Throughput of the KLA gated delta-rule recurrence on one GB300 (and N GPUs as replicas).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]

Headline workload (one timed "step" = one chunkwise prefill of the whole batch):
  gdn4k: B=8, H=16, T=4096, d_k=d_v=128, chunk 64, bf16 q/k/v ~ N(0,1), scalar gate
  alpha = exp(-softplus(N(-4,1))), eta = sigmoid(N(0,1)), eps 1e-6, S0 = 0, fp32 state.
Metric: prefill tokens/s (tokens = B*T, all heads included). Inputs are resident in HBM
when a timed step starts; L2 (129 MB) is flushed before every timed step, outside the timed
window, by writing a 256 MiB buffer and then reading another 256 MiB buffer (so the timed
kernel neither finds its inputs in L2 nor pays for writing back the flush's dirty lines). Each step is timed with CUDA events on the stream
the kernels are launched on.

Extras in the same JSON line: long131k prefill (B=1 H=16 T=131072), kda8k prefill
(per-key-channel gate, B=4 H=16 T=8192), decode (batch 64, H16, 1024 single-token
steps, L2 flushed before every step), decode_graph (the same steps as one CUDA graph, L2 not
flushed), verify4 / verify8 / verify16 (the decode batch advanced 4, 8 or 16 tokens per
call, as in speculative verification: the token loop at 4, the chunk form at 8 and 16), bwd_gdn4k and bwd_long131k (the backward passes of
the headline and the long-context workloads), each with its own roofline.

--impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the
same workload (whole sequences of some (b, h) chains) and reports the same metric.

Multi-GPU (torchrun): every rank runs its own independent batch (the recurrence shards
over sequences and heads with no exchange), so scaling is weak; value = all ranks' tokens
divided by the slowest rank's time.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "prefill tokens/s (T=4K, 131K) and decode tokens/s; % of roofline on 1 GB300"
L2_FLUSH_BYTES = 256 << 20

# Algorithmic bytes per token-head (d = 128): q, k, v, o in bf16 + alpha, eta fp32.
PREFILL_BYTES_PER_TOKEN_HEAD = 3 * 2 * 128 + 2 * 128 + 4 + 4            # 1032
PREFILL_BYTES_PER_TOKEN_HEAD_KDA = 3 * 2 * 128 + 2 * 128 + 4 * 128 + 4  # 1540
# Algorithmic flops per token-head at C = 64, d = 128 (S-products 6 d^2, in-chunk 5 C d, solve C^2/3).
PREFILL_FLOP_PER_TOKEN_HEAD = 6 * 128 * 128 + 5 * 64 * 128 + 64 * 64 / 3
# Decode: state read + write 8 d^2, q k v o 8 d (bf16), alpha, eta 8.
DECODE_BYTES_PER_HEAD_STEP = 8 * 128 * 128 + 4 * 2 * 128 + 8


# DRAM bytes (read + write) per launch of the tensor-core prefill kernel on the gdn4k
# workload, from an ncu capture of that kernel (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by the fingerprint of the kernel sources it was taken on. Any other source state
# reports null.
TC_SOURCES = ("gated_delta_rule_14_gb300/csrc/kla_chunk_tc.cu", "gated_delta_rule_14_gb300/csrc/sm103_ptx.cuh",
              "gated_delta_rule_14_gb300/csrc/kla_internal.cuh")
TC_TRAFFIC_GDN4K = {"064b64879e7b4310": 520.263936e6}
# sm__pipe_tensor_cycles_active (fraction of elapsed cycles) of the same kernel and capture:
# the algorithmic TFLOP/s divided by it is the rate of the MMA phases themselves.
TC_PIPE_ACTIVE_GDN4K = {"064b64879e7b4310": 0.1311}


def tc_fingerprint() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in TC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------------------ env
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(x: float, world: int, device=None) -> float:
    """Max over ranks (identity for one process)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []   # (t_start, t_end) windows of timed work

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.marks.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [ln for t, ln in self.lines if any(a - 0.1 <= t <= b + 0.25 for a, b in self.marks)]
        rows = [r.split(", ") for r in (inside or [ln for _, ln in self.lines])]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) >= 9:
                for n, val in zip(names, r[5:9]):
                    if val.strip() == "Active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------------------ GPU
def to_dev(a, dev, pin=False):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    if pin:
        return t.pin_memory()
    return t.to(dev)


def time_steps(fn, steps, warmup, flush, stream):
    """Run fn() warmup + steps times; L2 flushed before each; returns per-step ms (CUDA events)."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def prefill_inputs(name, seed, dev, **override):
    inp = synth.make_prefill(name, seed=seed, **override)
    d = {n: to_dev(getattr(inp, n), dev) for n in ("q", "k", "v", "alpha", "eta")}
    return inp, d


def bench_prefill(name, steps, warmup, seed, dev, flush, stream, pk):
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp, d = prefill_inputs(name, seed, dev)
    wl = inp.wl
    o = torch.empty((wl.B, wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=dev)
    ST = torch.empty((wl.B, wl.H, wl.d_k, wl.d_v), dtype=torch.float32, device=dev)

    def step():
        kla.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], wl.eps, None, chunk=wl.chunk, out=o, S_T=ST)

    ms = time_steps(step, steps, warmup, flush, stream)
    kla.device_status(dev)
    token_heads = wl.B * wl.T * wl.H
    per = PREFILL_BYTES_PER_TOKEN_HEAD_KDA if wl.gate == "channel" else PREFILL_BYTES_PER_TOKEN_HEAD
    alg_bytes = token_heads * per + wl.B * wl.H * wl.d_k * wl.d_v * 4      # + final state
    alg_flop = token_heads * PREFILL_FLOP_PER_TOKEN_HEAD
    mean_ms = statistics.fmean(ms)
    res = {"workload": name, "tokens": wl.B * wl.T, "ms": mean_ms, "ms_all": ms, "alg_bytes": alg_bytes,
           "alg_flop": alg_flop, "inp": inp, "dev_inputs": d, "o": o, "ST": ST}
    return res


def roofline(alg_bytes, ms, pk, traffic=None, bound="hbm"):
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    return {"bound": bound, "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": traffic, "peak_source": pk["source"]}


def bench_decode(steps_tok, seed, dev, flush, stream, pk, passes=1, warm_tokens=8):
    import torch

    import gated_delta_rule_14_gb300 as kla
    dd = synth.make_decode(seed=seed, steps=steps_tok)
    q, k, v, a, e = (to_dev(x, dev) for x in (dd.q, dd.k, dd.v, dd.alpha, dd.eta))
    S = to_dev(dd.S, dev)
    o = torch.empty(q.shape[:3] + (dd.wl.d_v,), dtype=torch.bfloat16, device=dev)
    for i in range(min(warm_tokens, steps_tok)):
        flush()
        kla.decode_step(q[i], k[i], v[i], a[i], e[i], S, dd.wl.eps, out=o[i])
    S.copy_(to_dev(dd.S, dev))
    torch.cuda.synchronize()
    total = 0.0
    per_step = []
    for _ in range(passes):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps_tok)]
        for i, (e0, e1) in enumerate(evs):
            flush()
            e0.record(stream)
            kla.decode_step(q[i], k[i], v[i], a[i], e[i], S, dd.wl.eps, out=o[i])
            e1.record(stream)
        torch.cuda.synchronize()
        t = [e0.elapsed_time(e1) for e0, e1 in evs]
        per_step += t
        total += sum(t)
    kla.device_status(dev)
    heads = dd.wl.B * dd.wl.H
    mean_ms = total / (passes * steps_tok)
    return {"tokens_per_s": dd.wl.B * steps_tok * passes / (total * 1e-3), "ms_per_token_step": mean_ms,
            "alg_bytes_per_step": heads * DECODE_BYTES_PER_HEAD_STEP, "per_step_ms": per_step,
            "launches": passes * steps_tok}


def bench_decode_graph(steps_tok, seed, dev, pk, replays=3):
    """The decode steps captured once in a CUDA graph and replayed back to back (no L2 flush:
    the 64 MB of state stays resident in the 129 MB L2 between steps, as it would for one layer
    decoding alone)."""
    import torch

    import gated_delta_rule_14_gb300 as kla
    dd = synth.make_decode(seed=seed, steps=steps_tok)
    q, k, v, a, e = (to_dev(x, dev) for x in (dd.q, dd.k, dd.v, dd.alpha, dd.eta))
    S = to_dev(dd.S, dev)
    o = torch.empty(q.shape[:3] + (dd.wl.d_v,), dtype=torch.bfloat16, device=dev)
    kla.decode_step(q[0], k[0], v[0], a[0], e[0], S, dd.wl.eps, out=o[0])   # first call outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(steps_tok):
                kla.decode_step(q[i], k[i], v[i], a[i], e[i], S, dd.wl.eps, out=o[i])
    torch.cuda.synchronize()
    g.replay()   # warm-up
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(dev)
    e0.record(cur)
    for _ in range(replays):
        g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    kla.device_status(dev)
    ms = e0.elapsed_time(e1) / replays
    heads = dd.wl.B * dd.wl.H
    gbs = heads * DECODE_BYTES_PER_HEAD_STEP * steps_tok / (ms * 1e-3) / 1e9
    return {"value": dd.wl.B * steps_tok / (ms * 1e-3), "unit": "tokens/s", "ms_per_token_step": ms / steps_tok,
            "token_steps": steps_tok, "batch": dd.wl.B, "launches": steps_tok * replays,
            "l2": "not flushed: the 64 MB state stays L2-resident between steps",
            "effective_gbs": round(gbs, 1),
            "note": "one CUDA graph of all steps; effective GB/s above the HBM peak means L2 hits"}


def bench_verify(ntok, calls, seed, dev, flush, stream, pk, channel=False):
    """Multi-token decode (speculative verification): every call advances the decode batch's
    states in place by `ntok` tokens; L2 flushed before every call. channel=True: the same batch
    (64 sequences x 16 heads) with the per-key-channel gates of the kda8k workload."""
    import torch

    import gated_delta_rule_14_gb300 as kla
    if channel:
        inp, d = prefill_inputs("kda8k", seed, dev, B=64, T=ntok, H=16, s0_sigma=0.02)
    else:
        inp, d = prefill_inputs("decode", seed, dev, T=ntok, chunk=64, s0_sigma=0.02)
    wl = inp.wl
    S = to_dev(inp.S0, dev)
    o = torch.empty((wl.B, wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=dev)

    def step():
        kla.chunk_fwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], wl.eps, S, chunk=64, out=o, S_T=S)

    ms = statistics.fmean(time_steps(step, calls, 3, flush, stream))
    kla.device_status(dev)
    heads = wl.B * wl.H
    per = PREFILL_BYTES_PER_TOKEN_HEAD_KDA if channel else PREFILL_BYTES_PER_TOKEN_HEAD
    alg_bytes = heads * (8 * wl.d_k * wl.d_v + ntok * per)
    if ntok < 5:
        kernel = "token loop (tokens_pipe_kernel: 128 x 32 state tiles in registers)"
    elif channel:
        kernel = "chunk form, per-channel gate (tokens_ch_kernel: one CTA per head, in-call decay factors <= 1)"
    else:
        kernel = "chunk form (tokens_tc_kernel: one CTA per head, warp-level tensor cores)"
    return {"value": wl.B * ntok / (ms * 1e-3), "unit": "tokens/s", "ms_per_call": ms, "calls": calls,
            "tokens_per_call": ntok, "batch": wl.B, "kernel": kernel, "roofline": roofline(alg_bytes, ms, pk),
            "l2": "flushed before every call (256 MiB write, then 256 MiB read)"}


BWD_BYTES_PER_TOKEN_HEAD = 4 * 2 * 128 + 8 + 3 * 4 * 128 + 8   # q, k, v, dO in; dq, dk, dv, dalpha, deta out
BWD_BYTES_PER_TOKEN_HEAD_KDA = BWD_BYTES_PER_TOKEN_HEAD + 2 * 4 * 127   # alpha and dalpha per key channel


BWD_KERNELS_PER_CALL = 4   # chunkwise path: prep, forward carry, reverse carry, gradients
# per-channel gate: range check, prep, two carries, gradients, the rerun launch (its CTAs return)
BWD_KDA_KERNELS_PER_CALL = 6
# long131k: prep, 2 x (value runs, transitions, combine, reruns), gradients
BWD_LONG_KERNELS_PER_CALL = 10


def bench_bwd(name, steps, seed, dev, flush, stream, pk, **override):
    """Backward pass of the named prefill workload (dL/do random bf16, dL/dS_T = 0)."""
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp, d = prefill_inputs(name, seed, dev, **override)
    wl = inp.wl
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    dO = torch.randn((wl.B, wl.T, wl.H, wl.d_v), device=dev, generator=g).to(torch.bfloat16)
    ws = torch.empty(kla.bwd_workspace_size(wl.B, wl.T, wl.H, wl.d_k, wl.d_v, torch.bfloat16,
                                            per_channel_gate=wl.gate == "channel"), dtype=torch.uint8, device=dev)

    def step():
        kla.chunk_bwd(d["q"], d["k"], d["v"], d["alpha"], d["eta"], dO, wl.eps, workspace=ws, want_dS0=False)

    ms = statistics.fmean(time_steps(step, steps, 1, flush, stream))
    kla.device_status(dev)
    alg = wl.B * wl.T * wl.H * (BWD_BYTES_PER_TOKEN_HEAD_KDA if wl.gate == "channel" else BWD_BYTES_PER_TOKEN_HEAD)
    return {"value": wl.B * wl.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "steps": steps,
            "workspace_bytes": ws.numel(), "roofline": roofline(alg, ms, pk),
            "note": "chunkwise backward: the chunk-parallel prep (T = (I+R)^-1, W, U, A) and the forward and "
                    "reverse chunk-state carries (one CTA per chain) on tcgen05 with TMA-staged tiles and TMA "
                    "record stores, the chunk-parallel gradients on warp-level bf16 MMAs; "
                    "~4.5 GB of DRAM traffic per call (ncu at B = 4, per-chunk S_c, dS_c, E_c, dE_c, W, U, A, T records) "
                    "against the algorithmic bytes"}


def e2e_prefill(res, steps, warmup, dev, stream, parts=8):
    """Same workload through the public host-buffer API (kla_chunk_fwd_host) with pinned host
    tensors: per step the H2D copies of q, k, v, alpha, eta, the prefill and the D2H copies of o
    and S_T, all inside the timed region; the work runs in `parts` parts (slices of whole chunks of
    every sequence for this bf16 / scalar-gate / d = 128 workload) so copies of one part overlap
    the prefill of another."""
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = res["inp"]
    wl = inp.wl
    host = {n: to_dev(getattr(inp, n), dev, pin=True) for n in ("q", "k", "v", "alpha", "eta")}
    bufs = kla.host_buffers(host["q"], host["v"], host["alpha"], device=dev)
    o_h = torch.empty(res["o"].shape, dtype=res["o"].dtype, pin_memory=True)
    ST_h = torch.empty(res["ST"].shape, dtype=res["ST"].dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_h.numel() * o_h.element_size() + ST_h.numel() * ST_h.element_size()

    def step():
        kla.chunk_fwd_host(host["q"], host["k"], host["v"], host["alpha"], host["eta"], wl.eps, chunk=wl.chunk,
                           parts=parts, out=o_h, S_T=ST_h, device=dev, buffers=bufs)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"ms": ms, "tokens_per_s": wl.B * wl.T / (ms * 1e-3), "h2d": h2d, "d2h": d2h, "parts": parts}


# ------------------------------------------------------------------------- CPU oracle
def oracle_sample(name, nchains, seed=0, threads=None, inp=None):
    """Time the fp64 oracle on `nchains` whole (b, h) sequences of the workload."""
    import oracle
    threads = threads or os.cpu_count() or 1
    inp = inp if inp is not None else synth.make_prefill(name, seed=seed)
    wl = inp.wl
    rng = np.random.default_rng(123)
    idx = rng.choice(wl.B * wl.H, size=min(nchains, wl.B * wl.H), replace=False)
    chains = [(int(i) // wl.H, int(i) % wl.H) for i in sorted(idx)]

    def pick(n):
        a = inp.as_f64(n)
        return np.stack([a[b, :, h] for b, h in chains])[:, :, None]
    args = [pick(n) for n in ("q", "k", "v", "alpha", "eta")]
    orc = oracle.load()
    t0 = time.perf_counter()
    orc.recurrent(*args, wl.eps, None, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"tokens": len(chains) * wl.T, "seconds": dt, "threads": min(threads, len(chains)),
            "chains": len(chains), "T": wl.T}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    name = "gdn4k"
    wl = synth.WORKLOADS[name]
    nchains = max(1, min(args.ref_chains, wl.B * wl.H))
    times = []
    tokens = 0
    inp = synth.make_prefill(name, seed=0)
    for i in range(args.warmup + args.steps):
        r = oracle_sample(name, nchains, inp=inp)
        if i >= args.warmup:
            times.append(r["seconds"])
            tokens = r["tokens"]
    ms = statistics.fmean(times) * 1e3
    value = tokens / (ms * 1e-3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(name, "none (CPU)"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": r["threads"], "kind": "oracle",
                         "sample": f"{nchains} whole (b,h) sequences of T={wl.T} from the {name} workload per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(name, l2):
    wl = synth.WORKLOADS[name]
    return {"workload": f"{name}: B={wl.B} H={wl.H} T={wl.T} d_k=d_v={wl.d_k} chunk={wl.chunk} "
                        f"{wl.dtype} q/k/v, fp32 state, {wl.gate} gate, S0=0",
            "B": wl.B, "T": wl.T, "H": wl.H, "d_k": wl.d_k, "d_v": wl.d_v, "chunk": wl.chunk,
            "global_batch": wl.B, "seq_len": wl.T, "l2": l2, "parallelism": "replicas (independent batch per GPU)"}


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--ref-chains", type=int, default=16)
    ap.add_argument("--cpu-chains", type=int, default=64)
    ap.add_argument("--decode-steps", type=int, default=1024)
    ap.add_argument("--verify-calls", type=int, default=256)
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--bwd-only", action="store_true",
                    help="time only the backward pass of --bwd-workload (a small case for profiling with --bwd-batch)")
    ap.add_argument("--bwd-workload", choices=["gdn4k", "kda8k"], default="gdn4k")
    ap.add_argument("--bwd-batch", type=int, default=8)
    ap.add_argument("--prefill-only", choices=["gdn4k", "kda8k", "long131k"], default=None,
                    help="time only the prefill of this workload (a command for profiling one kernel)")
    ap.add_argument("--verify-only", choices=["4", "8", "16", "16kda"], default=None,
                    help="time only this multi-token call on the decode batch (--verify-calls calls)")
    ap.add_argument("--e2e-parts", type=int, default=8,
                    help="time slices of the host-buffer prefill (the e2e number)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import gated_delta_rule_14_gb300 as kla
    kla._native.lib()
    pk = peaks()
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush():
        # write a buffer larger than L2, then read another one: the timed kernel starts with none
        # of its inputs in L2 and without the flush's dirty lines left to write back
        flush_buf.zero_()
        torch.sum(flush_rd, dim=0, out=flush_sink)

    if args.prefill_only:
        r = bench_prefill(args.prefill_only, args.steps, args.warmup, seed=rank, dev=dev, flush=flush, stream=stream,
                          pk=pk)
        if rank == 0:
            print(json.dumps({"prefill": args.prefill_only, "ms_per_step": r["ms"],
                              "roofline": roofline(r["alg_bytes"], r["ms"], pk)}), flush=True)
        return

    if args.verify_only:
        ntok, ch = int(args.verify_only.replace("kda", "")), args.verify_only.endswith("kda")
        r = bench_verify(ntok, args.verify_calls, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk, channel=ch)
        if rank == 0:
            print(json.dumps({f"verify{args.verify_only}": r}), flush=True)
        return

    if args.bwd_only:
        r = bench_bwd(args.bwd_workload, args.steps, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk,
                      B=args.bwd_batch)
        if rank == 0:
            print(json.dumps({f"bwd_{args.bwd_workload}": r, "batch": args.bwd_batch}), flush=True)
        return

    clocks = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    clocks.start()

    # ---- headline: gdn4k prefill
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    res = bench_prefill("gdn4k", args.steps, args.warmup, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk)
    clocks.mark(t0, time.time())
    barrier(world)
    ms_max = reduce_max(res["ms"], world, dev)
    tokens_all = reduce_sum(res["tokens"], world, dev)
    value = tokens_all / (ms_max * 1e-3)
    kern_ms = res["ms"]
    roof = roofline(res["alg_bytes"], kern_ms, pk, traffic=TC_TRAFFIC_GDN4K.get(tc_fingerprint()))
    tflops = res["alg_flop"] / (kern_ms * 1e-3) / 1e12
    active = TC_PIPE_ACTIVE_GDN4K.get(tc_fingerprint())
    tensor = {"achieved_tflops": round(tflops, 2), "peak_tflops": pk["bf16_tflops"],
              "frac": round(tflops / pk["bf16_tflops"], 4), "pipe_active": active}

    e2e = e2e_prefill(res, max(3, args.steps // 2), 3, dev, stream, parts=args.e2e_parts)
    e2e_val = reduce_sum(e2e["tokens_per_s"], world, dev) if world > 1 else e2e["tokens_per_s"]
    launches = args.steps * 1   # one kernel per prefill step

    extras = {}
    if not args.no_extras:
        for name, st in (("long131k", 3), ("kda8k", 3)):
            t0 = time.time()
            r = bench_prefill(name, st, 3, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk)
            clocks.mark(t0, time.time())
            extras[name] = {"value": r["tokens"] / (r["ms"] * 1e-3), "unit": "tokens/s", "ms_per_step": r["ms"],
                            "steps": st, "roofline": roofline(r["alg_bytes"], r["ms"], pk),
                            "tensor_tflops": round(r["alg_flop"] / (r["ms"] * 1e-3) / 1e12, 2)}
            launches += st
            del r
            torch.cuda.empty_cache()
        t0 = time.time()
        dr = bench_decode(args.decode_steps, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk)
        clocks.mark(t0, time.time())
        extras["decode"] = {"value": dr["tokens_per_s"], "unit": "tokens/s",
                            "ms_per_token_step": dr["ms_per_token_step"], "token_steps": args.decode_steps,
                            "batch": 64, "l2": "flushed before every token step (256 MiB write, then 256 MiB read)",
                            "roofline": roofline(dr["alg_bytes_per_step"], dr["ms_per_token_step"], pk)}
        launches += dr["launches"]
        t0 = time.time()
        dg = bench_decode_graph(args.decode_steps, seed=rank, dev=dev, pk=pk)
        clocks.mark(t0, time.time())
        extras["decode_graph"] = dg
        launches += dg["launches"]
        t0 = time.time()
        extras["verify4"] = bench_verify(4, args.verify_calls, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk)
        clocks.mark(t0, time.time())
        launches += args.verify_calls
        for ntok in (8, 16):
            t0 = time.time()
            extras[f"verify{ntok}"] = bench_verify(ntok, args.verify_calls, seed=rank, dev=dev, flush=flush,
                                                   stream=stream, pk=pk)
            clocks.mark(t0, time.time())
            launches += args.verify_calls
        t0 = time.time()
        extras["verify16_kda"] = bench_verify(16, args.verify_calls, seed=rank, dev=dev, flush=flush, stream=stream,
                                              pk=pk, channel=True)
        clocks.mark(t0, time.time())
        launches += args.verify_calls
        if not args.no_bwd:
            t0 = time.time()
            extras["bwd_gdn4k"] = bench_bwd("gdn4k", 3, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk)
            clocks.mark(t0, time.time())
            launches += 3 * BWD_KERNELS_PER_CALL
            torch.cuda.empty_cache()
            t0 = time.time()
            extras["bwd_long131k"] = bench_bwd("long131k", 3, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk)
            extras["bwd_long131k"]["note"] = ("chunkwise backward with the chunk-state carries split into "
                                              "segments run in parallel (16 chains of 2048 chunks)")
            clocks.mark(t0, time.time())
            launches += 3 * BWD_LONG_KERNELS_PER_CALL
            torch.cuda.empty_cache()
            t0 = time.time()
            extras["bwd_kda8k"] = bench_bwd("kda8k", 3, seed=rank, dev=dev, flush=flush, stream=stream, pk=pk)
            extras["bwd_kda8k"]["note"] = ("per-channel gate, chunkwise: gate range check, prep with the per-channel "
                                           "factor tiles (K e^{G-G_r}, K e^{G_r-G}, Q e^{G-G_r}), forward and reverse "
                                           "chunk-state carries on tcgen05 side by side, chunk-parallel gradients with dk, dq and the "
                                           "log-decay gradient per channel in registers; chains outside the "
                                           "factorised range rerun on the token-sequential path (none here)")
            clocks.mark(t0, time.time())
            launches += 3 * BWD_KDA_KERNELS_PER_CALL
            torch.cuda.empty_cache()
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        c = oracle_sample("gdn4k", args.cpu_chains, inp=res["inp"])
        c1 = oracle_sample("gdn4k", 4, inp=res["inp"], threads=1)
        cpu = {"value": c["tokens"] / c["seconds"], "unit": "tokens/s", "cores": c["threads"], "kind": "oracle",
               "sample": f"{c['chains']} whole (b,h) sequences of T={c['T']} of the gdn4k workload "
                         f"({c['seconds']:.1f} s wall)",
               "one_core": {"value": c1["tokens"] / c1["seconds"], "unit": "tokens/s", "cores": 1,
                            "sample": f"{c1['chains']} whole (b,h) sequences of T={c1['T']} of the gdn4k workload "
                                      f"({c1['seconds']:.1f} s wall)"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config("gdn4k", "flushed before every timed step (256 MiB write, then 256 MiB read)"),
            "roofline": roof, "tensor": tensor,
            "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": e2e["h2d"],
                    "d2h_bytes_per_step": e2e["d2h"], "api": "kla_chunk_fwd_host",
                    "parts": e2e["parts"]},
            "gpu_launches": launches, "clocks": clk, "cpu_baseline": cpu, "extras": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

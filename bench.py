"""Decode throughput of the fq library on GB300.

Workload (N=1 line): the full 28-layer Qwen3-0.6B-shaped decoder with Q8_0 weights
(seeded N(0, 0.02)), Q8_0 embedding and LM head, bf16 KV cache; 2048 positions are filled
by running the model on seeded random token ids; then greedy decode chains of 64 steps,
batch 1, each chain starting from those 2048 cached positions (the cache is rewound
between chains, so every timed step is the same workload).  One "step" = one decode token
through the whole hot path (embedding, 28 x [norm+QKV, QK-norm+rope+append+attention,
O-proj, norm+gate_up+SwiGLU, down], output norm, LM head, argmax).  At batch 1 the step is
one streamed persistent kernel, so the roofline kernel is the step itself.

The same line carries the other halves of the metric, measured the same way:
  q4k_batch1  the 36-layer Qwen3-8B shape with Q4_K weights, batch 1 at context 8192;
  batch32     the 8B shape with Q8_0 weights, 32 lockstep sequences at contexts U[512, 4096];
  layer_step  one 0.6B-shaped layer (f32 KV, 128 positions), hot and cold (16 rotated
              weight + cache copies, more than L2 holds).

Timing: W warm-up steps, then exactly K steps bracketed by a barrier and synchronisation,
CUDA events on the launching stream, max over ranks.  Every step streams ~0.87 GB
(weights + KV), far more than the 129 MB L2, so no flush is needed between steps.

--impl reference times the CPU oracle (the f64 restatement of the pages) on the same
workload: each of its steps is one of the 29 units of a decode token (28 layer steps at
context 2048, then the output norm + LM head), cycling, and tokens/s = (K / 29) / time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s at batch 1 and 32; achieved HBM GB/s vs GB300 peak"
WORKLOAD = "qwen3-0.6b"
CHAIN = 64
CONTEXT = 2048

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one streamed-step launch per
# workload, from a metrics-only ncu capture of that kernel inside the timed NVTX range.
# Reported only while the kernel's sources hash to the value they had when the counters were
# taken: a changed kernel has unmeasured traffic.
STEP_TRAFFIC = {
    "qwen3-0.6b": (869580160, "b6021b09d4d1df3c"),     # mean of 2 launches: 868.70 MB read + 0.88 MB written
    "qwen3-8b-q4k": (5502293248, "b6021b09d4d1df3c"),  # 5470.22 MB read + 32.08 MB written (exchange words)
}
STEP_SOURCES = ["stream_step.cu", "kernels.h", "quant.cuh", "tma.cuh", "common.cuh"]


def step_source_hash(base: str = None) -> str:
    """Hash of the streamed step's sources (in `base`, by default the package's csrc) with
    comments and blank lines removed, so that a comment edit does not count as a changed
    kernel."""
    import hashlib
    import re
    h = hashlib.sha256()
    if base is None:
        base = os.path.join(os.path.dirname(os.path.abspath(__file__)), "quantized_decoder_decode_gb300", "csrc")
    for f in STEP_SOURCES:
        with open(os.path.join(base, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())
        h.update(text.encode())
    return h.hexdigest()[:16]


def step_traffic(workload: str):
    t = STEP_TRAFFIC.get(workload)
    return t[0] if t and t[1] == step_source_hash() else None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KV_ELEM_BYTES = {"f32": 4.0, "bf16": 2.0, "q8_0": 34 / 32}   # per cached value (Q8_0: codes + fp16 scale)


def workload_of(args):
    """The named workload, with its cache dtype replaced when --kv asks for another, and its
    layer count when --layers asks for fewer (a small case of the same shapes for profilers)."""
    import dataclasses
    import synth.workloads as wl
    w = wl.WORKLOADS[args.workload]
    if getattr(args, "kv", None) and args.kv != w.kv_dtype:
        w = dataclasses.replace(w, kv_dtype=args.kv)
    if getattr(args, "layers", None):
        w = dataclasses.replace(w, dims=dataclasses.replace(w.dims, num_layers=args.layers))
    return w


def kv_tensor(a: np.ndarray, dev):
    """Prior cache rows as a device tensor of their raw bytes (bf16 bits, f32, Q8_0 blocks)."""
    import torch
    return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)


def step_bytes(dims, ctx: int) -> dict:
    """Algorithmic bytes of one batch-1 decode step at `ctx` cached positions."""
    q8 = 34 / 32
    H, F, L = dims.hidden_size, dims.intermediate_size, dims.num_layers
    qd, kvd = dims.q_dim, dims.kv_dim
    layer_w = (qd + 2 * kvd) * H + H * qd + 2 * F * H + H * F
    weights = L * layer_w * q8 + L * (2 * H + 2 * dims.head_dim) * 4
    head = dims.vocab_size * H * q8 + H * 4
    embd_row = H * q8
    kv_read = 2 * L * kvd * ctx * 2
    kv_write = 2 * L * kvd * 2
    return {"weights": weights, "lm_head": head, "embedding_row": embd_row, "kv_read": kv_read,
            "kv_write": kv_write, "total": weights + head + embd_row + kv_read + kv_write}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, ms: int = 100):
        self.index, self.ms = index, ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", f"-lms={self.ms}"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int, backend: str = "nccl"):
    """One process per GPU (torchrun env).  Replicas only: the process group carries the
    start/stop barriers and the max-over-ranks timing, never the data path."""
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(v: float, world: int, op: str) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def max_over_ranks(v: float, world: int) -> float:
    return _reduce(v, world, "max")


def sum_over_ranks(v: float, world: int) -> float:
    return _reduce(v, world, "sum")


def aggregate(units: float, seconds: float, world: int) -> tuple:
    """Whole-job throughput: units processed by all ranks / the slowest rank's time."""
    total = sum_over_ranks(units, world)
    dt = max_over_ranks(seconds, world)
    return total / dt, dt


# ---------------------------------------------------------------- CPU oracle (reference arm / baseline)

def oracle_setup(w, W):
    import oracle
    import synth.workloads as wl
    d = w.dims
    m = oracle.Model(d, W, w.weight_dtype, w.kv_dtype)
    c = m.new_cache(CONTEXT + 1)
    for L in range(d.num_layers):
        k, v = wl.make_kv_prior(w, 0, L, CONTEXT)
        c.write(L, 0, k, v)
    c.set_len(CONTEXT)
    return m, c


def oracle_unit(m, c, W, w, i, x):
    """Unit i % 29 of a decode token: a layer step at context 2048, or the LM head."""
    import oracle
    d = w.dims
    u = i % (d.num_layers + 1)
    if u < d.num_layers:
        m.layer_step(u, c, CONTEXT, x)
    else:
        xn = oracle.rmsnorm(x, W["output_norm"], d.rms_norm_eps)
        oracle.gemv(w.weight_dtype, W["output"], d.vocab_size, d.hidden_size, xn)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    import synth.workloads as wl
    w = wl.WORKLOADS[WORKLOAD]
    W = wl.make_weights(w)
    m, c = oracle_setup(w, W)
    threads = oracle.set_threads(0)
    x = wl.layer_input(w).astype(np.float64)
    for i in range(args.warmup):
        oracle_unit(m, c, W, w, i, x)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_unit(m, c, W, w, i, x)
    dt = time.perf_counter() - t0
    units = w.dims.num_layers + 1
    value = (args.steps / units) / dt
    sample = (f"{args.steps} oracle units (28 layer steps at context {CONTEXT} + output norm/LM head, cycling; "
              f"{units} units = one token), KV prior N(0,1) bf16")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def cpu_baseline(w, W, budget_s: float = 15.0) -> dict:
    """The oracle as it stands, full decode steps at context 2048 on this host's cores."""
    import oracle
    m, c = oracle_setup(w, W)
    threads = oracle.set_threads(0)
    c.set_len(CONTEXT)
    n, t0 = 0, time.perf_counter()
    while True:
        c.set_len(CONTEXT)
        m.decode_step(c, 1 + n, CONTEXT)
        n += 1
        if time.perf_counter() - t0 >= budget_s or n >= 64:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full oracle decode steps (28 layers + LM head, f64) at context {CONTEXT}, "
                      f"KV prior N(0,1) bf16 instead of a model prefill"}


def config_dict(w) -> dict:
    d = w.dims
    ctx = (f"{CONTEXT} positions filled by the model" if w.prefill_from_model else
           f"KV prior N(0,1) {w.kv_dtype} at context "
           + (f"U[{w.context_range[0]},{w.context_range[1]}]" if w.context_range else str(w.context)))
    moe = (f", {d.num_experts} experts top-{d.num_experts_used} (expert FFN {d.moe_intermediate_size})"
           if d.is_moe else f", FFN {d.intermediate_size}")
    return {"workload": f"{w.name}: {d.num_layers} layers, hidden {d.hidden_size}, {d.num_attention_heads}q/"
                        f"{d.num_key_value_heads}kv heads x {d.head_dim}{moe}, vocab {d.vocab_size}, "
                        f"{w.weight_dtype.upper()} weights, {w.kv_dtype} KV; batch {w.batch}; {ctx}; greedy chains "
                        f"of {w.steps} steps from that context",
            "batch": w.batch, "context": (list(w.context_range) if w.context_range else w.context),
            "chain": w.steps, "weights": w.weight_dtype, "kv": w.kv_dtype,
            "l2": "no flush: every step streams far more than the 129 MB L2 (weights + KV)"}


def weight_bytes(w, experts_per_layer=None) -> dict:
    """Algorithmic weight bytes touched by one step (ggml block sizes)."""
    d = w.dims
    bpw = 34 / 32 if w.weight_dtype == "q8_0" else 144 / 256
    H, L = d.hidden_size, d.num_layers
    attn = ((d.q_dim + 2 * d.kv_dim) * H + H * d.q_dim) * bpw
    norms = (2 * H + 2 * d.head_dim) * 4
    if d.is_moe:
        per_expert = 3 * H * d.moe_intermediate_size * bpw
        router = d.num_experts * H * 4
        ne = experts_per_layer if experts_per_layer is not None else [d.num_experts_used] * L
        ffn = sum(ne) * per_expert + L * router
    else:
        ffn = L * 3 * H * d.intermediate_size * bpw
    head = d.vocab_size * H * bpw + H * 4
    return {"layers": L * (attn + norms) + ffn, "lm_head": head, "embedding_rows": w.batch * H * bpw}


def load_workload(w, max_ctx_extra: int, dev, stream):
    """The workload's model on the device and one KV cache per sequence holding its context
    (filled by the model for the default workload, else the seeded N(0, 1) prior)."""
    import torch
    import synth.workloads as wl
    from quantized_decoder_decode_gb300 import fq
    d = w.dims
    n = w.batch
    chain = w.steps
    W = wl.make_weights(w)
    ctxs = [CONTEXT] * n if w.prefill_from_model else [int(c) for c in w.contexts()]
    cap_max = max(ctxs) + chain
    desc = fq.fq_desc_init(vocab_size=d.vocab_size, hidden_size=d.hidden_size, intermediate_size=d.intermediate_size,
                           num_layers=d.num_layers, num_attention_heads=d.num_attention_heads,
                           num_key_value_heads=d.num_key_value_heads, head_dim=d.head_dim,
                           rms_norm_eps=d.rms_norm_eps, rope_theta=d.rope_theta, num_experts=d.num_experts,
                           num_experts_used=d.num_experts_used, moe_intermediate_size=d.moe_intermediate_size,
                           max_positions=cap_max + max_ctx_extra)
    src, keep = fq.weight_src(desc, W, w.weight_dtype)
    model = fq.fq_load_weights(desc, src, stream)
    del src, keep
    kvs = [fq.fq_kv_init(model, c + chain, w.kv_dtype) for c in ctxs]
    toks = torch.empty((chain, n), dtype=torch.int32, device=dev)
    logits = torch.empty((n, d.vocab_size), dtype=torch.float32, device=dev)
    if w.prefill_from_model:
        # fill the context by running the model on seeded random ids (not timed)
        ids = wl.prefill_ids(w)
        for p in range(CONTEXT - 1):
            fq.fq_decode_step(model, kvs[0], int(ids[p]), p, 0, stream)
        fq.fq_decode_greedy(model, kvs, [int(ids[CONTEXT - 1])], 1, toks.data_ptr(), logits.data_ptr(), stream)
        torch.cuda.synchronize()
        first = [int(toks[0, 0].item())]
    else:
        for s_i, (kv, c) in enumerate(zip(kvs, ctxs)):
            for L in range(d.num_layers):
                k, v = wl.make_kv_prior(w, s_i, L, c)
                kt, vt = kv_tensor(k, dev), kv_tensor(v, dev)
                fq.fq_kv_append(kv, L, 0, c, kt.data_ptr(), vt.data_ptr(), stream)
            fq.fq_kv_commit(kv, c)
        torch.cuda.synchronize()
        first = [int(t) for t in wl.first_ids(w)]
    return W, model, kvs, ctxs, first, toks, logits


def free_workload(model, kvs):
    from quantized_decoder_decode_gb300 import fq
    for kv in kvs:
        fq.fq_kv_free(kv)
    fq.fq_model_free(model)


def step_bytes_of(w, ctxs, experts=None) -> dict:
    """Algorithmic bytes of one step (weights touched + KV read + KV written) averaged over a
    chain of w.steps steps from the contexts ctxs."""
    d = w.dims
    wb = weight_bytes(w, experts)
    eb = KV_ELEM_BYTES[w.kv_dtype]
    kv_read = sum(2 * d.num_layers * d.kv_dim * (c + (w.steps - 1) / 2) * eb for c in ctxs)
    kv_write = w.batch * 2 * d.num_layers * d.kv_dim * eb
    total = wb["layers"] + wb["lm_head"] + wb["embedding_rows"] + kv_read + kv_write
    return {"total": total, "weights_layers": wb["layers"], "lm_head": wb["lm_head"],
            "embedding_rows": wb["embedding_rows"], "kv_read": kv_read, "kv_write": kv_write}


def time_chains(model, kvs, ctxs, first, toks, logits, chain, steps, warmup, world, local, stream, st):
    """Greedy chains of `chain` steps from the cached contexts (rewound between chains):
    `warmup` untimed steps, then exactly `steps` steps between CUDA events on the launching
    stream, bracketed by a barrier and synchronisation; clocks sampled meanwhile."""
    import torch
    from quantized_decoder_decode_gb300 import fq

    def rewind():
        for kv, c in zip(kvs, ctxs):
            fq.fq_kv_rewind(kv, c)

    def chains(n_steps):
        done = 0
        while done < n_steps:
            s_ = min(chain, n_steps - done)
            rewind()
            fq.fq_decode_greedy(model, kvs, first, s_, toks.data_ptr(), logits.data_ptr(), stream)
            done += s_
        rewind()

    chains(max(warmup, 3))
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(world)
        ev0.record(st)
        torch.cuda.nvtx.range_push("timed")   # the region a profiler's NVTX filter selects
        chains(steps)
        torch.cuda.nvtx.range_pop()
        ev1.record(st)
        torch.cuda.synchronize()
        barrier(world)
    return ev0.elapsed_time(ev1) / 1e3, clk.summary(), fq.fq_step_kernels(model, stream), rewind


def sub_record(name: str, steps: int, warmup: int, dev, stream, st, peak, peak_kind) -> dict:
    """One more workload measured the same way as the main line (batch-1 8B Q4_K, or the
    batch-32 8B lockstep), for the same JSON line."""
    import synth.workloads as wl
    w = wl.WORKLOADS[name]
    W, model, kvs, ctxs, first, toks, logits = load_workload(w, 64, dev, stream)
    del W
    dt, clocks, kps, _ = time_chains(model, kvs, ctxs, first, toks, logits, w.steps, steps, warmup, 1, 0, stream, st)
    free_workload(model, kvs)
    sb = step_bytes_of(w, ctxs)
    gbs = sb["total"] / (dt / steps) / 1e9
    return {"workload": config_dict(w)["workload"], "batch": w.batch, "value": w.batch * steps / dt,
            "unit": "tokens/s", "steps": steps, "ms_per_step": dt / steps * 1e3, "kernels_per_step": kps,
            "step_roofline": {"bytes_per_step": sb["total"], "achieved_gbs": gbs, "peak": peak,
                              "frac": gbs / peak, "peak_kind": peak_kind,
                              "traffic": step_traffic(name) if kps == 1 else None},
            "clocks": clocks}


def layer_step_record(dev, stream, st, peak, peak_kind, copies: int = 16, reps: int = 6) -> dict:
    """The single 0.6B-shaped layer (one token, f32 KV with 128 prior positions): its 17.8 MB
    working set fits in L2, so it is timed hot (the same weights and cache every call) and
    cold (rotating over `copies` independent weight + cache copies, more than L2 holds)."""
    import torch
    import synth.workloads as wl
    from quantized_decoder_decode_gb300 import fq
    w = wl.WORKLOADS["qwen3-0.6b-layer"]
    d = w.dims
    side = torch.cuda.Stream(dev)
    ss = side.cuda_stream
    models, kvs, xs = [], [], []
    for i in range(copies):
        wi = wl.dataclasses.replace(w, seed=w.seed + 1000 * i)
        W = wl.make_weights(wi)
        desc = fq.fq_desc_init(vocab_size=d.vocab_size, hidden_size=d.hidden_size,
                               intermediate_size=d.intermediate_size, num_layers=1,
                               num_attention_heads=d.num_attention_heads, num_key_value_heads=d.num_key_value_heads,
                               head_dim=d.head_dim, max_positions=w.context + 8)
        src, keep = fq.weight_src(desc, W, w.weight_dtype)
        m = fq.fq_load_weights(desc, src, stream)
        kv = fq.fq_kv_init(m, w.context + 8, w.kv_dtype)
        k, v = wl.make_kv_prior(wi, 0, 0, w.context)
        kt, vt = kv_tensor(k, dev), kv_tensor(v, dev)
        fq.fq_kv_append(kv, 0, 0, w.context, kt.data_ptr(), vt.data_ptr(), stream)
        fq.fq_kv_commit(kv, w.context)
        models.append(m)
        kvs.append(kv)
        xs.append(torch.from_numpy(wl.layer_input(wi)).to(dev))
    torch.cuda.synchronize()

    def calls(order):
        for i in order:
            fq.fq_layer_step(models[i], 0, kvs[i], w.context, xs[i].data_ptr(), ss)
            fq.fq_kv_rewind(kvs[i], w.context)

    results = {}
    for kind, order in (("hot", [0] * copies), ("cold", list(range(copies)))):
        with torch.cuda.stream(side):
            calls(order)                       # per-stream workspaces exist before timing
        torch.cuda.synchronize()
        # every timed call is queued behind a short sleep kernel before the GPU reaches it,
        # so the events see the GPU time of the calls, not the host's launch rate
        n_calls = reps * copies
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            torch.cuda._sleep(50_000_000)
            e0.record(side)
            for _ in range(reps):
                calls(order)
            e1.record(side)
        torch.cuda.synchronize()
        results[kind] = {"us_per_layer_step": e0.elapsed_time(e1) * 1e3 / n_calls}
    wb = weight_bytes(w)
    nbytes = wb["layers"] + 2 * d.kv_dim * w.context * 4 + 2 * d.kv_dim * 4
    for kind in results:
        if "us_per_layer_step" in results[kind]:
            gbs = nbytes / (results[kind]["us_per_layer_step"] * 1e-6) / 1e9
            results[kind].update({"achieved_gbs": gbs, "frac": gbs / peak})
    for kv, m in zip(kvs, models):
        fq.fq_kv_free(kv)
        fq.fq_model_free(m)
    return {"workload": config_dict(w)["workload"].split(";")[0] + "; one token, f32 KV with 128 prior positions",
            "bytes_per_layer_step": nbytes, "copies_cold": copies, "peak": peak, "peak_kind": peak_kind, **results}


def run_fq(args):
    import torch
    import synth.workloads as wl
    from quantized_decoder_decode_gb300 import fq

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream(dev)
    stream = st.cuda_stream
    w = workload_of(args)
    d = w.dims
    n = w.batch
    chain = w.steps
    W, model, kvs, ctxs, first, toks, logits = load_workload(w, 64, dev, stream)

    # ---- timed region: exactly K steps (each step = one token for each of the n sequences)
    dt_dev, clocks, kernels_per_step, rewind = time_chains(model, kvs, ctxs, first, toks, logits, chain, args.steps,
                                                           args.warmup, world, local, stream, st)
    value, dt = aggregate(n * args.steps, dt_dev, world)
    streamed = fq.fq_step_path(model, n, w.kv_dtype)

    # ---- end to end through the public API with host buffers: per step the tokens go in
    # from pinned host memory (by value through the call) and the chosen tokens come back
    # to pinned host memory before the next step is issued
    host_tok = torch.empty(n, dtype=torch.int32, pin_memory=True)
    e2e_steps = min(args.steps, 4 * chain)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    done = 0
    while done < e2e_steps:
        s_ = min(chain, e2e_steps - done)
        rewind()
        cur = list(first)
        for _ in range(s_):
            fq.fq_decode_greedy(model, kvs, cur, 1, toks.data_ptr(), 0, stream)
            host_tok.copy_(toks[0], non_blocking=True)
            st.synchronize()
            cur = host_tok.tolist()
        done += s_
    rewind()
    e2e_value, e2e_dt = aggregate(n * e2e_steps, time.perf_counter() - t0, world)

    # ---- experts touched per layer (MoE): from one traced step
    experts = None
    if d.is_moe:
        ri = torch.empty((d.num_layers, n, d.num_experts_used), dtype=torch.int32, device=dev)
        rw = torch.empty_like(ri, dtype=torch.float32)
        fq.fq_decode_step_trace(model, kvs, first, 0, 0, ri.data_ptr(), rw.data_ptr(), stream)
        torch.cuda.synchronize()
        rewind()
        experts = [len(set(ri[L].flatten().tolist())) for L in range(d.num_layers)]

    peak, peak_kind = measured_peaks()
    sb = step_bytes_of(w, ctxs, experts)
    step_gbs = sb["total"] / (dt / args.steps) / 1e9
    # kernels inside the timed region: one launch per step (streamed) or one graph per step,
    # plus the state set-up launch of every chain
    n_chains = (args.steps + chain - 1) // chain
    if streamed:
        # the dominant kernel is the whole step: one launch per token, timed above
        kt = dt_dev / args.steps
        roof = {"bound": "hbm", "kernel": "streamed decode step (one persistent kernel per token)",
                "achieved": sb["total"] / kt / 1e9, "peak": peak, "unit": "GB/s",
                "frac": sb["total"] / kt / 1e9 / peak, "peak_kind": peak_kind, "bytes_per_launch": sb["total"],
                "us_per_launch": kt * 1e6, "traffic": step_traffic(w.name)}
    else:
        roof = None
    free_workload(model, kvs)
    del W

    subs = {}
    if rank == 0 and world == 1 and not args.no_subrecords and args.workload == WORKLOAD:
        subs["q4k_batch1"] = sub_record("qwen3-8b-q4k", 64, 8, dev, stream, st, peak, peak_kind)
        subs["batch32"] = sub_record("qwen3-8b-batch32", 32, 8, dev, stream, st, peak, peak_kind)
        subs["layer_step"] = layer_step_record(dev, stream, st, peak, peak_kind)

    if rank == 0:
        cb = None
        if world == 1 and not args.no_cpu_baseline and w.prefill_from_model:
            cb = cpu_baseline(w, wl.make_weights(w), budget_s=args.cpu_budget)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(w),
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 4 * n,
                    "d2h_bytes_per_step": 4 * n, "steps": e2e_steps},
            "gpu_launches": args.steps * kernels_per_step + n_chains,
            "kernels_per_step": kernels_per_step,
            "step_path": "streamed" if streamed else "kernel sequence",
            "roofline": roof,
            "step_roofline": {"bytes_per_step": sb["total"], "achieved_gbs": step_gbs, "peak": peak,
                              "frac": step_gbs / peak, "peak_kind": peak_kind,
                              "breakdown": {k: v for k, v in sb.items() if k != "total"},
                              "experts_per_layer": (sum(experts) / len(experts)) if experts else None},
            "clocks": clocks,
            "cpu_baseline": cb,
            **subs,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_kernel(args):
    """Kernel-level timing for profiling: the LM-head GEMV alone (--kernel lm_head), one
    decoder layer step at the workload's context (--kernel layer), or the layer's dense
    projections at the workload's batch (--kernel proj), `--steps` repetitions after
    `--warmup`, on one layer of the chosen workload's weights."""
    import dataclasses
    import torch
    import synth.workloads as wl
    from quantized_decoder_decode_gb300 import fq
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream(dev)
    stream = st.cuda_stream
    w = workload_of(args)
    d = w.dims
    ctx = CONTEXT if w.prefill_from_model else int(w.contexts().max())
    w1 = wl.scaled(w, num_layers=1)
    W = wl.make_weights(w1)
    desc = fq.fq_desc_init(vocab_size=d.vocab_size, hidden_size=d.hidden_size, intermediate_size=d.intermediate_size,
                           num_layers=1, num_attention_heads=d.num_attention_heads,
                           num_key_value_heads=d.num_key_value_heads, head_dim=d.head_dim,
                           num_experts=d.num_experts, num_experts_used=d.num_experts_used,
                           moe_intermediate_size=d.moe_intermediate_size, max_positions=ctx + 64)
    src, keep = fq.weight_src(desc, W, w.weight_dtype)
    model = fq.fq_load_weights(desc, src, stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    bpw = 34 / 32 if w.weight_dtype == "q8_0" else 144 / 256
    flops = None
    if args.kernel == "lm_head":
        x = torch.randn(d.hidden_size, device=dev)
        y = torch.empty(d.vocab_size, device=dev)
        call = lambda: fq.fq_gemv(model, 0, fq.W_OUTPUT, 1, x.data_ptr(), y.data_ptr(), stream)  # noqa: E731
        nbytes = d.vocab_size * d.hidden_size * bpw
    elif args.kernel == "proj":
        # every dense projection of one layer at the workload's batch (tensor-core GEMM for
        # batches of 8 or more); bytes = weights once + activations in and out
        n = w.batch
        mats = [(fq.W_Q, d.q_dim + 2 * d.kv_dim, d.hidden_size), (fq.W_O, d.hidden_size, d.q_dim)]
        if not d.is_moe:
            mats += [(fq.W_GATE, 2 * d.intermediate_size, d.hidden_size),
                     (fq.W_DOWN, d.hidden_size, d.intermediate_size)]
        bufs = [(wh, torch.randn(n, cols, device=dev), torch.empty(n, rows, device=dev)) for wh, rows, cols in mats]
        def call():
            for wh, xb, yb in bufs:
                fq.fq_gemv(model, 0, wh, n, xb.data_ptr(), yb.data_ptr(), stream)
        nbytes = sum(r * c * bpw + 4 * n * (r + c) for _, r, c in mats)
        flops = 2 * n * sum(r * c for _, r, c in mats)
    else:
        kv = fq.fq_kv_init(model, ctx + 1, w.kv_dtype)
        k, v = wl.make_kv_prior(w1, 0, 0, ctx)
        kt, vt = kv_tensor(k, dev), kv_tensor(v, dev)
        fq.fq_kv_append(kv, 0, 0, ctx, kt.data_ptr(), vt.data_ptr(), stream)
        fq.fq_kv_commit(kv, ctx)
        x = torch.from_numpy(wl.layer_input(w1)).to(dev)
        call = lambda: fq.fq_layer_step(model, 0, kv, ctx, x.data_ptr(), stream)  # noqa: E731
        wb = weight_bytes(dataclasses.replace(w1, batch=1))
        nbytes = wb["layers"] + 2 * d.kv_dim * ctx * 2
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    for a_, b_ in evs:
        a_.record(st)
        call()
        b_.record(st)
    torch.cuda.synchronize()
    t = [a_.elapsed_time(b_) / 1e3 for a_, b_ in evs]
    mean = sum(t) / len(t)
    peak, kind = measured_peaks()
    print(json.dumps({"kernel": args.kernel, "workload": w.name, "launches": len(t), "us_mean": mean * 1e6,
                      "us_min": min(t) * 1e6, "bytes": nbytes, "gbs": nbytes / mean / 1e9,
                      "frac": nbytes / mean / 1e9 / peak, "peak": peak, "peak_kind": kind,
                      "tflops": (flops / mean / 1e12) if flops else None}))
    fq.fq_model_free(model)
    return 0


def run_verify(args):
    """forwardStepAllLogits economics, as the qwen3 app page's verify benchmark measures them: one
    batched k-token pass that scores every position against k single-token steps, for k in
    {2, 4, 8, 16}, on the chosen workload's model at its context (seeded KV prior)."""
    import torch
    import synth.workloads as wl
    from quantized_decoder_decode_gb300 import fq
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream(dev)
    stream = st.cuda_stream
    w = workload_of(args)
    d = w.dims
    ctx = CONTEXT if w.prefill_from_model else int(w.contexts().max())
    W = wl.make_weights(w)
    desc = fq.fq_desc_init(vocab_size=d.vocab_size, hidden_size=d.hidden_size, intermediate_size=d.intermediate_size,
                           num_layers=d.num_layers, num_attention_heads=d.num_attention_heads,
                           num_key_value_heads=d.num_key_value_heads, head_dim=d.head_dim,
                           num_experts=d.num_experts, num_experts_used=d.num_experts_used,
                           moe_intermediate_size=d.moe_intermediate_size, max_positions=ctx + 64)
    src, keep = fq.weight_src(desc, W, w.weight_dtype)
    model = fq.fq_load_weights(desc, src, stream)
    del src, keep
    kv = fq.fq_kv_init(model, ctx + 32, w.kv_dtype)
    for L in range(d.num_layers):
        k, v = wl.make_kv_prior(w, 0, L, ctx)
        kt, vt = kv_tensor(k, dev), kv_tensor(v, dev)
        fq.fq_kv_append(kv, L, 0, ctx, kt.data_ptr(), vt.data_ptr(), stream)
    fq.fq_kv_commit(kv, ctx)
    logits = torch.empty((16, d.vocab_size), dtype=torch.float32, device=dev)
    ids = [int(t) for t in wl.first_ids(wl.scaled(w, batch=16))] if not w.prefill_from_model else \
        [int(t) for t in wl.prefill_ids(w)[:16]]
    reps = max(args.steps, 3)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fq.fq_kv_rewind(kv, ctx)
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a_, b_ in evs:
            fq.fq_kv_rewind(kv, ctx)
            a_.record(st)
            fn()
            b_.record(st)
        torch.cuda.synchronize()
        t = sorted(a_.elapsed_time(b_) * 1e3 for a_, b_ in evs)
        return t[len(t) // 2], t[0]

    for k in (2, 4, 8, 16):
        toks = ids[:k]
        v_med, v_best = timed(lambda: fq.fq_decode_step_all_logits(model, kv, toks, ctx, logits.data_ptr(), stream))

        def singles():
            for i, t in enumerate(toks):
                fq.fq_decode_step(model, kv, t, ctx + i, logits[i].data_ptr(), stream)
        s_med, s_best = timed(singles)
        print(json.dumps({"kernel": "verify", "workload": w.name, "k": k, "context": ctx,
                          "verify_us_median": v_med, "verify_us_best": v_best,
                          "single_steps_us_median": s_med, "single_steps_us_best": s_best,
                          "speedup_median": s_med / v_med, "verify_tokens_per_s": k / (v_med * 1e-6)}))
    fq.fq_kv_free(kv)
    fq.fq_model_free(model)
    return 0


def run_prefill(args):
    """Multi-token forwardStep (section 14.1) as a prefill: the 0.6B workload's 2048 prompt ids
    in one call (passes of 32 rows) against the same ids decoded one token at a time, both
    from an empty cache, both ending with the last row's logits."""
    import torch
    import synth.workloads as wl
    from quantized_decoder_decode_gb300 import fq
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    st = torch.cuda.current_stream(dev)
    stream = st.cuda_stream
    w = workload_of(args)
    if not w.prefill_from_model:
        print(json.dumps({"kernel": "prefill", "unavailable": f"{w.name} has no prompt; use the default workload"}))
        return 0
    d = w.dims
    ids = [int(t) for t in wl.prefill_ids(w)]
    n = len(ids)
    W = wl.make_weights(w)
    desc = fq.fq_desc_init(vocab_size=d.vocab_size, hidden_size=d.hidden_size, intermediate_size=d.intermediate_size,
                           num_layers=d.num_layers, num_attention_heads=d.num_attention_heads,
                           num_key_value_heads=d.num_key_value_heads, head_dim=d.head_dim,
                           num_experts=d.num_experts, num_experts_used=d.num_experts_used,
                           moe_intermediate_size=d.moe_intermediate_size, max_positions=n + 64)
    src, keep = fq.weight_src(desc, W, w.weight_dtype)
    model = fq.fq_load_weights(desc, src, stream)
    del src, keep
    kv = fq.fq_kv_init(model, n, w.kv_dtype)
    logits = torch.empty(d.vocab_size, dtype=torch.float32, device=dev)

    def timed(fn, reps):
        for _ in range(max(args.warmup, 3) if reps > 1 else 1):
            fq.fq_kv_rewind(kv, 0)
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a_, b_ in evs:
            fq.fq_kv_rewind(kv, 0)
            a_.record(st)
            fn()
            b_.record(st)
        torch.cuda.synchronize()
        t = sorted(a_.elapsed_time(b_) for a_, b_ in evs)
        return t[len(t) // 2]

    p_ms = timed(lambda: fq.fq_forward_step(model, kv, ids, 0, logits.data_ptr(), stream), 5)

    def tokenwise():
        for p, t in enumerate(ids):
            fq.fq_decode_step(model, kv, t, p, logits.data_ptr() if p == n - 1 else 0, stream)
    t_ms = timed(tokenwise, 2)
    print(json.dumps({"kernel": "prefill", "workload": w.name, "kv": w.kv_dtype, "tokens": n,
                      "forward_step_ms": p_ms, "token_by_token_ms": t_ms, "speedup": t_ms / p_ms,
                      "prefill_tokens_per_s": n / (p_ms * 1e-3)}))
    fq.fq_kv_free(kv)
    fq.fq_model_free(model)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["lm_head", "layer", "proj"], default=None,
                    help="time one kernel family instead of the decode loop (profiling)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["qwen3-0.6b", "qwen3-8b-q4k", "qwen3-8b-batch32", "qwen3-30b-a3b-batch16"],
                    help="the default is the benchmark line; the others are measured the same way")
    ap.add_argument("--steps", type=int, default=6400)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="fq", choices=["fq", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true",
                    help="skip the 8B batch-1 / batch-32 and single-layer records of the default line")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers of the workload's shapes: a small case for profilers, not a bench line")
    ap.add_argument("--kv", default=None, choices=["bf16", "q8_0"],
                    help="cache dtype in place of the workload's own (q8_0: the integer-score cache)")
    ap.add_argument("--verify", action="store_true",
                    help="all-logits verify pass of k tokens against k single steps, k in 2/4/8/16")
    ap.add_argument("--prefill", action="store_true",
                    help="the 2048-token prompt through one multi-token forwardStep against token-by-token decode")
    args = ap.parse_args()
    if args.prefill:
        return run_prefill(args)
    if args.verify:
        return run_verify(args)
    if args.kernel:
        return run_kernel(args)
    if args.impl == "reference":
        if args.workload != WORKLOAD:
            print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the default workload only"}))
            return 0
        return run_reference(args)
    return run_fq(args)


if __name__ == "__main__":
    sys.exit(main())

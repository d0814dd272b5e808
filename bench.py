"""Decode throughput of the fq library on GB300.

Workload (N=1 line): the full 28-layer Qwen3-0.6B-shaped decoder with Q8_0 weights
(seeded N(0, 0.02)), Q8_0 embedding and LM head, bf16 KV cache; 2048 positions are filled
by running the model on seeded random token ids; then greedy decode chains of 64 steps,
batch 1, each chain starting from those 2048 cached positions (the cache is rewound
between chains, so every timed step is the same workload).  One "step" = one decode token
through the whole hot path (embedding, 28 x [norm+QKV, QK-norm+rope+append+attention,
O-proj, norm+gate_up+SwiGLU, down], output norm, LM head, argmax).

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

# DRAM bytes (read + write) of one LM-head GEMV launch, from the ncu capture summarised in
# profiles/gemv_tma_q8_0_lm_head_qwen3-0.6b.md (its metrics-only recapture).  Reported only while the kernel's sources
# hash to the value they had when the counters were taken.
LM_HEAD_TRAFFIC = {"qwen3-0.6b": (168251392, "ae06facd60aae183")}
GEMV_SOURCES = ["gemv_tma.cu", "quant.cuh", "tma.cuh", "common.cuh"]


def gemv_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    base = os.path.join(os.path.dirname(os.path.abspath(__file__)), "quantized_decoder_decode_gb300", "csrc")
    for f in GEMV_SOURCES:
        with open(os.path.join(base, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def lm_head_traffic(workload: str):
    t = LM_HEAD_TRAFFIC.get(workload)
    return t[0] if t and t[1] == gemv_source_hash() else None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KV_ELEM_BYTES = {"f32": 4.0, "bf16": 2.0, "q8_0": 34 / 32}   # per cached value (Q8_0: codes + fp16 scale)


def workload_of(args):
    """The named workload, with its cache dtype replaced when --kv asks for another."""
    import dataclasses
    import synth.workloads as wl
    w = wl.WORKLOADS[args.workload]
    if getattr(args, "kv", None) and args.kv != w.kv_dtype:
        w = dataclasses.replace(w, kv_dtype=args.kv)
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
    W = wl.make_weights(w)
    ctxs = [CONTEXT] * n if w.prefill_from_model else [int(c) for c in w.contexts()]
    cap_max = max(ctxs) + chain
    desc = fq.fq_desc_init(vocab_size=d.vocab_size, hidden_size=d.hidden_size, intermediate_size=d.intermediate_size,
                           num_layers=d.num_layers, num_attention_heads=d.num_attention_heads,
                           num_key_value_heads=d.num_key_value_heads, head_dim=d.head_dim,
                           rms_norm_eps=d.rms_norm_eps, rope_theta=d.rope_theta, num_experts=d.num_experts,
                           num_experts_used=d.num_experts_used, moe_intermediate_size=d.moe_intermediate_size,
                           max_positions=cap_max + 64)
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

    chains(max(args.warmup, 3))
    torch.cuda.synchronize()
    barrier(world)

    # ---- timed region: exactly K steps (each step = one token for each of the n sequences)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.nvtx.range_push("timed")
        ev0.record(st)
        chains(args.steps)
        ev1.record(st)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        barrier(world)
    value, dt = aggregate(n * args.steps, ev0.elapsed_time(ev1) / 1e3, world)
    kernels_per_step = fq.fq_step_kernels(model, stream)

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

    # ---- roofline of the dominant kernel: the dequant GEMV, timed live on the LM head (the
    # largest single launch of the step) with CUDA events on its stream
    peak, peak_kind = measured_peaks()
    x = torch.randn(d.hidden_size, device=dev)
    y = torch.empty(d.vocab_size, device=dev)
    reps = 20
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for _ in range(3):
        fq.fq_gemv(model, 0, fq.W_OUTPUT, 1, x.data_ptr(), y.data_ptr(), stream)
    torch.cuda.synchronize()
    for a_, b_ in evs:
        a_.record(st)
        fq.fq_gemv(model, 0, fq.W_OUTPUT, 1, x.data_ptr(), y.data_ptr(), stream)
        b_.record(st)
    torch.cuda.synchronize()
    kt = sum(a_.elapsed_time(b_) for a_, b_ in evs) / reps / 1e3
    bpw = 34 / 32 if w.weight_dtype == "q8_0" else 144 / 256
    kbytes = d.vocab_size * d.hidden_size * bpw + d.hidden_size * 4 + d.vocab_size * 4
    achieved = kbytes / kt / 1e9

    wb = weight_bytes(w, experts)
    eb = KV_ELEM_BYTES[w.kv_dtype]
    kv_read = sum(2 * d.num_layers * d.kv_dim * (c + (chain - 1) / 2) * eb for c in ctxs)
    kv_write = n * 2 * d.num_layers * d.kv_dim * eb
    total = wb["layers"] + wb["lm_head"] + wb["embedding_rows"] + kv_read + kv_write
    step_gbs = total / (dt / args.steps) / 1e9
    # kernels inside the timed region: each step replays one captured graph; each chain adds
    # the one state-setup launch made before its replays
    n_chains = (args.steps + chain - 1) // chain

    if rank == 0:
        cb = None
        if world == 1 and not args.no_cpu_baseline and w.prefill_from_model:
            cb = cpu_baseline(w, W, budget_s=args.cpu_budget)
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(w),
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 4 * n,
                    "d2h_bytes_per_step": 4 * n, "steps": e2e_steps},
            "gpu_launches": args.steps * kernels_per_step + n_chains,
            "kernels_per_step": kernels_per_step,
            "roofline": {"bound": "hbm", "kernel": f"dequant GEMV ({w.weight_dtype}), LM head launch "
                                                   f"{d.vocab_size}x{d.hidden_size}",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind, "bytes_per_launch": kbytes, "us_per_launch": kt * 1e6,
                         "traffic": lm_head_traffic(w.name)},
            "step_roofline": {"bytes_per_step": total, "achieved_gbs": step_gbs, "peak": peak,
                              "frac": step_gbs / peak, "peak_kind": peak_kind,
                              "breakdown": {"weights_layers": wb["layers"], "lm_head": wb["lm_head"],
                                            "embedding_rows": wb["embedding_rows"], "kv_read": kv_read,
                                            "kv_write": kv_write},
                              "experts_per_layer": (sum(experts) / len(experts)) if experts else None},
            "clocks": clk.summary(),
            "cpu_baseline": cb,
        }
        print(json.dumps(line))
    for kv in kvs:
        fq.fq_kv_free(kv)
    fq.fq_model_free(model)
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

"""Parity of the CUDA decode path (through the C ABI) with the CPU oracle, on seeded
synthetic Qwen3-shaped inputs small enough for the oracle to finish in seconds while still
spanning several GEMV row tiles, several attention chunks and a ragged last tile."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import (DEV, Pair, assert_bf16_rows_close, assert_layer_close, assert_logits_close, check_routing,
                             max_err, stream, topk_ids)

pytestmark = pytest.mark.gpu

SMALL = wl.Dims(vocab_size=1000, hidden_size=256, intermediate_size=512, num_layers=2, num_attention_heads=4,
                num_key_value_heads=2)
SMALL_G4 = dataclasses.replace(SMALL, num_attention_heads=8, num_key_value_heads=2)
SMALL_MOE = dataclasses.replace(SMALL, num_attention_heads=8, num_key_value_heads=1, num_experts=16,
                                num_experts_used=4, moe_intermediate_size=256)


def workload(dims, wtype="q8_0", kv="bf16", seed=21, **kw):
    return wl.Workload("t", dims, wtype, kv, seed=seed, **kw)


@pytest.fixture
def pair_factory():
    made = []

    def make(*a, **k):
        p = Pair(*a, **k)
        made.append(p)
        return p
    yield make
    for p in made:
        p.close()


# ---------------------------------------------------------------- dequantisation (bit-exact)

@pytest.mark.parametrize("wtype,dims", [("q8_0", SMALL), ("q4_k", SMALL), ("q8_0", SMALL_MOE), ("q4_k", SMALL_MOE)])
def test_dequant_rows_bit_exact(pair_factory, wtype, dims):
    p = pair_factory(workload(dims, wtype), with_oracle=False)
    d = dims
    lw = p.W["layers"][1]
    cases = [(fq.W_TOK_EMBD, p.W["tok_embd"], d.vocab_size, d.hidden_size, 0),
             (fq.W_OUTPUT, p.W["output"], d.vocab_size, d.hidden_size, 0),
             (fq.W_Q, lw["wq"], d.q_dim, d.hidden_size, 1), (fq.W_K, lw["wk"], d.kv_dim, d.hidden_size, 1),
             (fq.W_V, lw["wv"], d.kv_dim, d.hidden_size, 1), (fq.W_O, lw["wo"], d.hidden_size, d.q_dim, 1)]
    if d.is_moe:
        E, Fe = d.num_experts, d.moe_intermediate_size
        cases += [(fq.W_GATE_EXPS, lw["gate_exps"], E * Fe, d.hidden_size, 1),
                  (fq.W_UP_EXPS, lw["up_exps"], E * Fe, d.hidden_size, 1),
                  (fq.W_DOWN_EXPS, lw["down_exps"], E * d.hidden_size, Fe, 1)]
    else:
        cases += [(fq.W_GATE, lw["w_gate"], d.intermediate_size, d.hidden_size, 1),
                  (fq.W_UP, lw["w_up"], d.intermediate_size, d.hidden_size, 1),
                  (fq.W_DOWN, lw["w_down"], d.hidden_size, d.intermediate_size, 1)]
    for which, host, rows, cols, layer in cases:
        for row0, n in [(0, 3), (rows - 5, 5), (rows // 2, 17)]:
            out = torch.empty((n, cols), dtype=torch.float32, device=DEV)
            fq.fq_dequant_rows(p.model, layer, which, row0, n, out.data_ptr(), stream())
            torch.cuda.synchronize()
            ref = oracle.dequant(wtype, host[row0:row0 + n].ravel(), n * cols).reshape(n, cols)
            assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (which, row0)


# ---------------------------------------------------------------- one decoder layer

def test_layer_step_qwen3_0p6b_layer(pair_factory):
    """The single 0.6B-shaped layer at its full size: T = 128 prior f32 positions."""
    w = wl.WORKLOADS["qwen3-0.6b-layer"]
    p = pair_factory(w, max_positions=1024)
    kv, oc = p.new_seq(capacity=w.context + 1, ctx=w.context, seq=0)
    x0 = wl.layer_input(w)
    x = torch.from_numpy(x0.copy()).to(DEV)
    fq.fq_layer_step(p.model, 0, kv, w.context, x.data_ptr(), stream())
    torch.cuda.synchronize()
    ref, _, _ = p.om.layer_step(0, oc, w.context, x0.astype(np.float64))
    assert_layer_close(x.cpu().numpy(), ref, "layer output")
    k, v = p.read_kv(kv, 0, w.context, 1)
    rk, rv = oc.read(0, w.context, 1)
    assert_layer_close(k, rk, "appended k")
    assert_layer_close(v, rv, "appended v")
    assert fq.fq_kv_len(kv) == w.context   # a layer step does not advance len
    # prior positions are untouched
    k0, _ = p.read_kv(kv, 0, 0, w.context)
    rk0, _ = oc.read(0, 0, w.context)
    assert np.array_equal(k0, rk0)


# ---------------------------------------------------------------- decode steps

def _oracle_step_from_gpu_rows(p, kvc, oc, token, pos, what):
    """The oracle's traced step at `pos`, attending over the GPU's appended k/v rows: its own
    rows are computed first and must equal the GPU's within one bf16 rounding; where any row
    differs (a value on a rounding boundary went the other way), the step is taken again
    over the GPU's rows, which then stay in the oracle's cache."""
    out = p.om.decode_step(oc, token, pos, trace=True)
    rows = [p.read_kv(kvc, L, pos, 1) for L in range(p.dims.num_layers)]
    same = True
    for L, (k, v) in enumerate(rows):
        ko, vo = oc.read(L, pos, 1)
        assert_bf16_rows_close(k, ko, f"{what} layer {L} appended k")
        assert_bf16_rows_close(v, vo, f"{what} layer {L} appended v")
        same = same and np.array_equal(k, ko) and np.array_equal(v, vo)
    if same:
        return out
    oc.set_len(pos)
    for L, (k, v) in enumerate(rows):
        oc.write(L, pos, k, v)
    oc.keep_current(True)
    try:
        return p.om.decode_step(oc, token, pos, trace=True)
    finally:
        oc.keep_current(False)


def _compare_step(p, kvs, ocs, tokens, what, gpu_rows=False):
    """One traced step against the oracle's step from the same caches: every layer's residual
    stream under the per-layer tolerance, the logits under 2e-2.  MoE: the expert ids are the
    exact top-k of the GPU's own router logits and equal the oracle's unless the oracle's
    k-th / (k+1)-th router-logit gap is within the measured router error (a near-tie: the
    trajectories then part, and the rest of that sequence's step is not compared).
    gpu_rows: the oracle attends over the GPU's appended rows (`_oracle_step_from_gpu_rows`)."""
    d = p.dims
    n = len(kvs)
    logits = torch.empty((n, d.vocab_size), dtype=torch.float32, device=DEV)
    lo = torch.empty((d.num_layers, n, d.hidden_size), dtype=torch.float32, device=DEV)
    ri = rw = rl = None
    if d.is_moe:
        ri = torch.empty((d.num_layers, n, d.num_experts_used), dtype=torch.int32, device=DEV)
        rw = torch.empty((d.num_layers, n, d.num_experts_used), dtype=torch.float32, device=DEV)
        rl = torch.empty((d.num_layers, n, d.num_experts), dtype=torch.float32, device=DEV)
    fq.fq_decode_step_trace(p.model, kvs, tokens, logits.data_ptr(), lo.data_ptr(),
                            ri.data_ptr() if ri is not None else 0, rw.data_ptr() if rw is not None else 0, stream(),
                            route_logits_ptr=rl.data_ptr() if rl is not None else 0)
    torch.cuda.synchronize()
    got_lg, got_lo = logits.cpu().numpy(), lo.cpu().numpy()
    refs = []
    for s in range(n):
        pos = ocs[s].len
        if gpu_rows:
            lg, lo_ref, rix, rwx = _oracle_step_from_gpu_rows(p, kvs[s], ocs[s], int(tokens[s]), pos, what)
        else:
            lg, lo_ref, rix, rwx = p.om.decode_step(ocs[s], int(tokens[s]), pos, trace=True)
        refs.append(lg)
        parted = False
        for L in range(d.num_layers):
            if d.is_moe:
                gi = ri[L, s].cpu().tolist()
                if sorted(gi) != sorted(rix[L].tolist()):
                    # the oracle's router logits on the GPU's own input to this layer decide
                    # whether this is a near-tie
                    oc2 = p.om.new_cache(ocs[s].capacity)
                    for LL in range(d.num_layers):
                        k, v = ocs[s].read(LL, 0, pos)
                        oc2.write(LL, 0, k, v)
                    oc2.set_len(pos)
                    x_in = got_lo[L - 1, s] if L else oracle.dequant(p.w.weight_dtype, p.W["tok_embd"][int(tokens[s])],
                                                                     d.hidden_size)
                    _, idx, _, rlog = p.om.layer_step(L, oc2, pos, np.asarray(x_in, np.float64), router_logits=True)
                    assert check_routing(gi, rl[L, s].cpu().numpy(), idx, rlog, d.num_experts_used,
                                         f"{what} seq {s} layer {L}") or sorted(gi) == sorted(idx.tolist()), \
                        f"{what} seq {s} layer {L}: routing"
                    parted = True
                    break
                assert sorted(gi) == topk_ids(rl[L, s].cpu().numpy(), d.num_experts_used), (what, s, L)
            assert_layer_close(got_lo[L, s], lo_ref[L], f"{what} seq {s} layer {L}")
            if d.is_moe:
                gw = dict(zip(ri[L, s].cpu().tolist(), rw[L, s].cpu().tolist()))
                assert_layer_close([gw[e] for e in rix[L].tolist()], rwx[L], f"{what} seq {s} layer {L} weights")
        if not parted:
            assert_logits_close(got_lg[s], lg, f"{what} seq {s} logits")
    return got_lg, np.stack(refs)


@pytest.mark.parametrize("dims,wtype,kv", [(SMALL, "q8_0", "bf16"), (SMALL_G4, "q4_k", "bf16"),
                                           (SMALL, "q8_0", "f32"), (SMALL_MOE, "q8_0", "bf16")])
def test_decode_steps_match_oracle(pair_factory, dims, wtype, kv):
    p = pair_factory(workload(dims, wtype, kv), max_positions=512)
    kvc, oc = p.new_seq(capacity=128, ctx=100, seq=0)    # 100 + steps spans two 64-position chunks
    tok = 17
    for step in range(3):
        got, ref = _compare_step(p, [kvc], [oc], [tok], f"step {step}")
        tok = oracle.argmax(ref[0])                      # teacher-forced on the oracle's token
    assert fq.fq_kv_len(kvc) == 103


@pytest.mark.parametrize("dims,ctxs", [(SMALL_G4, [37, 100, 250, 1, 64]), (SMALL_MOE, [37, 100, 250, 1, 64]),
                                       (SMALL_G4, [37, 100, 250, 1, 64, 5, 129, 200, 77, 33, 160, 2]),
                                       (SMALL_MOE, [70, 3, 250, 129, 64, 90, 11, 130, 190])])
def test_batch_ragged_matches_oracle(pair_factory, dims, ctxs):
    """Batches of 8+ run the dense projections on the tcgen05 GEMM."""
    p = pair_factory(workload(dims, "q8_0", "bf16", seed=33), max_positions=1024)
    kvs, ocs = [], []
    for s, c in enumerate(ctxs):
        kvc, oc = p.new_seq(capacity=300, ctx=c, seq=s)
        kvs.append(kvc)
        ocs.append(oc)
    toks = synth.uniform_i32(33, 99, len(ctxs), 0, dims.vocab_size)
    for step in range(2):
        _, ref = _compare_step(p, kvs, ocs, toks, f"batch step {step}")
        toks = ref.argmax(axis=1)


def test_moe_experts_shared_by_many_tokens(pair_factory):
    """Twelve sequences with the same token over the same cache route identically, so every
    chosen expert serves all twelve (three four-row passes of the expert GEMV each)."""
    p = pair_factory(workload(SMALL_MOE, "q8_0", "bf16", seed=34), max_positions=512)
    kvs, ocs = [], []
    for _ in range(12):
        kvc, oc = p.new_seq(capacity=128, ctx=40, seq=0)
        kvs.append(kvc)
        ocs.append(oc)
    got, ref = _compare_step(p, kvs, ocs, [123] * 12, "shared experts")
    for s in range(1, 12):
        assert np.array_equal(got[s], got[0]), f"sequence {s} differs from sequence 0"


@pytest.mark.parametrize("dims,wtype,rows", [(SMALL, "q8_0", 1), (SMALL, "q8_0", 3), (SMALL, "q8_0", 9),
                                             (SMALL_G4, "q4_k", 5), (SMALL_MOE, "q8_0", 4), (SMALL_MOE, "q8_0", 12)])
def test_all_logits_step_matches_sequential_oracle(pair_factory, dims, wtype, rows):
    """forwardStepAllLogits (section 14.1): the rows' logits equal the oracle's consecutive
    single-token steps; the cache ends where those steps leave it."""
    p = pair_factory(workload(dims, wtype, "bf16", seed=35), max_positions=512)
    ctx = 70                                        # rows cross the 64-position tile boundary
    kvc, oc = p.new_seq(capacity=128, ctx=ctx, seq=0)
    toks = [int(t) for t in synth.uniform_i32(35, 5, rows, 0, dims.vocab_size)]
    logits = torch.empty((rows, dims.vocab_size), dtype=torch.float32, device=DEV)
    fq.fq_decode_step_all_logits(p.model, kvc, toks, ctx, logits.data_ptr(), stream())
    torch.cuda.synchronize()
    assert fq.fq_kv_len(kvc) == ctx + rows
    got = logits.cpu().numpy()
    for i, t in enumerate(toks):
        ref = p.om.decode_step(oc, t, ctx + i)
        assert_logits_close(got[i], ref, f"row {i}")
    for L in range(dims.num_layers):
        k, v = p.read_kv(kvc, L, ctx, rows)
        kr, vr = oc.read(L, ctx, rows)
        for got_c, ref_c, name in ((k, kr, "k"), (v, vr, "v")):
            # stored bf16: a value on a rounding boundary may land one ulp (2^-7 of it) away
            # on top of the per-layer tolerance of the f32 arithmetic that produced it
            tol = 2.0 ** -7 * np.abs(ref_c) + 1e-3 * float(np.abs(ref_c).max()) + 1e-4
            assert np.all(np.abs(got_c - ref_c) <= tol), f"layer {L} appended {name}"


def test_all_logits_step_contract(pair_factory):
    p = pair_factory(workload(SMALL, "q8_0", "bf16", seed=36), max_positions=512, with_oracle=False)
    kvc, _ = p.new_seq(capacity=16, ctx=10, seq=0, oracle_cache=False)
    out = torch.empty((70, SMALL.vocab_size), dtype=torch.float32, device=DEV)
    for toks, pos0, status in [([1, 2], 9, fq.INVALID_SEQUENCE_LENGTH), ([], 10, fq.INVALID_SEQUENCE_LENGTH),
                               ([1] * 65, 10, fq.INVALID_SEQUENCE_LENGTH), ([1] * 7, 10, fq.KV_CACHE_OVERFLOW),
                               ([1, SMALL.vocab_size], 10, fq.INVALID_ARGUMENT)]:
        with pytest.raises(fq.FqError) as e:
            fq.fq_decode_step_all_logits(p.model, kvc, toks, pos0, out.data_ptr(), stream())
        assert e.value.status == status, (len(toks), pos0)
        assert fq.fq_kv_len(kvc) == 10             # a refused step leaves the cache as it was
    fq.fq_decode_step_all_logits(p.model, kvc, [1] * 6, 10, out.data_ptr(), stream())   # exactly fills it
    assert fq.fq_kv_len(kvc) == 16


def test_graph_replay_equals_direct_launches(pair_factory):
    # the kernel sequence captured once and replayed, against the same kernels launched directly
    p = pair_factory(workload(SMALL_G4, "q8_0", "bf16"), max_positions=512, with_oracle=False)
    fq.fq_set_option(p.model, fq.OPT_STEP_PATH, fq.PATH_KERNELS)
    a, _ = p.new_seq(capacity=256, ctx=150, seq=0, oracle_cache=False)
    b, _ = p.new_seq(capacity=256, ctx=150, seq=0, oracle_cache=False)
    la = torch.empty(SMALL_G4.vocab_size, dtype=torch.float32, device=DEV)
    lb = torch.empty_like(la)
    for t in (5, 6, 7):
        fq.fq_decode_step(p.model, a, t, fq.fq_kv_len(a), la.data_ptr(), stream())        # graph
        fq.fq_decode_step_trace(p.model, [b], [t], lb.data_ptr(), 0, 0, 0, stream())      # direct
        torch.cuda.synchronize()
        assert torch.equal(la, lb)


def test_cached_steps_equal_oracle_cacheless_forward(pair_factory):
    """The pages' own check: last logits of a cached prefill equal the no-cache forward."""
    p = pair_factory(workload(SMALL, "q8_0", "bf16", seed=44), max_positions=256)
    kvc, _ = p.new_seq(capacity=64, ctx=0, seq=0, oracle_cache=False)
    toks = synth.uniform_i32(44, 5, 40, 0, SMALL.vocab_size)
    logits = torch.empty(SMALL.vocab_size, dtype=torch.float32, device=DEV)
    for pos, t in enumerate(toks):
        fq.fq_decode_step(p.model, kvc, int(t), pos, logits.data_ptr(), stream())
    torch.cuda.synchronize()
    ref = p.om.forward_last_logits(toks)
    assert_logits_close(logits.cpu().numpy(), ref, "cached vs cacheless")


def test_greedy_chain_matches_oracle(pair_factory):
    p = pair_factory(workload(SMALL_G4, "q8_0", "bf16", seed=55), max_positions=512)
    ctxs = [90, 200]
    kvs, ocs = [], []
    for s, c in enumerate(ctxs):
        kvc, oc = p.new_seq(capacity=256, ctx=c, seq=s)
        kvs.append(kvc)
        ocs.append(oc)
    steps = 6
    out = torch.empty((steps, 2), dtype=torch.int32, device=DEV)
    logits = torch.empty((2, SMALL_G4.vocab_size), dtype=torch.float32, device=DEV)
    first = [3, 4]
    fq.fq_decode_greedy(p.model, kvs, first, steps, out.data_ptr(), logits.data_ptr(), stream())
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for s in range(2):
        tok, parted = first[s], False
        for i in range(steps):
            lg = p.om.decode_step(ocs[s], tok, ocs[s].len)
            order = np.argsort(-lg)
            if got[i, s] != order[0]:
                gap = lg[order[0]] - lg[order[1]]
                assert gap < 4e-2, f"seq {s} step {i}: token {got[i, s]} vs {order[0]} (gap {gap})"
                parted = True                             # a near-tie: the chains may part here
                break
            tok = int(order[0])
        assert fq.fq_kv_len(kvs[s]) == ctxs[s] + steps
        if not parted:                                    # the last step's logits are returned
            assert_logits_close(logits[s].cpu().numpy(), lg, f"greedy seq {s} last logits")


# ---------------------------------------------------------------- contract errors

def test_contract_errors_leave_state_unchanged(pair_factory):
    p = pair_factory(workload(SMALL, "q8_0", "bf16"), max_positions=256, with_oracle=False)
    q = pair_factory(workload(SMALL, "q8_0", "bf16"), max_positions=256, with_oracle=False)
    a, _ = p.new_seq(capacity=8, ctx=7, seq=0, oracle_cache=False)
    b, _ = p.new_seq(capacity=8, ctx=2, seq=1, oracle_cache=False)
    other, _ = q.new_seq(capacity=8, ctx=2, seq=0, oracle_cache=False)
    lg = torch.empty((2, SMALL.vocab_size), dtype=torch.float32, device=DEV)

    def status(fn):
        try:
            fn()
        except fq.FqError as e:
            return e.status
        return fq.OK

    assert status(lambda: fq.fq_decode_step(p.model, a, 1, 6, lg.data_ptr(), stream())) == fq.INVALID_SEQUENCE_LENGTH
    assert status(lambda: fq.fq_decode_step(p.model, a, SMALL.vocab_size, 7, lg.data_ptr(), stream())) == \
        fq.INVALID_ARGUMENT
    assert status(lambda: fq.fq_decode_step_batch(p.model, [a, a], [1, 2], lg.data_ptr(), stream())) == \
        fq.MISMATCHED_KV_CACHES
    assert status(lambda: fq.fq_decode_step_batch(p.model, [a, other], [1, 2], lg.data_ptr(), stream())) == \
        fq.MISMATCHED_KV_CACHES
    assert status(lambda: fq.fq_decode_greedy(p.model, [a], [1], 2, 0, 0, stream())) == fq.KV_CACHE_OVERFLOW
    assert status(lambda: fq.fq_decode_step_batch(p.model, [], [], lg.data_ptr(), stream())) == \
        fq.INVALID_SEQUENCE_LENGTH
    assert status(lambda: fq.fq_kv_append(a, 0, 3, 1, lg.data_ptr(), lg.data_ptr(), stream())) == \
        fq.INVALID_SEQUENCE_LENGTH
    assert fq.fq_kv_len(a) == 7 and fq.fq_kv_len(b) == 2
    fq.fq_decode_step(p.model, a, 1, 7, lg.data_ptr(), stream())     # fills the last slot
    assert fq.fq_kv_len(a) == 8
    assert status(lambda: fq.fq_decode_step(p.model, a, 1, 8, lg.data_ptr(), stream())) == fq.KV_CACHE_OVERFLOW
    assert fq.fq_kv_len(a) == 8
    torch.cuda.synchronize()

"""Stage-by-stage parity of one decoder layer: the raw QKV projection, the attention
output per head, the SwiGLU activations and each weight GEMV on its own, each against
the oracle's building blocks composed in the order the runner page gives."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import DEV, Pair, assert_layer_close, stream

pytestmark = pytest.mark.gpu

SMALL = wl.Dims(vocab_size=1000, hidden_size=256, intermediate_size=512, num_layers=2, num_attention_heads=4,
                num_key_value_heads=2)


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


def _gemv_ref(wtype, W, rows, cols, x):
    return oracle.gemv(wtype, W, rows, cols, x)


@pytest.mark.parametrize("wtype,n", [("q8_0", 1), ("q8_0", 3), ("q8_0", 6), ("q4_k", 1), ("q4_k", 3), ("q4_k", 6),
                                     ("q8_0", 8), ("q8_0", 13), ("q8_0", 32)])
def test_weight_gemv_matches_oracle(pair_factory, wtype, n):
    """n >= 8 on Q8_0 runs the tcgen05 GEMM (f16 weights, f16 hi/lo activations)."""
    d = dataclasses.replace(SMALL, hidden_size=512, intermediate_size=768 if wtype == "q8_0" else 1024)
    p = pair_factory(wl.Workload("g", d, wtype, "bf16", seed=71), with_oracle=False)
    lw = p.W["layers"][1]
    H, F = d.hidden_size, d.intermediate_size
    cases = [
        (fq.W_Q, [(lw["wq"], d.q_dim), (lw["wk"], d.kv_dim), (lw["wv"], d.kv_dim)], H, "concat"),
        (fq.W_O, [(lw["wo"], H)], d.q_dim, "concat"),
        (fq.W_GATE, [(lw["w_gate"], F), (lw["w_up"], F)], H, "interleave"),
        (fq.W_DOWN, [(lw["w_down"], H)], F, "concat"),
        (fq.W_OUTPUT, [(p.W["output"], d.vocab_size)], H, "concat"),
    ]
    for which, parts, cols, mode in cases:
        x = synth.normal_f32(5, 100 + which, n * cols).reshape(n, cols)
        rows = sum(r for _, r in parts)
        y = torch.empty((n, rows), dtype=torch.float32, device=DEV)
        xt = torch.from_numpy(x).to(DEV)
        fq.fq_gemv(p.model, 1, which, n, xt.data_ptr(), y.data_ptr(), stream())
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        for b in range(n):
            outs = [_gemv_ref(wtype, W, r, cols, x[b].astype(np.float64)) for W, r in parts]
            if mode == "concat":
                ref = np.concatenate(outs)
            else:
                ref = np.empty(rows)
                ref[0::2], ref[1::2] = outs[0], outs[1]
            assert_layer_close(got[b], ref, f"gemv which={which} row {b}")


@pytest.mark.parametrize("wtype,n", [("q8_0", 1), ("q8_0", 3), ("q4_k", 1), ("q4_k", 3)])
def test_tma_gemv_many_rows_matches_oracle(pair_factory, wtype, n):
    """8192 output rows give every SM a row tile, so the TMA-fed kernel serves this matrix
    (smaller ones go to the register-fed kernel, covered above)."""
    d = dataclasses.replace(SMALL, vocab_size=8192, hidden_size=512, intermediate_size=1024)
    p = pair_factory(wl.Workload("gt", d, wtype, "bf16", seed=73), with_oracle=False)
    x = synth.normal_f32(6, 7, n * d.hidden_size).reshape(n, d.hidden_size)
    y = torch.empty((n, d.vocab_size), dtype=torch.float32, device=DEV)
    xt = torch.from_numpy(x).to(DEV)
    fq.fq_gemv(p.model, 0, fq.W_OUTPUT, n, xt.data_ptr(), y.data_ptr(), stream())
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    for b in range(n):
        ref = _gemv_ref(wtype, p.W["output"], d.vocab_size, d.hidden_size, x[b].astype(np.float64))
        assert_layer_close(got[b], ref, f"LM-head rows, activation row {b}")


@pytest.mark.parametrize("kv", ["bf16", "f32"])
def test_layer_stages_match_oracle(pair_factory, kv):
    d = SMALL
    w = wl.Workload("s", d, "q8_0", kv, seed=72)
    p = pair_factory(w, max_positions=512)
    ctx = 100
    kvc, oc = p.new_seq(capacity=128, ctx=ctx, seq=0)
    x0 = synth.normal_f32(72, 9, d.hidden_size)
    x = torch.from_numpy(x0.copy()).to(DEV)
    qkv = torch.empty(d.q_dim + 2 * d.kv_dim, dtype=torch.float32, device=DEV)
    attn = torch.empty(d.q_dim, dtype=torch.float32, device=DEV)
    ffn = torch.empty(d.intermediate_size, dtype=torch.float32, device=DEV)
    fq.fq_layer_step_trace(p.model, 0, kvc, ctx, x.data_ptr(), qkv.data_ptr(), attn.data_ptr(), ffn.data_ptr(),
                           stream())
    torch.cuda.synchronize()

    lw = p.W["layers"][0]
    eps, D, G = d.rms_norm_eps, d.head_dim, d.num_attention_heads // d.num_key_value_heads
    xd = x0.astype(np.float64)
    xn = oracle.rmsnorm(xd, lw["attn_norm"], eps)
    q = oracle.gemv("q8_0", lw["wq"], d.q_dim, d.hidden_size, xn)
    k = oracle.gemv("q8_0", lw["wk"], d.kv_dim, d.hidden_size, xn)
    v = oracle.gemv("q8_0", lw["wv"], d.kv_dim, d.hidden_size, xn)
    assert_layer_close(qkv.cpu().numpy(), np.concatenate([q, k, v]), "raw qkv")

    x1, _, _ = p.om.layer_step(0, oc, ctx, xd)          # appends k/v at ctx in the oracle cache
    K, V = oc.read(0, 0, ctx + 1)
    o = np.empty(d.q_dim)
    for h in range(d.num_attention_heads):
        qh = oracle.rope(oracle.rmsnorm(q[h * D:(h + 1) * D], lw["q_norm"], eps), ctx, d.rope_theta)
        g = h // G
        o[h * D:(h + 1) * D] = oracle.attention(qh, K[:, g, :], V[:, g, :])
    assert_layer_close(attn.cpu().numpy(), o, "attention output")

    xa = xd + oracle.gemv("q8_0", lw["wo"], d.hidden_size, d.q_dim, o)
    xn2 = oracle.rmsnorm(xa, lw["ffn_norm"], eps)
    gt = oracle.gemv("q8_0", lw["w_gate"], d.intermediate_size, d.hidden_size, xn2)
    up = oracle.gemv("q8_0", lw["w_up"], d.intermediate_size, d.hidden_size, xn2)
    hh = np.array([oracle.silu(float(a)) for a in gt]) * up
    assert_layer_close(ffn.cpu().numpy(), hh, "swiglu activations")
    assert_layer_close(x.cpu().numpy(), x1, "layer output")

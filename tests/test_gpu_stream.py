"""The streamed batch-1 step (one persistent kernel per forwardStep, "14. Model families"
section 14.2) against the oracle and against the kernel sequence, over the cache lengths
that decide its work split: an empty cache (the new position alone), fewer positions than
attention chunks, a length inside one 32-position tile, and lengths with ragged tiles."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import DEV, assert_logits_close, stream
from tests.test_gpu_parity import SMALL, SMALL_G4, SMALL_MOE, _compare_step, pair_factory, workload  # noqa: F401

pytestmark = pytest.mark.gpu

SMALL_G1 = dataclasses.replace(SMALL, num_attention_heads=2, num_key_value_heads=2)
# attention chunks per kv head exceed the head_dim / 8 merge slices (S > 16 for 8 kv heads)
SMALL_KV8 = dataclasses.replace(SMALL, num_attention_heads=16, num_key_value_heads=8, intermediate_size=768)


@pytest.mark.parametrize("dims,wtype", [(SMALL, "q8_0"), (SMALL_G4, "q4_k"), (SMALL_G1, "q8_0"), (SMALL_KV8, "q8_0"),
                                        (SMALL_KV8, "q4_k")],
                         ids=["g2-q8_0", "g4-q4_k", "g1-q8_0", "kv8-q8_0", "kv8-q4_k"])
@pytest.mark.parametrize("ctx", [0, 1, 37, 300])
def test_streamed_steps_match_oracle_per_layer(pair_factory, dims, wtype, ctx):  # noqa: F811
    p = pair_factory(workload(dims, wtype, "bf16", seed=71 + ctx), max_positions=512)
    assert fq.fq_step_path(p.model, 1, "bf16")
    kvc, oc = p.new_seq(capacity=ctx + 8, ctx=ctx, seq=0)
    tok = 11
    for step in range(3):
        # the appended rows hold the oracle's k/v rounded to bf16 (a rounding decision at a
        # boundary may go either way); the oracle attends over the GPU's rows, in this step
        # and the later ones, so that every layer is compared from the same cache
        _, ref = _compare_step(p, [kvc], [oc], [tok], f"ctx {ctx} step {step}", gpu_rows=True)
        assert fq.fq_step_kernels(p.model, stream()) in (0, 1)
        tok = oracle.argmax(ref[0])


@pytest.mark.parametrize("dims,wtype", [(SMALL, "q8_0"), (SMALL_G4, "q4_k")], ids=["g2-q8_0", "g4-q4_k"])
def test_streamed_step_agrees_with_kernel_sequence(pair_factory, dims, wtype):  # noqa: F811
    p = pair_factory(workload(dims, wtype, "bf16", seed=5), max_positions=512, with_oracle=False)
    a, _ = p.new_seq(capacity=256, ctx=150, seq=0, oracle_cache=False)
    b, _ = p.new_seq(capacity=256, ctx=150, seq=0, oracle_cache=False)
    la = torch.empty(dims.vocab_size, dtype=torch.float32, device=DEV)
    lb = torch.empty_like(la)
    lc = torch.empty_like(la)
    for t in (5, 6, 7):
        pos = fq.fq_kv_len(a)
        fq.fq_decode_step(p.model, a, t, pos, la.data_ptr(), stream())
        assert fq.fq_step_kernels(p.model, stream()) == 1
        fq.fq_set_option(p.model, fq.OPT_STEP_PATH, fq.PATH_KERNELS)
        fq.fq_decode_step(p.model, b, t, pos, lb.data_ptr(), stream())
        assert fq.fq_step_kernels(p.model, stream()) > 1
        fq.fq_set_option(p.model, fq.OPT_STEP_PATH, fq.PATH_AUTO)
        torch.cuda.synchronize()
        assert_logits_close(la.cpu().numpy(), lb.cpu().numpy(), f"token {t}: streamed vs kernel sequence")
    # the streamed step is deterministic: the same inputs give the same bits
    fq.fq_kv_rewind(a, 150)
    for t in (5, 6, 7):
        fq.fq_decode_step(p.model, a, t, fq.fq_kv_len(a), lc.data_ptr(), stream())
    torch.cuda.synchronize()
    assert torch.equal(la, lc)


def test_streamed_greedy_chain_matches_oracle(pair_factory):  # noqa: F811
    p = pair_factory(workload(SMALL_KV8, "q8_0", "bf16", seed=57), max_positions=512)
    kvc, oc = p.new_seq(capacity=256, ctx=120, seq=0)
    steps = 8
    out = torch.empty(steps, dtype=torch.int32, device=DEV)
    logits = torch.empty(SMALL_KV8.vocab_size, dtype=torch.float32, device=DEV)
    fq.fq_decode_greedy(p.model, [kvc], [9], steps, out.data_ptr(), logits.data_ptr(), stream())
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert fq.fq_step_kernels(p.model, stream()) == 1
    tok, parted = 9, False
    for i in range(steps):
        lg = p.om.decode_step(oc, tok, oc.len)
        order = np.argsort(-lg)
        if got[i] != order[0]:
            gap = lg[order[0]] - lg[order[1]]
            assert gap < 4e-2, f"step {i}: token {got[i]} vs {order[0]} (gap {gap})"
            parted = True                        # a near-tie: the chains may part here
            break
        tok = int(order[0])
    assert fq.fq_kv_len(kvc) == 120 + steps
    if not parted:
        assert_logits_close(logits.cpu().numpy(), lg, "greedy last logits")


def test_step_path_choice(pair_factory):  # noqa: F811
    dense = pair_factory(workload(SMALL, "q8_0", "bf16"), max_positions=256, with_oracle=False)
    assert fq.fq_step_path(dense.model, 1, "bf16")
    assert not fq.fq_step_path(dense.model, 2, "bf16")        # lockstep batches: the kernel sequence
    assert not fq.fq_step_path(dense.model, 1, "f32")
    assert not fq.fq_step_path(dense.model, 1, "q8_0")
    fq.fq_set_option(dense.model, fq.OPT_STEP_PATH, fq.PATH_KERNELS)
    assert not fq.fq_step_path(dense.model, 1, "bf16")
    with pytest.raises(fq.FqError):
        fq.fq_set_option(dense.model, fq.OPT_STEP_PATH, 7)
    moe = pair_factory(workload(SMALL_MOE, "q8_0", "bf16"), max_positions=256, with_oracle=False)
    assert not fq.fq_step_path(moe.model, 1, "bf16")


@pytest.mark.parametrize("opt,value", [(fq.OPT_DEPENDENT_LAUNCH, 1), (fq.OPT_GRAPHS, 0), (fq.OPT_TENSOR_CORES, 0)],
                         ids=["dependent-launch", "no-graphs", "no-tensor-cores"])
def test_kernel_sequence_options_match_oracle(pair_factory, opt, value):  # noqa: F811
    # the options choose between equivalent launches of the same kernels; each must still
    # match the oracle (a batch of 9 reaches the tensor-core GEMM unless it is switched off)
    p = pair_factory(workload(SMALL_G4, "q8_0", "bf16", seed=13), max_positions=512)
    fq.fq_set_option(p.model, opt, value)
    kvs, ocs = [], []
    ctxs = [30, 90, 5, 64, 128, 1, 77, 33, 200]
    for s, c in enumerate(ctxs):
        kvc, oc = p.new_seq(capacity=256, ctx=c, seq=s)
        kvs.append(kvc)
        ocs.append(oc)
    logits = torch.empty((len(ctxs), SMALL_G4.vocab_size), dtype=torch.float32, device=DEV)
    toks = synth.uniform_i32(13, 2, len(ctxs), 0, SMALL_G4.vocab_size).tolist()
    for step in range(2):
        fq.fq_decode_step_batch(p.model, kvs, toks, logits.data_ptr(), stream())
        torch.cuda.synchronize()
        got = logits.cpu().numpy()
        for s in range(len(ctxs)):
            ref = p.om.decode_step(ocs[s], toks[s], ocs[s].len)
            assert_logits_close(got[s], ref, f"option {opt}={value} step {step} seq {s}")
            toks[s] = oracle.argmax(ref)

"""Multi-token forwardStep (section 14.1) on the CUDA path against the oracle: a prefill is
one call on a fresh cache at pos0 = 0, its logits equal forwardLastLogits over the same ids,
and the cache then holds what consecutive single steps append."""
import numpy as np
import pytest
import torch

import oracle
import synth
from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import DEV, assert_logits_close, assert_q8_rows_close, stream
from tests.test_gpu_parity import SMALL, SMALL_G4, SMALL_MOE, _compare_step, pair_factory, workload  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dims,wtype,kv,n", [(SMALL, "q8_0", "bf16", 77), (SMALL_G4, "q4_k", "bf16", 40),
                                             (SMALL_MOE, "q8_0", "bf16", 33), (SMALL, "q8_0", "q8_0", 70),
                                             (SMALL, "q8_0", "f32", 5), (SMALL, "q8_0", "bf16", 1)])
def test_prefill_matches_cacheless_oracle(pair_factory, dims, wtype, kv, n):
    """Section 14.1: a prefill is one forwardStep call on a fresh cache at pos0 = 0 and its
    logits equal forwardLastLogits over the same ids.  77 tokens run as passes of 32, 32 and
    13 rows; the cache then holds what consecutive steps append, and decoding continues."""
    p = pair_factory(workload(dims, wtype, kv, seed=37), max_positions=512)
    kvc, oc = p.new_seq(capacity=128, ctx=0, seq=0)
    toks = [int(t) for t in synth.uniform_i32(37, 7, n, 0, dims.vocab_size)]
    logits = torch.empty(dims.vocab_size, dtype=torch.float32, device=DEV)
    fq.fq_forward_step(p.model, kvc, toks, 0, logits.data_ptr(), stream())
    torch.cuda.synchronize()
    assert fq.fq_kv_len(kvc) == n
    ref = p.om.forward_last_logits(toks)
    assert_logits_close(logits.cpu().numpy(), ref, "prefill logits")
    for i, t in enumerate(toks):
        p.om.decode_step(oc, t, i, logits=False)
    for L in range(dims.num_layers):
        k, v = p.read_kv(kvc, L, 0, n)
        kr, vr = oc.read(L, 0, n)
        for got_c, ref_c, name in ((k, kr, "k"), (v, vr, "v")):
            if kv == "q8_0":
                assert_q8_rows_close(got_c, ref_c, f"layer {L} {name}")
            else:
                tol = 2.0 ** -7 * np.abs(ref_c) + 1e-3 * float(np.abs(ref_c).max()) + 1e-4
                assert np.all(np.abs(got_c - ref_c) <= tol), f"layer {L} prefilled {name}"
    # decoding continues from the prefilled cache (MoE routing checked for near-ties)
    _compare_step(p, [kvc], [oc], [oracle.argmax(ref)], "step after prefill")


def test_forward_step_contract(pair_factory):
    p = pair_factory(workload(SMALL, "q8_0", "bf16", seed=38), max_positions=512, with_oracle=False)
    kvc, _ = p.new_seq(capacity=40, ctx=10, seq=0, oracle_cache=False)
    out = torch.empty(SMALL.vocab_size, dtype=torch.float32, device=DEV)
    for toks, pos0, status in [([], 10, fq.INVALID_SEQUENCE_LENGTH), ([1, 2], 9, fq.INVALID_SEQUENCE_LENGTH),
                               ([1] * 31, 10, fq.KV_CACHE_OVERFLOW), ([1, SMALL.vocab_size], 10, fq.INVALID_ARGUMENT),
                               ([1, -1], 10, fq.INVALID_ARGUMENT)]:
        with pytest.raises(fq.FqError) as e:
            fq.fq_forward_step(p.model, kvc, toks, pos0, out.data_ptr(), stream())
        assert e.value.status == status, (toks, pos0)
        assert fq.fq_kv_len(kvc) == 10
    # logits may be omitted: the rows are appended all the same; a full cache then overflows
    fq.fq_forward_step(p.model, kvc, list(range(30)), 10, 0, stream())
    torch.cuda.synchronize()
    assert fq.fq_kv_len(kvc) == 40
    with pytest.raises(fq.FqError) as e:
        fq.fq_forward_step(p.model, kvc, [1], 40, out.data_ptr(), stream())
    assert e.value.status == fq.KV_CACHE_OVERFLOW

"""fq_layer_step_noalloc: the layer step for callers that cannot allocate device memory
(an allocator locked after start-up, a graph being captured, a host that plans every device
byte).  It must give the same results as fq_layer_step, call after call, while keeping all
scratch in the library's built-in array, and refuse shapes whose scratch does not fit."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
import synth.workloads as wl
from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import DEV, Pair, assert_layer_close, stream

pytestmark = pytest.mark.gpu

DENSE = wl.Dims(vocab_size=1000, hidden_size=256, intermediate_size=512, num_layers=2, num_attention_heads=8,
                num_key_value_heads=2)


def test_noalloc_layer_step_matches_layer_step_twice():
    p = Pair(wl.Workload("na", DENSE, "q8_0", "bf16", seed=91), max_positions=512, with_oracle=False)
    try:
        ctx = 100
        a, _ = p.new_seq(capacity=128, ctx=ctx, seq=0, oracle_cache=False)   # existing entry point
        b, _ = p.new_seq(capacity=128, ctx=ctx, seq=0, oracle_cache=False)   # allocation-free one
        x0 = synth.normal_f32(91, 7, DENSE.hidden_size)
        xa = torch.from_numpy(x0.copy()).to(DEV)
        xb = torch.from_numpy(x0.copy()).to(DEV)
        for call, layer in enumerate((0, 1)):
            pos = ctx + call
            fq.fq_layer_step(p.model, layer, a, pos, xa.data_ptr(), stream())
            fq.fq_layer_step_noalloc(p.model, layer, b, pos, xb.data_ptr(), stream())
            torch.cuda.synchronize()
            ga, gb = xa.cpu().numpy(), xb.cpu().numpy()
            assert_layer_close(gb, ga, f"call {call}: residual stream")
            ka, va = p.read_kv(a, layer, pos, 1)
            kb, vb = p.read_kv(b, layer, pos, 1)
            assert_layer_close(kb, ka, f"call {call}: appended k")
            assert_layer_close(vb, va, f"call {call}: appended v")
            fq.fq_kv_commit(a, pos + 1)
            fq.fq_kv_commit(b, pos + 1)
        fq.fq_check_device(p.model, stream())
    finally:
        p.close()


def test_noalloc_rejects_scratch_beyond_the_array():
    # 64 query heads at a 40960-position cache need ~2.7 MiB of split-K partials alone
    wide = dataclasses.replace(DENSE, num_layers=1, num_attention_heads=64, num_key_value_heads=8)
    p = Pair(wl.Workload("na-wide", wide, "q8_0", "bf16", seed=92), max_positions=40960, with_oracle=False)
    try:
        kv = fq.fq_kv_init(p.model, 40960, "bf16")
        p.kvs.append(kv)
        x = torch.zeros(wide.hidden_size, dtype=torch.float32, device=DEV)
        with pytest.raises(fq.FqError) as e:
            fq.fq_layer_step_noalloc(p.model, 0, kv, 0, x.data_ptr(), stream())
        assert e.value.status == fq.INVALID_ARGUMENT
        assert "scratch" in str(e.value)
    finally:
        p.close()

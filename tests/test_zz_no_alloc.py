"""fq_layer_step_noalloc: the layer step for callers that cannot allocate device memory when
they call it -- an engine whose allocator is sealed after start-up, a host that budgets
every device byte in advance, or code that runs where a cudaMalloc would stall or break
the surrounding work.  It must give the same bits as fq_layer_step (same kernels, same
splits), call after call, stay within the oracle's per-layer tolerance, keep all scratch in
the library's built-in array (no device memory is taken), and refuse shapes whose scratch
does not fit.  This file is collected last on purpose."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
import synth.workloads as wl
from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import DEV, Pair, assert_layer_close, assert_q8_rows_close

pytestmark = pytest.mark.gpu

DENSE = wl.Dims(vocab_size=1000, hidden_size=256, intermediate_size=512, num_layers=2, num_attention_heads=8,
                num_key_value_heads=2)
MOE = dataclasses.replace(DENSE, num_attention_heads=8, num_key_value_heads=1, num_experts=16, num_experts_used=4,
                          moe_intermediate_size=256)


def _free_device_bytes() -> int:
    free, _ = torch.cuda.mem_get_info(DEV)   # cudaMemGetInfo
    return int(free)


@pytest.mark.parametrize("dims,kv", [(DENSE, "bf16"), (MOE, "bf16"), (DENSE, "q8_0")],
                         ids=["dense-bf16", "moe-bf16", "dense-q8_0"])
def test_noalloc_layer_step_matches_layer_step_and_oracle(dims, kv):
    p = Pair(wl.Workload("na", dims, "q8_0", kv, seed=91), max_positions=512)
    ref_stream = torch.cuda.Stream(DEV)
    # a stream the library has never seen: if the call reached for a per-stream workspace,
    # it would have to allocate one
    na_stream = torch.cuda.Stream(DEV)
    try:
        ctx = 100
        a, oc = p.new_seq(capacity=128, ctx=ctx, seq=0)                   # existing entry point + oracle
        b, _ = p.new_seq(capacity=128, ctx=ctx, seq=0, oracle_cache=False)  # allocation-free one
        x0 = synth.normal_f32(91, 7, dims.hidden_size)
        xa = torch.from_numpy(x0.copy()).to(DEV)
        xb = torch.from_numpy(x0.copy()).to(DEV)
        x_in = x0.astype(np.float64)   # the oracle is teacher-forced on the GPU's layer input
        # a first call on this device finds the built-in array's device address (the driver may
        # load the library's module then); every later call must take no device memory
        warm, _ = p.new_seq(capacity=128, ctx=ctx, seq=1, oracle_cache=False)
        xw = torch.from_numpy(x0.copy()).to(DEV)
        fq.fq_layer_step_noalloc(p.model, 0, warm, ctx, xw.data_ptr(), na_stream.cuda_stream)
        torch.cuda.synchronize()
        for call, layer in enumerate((0, 1)):
            pos = ctx + call
            fq.fq_layer_step(p.model, layer, a, pos, xa.data_ptr(), ref_stream.cuda_stream)
            ref_stream.synchronize()
            free0 = _free_device_bytes()
            fq.fq_layer_step_noalloc(p.model, layer, b, pos, xb.data_ptr(), na_stream.cuda_stream)
            na_stream.synchronize()
            assert _free_device_bytes() == free0, f"call {call}: device memory was taken"
            ga, gb = xa.cpu().numpy(), xb.cpu().numpy()
            assert np.array_equal(gb, ga), f"call {call}: residual stream differs from fq_layer_step"
            ka, va = p.read_kv(a, layer, pos, 1)
            kb, vb = p.read_kv(b, layer, pos, 1)
            assert np.array_equal(kb, ka) and np.array_equal(vb, va), f"call {call}: appended k/v differ"
            xo, _, _ = p.om.layer_step(layer, oc, pos, x_in)
            oc.set_len(pos + 1)
            assert_layer_close(gb, xo, f"call {call}: residual stream vs oracle")
            ko, vo = oc.read(layer, pos, 1)
            if kv == "q8_0":
                assert_q8_rows_close(kb, ko, f"call {call}: appended k vs oracle")
                assert_q8_rows_close(vb, vo, f"call {call}: appended v vs oracle")
            else:
                assert_layer_close(kb, ko, f"call {call}: appended k vs oracle")
                assert_layer_close(vb, vo, f"call {call}: appended v vs oracle")
            x_in = gb.astype(np.float64)
            fq.fq_kv_commit(a, pos + 1)
            fq.fq_kv_commit(b, pos + 1)
        fq.fq_check_device(p.model, na_stream.cuda_stream)
    finally:
        torch.cuda.synchronize()
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
            fq.fq_layer_step_noalloc(p.model, 0, kv, 0, x.data_ptr(), torch.cuda.current_stream(DEV).cuda_stream)
        assert e.value.status == fq.INVALID_ARGUMENT
        assert "scratch" in str(e.value)
    finally:
        p.close()

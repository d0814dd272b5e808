"""The C ABI without a GPU: the library loads, exports every entry point include/fq.h
declares, and validates descriptors (section 14.2 rules) on the host."""
import os
import re

import pytest

from quantized_decoder_decode_gb300 import build as fqbuild
from quantized_decoder_decode_gb300 import fq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fqbuild.build()
    return fq.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fq.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fq_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("fq_desc_init", "fq_load_weights", "fq_layer_step", "fq_decode_step", "fq_decode_step_batch",
                     "fq_kv_append"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(fq.EXPORTED) <= set(declared_symbols())


QWEN3_0P6B = dict(vocab_size=151936, hidden_size=1024, intermediate_size=3072, num_layers=28,
                  num_attention_heads=16, num_key_value_heads=8, head_dim=128)


def status_of(**p):
    try:
        fq.fq_desc_init(**p)
    except fq.FqError as e:
        return e.status
    return fq.OK


def test_desc_validation(lib):
    assert status_of(**QWEN3_0P6B) == fq.OK
    moe = dict(QWEN3_0P6B, hidden_size=2048, num_attention_heads=32, num_key_value_heads=4, num_layers=48,
               num_experts=128, num_experts_used=8, moe_intermediate_size=768)
    assert status_of(**moe) == fq.OK
    bad = [dict(QWEN3_0P6B, num_attention_heads=0), dict(QWEN3_0P6B, num_key_value_heads=0),
           dict(QWEN3_0P6B, num_key_value_heads=3), dict(QWEN3_0P6B, head_dim=127),
           dict(QWEN3_0P6B, num_experts=8), dict(moe, num_experts_used=129), dict(moe, moe_expert_top_p=0.5),
           dict(QWEN3_0P6B, vocab_size=0), dict(QWEN3_0P6B, intermediate_size=0)]
    for b in bad:
        assert status_of(**b) == fq.INVALID_CONFIG, b
    unsupported = [dict(QWEN3_0P6B, head_dim=64), dict(QWEN3_0P6B, hidden_size=1000),
                   dict(QWEN3_0P6B, num_attention_heads=48, num_key_value_heads=3)]
    for u in unsupported:
        assert status_of(**u) == fq.UNSUPPORTED, u


def test_status_strings(lib):
    assert lib.fq_status_str(fq.KV_CACHE_OVERFLOW) == b"kv cache overflow"
    assert lib.fq_status_str(fq.OK) == b"ok"


def test_null_arguments_are_rejected_without_a_gpu(lib):
    import ctypes
    assert lib.fq_desc_init(None, None) == fq.INVALID_ARGUMENT
    assert lib.fq_load_weights(None, None, None, None) == fq.INVALID_ARGUMENT
    assert lib.fq_decode_step_batch(None, None, 0, None, None, None) == fq.INVALID_ARGUMENT
    assert lib.fq_decode_step_all_logits(None, None, None, 1, 0, None, None) == fq.INVALID_ARGUMENT
    assert lib.fq_forward_step(None, None, None, 1, 0, None, None) == fq.INVALID_ARGUMENT
    assert lib.fq_quantize_q8_0(None, 128, None, None) == fq.INVALID_ARGUMENT
    out = ctypes.c_void_p()
    assert lib.fq_kv_init(None, 4, fq.BF16, ctypes.byref(out)) == fq.INVALID_ARGUMENT

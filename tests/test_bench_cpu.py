"""Host-side accounting of bench.py, without a GPU: the algorithmic bytes a step moves (the
numerator of every roofline figure the bench reports) against the per-configuration totals
derived from the Qwen3 shapes and the ggml block sizes, the --kv and --layers workload
switches, and the source hash that keeps a DRAM-traffic record tied to the kernel it was
taken on."""
import argparse
import os
import shutil

import numpy as np
import pytest
import torch

import bench
import synth.workloads as wl

MB = 1e6


def test_step_bytes_of_the_0p6b_decode_step():
    # Qwen3-0.6B Q8_0: 633.5 MB of weights (165 MB of them the LM head), bf16 KV of 28 layers
    # x 8 kv heads x 128 x 2 bytes x (K, V) = 114,688 bytes per cached position
    b = bench.step_bytes(wl.QWEN3_0P6B, 2048)
    assert (b["weights"] + b["lm_head"]) / MB == pytest.approx(633.5, rel=1e-3)
    assert b["lm_head"] / MB == pytest.approx(165.3, rel=1e-3)
    assert b["kv_read"] == 2048 * 114688 and b["kv_write"] == 114688
    assert b["total"] / MB == pytest.approx(868.5, rel=1e-3)


def test_weight_bytes_of_the_8b_q8_0_model():
    # Qwen3-8B Q8_0: 8.04 GB of weights touched per step, of which the LM head is
    # 151936 x 4096 x 34/32 bytes
    wb = bench.weight_bytes(wl.WORKLOADS["qwen3-8b-batch32"])
    assert (wb["layers"] + wb["lm_head"]) / 1e9 == pytest.approx(8.04, rel=2e-3)
    assert wb["lm_head"] == pytest.approx(151936 * 4096 * 34 / 32 + 4096 * 4)


def test_q8_0_cache_rows_cost_34_bytes_per_32_values():
    # a head's cached row of 128 values: 4 blocks of 34 bytes = 136 bytes (bf16: 256)
    assert bench.KV_ELEM_BYTES["q8_0"] * 128 == 136
    assert bench.KV_ELEM_BYTES["bf16"] * 128 == 256


def test_kv_switch_replaces_only_the_cache_dtype():
    base = wl.WORKLOADS["qwen3-8b-batch32"]
    w = bench.workload_of(argparse.Namespace(workload="qwen3-8b-batch32", kv="q8_0"))
    assert w.kv_dtype == "q8_0" and w.dims == base.dims and w.seed == base.seed and w.batch == base.batch
    assert bench.workload_of(argparse.Namespace(workload="qwen3-8b-batch32", kv=None)) is base


def test_kv_tensor_keeps_the_bytes():
    bf = np.array([0x3F80, 0xBF80], dtype=np.uint16)
    t = bench.kv_tensor(bf, torch.device("cpu"))
    assert t.dtype == torch.int16 and t.numpy().view(np.uint16).tolist() == [0x3F80, 0xBF80]
    blocks = np.arange(34, dtype=np.uint8)
    assert bench.kv_tensor(blocks, torch.device("cpu")).dtype == torch.uint8


def test_step_bytes_of_a_chain_counts_the_growing_context():
    # a chain of 64 steps from 2048 cached positions reads 2048 + 31.5 positions per step on
    # average; the weights are the same every step
    w = wl.WORKLOADS["qwen3-0.6b"]
    sb = bench.step_bytes_of(w, [2048])
    per_pos = 2 * 28 * 8 * 128 * 2
    assert sb["kv_read"] == pytest.approx(per_pos * (2048 + 31.5))
    assert sb["kv_write"] == per_pos
    assert sb["total"] == pytest.approx(sb["weights_layers"] + sb["lm_head"] + sb["embedding_rows"] + sb["kv_read"]
                                        + sb["kv_write"])
    b32 = bench.step_bytes_of(wl.WORKLOADS["qwen3-8b-batch32"], [512, 4096])
    assert b32["kv_write"] == 32 * 2 * 36 * 8 * 128 * 2


def test_layers_switch_keeps_the_shapes_and_names_the_reduced_model():
    # a small profiling case: only the layer count changes, and the workload string says so
    args = argparse.Namespace(workload="qwen3-8b-q4k", kv=None, layers=4)
    w = bench.workload_of(args)
    full = bench.workload_of(argparse.Namespace(workload="qwen3-8b-q4k", kv=None, layers=None))
    assert w.dims.num_layers == 4 and full.dims.num_layers == 36
    assert w.dims.hidden_size == full.dims.hidden_size and w.weight_dtype == full.weight_dtype
    assert w.context == full.context
    assert "4 layers" in bench.config_dict(w)["workload"]


def test_step_source_hash_ignores_comments_but_not_code(tmp_path):
    src = os.path.join(os.path.dirname(os.path.abspath(bench.__file__)), "quantized_decoder_decode_gb300", "csrc")
    for f in bench.STEP_SOURCES:
        shutil.copy(os.path.join(src, f), tmp_path / f)
    h0 = bench.step_source_hash(str(tmp_path))
    assert h0 == bench.step_source_hash()
    k = tmp_path / "stream_step.cu"
    text = k.read_text()
    k.write_text("// a comment line\n/* a block\n   comment */\n\n" + text.replace("{", "{  // trailing", 1))
    assert bench.step_source_hash(str(tmp_path)) == h0
    k.write_text(text.replace("constexpr int SLOT = 16384;", "constexpr int SLOT = 32768;"))
    assert bench.step_source_hash(str(tmp_path)) != h0

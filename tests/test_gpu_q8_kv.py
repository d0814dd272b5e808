"""The q8_0 KvCache on the CUDA path against the oracle.

The fucina runner page ("KV cache") describes a cache that stores K and V as ggml Q8_0
blocks and scores decode through the integer q8 x q8 path; section 14.2 names the same
option for Qwen3.  Checked here: the device quantiser byte for byte, the cache copies byte
for byte, and the layer, decode, lockstep-batch and all-logits steps under the per-layer and
logit tolerances, with the new rows within one code step of the oracle's."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
from quantized_decoder_decode_gb300 import fq
from tests.gpu_util import DEV, Pair, assert_layer_close, assert_logits_close, assert_q8_rows_close, stream
from tests.test_gpu_parity import SMALL, SMALL_G4, SMALL_MOE, _compare_step, workload

pytestmark = pytest.mark.gpu


@pytest.fixture
def pairs():
    made = []

    def make(*a, **k):
        p = Pair(*a, **k)
        made.append(p)
        return p
    yield make
    for p in made:
        p.close()


def _quantiser_input() -> np.ndarray:
    rng = np.random.default_rng(5)
    scale = np.repeat(10.0 ** rng.uniform(-3, 2, 48 * 4), 32)
    blocks = (rng.standard_normal(128 * 48) * scale).astype(np.float32).reshape(-1, 32)
    d = np.float32(2.0 ** -4)
    half = ((np.arange(1, 16) + 0.5) * d).astype(np.float32)
    blocks[0] = 0
    blocks[0, 0] = 127 * d                                   # scale exactly d
    blocks[0, 1:16], blocks[0, 16:31] = half, -half         # ties round away from zero
    blocks[1] = 0                                           # zero block
    blocks[2] = rng.standard_normal(32) * 1e-7              # amax / 127 underflows fp16: d = 0
    blocks[3] = rng.standard_normal(32) * 1e-5              # subnormal fp16 scale
    blocks[4] = rng.standard_normal(32) * 3e6
    blocks[4, 0] = 1e7                                      # amax / 127 overflows fp16: d = inf
    blocks[5] = 5.0                                         # every value equals amax
    blocks[6] = 0
    blocks[6, 0] = -127 * d
    blocks[6, 1:16] = np.nextafter(half, np.float32(np.inf))   # one f32 ulp past the tie
    blocks[6, 16:31] = np.nextafter(half, np.float32(0))       # one f32 ulp short of it
    return blocks.ravel()


def test_quantiser_matches_oracle_bitwise():
    x = _quantiser_input()
    xt = torch.from_numpy(x).to(DEV)
    out = torch.empty(x.size // 32 * 34, dtype=torch.uint8, device=DEV)
    fq.fq_quantize_q8_0(xt.data_ptr(), x.size, out.data_ptr(), stream())
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.quant("q8_0", x))
    with pytest.raises(fq.FqError) as e:
        fq.fq_quantize_q8_0(xt.data_ptr(), 96, out.data_ptr(), stream())
    assert e.value.status == fq.INVALID_ARGUMENT


def test_cache_copies_are_byte_exact(pairs):
    w = workload(SMALL, "q8_0", "q8_0", seed=41)
    p = pairs(w, max_positions=512, with_oracle=False)
    cap = 37                                                # odd: the scale plane pads to 38 rows
    kv = fq.fq_kv_init(p.model, cap, "q8_0")
    p.kvs.append(kv)
    priors = [wl.make_kv_prior(w, 0, L, cap) for L in range(SMALL.num_layers)]
    for L, (k, v) in enumerate(priors):
        kt, vt = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)   # alive until the copy ran
        fq.fq_kv_append(kv, L, 0, cap, kt.data_ptr(), vt.data_ptr(), stream())
        torch.cuda.synchronize()
    fq.fq_kv_commit(kv, cap)
    for L, (k, v) in enumerate(priors):
        gk, gv = p.read_kv_blocks(kv, L, 0, cap)
        assert np.array_equal(gk, k) and np.array_equal(gv, v)
        sk, sv = p.read_kv_blocks(kv, L, 5, 7)
        assert np.array_equal(sk, k[5:12]) and np.array_equal(sv, v[5:12])


@pytest.mark.parametrize("ctx", [0, 1, 63, 64, 127, 128, 129, 1000, 2047])
def test_layer_step_0p6b_layer(pairs, ctx):
    """The 0.6B-shaped layer (two q heads per kv head) at contexts on and off the 64-row
    tiles and across several attention chunks; odd and even capacities."""
    w = dataclasses.replace(wl.WORKLOADS["qwen3-0.6b-layer"], kv_dtype="q8_0", context=ctx)
    p = pairs(w, max_positions=4096)
    kv, oc = p.new_seq(capacity=ctx + 1, ctx=ctx, seq=0)
    x0 = wl.layer_input(w)
    x = torch.from_numpy(x0.copy()).to(DEV)
    fq.fq_layer_step(p.model, 0, kv, ctx, x.data_ptr(), stream())
    torch.cuda.synchronize()
    ref, _, _ = p.om.layer_step(0, oc, ctx, x0.astype(np.float64))
    assert_layer_close(x.cpu().numpy(), ref, f"layer output at context {ctx}")
    k, v = p.read_kv(kv, 0, ctx, 1)
    rk, rv = oc.read(0, ctx, 1)
    assert_q8_rows_close(k, rk, "appended k")
    assert_q8_rows_close(v, rv, "appended v")
    if ctx:
        k0, _ = p.read_kv(kv, 0, 0, ctx)                    # prior rows untouched
        rk0, _ = oc.read(0, 0, ctx)
        assert np.array_equal(k0, rk0)


@pytest.mark.parametrize("dims", [SMALL, SMALL_G4, SMALL_MOE])
def test_decode_steps_match_oracle(pairs, dims):
    """Two, four and eight q heads per kv head (eight runs as two CTAs of four)."""
    p = pairs(workload(dims, "q8_0", "q8_0", seed=42), max_positions=512)
    kvc, oc = p.new_seq(capacity=128, ctx=100, seq=0)
    tok = 17
    for step in range(3):
        _, ref = _compare_step(p, [kvc], [oc], [tok], f"q8 kv step {step}")
        tok = oracle.argmax(ref[0])
    for L in range(dims.num_layers):
        k, v = p.read_kv(kvc, L, 100, 3)
        rk, rv = oc.read(L, 100, 3)
        assert_q8_rows_close(k, rk, f"layer {L} k")
        assert_q8_rows_close(v, rv, f"layer {L} v")


def test_batch_ragged_matches_oracle(pairs):
    """Ten sequences (tensor-core projections) of ragged lengths over q8_0 caches."""
    ctxs = [37, 100, 250, 1, 64, 5, 129, 200, 77, 33]
    p = pairs(workload(SMALL_G4, "q8_0", "q8_0", seed=43), max_positions=1024)
    kvs, ocs = [], []
    for s, c in enumerate(ctxs):
        kvc, oc = p.new_seq(capacity=300, ctx=c, seq=s)
        kvs.append(kvc)
        ocs.append(oc)
    toks = synth.uniform_i32(43, 99, len(ctxs), 0, SMALL_G4.vocab_size)
    for step in range(2):
        _, ref = _compare_step(p, kvs, ocs, toks, f"q8 kv batch step {step}")
        toks = ref.argmax(axis=1)


@pytest.mark.parametrize("rows", [3, 9])
def test_all_logits_step_matches_sequential_oracle(pairs, rows):
    p = pairs(workload(SMALL, "q8_0", "q8_0", seed=44), max_positions=512)
    ctx = 61                                                # rows cross the 64-row tile boundary
    kvc, oc = p.new_seq(capacity=128, ctx=ctx, seq=0)
    toks = [int(t) for t in synth.uniform_i32(44, 5, rows, 0, SMALL.vocab_size)]
    logits = torch.empty((rows, SMALL.vocab_size), dtype=torch.float32, device=DEV)
    fq.fq_decode_step_all_logits(p.model, kvc, toks, ctx, logits.data_ptr(), stream())
    torch.cuda.synchronize()
    assert fq.fq_kv_len(kvc) == ctx + rows
    got = logits.cpu().numpy()
    for i, t in enumerate(toks):
        assert_logits_close(got[i], p.om.decode_step(oc, t, ctx + i), f"row {i}")
    for L in range(SMALL.num_layers):
        k, v = p.read_kv(kvc, L, ctx, rows)
        rk, rv = oc.read(L, ctx, rows)
        assert_q8_rows_close(k, rk, f"layer {L} k")
        assert_q8_rows_close(v, rv, f"layer {L} v")


def test_caches_of_different_dtypes_do_not_batch(pairs):
    p = pairs(workload(SMALL, "q8_0", "bf16", seed=45), max_positions=512, with_oracle=False)
    a = fq.fq_kv_init(p.model, 16, "bf16")
    b = fq.fq_kv_init(p.model, 16, "q8_0")
    p.kvs += [a, b]
    logits = torch.empty((2, SMALL.vocab_size), dtype=torch.float32, device=DEV)
    with pytest.raises(fq.FqError) as e:
        fq.fq_decode_step_batch(p.model, [a, b], [1, 2], logits.data_ptr(), stream())
    assert e.value.status == fq.MISMATCHED_KV_CACHES
    assert fq.fq_kv_len(a) == 0 and fq.fq_kv_len(b) == 0

"""Pins of the CPU oracle against facts outside itself (no GPU needed).

Each test checks the oracle against something it cannot agree with by construction:
library conversions (numpy float16, torch bfloat16), hand-computed block fixtures,
closed forms, invariants of the mathematics, library routines for special cases, and the
pages' own cross-checks (no-cache last logits == cached prefill-then-step; batch row ==
single stream).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.workloads as wl
from tests.conftest import read_golden

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- number formats

def test_fp16_decode_exhaustive_matches_numpy():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_f64(int(h)) for h in codes])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(ref[~both_nan], got[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_fp16_encode_matches_numpy_rounding():
    vals = list(RNG.normal(0, 1, 3000)) + list(RNG.normal(0, 1e-5, 2000)) + list(RNG.normal(0, 2e4, 500))
    # exact halfway points between fp16 neighbours (ties to even), subnormal boundaries, overflow
    vals += [1 + 2 ** -11, 1 + 3 * 2 ** -11, 2 ** -25, 3 * 2 ** -25, 2 ** -24, 65504.0, 65519.99, 65520.0, -65520.0,
             2 ** -14 - 2 ** -25, 0.0, -0.0, 1e-9]
    for v in vals:
        ref = int(np.array([v], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
        assert oracle.f64_to_fp16(float(v)) == ref, v


def test_bf16_decode_and_encode_match_torch():
    codes = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    ref = codes.to(torch.float64).numpy()
    for h in range(0, 65536, 7):
        if np.isnan(ref[h]):
            continue
        assert oracle.bf16_to_f64(h) == ref[h]
    # f32-representable inputs: torch rounds f32 -> bf16 to nearest even
    vals = np.concatenate([RNG.normal(0, 1, 4000), RNG.normal(0, 1e-30, 200)]).astype(np.float32)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], dtype=np.float32)
    vals = np.concatenate([vals, ties])
    ref_bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(ref_bits, got)


# ---------------------------------------------------------------- Q8_0

def test_q8_0_hand_built_block(golden_dir):
    g = read_golden(f"{golden_dir}/q8_0_block.txt")
    blk = np.array([int(b, 16) for b in g["bytes"][0].split()], dtype=np.uint8)
    assert blk.size == 34
    out = oracle.dequant("q8_0", blk, 32)
    for e in g["expect"]:
        i, v = e.split()
        assert out[int(i)] == float(v)
    assert np.array_equal(out, 0.5 * (np.arange(32) - 16))


def test_q8_0_scale_is_fp16_of_amax_over_127():
    x = RNG.normal(0, 0.02, 32 * 200).astype(np.float32)
    packed = oracle.quant("q8_0", x).reshape(200, 34)
    amax = np.abs(x.reshape(200, 32).astype(np.float64)).max(axis=1)
    ref = (amax / 127.0).astype(np.float16).view(np.uint16)
    got = packed[:, 0].astype(np.uint16) | (packed[:, 1].astype(np.uint16) << 8)
    assert np.array_equal(ref, got)
    # the largest-magnitude element gets code +-127
    q = packed[:, 2:].view(np.int8)
    assert np.all(np.abs(q).max(axis=1) == 127)


def test_q8_0_requant_of_dequant_is_byte_identical():
    x = RNG.normal(0, 0.02, 32 * 500).astype(np.float32)
    x[:32] = 0.0                                   # an all-zero block
    packed = oracle.quant("q8_0", x)
    again = oracle.quant("q8_0", oracle.dequant("q8_0", packed, x.size))
    assert np.array_equal(packed, again)


def test_q8_0_error_within_half_step():
    x = RNG.normal(0, 0.02, 32 * 300).astype(np.float32)
    packed = oracle.quant("q8_0", x)
    y = oracle.dequant("q8_0", packed, x.size).astype(np.float64)
    d = packed.reshape(-1, 34)[:, :2].copy().view(np.float16).astype(np.float64).repeat(32)
    assert np.all(np.abs(y - x) <= d / 2 * (1 + 1e-12))


def test_generator_q8_0_packing_equals_oracle_quantiser():
    rows, cols = 37, 256
    packed = synth.q8_0(7, 99, rows, cols, 0.02)
    floats = synth.normal_f32(7, 99, rows * cols, std=0.02)
    assert np.array_equal(packed.ravel(), oracle.quant("q8_0", floats))


# ---------------------------------------------------------------- Q4_K

def _q4k_golden_block(golden_dir):
    g = read_golden(f"{golden_dir}/q4_k_block.txt")
    header = [int(b, 16) for b in g["header"][0].split()]
    scales = [int(b, 16) for b in g["scales"][0].split()]
    chunks = [int(b, 16) for b in g["chunks"][0].split()]
    blk = np.array(header + scales + [c for c in chunks for _ in range(32)], dtype=np.uint8)
    sc = [int(v) for v in g["sc"][0].split()]
    mn = [int(v) for v in g["mn"][0].split()]
    expect = [float(v) for v in g["expect_sub"][0].split()]
    return blk, sc, mn, expect


def test_q4_k_hand_built_block(golden_dir):
    blk, sc, mn, expect = _q4k_golden_block(golden_dir)
    assert blk.size == 144
    for j in range(8):
        assert oracle.q4k_scale_min(blk[4:16], j) == (sc[j], mn[j])
    out = oracle.dequant("q4_k", blk, 256)
    for j in range(8):
        assert np.all(out[32 * j:32 * j + 32] == expect[j]), j


def test_q4_k_element_order_inside_sub_blocks(golden_dir):
    # 128 distinct nibble bytes: any other byte <-> element map inside a chunk moves some byte
    # to another element and changes its low or its high nibble
    g = read_golden(f"{golden_dir}/q4_k_block_distinct.txt")
    blk = np.array([int(b, 16) for key in ("header", "scales", "nibbles") for b in g[key][0].split()],
                   dtype=np.uint8)
    assert blk.size == 144 and len(set(blk[16:].tolist())) == 128
    expect = np.array([float(v) for v in g["expect"][0].split()])
    out = oracle.dequant("q4_k", blk, 256)
    assert np.array_equal(out, expect)


def test_q4_k_scale_min_pack_roundtrip_exhaustive():
    # every (scale, min) value in every sub-block slot, with the other slots holding
    # distinct values so that a crossed bit field shows up
    base_sc = np.array([5, 10, 15, 20, 25, 30, 35, 40])
    base_mn = np.array([41, 37, 33, 29, 21, 17, 13, 9])
    for j in range(8):
        for v in range(64):
            for w in (0, 63, v, 63 - v):
                sc, mn = base_sc.copy(), base_mn.copy()
                sc[j], mn[j] = v, w
                s12 = oracle.q4k_pack_scale_min(sc, mn)
                got = [oracle.q4k_scale_min(s12, i) for i in range(8)]
                assert got == list(zip(sc.tolist(), mn.tolist()))


def test_q4_k_pack_matches_hand_built_bytes(golden_dir):
    blk, sc, mn, _ = _q4k_golden_block(golden_dir)
    assert np.array_equal(oracle.q4k_pack_scale_min(sc, mn), blk[4:16])


def test_q4_k_reconstruction_error_bounded():
    x = RNG.normal(0, 0.02, 256 * 64).astype(np.float32)
    packed = oracle.quant("q4_k", x).reshape(64, 144)
    y = oracle.dequant("q4_k", packed, x.size).astype(np.float64).reshape(64, 8, 32)
    xs = x.astype(np.float64).reshape(64, 8, 32)
    d = packed[:, 0:2].copy().view(np.float16).astype(np.float64)[:, 0]
    dmin = packed[:, 2:4].copy().view(np.float16).astype(np.float64)[:, 0]
    for b in range(64):
        for j in range(8):
            sc, mn = oracle.q4k_scale_min(packed[b, 4:16], j)
            step = d[b] * sc
            # half a step of rounding plus the min offset's own rounding (half of dmin) plus
            # the scale's rounding stretched over 15 steps
            bound = step / 2 + dmin[b] / 2 + 15 * d[b] / 2 + 1e-9
            assert np.abs(y[b, j] - xs[b, j]).max() <= bound


def test_generator_q4_k_packing_equals_oracle_quantiser():
    rows, cols = 9, 512
    packed = synth.q4_k(3, 42, rows, cols, 0.02)
    floats = synth.normal_f32(3, 42, rows * cols, std=0.02)
    assert np.array_equal(packed.ravel(), oracle.quant("q4_k", floats))


# ---------------------------------------------------------------- building blocks

def test_rmsnorm_matches_torch():
    x = RNG.normal(0, 3, 1024)
    g = (1 + RNG.normal(0, 0.1, 1024)).astype(np.float32)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (1024,), torch.from_numpy(g.astype(np.float64)),
                                       eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(x, g, 1e-6), ref, rtol=1e-14, atol=0)


def test_rmsnorm_constant_vector_closed_form():
    c, eps = -2.5, 1e-6
    y = oracle.rmsnorm(np.full(64, c), np.ones(64, np.float32), eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-15)


@pytest.mark.parametrize("D", [2, 8, 128])
def test_rope_equals_complex_rotation(D):
    # rotate-half pairing (i, i + D/2): z_i = v_i + 1j v_{i+D/2} is multiplied by e^{1j pos f_i}
    theta, pos = 1e6, 777
    v = RNG.normal(0, 1, D)
    got = oracle.rope(v, pos, theta)
    i = np.arange(D // 2)
    z = (v[:D // 2] + 1j * v[D // 2:]) * np.exp(1j * pos * np.power(theta, -2.0 * i / D))
    np.testing.assert_allclose(got[:D // 2], z.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[D // 2:], z.imag, rtol=0, atol=1e-12)


def test_rope_preserves_norm_and_pos0_is_identity():
    v = RNG.normal(0, 1, 128)
    assert np.array_equal(oracle.rope(v, 0, 1e6), v)
    for pos in (1, 100, 8191, 40000):
        r = oracle.rope(v, pos, 1e6)
        assert abs(np.linalg.norm(r) - np.linalg.norm(v)) <= 1e-12 * np.linalg.norm(v)


def test_rope_relative_position_identity():
    q, k = RNG.normal(0, 1, 128), RNG.normal(0, 1, 128)
    for p, pp, s in [(5, 3, 100), (0, 17, 4000), (2048, 1, 7)]:
        a = oracle.rope(q, p, 1e6) @ oracle.rope(k, pp, 1e6)
        b = oracle.rope(q, p + s, 1e6) @ oracle.rope(k, pp + s, 1e6)
        assert abs(a - b) <= 1e-9 * (1 + abs(a))


def _q8_rows_of_equal_codes(codes, d_bits=0x2800):
    """Q8_0 rows of one block each: fp16 scale d_bits, then 32 copies of the row's code."""
    rows = []
    for c in codes:
        rows.append([d_bits & 0xFF, d_bits >> 8] + [int(c) & 0xFF] * 32)
    return np.array(rows, dtype=np.uint8)


def test_qk_norm_then_rope_worked_example(golden_dir):
    # the worked example of the golden file: per-head RMSNorm with non-constant gains, then
    # the rotate-half RoPE at position 2 (rotating first would change elements 2 and 3)
    g = read_golden(f"{golden_dir}/qk_norm_rope_order.txt")
    vec = lambda key: np.array([float(v) for v in g[key][0].split()])  # noqa: E731
    # eight heads of dim 4 so that every matrix has whole Q8_0 blocks; heads 1-7 project to
    # zero (all-zero rows) and must stay zero through the norm and the rotation
    dims = wl.Dims(vocab_size=40, hidden_size=32, intermediate_size=32, num_layers=1, num_attention_heads=8,
                   num_key_value_heads=8, head_dim=4)
    W = wl.make_weights(wl.Workload("qk-order", dims, "q8_0", "f32", seed=3))
    lw = W["layers"][0]
    pad = lambda c: np.concatenate([c, np.zeros(28)]).astype(int)  # noqa: E731
    lw["wq"] = _q8_rows_of_equal_codes(pad(vec("wq_codes")))
    lw["wk"] = _q8_rows_of_equal_codes(pad(vec("wk_codes")))
    lw["wv"] = _q8_rows_of_equal_codes(pad(vec("wv_codes")))
    lw["q_norm"] = vec("q_norm").astype(np.float32)
    lw["k_norm"] = vec("k_norm").astype(np.float32)
    m = oracle.Model(dims, W, "q8_0", "f32")
    q, k, v = m.qkv_project(0, np.ones(32), int(g["pos"][0]))
    np.testing.assert_allclose(q[0], vec("q"), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(k[0], vec("k"), rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(v[0], vec("v"))
    assert not q[1:].any() and not k[1:].any() and not v[1:].any()


def test_attention_matches_torch_sdpa():
    for T, D in [(1, 4), (5, 4), (8, 16), (300, 128)]:
        q = RNG.normal(0, 1, D)
        K = RNG.normal(0, 1, (T, D)).astype(np.float32)
        V = RNG.normal(0, 1, (T, D)).astype(np.float32)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q).view(1, 1, 1, D), torch.from_numpy(K.astype(np.float64)).view(1, 1, T, D),
            torch.from_numpy(V.astype(np.float64)).view(1, 1, T, D)).view(D).numpy()
        np.testing.assert_allclose(oracle.attention(q, K, V), ref, rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    D = 16
    V = RNG.normal(0, 1, (6, D)).astype(np.float32)
    K = RNG.normal(0, 1, (6, D)).astype(np.float32)
    # a single position returns its value row exactly
    assert np.array_equal(oracle.attention(RNG.normal(0, 1, D), K[:1], V[:1]), V[0].astype(np.float64))
    # a zero query weights all positions equally
    np.testing.assert_allclose(oracle.attention(np.zeros(D), K, V), V.astype(np.float64).mean(0), rtol=1e-14)
    # permuting the (k, v) pairs changes nothing
    perm = RNG.permutation(6)
    q = RNG.normal(0, 1, D)
    np.testing.assert_allclose(oracle.attention(q, K[perm], V[perm]), oracle.attention(q, K, V), rtol=1e-13)


# ---------------------------------------------------------------- q8_0 KV cache

def _q8_block_scale(x32: np.ndarray) -> float:
    """fp16 of amax / 127 for one block of f32 values (numpy's float16 conversion)."""
    return float(np.float16(np.abs(x32.astype(np.float64)).max() / 127.0))


def test_q8_cache_row_holds_whole_codes_of_the_fp16_block_scale():
    x = RNG.normal(0, 1, 256) * np.repeat([1e-3, 1.0, 30.0, 0.2, 5.0, 1e-6, 7.0, 0.5], 32)
    r = oracle.kv_round_row("q8_0", x).astype(np.float64)
    xf = x.astype(np.float32).astype(np.float64)
    for b in range(8):
        d = _q8_block_scale(xf[32 * b:32 * b + 32])
        if d == 0.0:                     # amax / 127 below half the smallest fp16: zero block
            assert b == 5 and np.all(r[32 * b:32 * b + 32] == 0)
            continue
        codes = r[32 * b:32 * b + 32] / d
        assert np.array_equal(codes, np.round(codes)) and np.abs(codes).max() <= 127
        assert np.abs(xf[32 * b:32 * b + 32] - r[32 * b:32 * b + 32]).max() <= d / 2
    # quantising a cached row again changes nothing
    assert np.array_equal(oracle.kv_round_row("q8_0", r), r.astype(np.float32))


def test_q8_cache_blocks_are_independent_and_zero_blocks_stay_zero():
    x = RNG.normal(0, 1, 128)
    x[32:64] = 0.0
    r = oracle.kv_round_row("q8_0", x)
    assert np.all(r[32:64] == 0)
    y = x.copy()
    y[96:128] *= 50.0
    ry = oracle.kv_round_row("q8_0", y)
    assert np.array_equal(ry[:96], r[:96]) and not np.array_equal(ry[96:], r[96:])


def test_q8_cache_ties_round_away_and_decisions_are_taken_in_f32():
    d = 2.0 ** -4
    x = np.zeros(32)
    x[0] = 127 * d                       # sets the scale to d exactly
    x[1], x[2], x[3], x[4] = 3.5 * d, -3.5 * d, 2.25 * d, -0.5 * d
    # just below the tie in f64, but the f32 rounding of the value lands on the tie
    x[5] = 5.5 * d - 2.0 ** -40
    r = oracle.kv_round_row("q8_0", x) / d
    assert list(r[:6]) == [127, 4, -4, 2, -1, 6]


def test_q8_attention_equals_the_integer_score_path():
    D, T = 128, 37
    q = RNG.normal(0, 1, D)
    kc = RNG.integers(-127, 128, (T, D)).astype(np.int64)
    vc = RNG.integers(-127, 128, (T, D)).astype(np.int64)
    kd = np.float16(RNG.uniform(0.005, 0.03, (T, D // 32))).astype(np.float64)
    vd = np.float16(RNG.uniform(0.005, 0.03, (T, D // 32))).astype(np.float64)
    K = (kc * np.repeat(kd, 32, axis=1)).astype(np.float32)
    V = (vc * np.repeat(vd, 32, axis=1)).astype(np.float32)
    qb = oracle.quant("q8_0", q.astype(np.float32)).reshape(D // 32, 34)
    qdd = qb[:, :2].copy().view(np.float16).astype(np.float64).ravel()
    qc = qb[:, 2:].view(np.int8).astype(np.int64)
    # integer dot per block, then the two fp16 scales, then 1/sqrt(D)
    isum = np.einsum("bi,tbi->tb", qc, kc.reshape(T, D // 32, 32))
    s = (isum * qdd[None, :] * kd).sum(1) / math.sqrt(D)
    p = np.exp(s - s.max())
    ref = (p[:, None] * V.astype(np.float64)).sum(0) / p.sum()
    np.testing.assert_allclose(oracle.attention_q8(q, K, V), ref, rtol=1e-12, atol=1e-14)


def test_q8_attention_ignores_changes_of_q_inside_its_codes():
    D = 64
    K = oracle.kv_round_row("q8_0", RNG.normal(0, 1, 8 * D)).reshape(8, D)
    V = oracle.kv_round_row("q8_0", RNG.normal(0, 1, 8 * D)).reshape(8, D)
    q = RNG.normal(0, 1, D)
    q[0], q[32] = 3.0, -3.0                  # block maxima stay put
    base = oracle.attention_q8(q, K, V)
    nudged = q.copy()
    nudged[1:32] += 1e-7                     # far inside the code cells (step 3/127)
    assert np.array_equal(oracle.attention_q8(nudged, K, V), base)
    assert not np.array_equal(oracle.attention(nudged, K, V), oracle.attention(q, K, V))
    # a single position returns its (dequantised) value row exactly
    assert np.array_equal(oracle.attention_q8(q, K[:1], V[:1]), V[0].astype(np.float64))


def test_silu_matches_torch():
    z = RNG.normal(0, 4, 200)
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    np.testing.assert_allclose([oracle.silu(float(v)) for v in z], ref, rtol=1e-15, atol=1e-300)


def test_router_topk_properties():
    for _ in range(50):
        logits = RNG.normal(0, 1, 128)
        idx, w = oracle.router(logits, 8, True)
        assert len(set(idx.tolist())) == 8
        assert abs(w.sum() - 1.0) <= 1e-12
        ref = np.argsort(-logits, kind="stable")[:8]
        assert np.array_equal(idx, ref)
        assert np.all(np.diff(w) <= 0)
    # without renormalisation the weights are the softmax probabilities
    logits = RNG.normal(0, 1, 16)
    idx, w = oracle.router(logits, 4, False)
    p = torch.softmax(torch.from_numpy(logits), 0).numpy()
    np.testing.assert_allclose(w, p[idx], rtol=1e-13)


def test_router_ties_go_to_lower_index():
    logits = np.zeros(10)
    logits[[2, 5, 7]] = 1.0
    idx, _ = oracle.router(logits, 2, True)
    assert idx.tolist() == [2, 5]
    idx, w = oracle.router(np.zeros(6), 3, True)
    assert idx.tolist() == [0, 1, 2] and np.allclose(w, 1 / 3)


@pytest.mark.parametrize("wtype,cols", [("q8_0", 96), ("q4_k", 512)])
def test_gemv_matches_numpy_matmul_of_dequantised(wtype, cols):
    rows = 300
    W = (synth.q8_0 if wtype == "q8_0" else synth.q4_k)(11, 5, rows, cols, 0.02)
    x = RNG.normal(0, 1, cols)
    Wf = oracle.dequant(wtype, W, rows * cols).astype(np.float64).reshape(rows, cols)
    np.testing.assert_allclose(oracle.gemv(wtype, W, rows, cols, x), Wf @ x, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- model level

TINY = wl.Dims(vocab_size=97, hidden_size=64, intermediate_size=96, num_layers=2, num_attention_heads=4,
               num_key_value_heads=2, head_dim=16)
TINY_MOE = dataclasses.replace(TINY, num_experts=6, num_experts_used=2, moe_intermediate_size=32)


def tiny_model(dims=TINY, wtype="q8_0", kv="bf16", seed=5):
    hid = dims.hidden_size
    if wtype == "q4_k":
        dims = dataclasses.replace(dims, hidden_size=256, intermediate_size=512, head_dim=64,
                                   moe_intermediate_size=256 if dims.num_experts else 0)
        hid = 256
    w = wl.Workload("tiny", dims, wtype, kv, seed=seed)
    W = wl.make_weights(w)
    return oracle.Model(dims, W, wtype, kv), W, dims, hid


TINY_Q8KV = dataclasses.replace(TINY, head_dim=32)   # whole Q8_0 blocks per cached row


@pytest.mark.parametrize("dims,wtype,kv", [(TINY, "q8_0", "bf16"), (TINY, "q4_k", "f32"), (TINY_MOE, "q8_0", "bf16"),
                                           (TINY_Q8KV, "q8_0", "q8_0")])
def test_no_cache_logits_equal_cached_prefill_then_step(dims, wtype, kv):
    m, _, d, _ = tiny_model(dims, wtype, kv)
    toks = synth.uniform_i32(9, 1, 7, 0, d.vocab_size)
    ref = m.forward_last_logits(toks)
    cache = m.new_cache(16)
    for p, t in enumerate(toks):
        lg = m.decode_step(cache, int(t), p)
    assert cache.len == len(toks)
    np.testing.assert_allclose(lg, ref, rtol=1e-12, atol=1e-12)


def test_batch_rows_equal_single_streams():
    m, _, d, _ = tiny_model(TINY_MOE)
    prompts = [synth.uniform_i32(4, s, 3 + s, 0, d.vocab_size) for s in range(3)]
    caches, singles = [], []
    for pr in prompts:
        c1, c2 = m.new_cache(12), m.new_cache(12)
        for p, t in enumerate(pr):
            m.decode_step(c1, int(t), p, logits=False)
            m.decode_step(c2, int(t), p, logits=False)
        caches.append(c1)
        singles.append(c2)
    nxt = [11, 22, 33]
    batch = m.decode_step_batch(caches, nxt)
    for s in range(3):
        ref = m.decode_step(singles[s], nxt[s], singles[s].len)
        assert np.array_equal(batch[s], ref)
        assert caches[s].len == singles[s].len


def test_cache_holds_bf16_values_after_step():
    m, _, d, _ = tiny_model()
    c = m.new_cache(4)
    m.decode_step(c, 3, 0, logits=False)
    k, v = c.read(1, 0, 1)
    assert np.all((k.view(np.uint32) & 0xFFFF) == 0) and np.all((v.view(np.uint32) & 0xFFFF) == 0)
    assert np.any(k != 0)


def test_keep_current_attends_over_the_rows_written_at_the_position():
    m, _, d, _ = tiny_model()
    a, b, c = m.new_cache(8), m.new_cache(8), m.new_cache(8)
    for p, t in enumerate([3, 17, 40]):
        for cache in (a, b, c):
            m.decode_step(cache, t, p, logits=False)
    ref, ref_lo, _, _ = m.decode_step(a, 5, 3, trace=True)
    # the step's own rows, written beforehand and kept: the same step bit for bit
    for L in range(d.num_layers):
        k, v = a.read(L, 3, 1)
        b.write(L, 3, k, v)
        c.write(L, 3, k, 2 * v if L == 1 else v)
    b.keep_current(True)
    lg = m.decode_step(b, 5, 3)
    b.keep_current(False)
    assert np.array_equal(lg, ref) and b.len == 4
    # other rows: layer 0 is untouched, layer 1 attends over the doubled v row, which stays
    c.keep_current(True)
    lg2, lo2, _, _ = m.decode_step(c, 5, 3, trace=True)
    c.keep_current(False)
    assert np.array_equal(lo2[0], ref_lo[0]) and not np.array_equal(lo2[1], ref_lo[1])
    assert np.array_equal(c.read(1, 3, 1)[1], 2 * a.read(1, 3, 1)[1])
    # without the flag the step stores its own rows again
    c.set_len(3)
    assert np.array_equal(m.decode_step(c, 5, 3), ref)


def test_q8_cache_holds_quantised_rows_after_step():
    m, _, d, _ = tiny_model(TINY_Q8KV, kv="q8_0")
    mf, _, _, _ = tiny_model(TINY_Q8KV, kv="f32")
    c, cf = m.new_cache(4), mf.new_cache(4)
    for p, t in enumerate([3, 17]):
        m.decode_step(c, t, p, logits=False)
        mf.decode_step(cf, t, p, logits=False)
    k, v = c.read(0, 0, 2)          # layer 0 saw identical inputs in both models
    kf, vf = cf.read(0, 0, 2)
    for got, exact in ((k, kf), (v, vf)):
        assert np.array_equal(got.ravel(), oracle.kv_round_row("q8_0", exact.ravel().astype(np.float64)))
    # the q8_0 cache perturbs the step by the size of its rounding, not more
    lq = m.decode_step(c, 5, 2)
    lf = mf.decode_step(cf, 5, 2)
    assert 0 < np.abs(lq - lf).max() <= 2e-2 * np.abs(lf).max()


def _zeros_like_packed(a):
    return np.zeros_like(a)   # Q8_0 / Q4_K blocks of zero bytes decode to exact zeros


def test_zero_weights_give_zero_logits():
    _, W, d, _ = tiny_model()
    Z = {k: (_zeros_like_packed(v) if v.dtype == np.uint8 else v) for k, v in W.items() if k != "layers"}
    Z["layers"] = [{k: (_zeros_like_packed(v) if v.dtype == np.uint8 else v) for k, v in lw.items()}
                   for lw in W["layers"]]
    m = oracle.Model(d, Z, "q8_0", "bf16")
    lg = m.decode_step(m.new_cache(2), 5, 0)
    assert np.all(lg == 0)


def test_zero_output_projections_leave_residual_unchanged():
    _, W, d, _ = tiny_model(TINY_MOE)
    for lw in W["layers"]:
        lw["wo"] = np.zeros_like(lw["wo"])
        lw["down_exps"] = np.zeros_like(lw["down_exps"])
    m = oracle.Model(d, W, "q8_0", "bf16")
    c = m.new_cache(2)
    x0 = RNG.normal(0, 1, d.hidden_size)
    x1, _, _ = m.layer_step(0, c, 0, x0)
    assert np.array_equal(x0, x1)


def test_moe_with_identical_experts_equals_dense_swiglu():
    # norm_topk_prob renormalises the selected weights to 1, so identical experts collapse
    # to one dense SwiGLU block with the same matrices
    m_moe, W, d, _ = tiny_model(TINY_MOE)
    E, Fe, H = d.num_experts, d.moe_intermediate_size, d.hidden_size
    dense = dataclasses.replace(d, num_experts=0, num_experts_used=0, moe_intermediate_size=0,
                                intermediate_size=Fe)
    Wd = {k: v for k, v in W.items() if k != "layers"}
    Wd["layers"] = []
    for lw in W["layers"]:
        g1 = lw["gate_exps"][:Fe]
        u1 = lw["up_exps"][:Fe]
        d1 = lw["down_exps"][:H]
        lw["gate_exps"] = np.ascontiguousarray(np.tile(g1, (E, 1)))
        lw["up_exps"] = np.ascontiguousarray(np.tile(u1, (E, 1)))
        lw["down_exps"] = np.ascontiguousarray(np.tile(d1, (E, 1)))
        ld = {k: v for k, v in lw.items() if k not in ("router", "gate_exps", "up_exps", "down_exps")}
        ld.update(w_gate=g1, w_up=u1, w_down=d1)
        Wd["layers"].append(ld)
    m_moe = oracle.Model(d, W, "q8_0", "bf16")
    m_dense = oracle.Model(dense, Wd, "q8_0", "bf16")
    a = m_moe.decode_step(m_moe.new_cache(2), 7, 0)
    b = m_dense.decode_step(m_dense.new_cache(2), 7, 0)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_gqa_grouping_uses_consecutive_q_heads():
    # q head h must read kv head h // (n_q / n_kv): with V = +1 for kv head 0 and -1 for kv
    # head 1, q head 1 (group 0) sees +1 whatever the softmax weights are.
    _, W, d, _ = tiny_model(TINY)
    D, H = d.head_dim, d.hidden_size
    lw = W["layers"][0]
    wo = np.zeros((H, d.q_dim), dtype=np.float32)
    wo[:, D:2 * D] = np.eye(H, D)          # x[r] += o_head1[r] for r < D
    lw["wo"] = synth.pack_q8_0(wo).reshape(H, -1)
    lw["w_down"] = np.zeros_like(lw["w_down"])
    # the new position's value row is W_v xn with xn = rmsnorm(e_0) = sqrt(H) g_0 e_0: make it
    # about +1 for kv head 0 and -1 for kv head 1 as well, so no softmax weight can flip the sign
    wv = np.zeros((d.kv_dim, H), dtype=np.float32)
    wv[:D, 0] = 1.0 / (math.sqrt(H) * lw["attn_norm"][0])
    wv[D:, 0] = -wv[0, 0]
    lw["wv"] = synth.pack_q8_0(wv).reshape(d.kv_dim, -1)
    m = oracle.Model(d, W, "q8_0", "f32")
    c = m.new_cache(8)
    K = np.random.default_rng(77).normal(0, 1, (5, d.num_key_value_heads, D)).astype(np.float32)
    V = np.ones((5, d.num_key_value_heads, D), dtype=np.float32)
    V[:, 1, :] = -1
    c.write(0, 0, K, V)
    c.set_len(5)
    x0 = np.zeros(H)
    x0[0] = 1.0
    x1, _, _ = m.layer_step(0, c, 5, x0)
    delta = (x1 - x0)[:D]
    assert np.all(delta > 0.9), delta


def test_validation_rejects_bad_configs():
    assert oracle.validate(TINY) == oracle.OK
    assert oracle.validate(TINY_MOE) == oracle.OK
    bad = [dataclasses.replace(TINY, num_attention_heads=0), dataclasses.replace(TINY, num_key_value_heads=3),
           dataclasses.replace(TINY, head_dim=15), dataclasses.replace(TINY, num_experts=4),
           dataclasses.replace(TINY_MOE, num_experts_used=7)]
    for b in bad:
        assert oracle.validate(b) == oracle.INVALID_CONFIG, b
    # a q8_0 cache stores whole blocks of 32 per row
    assert oracle.validate(TINY, kv_dtype="q8_0") == oracle.INVALID_CONFIG
    assert oracle.validate(dataclasses.replace(TINY, head_dim=32), kv_dtype="q8_0") == oracle.OK


def test_step_contract_errors():
    m, _, d, _ = tiny_model()
    c = m.new_cache(2)
    with pytest.raises(oracle.OracleError) as e:
        m.decode_step(c, 1, 1)
    assert e.value.code == oracle.INVALID_SEQUENCE_LENGTH
    m.decode_step(c, 1, 0, logits=False)
    m.decode_step(c, 1, 1, logits=False)
    with pytest.raises(oracle.OracleError) as e:
        m.decode_step(c, 1, 2)
    assert e.value.code == oracle.KV_CACHE_OVERFLOW
    c2 = m.new_cache(4)
    with pytest.raises(oracle.OracleError) as e:
        m.decode_step_batch([c2, c2], [1, 2])
    assert e.value.code == oracle.MISMATCHED_KV_CACHES
    with pytest.raises(oracle.OracleError) as e:
        m.forward_last_logits(np.array([], dtype=np.int32))
    assert e.value.code == oracle.INVALID_SEQUENCE_LENGTH


# ---------------------------------------------------------------- sampling

def _freqs(z, n_grid=1 << 14, **kw):
    """How often each token is drawn as u sweeps a uniform grid of [0, 1)."""
    counts = np.zeros(len(z))
    for i in range(n_grid):
        counts[oracle.sample(z, (i + 0.5) / n_grid, **kw)] += 1
    return counts / n_grid


def test_uniform24_is_the_top_of_splitmix64():
    # SplitMix64 from seed 0 begins 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F
    for c, out in enumerate((0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F)):
        assert oracle.uniform24(0, c) == (out >> 40) / 2.0 ** 24
    us = [oracle.uniform24(12345, c) for c in range(1000)]
    assert all(0.0 <= u < 1.0 and (u * 2 ** 24).is_integer() for u in us)
    assert abs(np.mean(us) - 0.5) < 0.05


def test_greedy_cases_are_argmax():
    z = RNG.normal(0, 1, 40)
    z[[7, 21]] = z.max() + 1.0                  # a tie: the lower id wins
    for u in (0.0, 0.3, 0.999):
        assert oracle.sample(z, u, temp=0.0, top_p=0.5, min_p=0.2) == 7
        assert oracle.sample(z, u, temp=0.8, top_k=1) == 7


def test_inverse_cdf_draws_follow_the_tempered_softmax():
    from scipy.special import softmax
    z = RNG.normal(0, 2, 30)
    for temp in (1.0, 0.6, 1.7):
        np.testing.assert_allclose(_freqs(z, temp=temp), softmax(z / temp), atol=2.0 / (1 << 14))


def test_cutoffs_on_a_hand_built_distribution():
    z = np.log([0.5, 0.3, 0.15, 0.05])
    np.testing.assert_allclose(_freqs(z, top_p=0.75), [0.5 / 0.8, 0.3 / 0.8, 0, 0], atol=1e-3)
    np.testing.assert_allclose(_freqs(z, top_p=0.81), [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0], atol=1e-3)
    # top-k first, then top-p of the kept mass: 0.9 * 0.95 is reached at the third candidate
    np.testing.assert_allclose(_freqs(z, top_k=3, top_p=0.9), [0.5 / 0.95, 0.3 / 0.95, 0.15 / 0.95, 0], atol=1e-3)
    np.testing.assert_allclose(_freqs(z, top_k=2), [0.5 / 0.8, 0.3 / 0.8, 0, 0], atol=1e-3)
    # min-p relative to the top probability: 0.35 * 0.5 = 0.175 drops the last two
    np.testing.assert_allclose(_freqs(z, min_p=0.35), [0.5 / 0.8, 0.3 / 0.8, 0, 0], atol=1e-3)
    assert _freqs(z, min_p=0.1)[3] > 0          # 0.05 >= 0.1 * 0.5 stays
    # at least one candidate always stays
    assert oracle.sample(z, 0.99, top_p=1e-9) == 0 and oracle.sample(z, 0.99, min_p=1.0) == 0


def test_candidates_run_in_probability_order_with_ties_to_the_lower_id():
    z = np.log([0.2, 0.4, 0.2, 0.2])
    assert oracle.sample(z, 0.0) == 1           # the most probable first
    assert oracle.sample(z, 0.45) == 0          # then the tied ones by id: 0, 2, 3
    assert oracle.sample(z, 0.65) == 2 and oracle.sample(z, 0.85) == 3


def test_repeat_penalty_divides_positive_and_multiplies_negative_logits():
    z = np.array([2.0, 1.0, -1.0])
    assert oracle.sample(z, 0.5, temp=0.0, repeat_penalty=2.0, history=[0, 2, 0]) == 0   # [1, 1, -2]: tie
    assert oracle.sample(z, 0.5, temp=0.0, repeat_penalty=4.0, history=[0, 2]) == 1      # [0.5, 1, -4]
    from scipy.special import softmax
    np.testing.assert_allclose(_freqs(z, repeat_penalty=2.0, history=[0, 2]), softmax([1.0, 1.0, -2.0]),
                               atol=2.0 / (1 << 14))

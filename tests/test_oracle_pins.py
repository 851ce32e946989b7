"""Pins of the CPU oracle against facts that do not come from the oracle itself: closed forms,
invariants, hand-computed cases, library routines for the number formats, brute force on tiny
inputs and the byte counts the pages print. Each test names the mistake it is there to catch."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import Oracle, ERR_NONFINITE, ERR_INVALID

ORC = Oracle("f64")


def bf16_bits(values):
    """float values that are exactly bf16 -> bit patterns (via torch, a library routine)."""
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


# ------------------------------------------------------------------ number formats

def test_bf16_decode_exhaustive_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_vals(bits)
    got = np.array([ORC.bf16_value(int(b)) for b in bits[::1]])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_fp16_decode_exhaustive_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([ORC.fp16_value(int(b)) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_round_bf16_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1e-40, -3e-39, 3.3e38, 3.4e38, 1.0 + 2 ** -8])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([ORC.round_bf16(float(v)) for v in x], dtype=np.uint16)
    assert (got == ref).all()


def test_round_bf16_rounds_once_from_double():
    # 1 + 2^-8 is a tie (rounds to even: 1.0). Just above the tie must round up. Going through
    # float32 first would land on the tie and round down: the single-rounding reading catches it.
    assert ORC.round_bf16(1.0 + 2 ** -8) == 0x3F80
    assert ORC.round_bf16(1.0 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert ORC.round_bf16(1.0 + 3 * 2 ** -8) == 0x3F82     # tie between 0x3F81 and 0x3F82 -> even
    assert ORC.round_bf16(-2.0) == 0xC000
    assert ORC.round_bf16(float("inf")) == 0x7F80


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_constant_vector_closed_form():
    n, c, eps = 64, 0.37, 1e-5
    g = bf16_bits(np.linspace(0.5, 1.5, n))
    y = ORC.rmsnorm(np.full(n, c), g, eps)
    expect = bf16_vals(g) * c / math.sqrt(c * c + eps)
    np.testing.assert_allclose(y, expect, rtol=1e-14)


def test_rmsnorm_hand_case_uses_mean_not_sum_and_applies_gain():
    g = bf16_bits([1.5, 0.5])
    y = ORC.rmsnorm(np.array([3.0, 4.0]), g, 0.0)
    r = math.sqrt((9 + 16) / 2)
    np.testing.assert_allclose(y, [1.5 * 3 / r, 0.5 * 4 / r], rtol=1e-14)


def test_rmsnorm_scale_invariance():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(300)
    g = bf16_bits(1 + 0.02 * rng.standard_normal(300))
    np.testing.assert_allclose(ORC.rmsnorm(x, g, 0.0), ORC.rmsnorm(x * 1234.5, g, 0.0), rtol=1e-12)


# ------------------------------------------------------------------ GEMV

def test_gemv_permutation_matrix_is_exact():
    n = 37
    perm = np.random.default_rng(3).permutation(n)
    W = np.zeros((n, n), np.float32)
    W[np.arange(n), perm] = 1.0
    x = np.random.default_rng(4).standard_normal(n)
    assert np.array_equal(ORC.gemv_bf16(bf16_bits(W), x), x[perm])


@pytest.mark.parametrize("rows,cols", [(333, 1100), (7, 11008), (1, 8), (64, 3)])
def test_gemv_odd_shapes_match_brute_force(rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    W = bf16_bits(0.02 * rng.standard_normal((rows, cols)))
    x = rng.standard_normal(cols)
    ref = bf16_vals(W) @ x  # library matmul of the decoded matrix
    np.testing.assert_allclose(ORC.gemv_bf16(W, x), ref, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ int4

def test_int4_every_nibble_both_positions_every_scale_kind():
    # one row per scale kind; each row's bytes run over all 256 values, so every nibble appears as
    # a low (even input) and high (odd input) element. Scale bits: +s, -s, 0, fp16 subnormal, max.
    scale_bits = np.array([0x2E66, 0xAE66, 0x0000, 0x0001, 0x7BFF], np.uint16)  # fp16
    rows, cols, group = len(scale_bits), 512, 512
    wq = np.tile(np.arange(256, dtype=np.uint8), (rows, 1))
    scales = scale_bits.reshape(rows, 1)
    w = ORC.dequant_int4(wq, scales, scale_is_bf16=False, group=group)
    s = scale_bits.view(np.float16).astype(np.float64)
    for r in range(rows):
        for c in range(cols):
            b = c // 2
            q = (b & 0xF) if c % 2 == 0 else (b >> 4)
            assert w[r, c] == (q - 8) * s[r]


def test_int4_group_index_runs_along_the_input_dimension():
    rows, cols, group = 3, 256, 64
    wq = np.full((rows, cols // 2), 0x99, np.uint8)  # q = 9 -> (q - 8) = 1 everywhere
    scales = bf16_bits(np.arange(rows * (cols // group), dtype=np.float32).reshape(rows, -1) + 1)
    w = ORC.dequant_int4(wq, scales, scale_is_bf16=True, group=group)
    expect = np.repeat(bf16_vals(scales), group, axis=1)
    assert np.array_equal(w, expect)


def test_int4_gemv_matches_brute_force():
    rng = np.random.default_rng(5)
    rows, cols, group = 45, 640, 128
    wq = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    s16 = np.abs(0.005 * rng.standard_normal((rows, cols // group))).astype(np.float16)
    x = rng.standard_normal(cols)
    lo, hi = (wq & 0xF).astype(np.int64) - 8, (wq >> 4).astype(np.int64) - 8
    q = np.stack([lo, hi], axis=2).reshape(rows, cols)
    W = q * np.repeat(s16.astype(np.float64), group, axis=1)
    np.testing.assert_allclose(ORC.gemv_int4(wq, s16.view(np.uint16), False, group, x), W @ x,
                               rtol=1e-12, atol=1e-14)


def test_exponent_trick_identity_for_every_nibble():
    # tinyinfer's dequant: OR the nibble into the mantissa of 2^23 and subtract. In binary32,
    # bits 0x4B000000 | q encode 2^23 + q exactly, so subtracting 2^23 + 8 gives q - 8 exactly.
    for q in range(16):
        f = np.array([0x4B000000 | q], np.uint32).view(np.float32)[0]
        assert float(f) - 8388616.0 == q - 8
        # 16-bit form: 0x6400 | q is 1024 + q in fp16
        h = np.array([0x6400 | q], np.uint16).view(np.float16)[0]
        assert float(h) - 1032.0 == q - 8


# ------------------------------------------------------------------ RoPE

def test_rope_hand_case_d4_half_split():
    v = np.array([1.0, 2.0, 3.0, 4.0])
    out = ORC.rope(v, pos=1, theta=10000.0)
    a0, a1 = 1.0, 1.0 / 100.0  # theta_i = pos * 10000^(-2i/4)
    expect = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
              3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    np.testing.assert_allclose(out, expect, rtol=1e-15, atol=1e-15)


def test_rope_position_zero_is_identity_and_norm_preserved():
    rng = np.random.default_rng(6)
    v = rng.standard_normal(128)
    assert np.array_equal(ORC.rope(v, 0, 1e6), v)
    out = ORC.rope(v, 4095, 1e6)
    half = 64
    np.testing.assert_allclose(out[:half] ** 2 + out[half:] ** 2, v[:half] ** 2 + v[half:] ** 2,
                               rtol=1e-12)


def test_rope_composes_and_scores_depend_on_offset_only():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    np.testing.assert_allclose(ORC.rope(ORC.rope(q, 300, 5e5), 21, 5e5), ORC.rope(q, 321, 5e5),
                               rtol=1e-9, atol=1e-12)
    s1 = ORC.rope(q, 1000, 1e4) @ ORC.rope(k, 990, 1e4)
    s2 = ORC.rope(q, 17, 1e4) @ ORC.rope(k, 7, 1e4)
    assert abs(s1 - s2) < 1e-9


# ------------------------------------------------------------------ softmax / attention

def test_softmax_hand_values_and_overflow_safety():
    np.testing.assert_allclose(ORC.softmax(np.array([0.0, math.log(2.0)])), [1 / 3, 2 / 3], rtol=1e-15)
    p = ORC.softmax(np.array([1000.0, 1000.0, 0.0]))   # needs the max subtracted first
    np.testing.assert_allclose(p, [0.5, 0.5, 0.0], atol=1e-300)
    p = ORC.softmax(np.random.default_rng(8).standard_normal(777) * 5)
    assert abs(p.sum() - 1) < 1e-12


def _kv(nkv, ctx, d, rng, std=1.0):
    return (bf16_bits(std * rng.standard_normal((nkv, ctx, d))),
            bf16_bits(std * rng.standard_normal((nkv, ctx, d))))


def test_attention_single_position_returns_v0_exactly():
    rng = np.random.default_rng(9)
    K, V = _kv(2, 5, 64, rng)
    q = rng.standard_normal(4 * 64)
    out = ORC.attention(q, K, V, 4, 2, 64, n_ctx=1).reshape(4, 64)
    vals = bf16_vals(V)
    for h in range(4):
        assert np.array_equal(out[h], vals[h // 2, 0])


def test_attention_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(10)
    K = np.tile(bf16_bits(rng.standard_normal(64)), (1, 9, 1)).reshape(1, 9, 64)
    V = bf16_bits(rng.standard_normal((1, 9, 64)))
    out = ORC.attention(rng.standard_normal(64 * 3), K, V, 3, 1, 64, n_ctx=9).reshape(3, 64)
    for h in range(3):
        np.testing.assert_allclose(out[h], bf16_vals(V)[0].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attention_two_key_hand_case_pins_the_scale():
    d, a, b = 64, 2.0, 3.0
    q = np.zeros(d); q[0] = a
    K = np.zeros((1, 2, d), np.float32); K[0, 0, 0] = b
    V = np.zeros((1, 2, d), np.float32); V[0, 0, :] = 1.0
    out = ORC.attention(q, bf16_bits(K), bf16_bits(V), 1, 1, d, n_ctx=2)
    p0 = 1.0 / (1.0 + math.exp(-a * b / math.sqrt(d)))
    np.testing.assert_allclose(out, np.full(d, p0), rtol=1e-14)


def test_attention_gqa_groups_are_contiguous():
    # each KV head j holds a constant value row j+1: head h must return exactly (h // group) + 1
    nq, nkv, d, ctx = 12, 4, 64, 6
    rng = np.random.default_rng(11)
    K = bf16_bits(rng.standard_normal((nkv, ctx, d)))
    V = bf16_bits(np.repeat(np.arange(1, nkv + 1, dtype=np.float32), ctx * d).reshape(nkv, ctx, d))
    out = ORC.attention(rng.standard_normal(nq * d), K, V, nq, nkv, d, n_ctx=ctx).reshape(nq, d)
    for h in range(nq):
        np.testing.assert_allclose(out[h], h // (nq // nkv) + 1, rtol=1e-14)


def test_attention_one_dominant_key_selects_its_value():
    d, ctx = 64, 40
    rng = np.random.default_rng(12)
    K = rng.standard_normal((1, ctx, d)) * 0.01
    q = np.zeros(d); q[3] = 100.0
    K[0, 17, 3] = 30.0
    V = rng.standard_normal((1, ctx, d))
    out = ORC.attention(q, bf16_bits(K), bf16_bits(V), 1, 1, d, n_ctx=ctx)
    np.testing.assert_allclose(out, bf16_vals(bf16_bits(V))[0, 17], rtol=1e-9, atol=1e-9)


def test_attention_reads_only_the_first_n_ctx_slots():
    rng = np.random.default_rng(13)
    K, V = _kv(2, 30, 64, rng)
    q = rng.standard_normal(4 * 64)
    a = ORC.attention(q, K, V, 4, 2, 64, n_ctx=11)
    K2, V2 = K.copy(), V.copy()
    K2[:, 11:] = 0x7FC0  # NaN beyond the length must not be touched
    V2[:, 11:] = 0x7FC0
    assert np.array_equal(ORC.attention(q, K2, V2, 4, 2, 64, n_ctx=11), a)


@pytest.mark.parametrize("n_ctx,chunk_len,n_chunks", [
    (1, 1, 1), (1, 64, 3), (57, 8, 8), (57, 10, 6), (128, 128, 1), (129, 128, 2),
    (300, 7, 50), (300, 1000, 1), (77, 30, 5)])  # the last cases leave whole chunks empty
def test_split_k_partials_and_combine_equal_plain_attention(n_ctx, chunk_len, n_chunks):
    rng = np.random.default_rng(n_ctx + chunk_len)
    nq, nkv, d = 8, 2, 64
    K, V = _kv(nkv, 320, d, rng)
    q = rng.standard_normal(nq * d)
    m, l, o = ORC.attention_partials(q, K, V, nq, nkv, d, n_ctx, chunk_len, n_chunks)
    if n_chunks * chunk_len > n_ctx:
        empty = [c for c in range(n_chunks) if c * chunk_len >= n_ctx]
        for c in empty:
            assert np.all(m[:, c] == -np.inf) and np.all(l[:, c] == 0) and np.all(o[:, c] == 0)
    np.testing.assert_allclose(ORC.attention_combine(m, l, o),
                               ORC.attention(q, K, V, nq, nkv, d, n_ctx), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ SwiGLU / argmax

def test_swiglu_known_values():
    g = np.array([0.0, 1.0, -1.0, 40.0, -40.0])
    u = np.array([5.0, 2.0, 3.0, 0.5, 7.0])
    a = ORC.swiglu(g, u)
    sig = lambda z: 1 / (1 + math.exp(-z))
    np.testing.assert_allclose(a, [0.0, 2 * sig(1.0), -3 * sig(-1.0), 0.5 * 40 * sig(40), 7 * -40 * sig(-40)],
                               rtol=1e-14, atol=1e-30)
    assert abs(ORC.swiglu(np.array([1.0]), np.array([1.0]))[0] - 0.7310585786300049) < 1e-15


def test_argmax_lowest_index_on_ties_and_errors_on_nonfinite():
    assert ORC.argmax(np.array([1.0, 3.0, 3.0, 2.0])) == (1, 0)
    x = np.random.default_rng(14).standard_normal(5000)
    assert ORC.argmax(x)[0] == int(np.argmax(x))
    x[4000] = np.nan
    assert ORC.argmax(x) == (-1, ERR_NONFINITE)
    x[4000] = np.inf
    assert ORC.argmax(x)[1] == ERR_NONFINITE


def test_oracle_f32_build_is_float():
    o32 = Oracle("f32")
    assert o32.real == np.float32
    x = np.random.default_rng(15).standard_normal(100)
    W = bf16_bits(0.02 * np.random.default_rng(16).standard_normal((50, 100)))
    np.testing.assert_allclose(o32.gemv_bf16(W, x), ORC.gemv_bf16(W, x), rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------- gathered-expert MLP

def _moe(fmt="bf16", E=6, k=3, H=64, F=96, seed=0):
    return synth.make_moe(E, k, H, F, fmt, 32, "bf16" if fmt == "int4" else "fp16", seed)


def _dense_mlp(orc, m, e, fmt):
    # the dense SwiGLU MLP of expert e from the pinned blocks
    if fmt == "int4":
        g = orc.gemv_int4(m["wg"][e], m["sg"][e], 1, 32, m["x"])
        u = orc.gemv_int4(m["wu"][e], m["su"][e], 1, 32, m["x"])
        return orc.gemv_int4(m["wd"][e], m["sd"][e], 1, 32, orc.swiglu(g, u))
    g = orc.gemv_bf16(m["wg"][e], m["x"])
    u = orc.gemv_bf16(m["wu"][e], m["x"])
    return orc.gemv_bf16(m["wd"][e], orc.swiglu(g, u))


def _moe_call(orc, m, fmt, ids, weights):
    f = 1 if fmt == "int4" else 0
    return orc.moe_mlp(f, 32, 1, m["wg"], m["sg"], m["wu"], m["su"], m["wd"], m["sd"], ids, weights, m["x"])


@pytest.mark.parametrize("fmt", ["bf16", "int4"])
def test_moe_one_expert_is_the_dense_mlp(fmt):
    # top-1 with weight 1 reduces to the dense SwiGLU MLP of that expert, gathered by its id
    m = _moe(fmt)
    for e in (0, 4):
        got = _moe_call(ORC, m, fmt, [e], [1.0])
        assert np.array_equal(got, _dense_mlp(ORC, m, e, fmt))


@pytest.mark.parametrize("fmt", ["bf16", "int4"])
def test_moe_is_the_weighted_sum_of_the_chosen_experts(fmt):
    m = _moe(fmt, seed=1)
    ids, w = m["ids"], m["weights"].astype(np.float64)
    got = _moe_call(ORC, m, fmt, ids, w)
    want = sum(wi * _dense_mlp(ORC, m, int(e), fmt) for e, wi in zip(ids, w))
    assert np.allclose(got, want, rtol=1e-13, atol=1e-15)
    # each expert is read at its own id: a gather from the wrong slot fails this
    assert not np.allclose(got, sum(wi * _dense_mlp(ORC, m, (int(e) + 1) % 6, fmt) for e, wi in zip(ids, w)))


def test_moe_routing_invariants():
    m = _moe(seed=2)
    ids, w = m["ids"], m["weights"].astype(np.float64)
    base = _moe_call(ORC, m, "bf16", ids, w)
    # the order of the chosen experts does not matter
    perm = np.array([2, 0, 1])
    assert np.allclose(_moe_call(ORC, m, "bf16", ids[perm], w[perm]), base, rtol=1e-13, atol=1e-15)
    # an expert chosen with weight 0 adds nothing (exactly)
    got = _moe_call(ORC, m, "bf16", np.append(ids, 5), np.append(w, 0.0))
    assert np.array_equal(got, base)
    # linear in the routing weights: one id twice counts as once with the summed weight
    two = _moe_call(ORC, m, "bf16", [ids[0], ids[0]], [0.25, 0.5])
    assert np.allclose(two, _moe_call(ORC, m, "bf16", [ids[0]], [0.75]), rtol=1e-13, atol=1e-15)


def test_moe_synthetic_case_is_valid():
    m = synth.make_moe(64, 8, 2048, 1024)
    assert len(set(m["ids"].tolist())) == 8 and m["ids"].min() >= 0 and m["ids"].max() < 64
    assert abs(float(m["weights"].sum()) - 1.0) < 1e-6 and (m["weights"] > 0).all()
    assert m["wg"].shape == (64, 1024, 2048) and m["wd"].shape == (64, 2048, 1024)

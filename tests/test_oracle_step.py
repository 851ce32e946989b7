"""The oracle's whole decode step: its wiring, checked against the pinned building blocks and
against closed forms; the byte accounting against the numbers the pages print."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import Oracle, ERR_INVALID

ORC = Oracle("f64")
GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_byte_accounting.json")))


def f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tiny(**kw):
    return synth.config("tiny", **kw)


# ---------------------------------------------------------------- byte accounting (pages' numbers)

def test_llama1b_weight_bytes_match_the_page():
    mb = synth.model_bytes(synth.config("llama1b"))
    total = mb["layers"] + mb["embed"] + mb["final_norm"]   # tied: the table is streamed once
    assert total == GOLDEN["llama32_1b_weight_bytes"]["value"]


def test_llama1b_layer_bytes_mlp_share_and_kv_per_position():
    cfg = synth.config("llama1b")
    sh = synth.linear_shapes(cfg)
    mat = sum(r * c * 2 for r, c in sh.values())
    assert round(mat / 1e6, 1) == GOLDEN["llama32_1b_layer_matmul_mb"]["value"]
    mlp = sum(sh[w][0] * sh[w][1] * 2 for w in ("wg", "wu", "wd"))
    assert round(mlp / mat, 2) == GOLDEN["llama32_1b_mlp_share"]["value"]
    kv = cfg["n_layers"] * cfg["n_kv_heads"] * cfg["head_dim"] * 2 * 2
    assert kv == GOLDEN["llama32_1b_kv_bytes_per_position"]["value"]
    assert round(kv * 4096 / 1e6) == GOLDEN["llama32_1b_kv_mb_at_4096"]["value"]


def test_llama1b_floor_at_the_pages_bandwidth():
    bw = GOLDEN["rtx3050_stream_gbs"]["value"] * 1e9
    w = GOLDEN["llama32_1b_weight_bytes"]["value"]
    assert round(w / bw * 1e3, 2) == GOLDEN["llama32_1b_floor_ms"]["value"]
    kv = GOLDEN["llama32_1b_kv_bytes_per_position"]["value"] * 4096
    assert round((w + kv) / bw * 1e3, 2) == GOLDEN["llama32_1b_floor_ms_ctx4096"]["value"]


def test_tinyllama_bytes_match_the_page():
    cfg = synth.config("tinyllama_int4")
    bf = dict(cfg, weight_format="bf16")
    mb = synth.model_bytes(bf)
    # 16-bit: layers plus the output head (the input side reads one row)
    assert round((mb["layers"] + mb["lm_head"]) / 1e9, 2) == GOLDEN["tinyllama_bf16_gb_per_token"]["value"]
    # int4 at 4.25 bits per weight, head included in int4 on that page
    n_w = sum(r * c for r, c in synth.linear_shapes(cfg).values()) * cfg["n_layers"] + cfg["vocab"] * cfg["hidden"]
    assert round(n_w * 4.25 / 8 / 1e9, 2) == GOLDEN["tinyllama_int4_gb_per_token"]["value"]


# ---------------------------------------------------------------- step wiring

@pytest.fixture(scope="module")
def tiny_bias():
    cfg = tiny(qkv_bias=True, n_layers=1, max_ctx=8)
    return cfg, synth.make_model(cfg, seed=3)


def test_first_layer_equals_composition_of_pinned_blocks(tiny_bias):
    cfg, w = tiny_bias
    om = ORC.model(cfg, w)
    K, V = synth.make_kv(cfg, prefill=3, seed=3)
    tok, pos = 77, 3
    K0, V0 = K.copy(), V.copy()
    logits, am, rc, tr = ORC.decode_step(om, tok, pos, K, V, trace=True)
    assert rc == 0
    H, nq, nkv, d = cfg["hidden"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    L = w["layers"][0]
    x = f64(w["embed"][tok])
    n = ORC.rmsnorm(x, L["g1"], cfg["rms_eps"])
    q = ORC.gemv_bf16(L["wq"], n) + f64(L["bq"])
    k = ORC.gemv_bf16(L["wk"], n) + f64(L["bk"])
    v = ORC.gemv_bf16(L["wv"], n) + f64(L["bv"])
    q = np.concatenate([ORC.rope(q[h * d:(h + 1) * d], pos, cfg["rope_theta"]) for h in range(nq)])
    k = np.concatenate([ORC.rope(k[j * d:(j + 1) * d], pos, cfg["rope_theta"]) for j in range(nkv)])
    kb = np.array([ORC.round_bf16(t) for t in k], np.uint16).reshape(nkv, d)
    vb = np.array([ORC.round_bf16(t) for t in v], np.uint16).reshape(nkv, d)
    # the step writes exactly slot pos of layer 0 and nothing else
    assert np.array_equal(K[0, :, pos], kb) and np.array_equal(V[0, :, pos], vb)
    mask = np.ones(K.shape, bool); mask[0, :, pos] = False
    assert np.array_equal(K[mask], K0[mask]) and np.array_equal(V[mask], V0[mask])
    att = ORC.attention(q, K[0], V[0], nq, nkv, d, pos + 1)
    x = x + ORC.gemv_bf16(L["wo"], att)
    n2 = ORC.rmsnorm(x, L["g2"], cfg["rms_eps"])
    a = ORC.swiglu(ORC.gemv_bf16(L["wg"], n2), ORC.gemv_bf16(L["wu"], n2))
    x = x + ORC.gemv_bf16(L["wd"], a)
    np.testing.assert_allclose(tr[0], x, rtol=1e-13, atol=1e-13)
    nf = ORC.rmsnorm(x, w["final_norm"], cfg["rms_eps"])
    np.testing.assert_allclose(logits, ORC.gemv_bf16(w["lm_head"], nf), rtol=1e-13, atol=1e-13)
    assert am == int(np.argmax(logits))


def test_zero_blocks_leave_the_embedding_row():
    cfg = tiny(n_layers=2, max_ctx=4)
    w = synth.make_model(cfg, seed=4)
    for L in w["layers"]:
        L["wo"] = np.zeros_like(L["wo"])
        L["wd"] = np.zeros_like(L["wd"])
    K, V = synth.make_kv(cfg, prefill=0)
    logits, am, rc, tr = ORC.decode_step(ORC.model(cfg, w), 5, 0, K, V, trace=True)
    x = f64(w["embed"][5])
    assert np.array_equal(tr[1], x)
    g = f64(w["final_norm"])
    nf = x / np.sqrt(np.mean(x * x) + cfg["rms_eps"]) * g
    np.testing.assert_allclose(logits, f64(w["lm_head"]) @ nf, rtol=1e-12, atol=1e-14)


def test_tied_head_uses_the_embedding():
    cfg = tiny(tied=True, max_ctx=4)
    w = synth.make_model(cfg)
    assert w["lm_head"] is w["embed"]


def test_invalid_arguments_are_rejected():
    cfg = tiny(max_ctx=4)
    om = ORC.model(cfg, synth.make_model(cfg))
    K, V = synth.make_kv(cfg, 0)
    assert ORC.decode_step(om, cfg["vocab"], 0, K, V)[2] == ERR_INVALID
    assert ORC.decode_step(om, 0, 4, K, V)[2] == ERR_INVALID
    assert ORC.decode_step(om, -1, 0, K, V)[2] == ERR_INVALID


def test_int4_step_matches_composition():
    cfg = tiny(weight_format="int4", group_size=64, scale_dtype="fp16", n_layers=1, max_ctx=4)
    w = synth.make_model(cfg, seed=5)
    K, V = synth.make_kv(cfg, 0)
    _, _, rc, tr = ORC.decode_step(ORC.model(cfg, w), 9, 0, K, V, trace=True)
    assert rc == 0
    L = w["layers"][0]
    x = f64(w["embed"][9])
    n = ORC.rmsnorm(x, L["g1"], cfg["rms_eps"])
    v = ORC.gemv_int4(L["wv"], L["sv"], False, 64, n)
    vb = np.array([ORC.round_bf16(t) for t in v], np.uint16)
    att = np.concatenate([f64(vb.reshape(2, 64)[h // 2]) for h in range(4)])  # pos 0: o = V[0]
    x = x + ORC.gemv_int4(L["wo"], L["so"], False, 64, att)
    n2 = ORC.rmsnorm(x, L["g2"], cfg["rms_eps"])
    a = ORC.swiglu(ORC.gemv_int4(L["wg"], L["sg"], False, 64, n2), ORC.gemv_int4(L["wu"], L["su"], False, 64, n2))
    x = x + ORC.gemv_int4(L["wd"], L["sd"], False, 64, a)
    np.testing.assert_allclose(tr[0], x, rtol=1e-13, atol=1e-13)


def test_fp32_and_fp64_oracles_agree_on_the_tiny_model():
    """Same bytes in, fp32 vs fp64 arithmetic: logits within 1e-5 relative. The bf16 KV store can
    round a value to the neighbouring bf16 in one precision and not the other; such a slot must
    differ by exactly one bf16 step, it must be rare, and the caches are re-synchronised so that
    every step starts from the same bytes."""
    cfg = tiny()
    w = synth.make_model(cfg)
    toks = synth.make_tokens(cfg, cfg["prompt"])
    o32 = Oracle("f32")
    m64, m32 = ORC.model(cfg, w), o32.model(cfg, w)
    K64, V64 = synth.make_kv(cfg, 0)
    flips = 0
    for pos in range(cfg["prompt"] + cfg["steps"]):
        tok = int(toks[pos]) if pos < cfg["prompt"] else am
        K32, V32 = K64.copy(), V64.copy()
        l64, am, rc = ORC.decode_step(m64, tok, pos, K64, V64)
        l32, _, _ = o32.decode_step(m32, tok, pos, K32, V32)
        assert rc == 0
        d = np.concatenate([(K32 != K64).ravel(), (V32 != V64).ravel()])
        if d.any():
            flips += int(d.sum())
            for a, b in ((K32, K64), (V32, V64)):
                diff = a != b
                assert np.all(np.abs(a[diff].astype(np.int32) - b[diff].astype(np.int32)) == 1)
            continue
        rel = np.linalg.norm(l32 - l64) / np.linalg.norm(l64)
        assert rel < 1e-5, (pos, rel)
    written = 2 * cfg["n_layers"] * cfg["n_kv_heads"] * cfg["head_dim"] * (cfg["prompt"] + cfg["steps"])
    assert flips <= 0.002 * written  # fp32 dot products carry ~1e-6 relative error

"""Per-kernel parity on the GPU: the packer, the streaming GEMV (bf16 and int4, every epilogue) and
split-K attention, each called through the C ABI and compared with the CPU oracle element by
element on seeded inputs, on shapes that span several ring stages and end in ragged tails."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402
from util import bf16_to_f64, kv_close  # noqa: E402

pytestmark = pytest.mark.gpu
ORC = Oracle("f64")


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host_u16(t):
    return t.cpu().numpy().view(np.uint16)


def pack(fmt, group, sdt, W, S=None):
    rows = W.shape[0]
    cols = W.shape[1] * (2 if fmt == T.TINFER_INT4 else 1)
    rb = T.tinfer_packed_row_bytes(fmt, cols, group)
    assert rb > 0
    out = torch.empty(rows * rb, dtype=torch.uint8, device="cuda")
    rc = T.tinfer_pack_matrix(fmt, group, sdt, rows, cols, dev(W), dev(S) if S is not None else None, out)
    assert rc == 0
    return out


def gemv(fmt, group, sdt, packed, rows, cols, x, gain=None, bias=None, epi=T.TINFER_EPI_STORE, y=None,
         eps=1e-5):
    xd = torch.from_numpy(np.asarray(x, np.float32)).cuda()
    gd = torch.from_numpy(np.asarray(gain, np.float32)).cuda() if gain is not None else None
    bd = torch.from_numpy(np.asarray(bias, np.float32)).cuda() if bias is not None else None
    n_out = rows // 2 if epi == T.TINFER_EPI_SWIGLU else rows
    yd = torch.from_numpy(np.asarray(y, np.float32)).cuda() if y is not None else \
        torch.full((n_out,), np.nan, dtype=torch.float32, device="cuda")
    am = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    rc = T.tinfer_op_gemv(fmt, group, sdt, rows, cols, packed, xd, gd, eps, bd, epi, yd, am)
    torch.cuda.synchronize()
    return rc, yd.cpu().numpy().astype(np.float64), int(am.item())


# ------------------------------------------------------------------ packer

@pytest.mark.parametrize("name,over", [
    ("tiny", {}), ("tiny", dict(qkv_bias=True)),
    ("tiny", dict(weight_format="int4", group_size=64, scale_dtype="fp16", ffn=704)),
    ("tiny", dict(weight_format="int4", group_size=128, scale_dtype="bf16", ffn=768))])
def test_pack_unpack_layer_round_trip_is_bit_exact(name, over):
    c = synth.config(name, n_layers=1, max_ctx=8, **over)
    w = synth.make_model(c, seed=11)
    eng = T.Engine(c, w)
    L = w["layers"][0]
    back = {k: torch.zeros_like(dev(v)) for k, v in L.items()}
    dst = T.tinfer_layer_src()
    for k, t in back.items():
        setattr(dst, k, t.data_ptr())
    assert T.tinfer_unpack_layer(eng.cfg, eng.blobs[0], dst) == 0
    torch.cuda.synchronize()
    for k, v in L.items():
        assert np.array_equal(back[k].cpu().numpy().view(v.dtype), v), k
    eng.close()


# ------------------------------------------------------------------ GEMV bf16

@pytest.mark.parametrize("rows,cols", [(333, 1104), (2048, 2048), (97, 8192), (40, 8960), (1376, 256),
                                       (256, 688), (7, 64), (1, 2048)])
def test_gemv_bf16_matches_oracle(rows, cols):
    rng = np.random.default_rng(rows * 31 + cols)
    W = synth.normal_bf16(f"gemv{rows}x{cols}", (rows, cols), 0.0, 0.02)
    x = rng.standard_normal(cols).astype(np.float32)
    bias = rng.standard_normal(rows).astype(np.float32)
    p = pack(T.TINFER_BF16, 0, 0, W)
    rc, y, _ = gemv(T.TINFER_BF16, 0, 0, p, rows, cols, x, bias=bias)
    assert rc == 0
    ref = ORC.gemv_bf16(W, x.astype(np.float64)) + bias
    np.testing.assert_allclose(y, ref, rtol=1e-4, atol=2e-5 * np.sqrt(cols / 256))


@pytest.mark.parametrize("cols", [2048, 2560, 8192])  # one, two and four row segments
def test_gemv_rmsnorm_prologue_matches_oracle(cols):
    rows = 515
    rng = np.random.default_rng(3)
    W = synth.normal_bf16("gemvnorm", (rows, cols), 0.0, 0.02)
    x = (3 * rng.standard_normal(cols)).astype(np.float32)
    g_bits = synth.normal_bf16("gain", (cols,), 1.0, 0.02)
    g = bf16_to_f64(g_bits).astype(np.float32)
    p = pack(T.TINFER_BF16, 0, 0, W)
    rc, y, _ = gemv(T.TINFER_BF16, 0, 0, p, rows, cols, x, gain=g, eps=1e-5)
    assert rc == 0
    n = ORC.rmsnorm(x.astype(np.float64), g_bits, 1e-5)
    np.testing.assert_allclose(y, ORC.gemv_bf16(W, n), rtol=1e-4, atol=1e-4)


def test_gemv_residual_and_swiglu_epilogues():
    rows, cols = 300, 1536
    rng = np.random.default_rng(4)
    W = synth.normal_bf16("gemvres", (rows, cols), 0.0, 0.02)
    x = rng.standard_normal(cols).astype(np.float32)
    y0 = rng.standard_normal(rows).astype(np.float32)
    p = pack(T.TINFER_BF16, 0, 0, W)
    rc, y, _ = gemv(T.TINFER_BF16, 0, 0, p, rows, cols, x, epi=T.TINFER_EPI_RESIDUAL, y=y0)
    assert rc == 0
    np.testing.assert_allclose(y, y0 + ORC.gemv_bf16(W, x.astype(np.float64)), rtol=1e-4, atol=5e-5)
    # gate/up interleaved rows: (g0, u0, g1, u1, ...)
    rc, a, _ = gemv(T.TINFER_BF16, 0, 0, p, rows, cols, x, epi=T.TINFER_EPI_SWIGLU)
    assert rc == 0
    full = ORC.gemv_bf16(W, x.astype(np.float64))
    np.testing.assert_allclose(a, ORC.swiglu(full[0::2], full[1::2]), rtol=1e-4, atol=5e-5)


def test_gemv_argmax_ties_lowest_index_and_nonfinite():
    rows, cols = 5000, 256
    W = synth.normal_bf16("argmax", (rows, cols), 0.0, 0.02)
    W[4321] = W[17] = f_row = synth.normal_bf16("hot", (cols,), 0.5, 0.0)  # two equal maxima
    x = np.ones(cols, np.float32)
    p = pack(T.TINFER_BF16, 0, 0, W)
    rc, y, am = gemv(T.TINFER_BF16, 0, 0, p, rows, cols, x, epi=T.TINFER_EPI_ARGMAX)
    assert rc == 0 and am == 17 and y[17] == y[4321]
    ref = ORC.gemv_bf16(W, x.astype(np.float64))
    assert ORC.argmax(ref)[0] == 17
    # the same with rows wider than one segment (the LM head of a 2560-wide model)
    W3 = synth.normal_bf16("argmax3", (3000, 2560), 0.0, 0.02)
    W3[2999] = W3[1500] = synth.normal_bf16("hot3", (2560,), 0.25, 0.0)
    rc, y3, am3 = gemv(T.TINFER_BF16, 0, 0, pack(T.TINFER_BF16, 0, 0, W3), 3000, 2560,
                       np.ones(2560, np.float32), epi=T.TINFER_EPI_ARGMAX)
    assert rc == 0 and am3 == 1500
    np.testing.assert_allclose(y3, ORC.gemv_bf16(W3, np.ones(2560)), rtol=1e-4, atol=1e-4)
    W2 = W.copy()
    W2[999, 5] = 0x7FC0  # NaN
    p2 = pack(T.TINFER_BF16, 0, 0, W2)
    rc, _, am = gemv(T.TINFER_BF16, 0, 0, p2, rows, cols, x, epi=T.TINFER_EPI_ARGMAX)
    assert rc == T.TINFER_ERR_NONFINITE and am == -1
    del f_row


# ------------------------------------------------------------------ GEMV int4

@pytest.mark.parametrize("rows,cols,group,sdt", [
    (333, 2048, 64, "fp16"), (100, 5632, 64, "fp16"), (77, 2560, 128, "bf16"), (50, 8192, 128, "bf16"),
    (64, 256, 32, "fp16"), (2561, 2048, 64, "fp16")])
def test_gemv_int4_matches_oracle(rows, cols, group, sdt):
    key = f"i4_{rows}_{cols}"
    Wq = synth.nibbles(key, (rows, cols // 2))
    S = synth.abs_normal_16(key + ".s", (rows, cols // group), 0.005, sdt)
    x = np.random.default_rng(rows).standard_normal(cols).astype(np.float32)
    fmt_s = T.TINFER_SCALE_BF16 if sdt == "bf16" else T.TINFER_SCALE_FP16
    p = pack(T.TINFER_INT4, group, fmt_s, Wq, S)
    rc, y, _ = gemv(T.TINFER_INT4, group, fmt_s, p, rows, cols, x)
    assert rc == 0
    ref = ORC.gemv_int4(Wq, S, sdt == "bf16", group, x.astype(np.float64))
    np.testing.assert_allclose(y, ref, rtol=1e-4, atol=3e-5 * np.sqrt(cols / 256))


@pytest.mark.parametrize("sdt", ["fp16", "bf16"])
def test_int4_dequant_is_bit_exact(sdt):
    # x = e_k extracts column k: y[r] = (q - 8) * s exactly, the oracle's dequantised value
    rows, cols, group = 96, 512, 64
    Wq = synth.nibbles("dq" + sdt, (rows, cols // 2))
    S = synth.abs_normal_16("dq.s" + sdt, (rows, cols // group), 0.005, sdt)
    fmt_s = T.TINFER_SCALE_BF16 if sdt == "bf16" else T.TINFER_SCALE_FP16
    p = pack(T.TINFER_INT4, group, fmt_s, Wq, S)
    deq = ORC.dequant_int4(Wq, S, sdt == "bf16", group)
    for k in (0, 1, 2, 3, 4, 5, 6, 7, 8, 15, 16, 31, 32, 63, 64, 200, 511):
        x = np.zeros(cols, np.float32)
        x[k] = 1.0
        rc, y, _ = gemv(T.TINFER_INT4, group, fmt_s, p, rows, cols, x)
        assert rc == 0
        assert np.array_equal(y, deq[:, k]), k


# ------------------------------------------------------------------ attention

def attention_case(nq, nkv, d, pos, n_chunks, max_ctx=None, seed=0, theta=10000.0):
    max_ctx = max_ctx or pos + 3
    rng = np.random.default_rng(seed + pos)
    K = synth.normal_bf16(f"attK{nq}{nkv}{d}{pos}", (nkv, max_ctx, d), 0.0, 1.0)
    V = synth.normal_bf16(f"attV{nq}{nkv}{d}{pos}", (nkv, max_ctx, d), 0.0, 1.0)
    qkv = rng.standard_normal((nq + 2 * nkv) * d).astype(np.float32)
    Kd, Vd = dev(K), dev(V)
    out = torch.full((nq * d,), np.nan, dtype=torch.float32, device="cuda")
    parts = None
    if n_chunks > 0:
        parts = (torch.zeros(nq * n_chunks, device="cuda"), torch.zeros(nq * n_chunks, device="cuda"),
                 torch.zeros(nq * n_chunks * d, device="cuda"))
    rc = T.tinfer_op_attention(nq, nkv, d, max_ctx, theta, pos, n_chunks, torch.from_numpy(qkv).cuda(),
                               Kd, Vd, out, *(parts or (None, None, None)))
    torch.cuda.synchronize()
    assert rc == 0
    Kg, Vg = host_u16(Kd), host_u16(Vd)
    # the slot at pos holds bf16(RoPE(k)) and bf16(v) (close to the oracle's rounding, kv_close);
    # every other slot is untouched
    q = qkv[:nq * d].astype(np.float64)
    k = qkv[nq * d:(nq + nkv) * d].astype(np.float64)
    v = qkv[(nq + nkv) * d:].astype(np.float64)
    k_rot = np.concatenate([ORC.rope(k[j * d:(j + 1) * d], pos, theta) for j in range(nkv)])
    kb = np.array([ORC.round_bf16(t) for t in k_rot], np.uint16).reshape(nkv, d)
    vb = np.array([ORC.round_bf16(t) for t in v], np.uint16).reshape(nkv, d)
    assert kv_close(Kg[:, pos], kb) <= 0 and kv_close(Vg[:, pos], vb) <= 0
    mask = np.ones(K.shape, bool)
    mask[:, pos] = False
    assert np.array_equal(Kg[mask], K[mask]) and np.array_equal(Vg[mask], V[mask])
    # attention over the cache as written, against the oracle
    q_rot = np.concatenate([ORC.rope(q[h * d:(h + 1) * d], pos, theta) for h in range(nq)])
    ref = ORC.attention(q_rot, Kg, Vg, nq, nkv, d, pos + 1)
    np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=1e-4, atol=3e-5)
    if parts is not None:
        m, l, o = ORC.attention_partials(q_rot, Kg, Vg, nq, nkv, d, pos + 1,
                                         (pos + n_chunks) // n_chunks, n_chunks)
        gm = parts[0].cpu().numpy().reshape(nq, n_chunks)
        gl = parts[1].cpu().numpy().reshape(nq, n_chunks)
        go = parts[2].cpu().numpy().reshape(nq, n_chunks, d)
        empty = np.isneginf(m)
        assert np.array_equal(np.isneginf(gm), empty)
        np.testing.assert_allclose(gm[~empty], m[~empty], rtol=1e-5, atol=1e-5)
        np.testing.assert_allclose(gl, l, rtol=1e-4, atol=1e-5)
        np.testing.assert_allclose(go, o, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("nq,nkv,d,pos", [
    (4, 2, 64, 0), (4, 2, 64, 31), (32, 8, 64, 1100), (12, 2, 128, 300), (12, 2, 128, 4100),
    (40, 8, 64, 700), (6, 6, 64, 77), (24, 8, 64, 513), (32, 4, 64, 2100), (16, 2, 64, 255)])
def test_attention_engine_chunking_matches_oracle(nq, nkv, d, pos):
    attention_case(nq, nkv, d, pos, n_chunks=0)


@pytest.mark.parametrize("nq,nkv,d,pos,n_chunks", [
    (8, 2, 64, 57, 8), (12, 4, 64, 129, 2), (4, 2, 64, 9, 8), (8, 2, 64, 0, 3), (10, 2, 128, 300, 3),
    (8, 1, 64, 255, 1)])
def test_attention_explicit_chunks_and_partials(nq, nkv, d, pos, n_chunks):
    attention_case(nq, nkv, d, pos, n_chunks)

"""The GEMV over a batch of m activation vectors (tinfer_op_gemv_batch), the verify shape of
speculative decoding: every output against the oracle's GEMV of each vector on its own."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402

pytestmark = pytest.mark.gpu
ORC = Oracle("f64")


def packed_matrix(fmt, rows, cols, group, sdt, seed):
    key = f"gemvm.{rows}.{cols}.{seed}"
    if fmt == "int4":
        W = synth.nibbles(key, (rows, cols // 2), seed)
        S = synth.abs_normal_16(key + ".s", (rows, cols // group), 0.005, sdt, seed)
        f = T.TINFER_INT4
    else:
        W = synth.normal_bf16(key, (rows, cols), 0.0, 0.02, seed)
        S = None
        f = T.TINFER_BF16
    sd = T.TINFER_SCALE_BF16 if sdt == "bf16" else T.TINFER_SCALE_FP16
    rb = T.tinfer_packed_row_bytes(f, cols, group)
    packed = torch.empty(rows * rb, dtype=torch.uint8, device="cuda")
    w_d = torch.from_numpy(W.view(np.int16) if W.dtype == np.uint16 else W).cuda()
    s_d = torch.from_numpy(S.view(np.int16)).cuda() if S is not None else None
    assert T.tinfer_pack_matrix(f, group, sd, rows, cols, w_d, s_d, packed) == 0

    def ref(x):
        x = np.asarray(x, np.float64)
        if fmt == "int4":
            return ORC.gemv_int4(W, S, sdt == "bf16", group, x)
        return ORC.gemv_bf16(W, x)
    return f, sd, packed, ref


@pytest.mark.parametrize("fmt,group,sdt", [("bf16", 64, "fp16"), ("int4", 64, "fp16"), ("int4", 128, "bf16")])
@pytest.mark.parametrize("m", [1, 2, 4, 8])
@pytest.mark.parametrize("rows,cols", [(3072, 2048), (1000, 1536), (333, 1024)])
def test_gemv_batch_matches_oracle(fmt, group, sdt, m, rows, cols):
    if cols % group:
        pytest.skip("group does not divide the row")
    f, sd, packed, ref = packed_matrix(fmt, rows, cols, group, sdt, seed=m)
    x = synth.normals(f"gemvm.x.{m}.{cols}", m * cols, seed=m).astype(np.float32).reshape(m, cols)
    bias = (synth.normals("gemvm.b", rows, seed=m) * 0.1).astype(np.float32)
    y = torch.empty(m * rows, dtype=torch.float32, device="cuda")
    rc = T.tinfer_op_gemv_batch(f, group, sd, rows, cols, m, packed, torch.from_numpy(x).cuda(),
                                torch.from_numpy(bias).cuda(), T.TINFER_EPI_STORE, y)
    if rc == T.TINFER_ERR_UNSUPPORTED:
        assert fmt == "int4" and (cols // max(1, 2 ** int(np.ceil(np.log2(max(1, cols * m / 2048)))))) % (64 // m)
        pytest.skip("segment does not hold whole runs of words")
    assert rc == 0
    got = y.cpu().numpy().reshape(m, rows).astype(np.float64)
    for j in range(m):
        np.testing.assert_allclose(got[j], ref(x[j]) + bias, rtol=1e-4, atol=3e-5 * np.sqrt(cols / 256))
    # the residual epilogue adds to y
    y0 = got.astype(np.float32).ravel()
    y = torch.from_numpy(y0.copy()).cuda()
    assert T.tinfer_op_gemv_batch(f, group, sd, rows, cols, m, packed, torch.from_numpy(x).cuda(), None,
                                  T.TINFER_EPI_RESIDUAL, y) == 0
    got2 = y.cpu().numpy().reshape(m, rows).astype(np.float64)
    for j in range(m):
        np.testing.assert_allclose(got2[j] - got[j], ref(x[j]), rtol=1e-4, atol=6e-5 * np.sqrt(cols / 256))


@pytest.mark.parametrize("fmt,rows,cols,m", [("bf16", 3072, 2048, 8), ("int4", 11264, 2048, 4),
                                             ("bf16", 2048, 8192, 2)])
def test_gemv_batch_verify_shapes(fmt, rows, cols, m):
    # Llama-shaped QKV at m = 8, TinyLlama-shaped int4 gate/up at m = 4, Llama-shaped down at m = 2
    f, sd, packed, ref = packed_matrix(fmt, rows, cols, 64, "fp16", seed=11)
    x = synth.normals("gemvm.vx", m * cols, seed=11).astype(np.float32).reshape(m, cols)
    y = torch.empty(m * rows, dtype=torch.float32, device="cuda")
    assert T.tinfer_op_gemv_batch(f, 64, sd, rows, cols, m, packed, torch.from_numpy(x).cuda(), None,
                                  T.TINFER_EPI_STORE, y) == 0
    got = y.cpu().numpy().reshape(m, rows).astype(np.float64)
    for j in range(m):
        np.testing.assert_allclose(got[j], ref(x[j]), rtol=1e-4, atol=3e-5 * np.sqrt(cols / 256))


def test_gemv_batch_rejects_unsupported_shapes():
    f, sd, packed, _ = packed_matrix("bf16", 64, 4096, 64, "fp16", seed=3)
    x = torch.zeros(8 * 4096, device="cuda")
    y = torch.empty(8 * 64, device="cuda")
    assert T.tinfer_op_gemv_batch(f, 64, sd, 64, 4096, 8, packed, x, None, 0, y) == T.TINFER_ERR_UNSUPPORTED  # m * cols
    assert T.tinfer_op_gemv_batch(f, 64, sd, 64, 4096, 3, packed, x, None, 0, y) == T.TINFER_ERR_UNSUPPORTED  # m
    assert T.tinfer_op_gemv_batch(f, 64, sd, 64, 4096, 2, packed, x, None, 2, y) == T.TINFER_ERR_INVALID_ARG  # epilogue

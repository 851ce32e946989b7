"""The batched-prefill matrix product on the tensor cores (tinfer_op_gemm_bf16): every output row
against the oracle's pinned bf16 GEMV of that row, single tiles, several tiles, ragged edges in M, N
and K, a prefill-shaped QKV product, several tiles per persistent CTA (both tensor-memory
accumulators reused), and rejected arguments."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402
from util import bf16_to_f64  # noqa: E402

pytestmark = pytest.mark.gpu
ORC = Oracle("f64")


def run_gemm(m, n, k, seed):
    X = synth.normal_bf16(f"gemm.x.{m}.{k}.{seed}", (m, k), 0.0, 1.0, seed)
    W = synth.normal_bf16(f"gemm.w.{n}.{k}.{seed}", (n, k), 0.0, 0.02, seed)
    x_d = torch.from_numpy(X.view(np.int16)).cuda()
    w_d = torch.from_numpy(W.view(np.int16)).cuda()
    y_d = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    assert T.tinfer_op_gemm_bf16(m, n, k, x_d, w_d, y_d) == T.TINFER_OK
    return X, W, y_d.cpu().numpy()


def check_rows(X, W, Y, rows):
    """Each output within the rounding bound of an fp32 sum of its k exact bf16 products: the
    products are exact in fp32 (8-bit significands), and k additions round by at most 2^-23
    relative each (allowing truncation as well as rounding to nearest), so
    |y - y_exact| <= k 2^-23 sum_c |w_rc x_ic|."""
    k = X.shape[1]
    Wf = bf16_to_f64(W)
    worst = 0.0
    for i in rows:
        x = bf16_to_f64(X[i])
        ref = ORC.gemv_bf16(W, x)
        bound = k * 2.0 ** -23 * (np.abs(Wf) @ np.abs(x)) + 1e-30
        err = np.abs(Y[i].astype(np.float64) - ref)
        assert np.all(np.isfinite(Y[i])), i
        assert np.all(err <= bound), (i, float((err / bound).max()))
        worst = max(worst, float((err / bound).max()))
    return worst


@pytest.mark.parametrize("m,n,k", [(128, 128, 64), (128, 256, 2048), (200, 300, 2048), (7, 64, 8),
                                   (1, 1, 64), (300, 1000, 200), (129, 129, 1000)])
def test_gemm_matches_oracle_rows(m, n, k):
    X, W, Y = run_gemm(m, n, k, seed=1)
    check_rows(X, W, Y, range(m))


def test_gemm_prefill_qkv_shape_sampled_rows():
    # a 512-token prompt through the Llama-shaped fused QKV projection (3072 x 2048): 12 x 4 tiles of
    # 32 K blocks each; rows sampled from every tile row, all columns checked
    m, n, k = 512, 3072, 2048
    X, W, Y = run_gemm(m, n, k, seed=2)
    rows = sorted(set(list(range(0, m, 37)) + [127, 128, 255, 256, 383, 384, 511]))
    check_rows(X, W, Y, rows)


def test_gemm_several_tiles_per_cta_sampled_rows():
    # 16 x 32 tiles of 128 x 256 on at most one CTA per SM: every CTA computes three or four tiles,
    # alternating its two tensor-memory accumulators; rows sampled from every tile row
    m, n, k = 2048, 8192, 256
    X, W, Y = run_gemm(m, n, k, seed=3)
    rows = sorted(set(list(range(0, m, 61)) + [127, 128, 1023, 1024, 2047]))
    check_rows(X, W, Y, rows)


def test_gemm_rejects_bad_arguments():
    x = torch.zeros((4, 64), dtype=torch.int16, device="cuda")
    w = torch.zeros((4, 64), dtype=torch.int16, device="cuda")
    y = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    assert T.tinfer_op_gemm_bf16(4, 4, 12, x, w, y) == T.TINFER_ERR_INVALID_ARG      # k not a multiple of 8
    assert T.tinfer_op_gemm_bf16(0, 4, 64, x, w, y) == T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_op_gemm_bf16(4, 4, 64, x.data_ptr() + 2, w, y) == T.TINFER_ERR_INVALID_ARG  # misaligned x
    assert T.tinfer_op_gemm_bf16(4, 4, 64, None, w, y) == T.TINFER_ERR_INVALID_ARG

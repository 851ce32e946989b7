"""The attention entry point that allocates nothing (its scratch is a fixed array inside the
library), through the C ABI: on the same inputs it must give what tinfer_op_attention gives, on two
calls in a row, and it must refuse problems larger than its scratch. The file name sorts last so
that the suite runs it after everything else; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import decode_persistent_megakernel_gb300 as T
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    T.build()


def _case(nq, nkv, d, pos, max_ctx, seed):
    K = synth.normal_bf16(f"naK{nq}{nkv}{d}{pos}", (nkv, max_ctx, d), 0.0, 1.0)
    V = synth.normal_bf16(f"naV{nq}{nkv}{d}{pos}", (nkv, max_ctx, d), 0.0, 1.0)
    qkv = np.random.default_rng(seed).standard_normal((nq + 2 * nkv) * d).astype(np.float32)
    return K, V, qkv


def _u16_dev(a):
    return torch.from_numpy(a.view(np.int16).copy()).cuda()


@pytest.mark.parametrize("nq,nkv,d,pos,n_chunks", [
    (32, 8, 64, 1030, 0),     # Llama-3.2-1B-shaped heads, the engine's own chunking
    (12, 2, 128, 700, 0),     # head_dim 128, 6 query heads per KV head
    (8, 2, 64, 57, 5),        # explicit chunks with a ragged last chunk
])
def test_noalloc_attention_matches_allocating_entry(nq, nkv, d, pos, n_chunks):
    max_ctx = pos + 9
    theta = 500000.0
    K, V, qkv = _case(nq, nkv, d, pos, max_ctx, seed=pos)
    q_dev = torch.from_numpy(qkv).cuda()

    Kr, Vr = _u16_dev(K), _u16_dev(V)
    ref = torch.full((nq * d,), float("nan"), device="cuda")
    assert T.tinfer_op_attention(nq, nkv, d, max_ctx, theta, pos, n_chunks, q_dev, Kr, Vr, ref) == 0

    for call in range(2):  # two calls in a row reuse the same scratch
        Kn, Vn = _u16_dev(K), _u16_dev(V)
        out = torch.full((nq * d,), float("nan"), device="cuda")
        rc = T.tinfer_op_attention_noalloc(nq, nkv, d, max_ctx, theta, pos, n_chunks, q_dev, Kn, Vn, out)
        torch.cuda.synchronize()
        assert rc == 0, (call, T.status_string(rc))
        torch.testing.assert_close(out, ref, rtol=1e-5, atol=1e-6)
        # the cache slot at pos is written the same way; the rest of the cache is untouched
        assert torch.equal(Kn, Kr) and torch.equal(Vn, Vr)


def test_noalloc_attention_rejects_problems_beyond_its_scratch():
    nq, nkv, d = 64, 8, 128
    cap = T.TINFER_NOALLOC_SCRATCH_BYTES - 2048
    n_chunks = 64
    assert nq * n_chunks * (d + 2) * 4 > cap
    K, V, qkv = _case(nq, nkv, d, 100, 128, seed=1)
    out = torch.zeros(nq * d, device="cuda")
    rc = T.tinfer_op_attention_noalloc(nq, nkv, d, 128, 10000.0, 100, n_chunks,
                                       torch.from_numpy(qkv).cuda(), _u16_dev(K), _u16_dev(V), out)
    assert rc == T.TINFER_ERR_UNSUPPORTED
    assert torch.count_nonzero(out) == 0

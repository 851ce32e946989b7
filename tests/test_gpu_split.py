"""The column-split down projection ("Decoding in tiles", section 4: FFN tasks multiply their
SwiGLU rows by the matching columns of the down projection, and an FFN-reduce sums the per-task
partials in a fixed order): the same step against the oracle, its packed layer round trip, and its
reproducibility (the fixed-order reduce gives the same bits on every run)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402
from util import ARGMAX_MARGIN, LOGIT_MAX_ABS, LOGIT_REL_L2, compare_logits, kv_close  # noqa: E402

pytestmark = pytest.mark.gpu
ORC = Oracle("f64")


def run_split(c, w, n_prompt, n_steps, prefill=0, seed=0):
    K, V = synth.make_kv(c, prefill, seed)
    eng = T.Engine(c, w, T.TINFER_MEGAKERNEL, kv=(K, V))
    om = ORC.model(c, w)
    prompt = synth.make_tokens(c, max(n_prompt, 1), seed)
    tok = int(prompt[0])
    out = []
    for k in range(n_prompt + n_steps):
        pos = prefill + k
        if k < n_prompt:
            tok = int(prompt[k])
        eng.step(tok, pos)
        torch.cuda.synchronize()
        ref, am_ref, rc = ORC.decode_step(om, tok, pos, K, V)
        assert rc == 0
        got = eng.logits.cpu().numpy()
        out.append(got.copy())
        err, rel, margin = compare_logits(got, ref)
        assert err <= LOGIT_MAX_ABS and rel <= LOGIT_REL_L2, (k, err, rel)
        if margin > ARGMAX_MARGIN:
            assert int(eng.argmax.item()) == am_ref
        Kg = eng.k[:, :, pos].cpu().numpy().view(np.uint16)
        assert kv_close(Kg, K[:, :, pos]) <= 0
        tok = am_ref
    assert eng.error() == T.TINFER_OK
    eng.close()
    return np.stack(out)


@pytest.mark.parametrize("over", [dict(), dict(qkv_bias=True, tied=True),
                                  dict(n_heads=6, n_kv_heads=2, head_dim=128, hidden=384, ffn=1024)])
def test_split_tiny_variants_match_oracle(over):
    c = synth.config("tiny", ffn_split=True, max_ctx=300, **over)
    w = synth.make_model(c, seed=1)
    a = run_split(c, w, 2, 4, prefill=280, seed=1)
    b = run_split(c, w, 2, 4, prefill=280, seed=1)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))  # the fixed-order reduce


@pytest.mark.parametrize("name,steps", [("llama1b", 2), ("qwen1.5b", 2)])
def test_split_full_size_matches_oracle(name, steps):
    c = synth.config(name, ffn_split=True)
    w = synth.make_model(c, seed=0)
    P = c["prefill"]
    K, V = synth.make_kv(c, P, seed=0)
    eng = T.Engine(c, w, T.TINFER_MEGAKERNEL, kv=(K, V))
    om = ORC.model(c, w)
    tok = int(synth.make_tokens(c, 1, seed=0)[0])
    for k in range(steps):
        eng.step(tok, P + k)
        torch.cuda.synchronize()
        ref, am_ref, rc = ORC.decode_step(om, tok, P + k, K, V)
        err, rel, margin = compare_logits(eng.logits.cpu().numpy(), ref)
        assert err <= LOGIT_MAX_ABS and rel <= LOGIT_REL_L2, (name, k, err, rel)
        if margin > ARGMAX_MARGIN:
            assert int(eng.argmax.item()) == am_ref
        tok = am_ref
    assert eng.error() == T.TINFER_OK
    eng.close()


def test_split_pack_round_trip_and_unsupported_forms():
    c = synth.config("tiny", ffn_split=True)
    w = synth.make_model(c, seed=2)
    eng = T.Engine(c, w)
    L = w["layers"][1]
    dst = T.tinfer_layer_src()
    keep = {}
    for name, arr in L.items():
        t = torch.empty(arr.size, dtype=torch.uint8 if arr.dtype == np.uint8 else torch.int16, device="cuda")
        keep[name] = t
        setattr(dst, name, t.data_ptr())
    assert T.tinfer_unpack_layer(eng.cfg, eng.blobs[1], dst) == 0
    torch.cuda.synchronize()
    for name, arr in L.items():
        got = keep[name].cpu().numpy().view(arr.dtype).reshape(arr.shape)
        assert np.array_equal(got, arr), name
    eng.close()
    for bad in (dict(weight_format="int4", group_size=64, scale_dtype="fp16", ffn=704),):
        cb = synth.config("tiny", ffn_split=True, **bad)
        assert T.tinfer_check_config(T.make_config(cb)) == T.TINFER_ERR_UNSUPPORTED
    assert T.tinfer_check_config(T.make_config(c, T.TINFER_GRAPH)) == T.TINFER_ERR_UNSUPPORTED

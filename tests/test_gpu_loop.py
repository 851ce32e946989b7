"""The in-kernel token loop (tinfer_generate_dev): one cooperative launch decodes several tokens,
each step's greedy choice combined on the device and fed to the next step ("Decoding in tiles",
section 5, Figure 10). Checked against the oracle's greedy run, against per-step launches of the
same kernel (bitwise, on the KV cache), and on its stop conditions."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402
from util import ARGMAX_MARGIN  # noqa: E402

pytestmark = pytest.mark.gpu
ORC = Oracle("f64")


def oracle_greedy(c, w, K, V, first, pos0, n):
    om = ORC.model(c, w)
    K, V = K.copy(), V.copy()
    out, tok = [], first
    for k in range(n):
        _, tok, rc = ORC.decode_step(om, tok, pos0 + k, K, V)
        assert rc == 0
        out.append(tok)
    return out


@pytest.mark.parametrize("mode", [T.TINFER_MEGAKERNEL, T.TINFER_GRAPH])
def test_tiny_model_loop_equals_oracle_greedy(mode):
    c = synth.config("tiny", max_ctx=40)
    w = synth.make_model(c, seed=3)
    K, V = synth.make_kv(c, 0)
    first = int(synth.make_tokens(c, 1, seed=3)[0])
    n = 24
    ref = oracle_greedy(c, w, K, V, first, 0, n)
    eng = T.Engine(c, w, mode)
    toks = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda") if mode == T.TINFER_MEGAKERNEL else None
    assert T.tinfer_generate_dev(eng.ctx, first, 0, n, -1, None, toks, count) == 0
    assert eng.error() == T.TINFER_OK
    assert toks.cpu().tolist() == ref
    if count is not None:
        assert int(count.item()) == n
    eng.close()


def test_loop_writes_the_same_cache_as_per_step_launches():
    # a prefilled context so that the attention runs several chunks; the loop's steps and single
    # launches run the same arithmetic, so the cache agrees bit for bit
    c = synth.config("tiny", max_ctx=320)
    w = synth.make_model(c, seed=4)
    K, V = synth.make_kv(c, 290, seed=4)
    first = int(synth.make_tokens(c, 1, seed=4)[0])
    n = 20
    eng = T.Engine(c, w, kv=(K, V))
    toks = torch.zeros(n, dtype=torch.int32, device="cuda")
    assert T.tinfer_generate_dev(eng.ctx, first, 290, n, -1, None, toks, None) == 0
    assert eng.error() == T.TINFER_OK
    k_loop, v_loop, t_loop = eng.k.cpu().numpy(), eng.v.cpu().numpy(), toks.cpu().tolist()
    eng.close()
    eng = T.Engine(c, w, kv=(K, V))
    chain = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    chain[0] = first
    for k in range(n):
        eng.step_dev(chain[k:k + 1], 290 + k, logits=False, argmax=chain[k + 1:k + 2])
    assert eng.error() == T.TINFER_OK
    assert chain[1:].cpu().tolist() == t_loop
    assert np.array_equal(eng.k.cpu().numpy(), k_loop) and np.array_equal(eng.v.cpu().numpy(), v_loop)
    eng.close()


def test_loop_stops_after_the_end_token():
    c = synth.config("tiny", max_ctx=40)
    w = synth.make_model(c, seed=3)
    K, V = synth.make_kv(c, 0)
    first = int(synth.make_tokens(c, 1, seed=3)[0])
    ref = oracle_greedy(c, w, K, V, first, 0, 16)
    # the end token: one chosen for the first time at step `stop` (as late as possible up to 8)
    firsts = [s for s in range(16) if ref[s] not in ref[:s]]
    stop = max(s for s in firsts if s <= 8)
    eos = ref[stop]
    eng = T.Engine(c, w)
    toks = torch.full((16,), -7, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert T.tinfer_generate_dev(eng.ctx, first, 0, 16, eos, None, toks, count) == 0
    assert eng.error() == T.TINFER_OK
    got = toks.cpu().tolist()
    assert int(count.item()) == stop + 1
    assert got[:stop + 1] == ref[:stop + 1] and got[stop + 1:] == [-7] * (16 - stop - 1)
    eng.close()


def test_loop_stops_on_a_nonfinite_logit():
    c = synth.config("tiny", max_ctx=16)
    w = synth.make_model(c)
    w["lm_head"] = w["lm_head"].copy()
    w["lm_head"][1234, 7] = 0x7F80  # +inf weight -> an infinite or NaN logit on the first step
    eng = T.Engine(c, w)
    toks = torch.full((8,), -7, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert T.tinfer_generate_dev(eng.ctx, 5, 0, 8, -1, None, toks, count) == 0
    assert eng.error() == T.TINFER_ERR_NONFINITE
    assert toks.cpu().tolist() == [-1] + [-7] * 7 and int(count.item()) == 1
    eng.close()


def test_loop_host_validation():
    c = synth.config("tiny", max_ctx=16)
    eng = T.Engine(c, synth.make_model(c))
    toks = torch.zeros(16, dtype=torch.int32, device="cuda")
    E = T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_generate_dev(eng.ctx, 1, 0, 0, -1, None, toks, None) == E       # no steps
    assert T.tinfer_generate_dev(eng.ctx, 1, 10, 7, -1, None, toks, None) == E      # past max_ctx
    assert T.tinfer_generate_dev(eng.ctx, c["vocab"], 0, 4, -1, None, toks, None) == E
    assert T.tinfer_generate_dev(eng.ctx, 1, 0, 4, c["vocab"], None, toks, None) == E
    assert T.tinfer_generate_dev(eng.ctx, 1, 0, 4, -1, None, None, None) == E
    eng.close()


def test_llama1b_loop_choices_match_the_oracle():
    """Full size: 16 tokens in one launch from the prefilled context. The oracle is fed the GPU's
    own choices (teacher forcing on the GPU's trajectory) and must agree with each of them wherever
    its top-1 / top-2 margin exceeds the tolerance."""
    c = synth.config("llama1b")
    w = synth.make_model(c, seed=0)
    P = c["prefill"]
    K, V = synth.make_kv(c, P, seed=0)
    first = int(synth.make_tokens(c, 1, seed=0)[0])
    n = 16
    eng = T.Engine(c, w, kv=(K, V))
    toks = torch.zeros(n, dtype=torch.int32, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert T.tinfer_generate_dev(eng.ctx, first, P, n, -1, None, toks, count) == 0
    assert eng.error() == T.TINFER_OK and int(count.item()) == n
    got = toks.cpu().tolist()
    eng.close()
    om = ORC.model(c, w)
    tok = first
    for k in range(n):
        ref, am, rc = ORC.decode_step(om, tok, P + k, K, V)
        assert rc == 0
        srt = np.sort(ref)
        if srt[-1] - srt[-2] > ARGMAX_MARGIN:
            assert got[k] == am, (k, got[k], am)
        tok = got[k]

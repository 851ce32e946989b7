"""Whole-step parity on the GPU through the C ABI: teacher-forced decode of small models against the
fp64 oracle, in both execution modes (persistent megakernel, CUDA graph of per-phase kernels), plus
determinism, the KV-cache write contract, the host-loop generate call and the error paths."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402
from util import ARGMAX_MARGIN, LOGIT_MAX_ABS, LOGIT_REL_L2, compare_logits, kv_close  # noqa: E402

pytestmark = pytest.mark.gpu
ORC = Oracle("f64")
MODES = [T.TINFER_MEGAKERNEL, T.TINFER_GRAPH]


def run_teacher_forced(c, w, mode, n_prompt, n_steps, prefill=0, seed=0, check_kv=True):
    """Feeds both sides the same tokens: the prompt, then the oracle's greedy choices."""
    K, V = synth.make_kv(c, prefill, seed)
    eng = T.Engine(c, w, mode, kv=(K, V))
    om = ORC.model(c, w)
    prompt = synth.make_tokens(c, max(n_prompt, 1), seed)
    tok = int(prompt[0])
    worst = (0.0, 0.0)
    logits_all = []
    for k in range(n_prompt + n_steps):
        pos = prefill + k
        if k < n_prompt:
            tok = int(prompt[k])
        eng.step(tok, pos)
        torch.cuda.synchronize()
        ref, am_ref, rc = ORC.decode_step(om, tok, pos, K, V)
        assert rc == 0
        got = eng.logits.cpu().numpy()
        logits_all.append(got.copy())
        err, rel, margin = compare_logits(got, ref)
        assert err <= LOGIT_MAX_ABS and rel <= LOGIT_REL_L2, (k, err, rel)
        worst = (max(worst[0], err), max(worst[1], rel))
        if margin > ARGMAX_MARGIN:
            assert int(eng.argmax.item()) == am_ref, (k, int(eng.argmax.item()), am_ref, margin)
        if check_kv:
            # slots [0, pos]: close to the oracle's own rounding (kv_close); later slots untouched
            Kg = eng.k.cpu().numpy().view(np.uint16)
            Vg = eng.v.cpu().numpy().view(np.uint16)
            assert kv_close(Kg[:, :, :pos + 1], K[:, :, :pos + 1]) <= 0
            assert kv_close(Vg[:, :, :pos + 1], V[:, :, :pos + 1]) <= 0
            assert np.array_equal(Kg[:, :, pos + 1:], K[:, :, pos + 1:])
            assert np.array_equal(Vg[:, :, pos + 1:], V[:, :, pos + 1:])
        tok = am_ref
    assert eng.error() == T.TINFER_OK
    eng.close()
    return worst, np.stack(logits_all)


@pytest.mark.parametrize("mode", MODES)
def test_tiny_model_teacher_forced(mode):
    c = synth.config("tiny")
    w = synth.make_model(c, seed=0)
    run_teacher_forced(c, w, mode, c["prompt"], c["steps"])


@pytest.mark.parametrize("over", [
    dict(qkv_bias=True, tied=True),
    dict(n_heads=8, n_kv_heads=1, head_dim=32 * 2),        # group 8
    dict(n_heads=6, n_kv_heads=2, head_dim=128, hidden=384, ffn=1024),  # group 3, d 128
    dict(weight_format="int4", group_size=64, scale_dtype="fp16", ffn=704),
    dict(weight_format="int4", group_size=128, scale_dtype="bf16", ffn=768, tied=True),
])
@pytest.mark.parametrize("mode", MODES)
def test_variants_teacher_forced(over, mode):
    c = synth.config("tiny", n_layers=2, max_ctx=300, **over)
    w = synth.make_model(c, seed=1)
    # a prefilled cache so that attention spans several chunks
    run_teacher_forced(c, w, mode, 1, 3, prefill=280, seed=1)


def test_megakernel_and_graph_are_bitwise_equal_and_deterministic():
    c = synth.config("tiny", max_ctx=40)
    w = synth.make_model(c, seed=2)
    outs = []
    for mode in (T.TINFER_MEGAKERNEL, T.TINFER_MEGAKERNEL, T.TINFER_GRAPH):
        K, V = synth.make_kv(c, 20, seed=2)
        eng = T.Engine(c, w, mode, kv=(K, V))
        toks = synth.make_tokens(c, 8, seed=2)
        seq = []
        for k, t in enumerate(toks.tolist()):
            eng.step(t, 20 + k)
            seq.append(eng.logits.cpu().numpy().copy())
        outs.append((np.stack(seq), eng.k.cpu().numpy().copy()))
        eng.close()
    for o in outs[1:]:
        assert np.array_equal(o[0].view(np.uint32), outs[0][0].view(np.uint32))
        assert np.array_equal(o[1], outs[0][1])


def test_device_token_chaining_and_generate_match_oracle_greedy():
    c = synth.config("tiny", max_ctx=24)
    w = synth.make_model(c, seed=3)
    K, V = synth.make_kv(c, 0)
    om = ORC.model(c, w)
    first = int(synth.make_tokens(c, 1, seed=3)[0])
    greedy, tok = [], first
    for pos in range(12):
        _, tok, rc = ORC.decode_step(om, tok, pos, K, V)
        greedy.append(tok)
    for mode in MODES:
        eng = T.Engine(c, w, mode)
        out = (ctypes.c_int32 * 12)()
        assert T.tinfer_generate(eng.ctx, first, 0, 12, None, out) == 0
        assert list(out) == greedy
        eng.close()
        # device-side chaining: the argmax buffer of one step is the token input of the next
        eng = T.Engine(c, w, mode)
        toks = torch.zeros(13, dtype=torch.int32, device="cuda")
        toks[0] = first
        for pos in range(12):
            eng.step_dev(toks[pos:pos + 1], pos, argmax=toks[pos + 1:pos + 2], logits=False)
        assert toks[1:].cpu().tolist() == greedy
        eng.close()


def test_host_validation_errors():
    c = synth.config("tiny", max_ctx=8)
    w = synth.make_model(c)
    eng = T.Engine(c, w)
    assert T.tinfer_decode_step(eng.ctx, c["vocab"], 0, None, None, eng.argmax) == T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_decode_step(eng.ctx, 0, 8, None, None, eng.argmax) == T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_decode_step(eng.ctx, -1, 0, None, None, eng.argmax) == T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_decode_step_dev(eng.ctx, None, 0, None, None, eng.argmax) == T.TINFER_ERR_INVALID_ARG
    bad = T.make_config(c)
    bad.n_kv_heads = 3
    assert T.tinfer_check_config(bad) == T.TINFER_ERR_INVALID_ARG
    rc, ctx = T.tinfer_create(eng.cfg, T.tinfer_weights(), eng.k, eng.v)
    assert rc == T.TINFER_ERR_INVALID_ARG
    eng.close()


@pytest.mark.parametrize("mode", MODES)
def test_bad_device_token_is_reported_and_cleared(mode):
    c = synth.config("tiny", max_ctx=8)
    eng = T.Engine(c, synth.make_model(c), mode)
    tok = torch.tensor([c["vocab"] + 5], dtype=torch.int32, device="cuda")
    eng.step_dev(tok, 0)
    assert eng.error() == T.TINFER_ERR_INVALID_ARG
    eng.step(3, 0)
    assert eng.error() == T.TINFER_OK
    eng.close()


@pytest.mark.parametrize("mode", MODES)
def test_nonfinite_logit_sets_error_word_then_recovers(mode):
    c = synth.config("tiny", max_ctx=8)
    w = synth.make_model(c)
    w["lm_head"] = w["lm_head"].copy()
    w["lm_head"][1234, 7] = 0x7F80  # +inf weight -> an infinite or NaN logit
    eng = T.Engine(c, w, mode)
    eng.step(5, 0)
    torch.cuda.synchronize()
    assert int(eng.argmax.item()) == -1
    # the next step is refused with the recorded error, without launching
    assert T.tinfer_decode_step(eng.ctx, 5, 1, None, None, eng.argmax) == T.TINFER_ERR_NONFINITE
    assert eng.error() == T.TINFER_ERR_NONFINITE
    assert eng.error() == T.TINFER_OK
    eng.close()


def test_barrier_timeout_is_reported_and_the_context_recovers():
    # a fault made on the host side of the contract: one CTA withholds its results of one phase, the
    # bounded waits of the CTAs that need them run out, the step ends with TINFER_ERR_TIMEOUT and the
    # GPU stays usable
    c = synth.config("tiny", max_ctx=8)
    w = synth.make_model(c)
    eng = T.Engine(c, w)
    assert T.tinfer_set_timeout_ns(eng.ctx, 20_000_000) == 0
    assert T.tinfer_debug_withhold_results(eng.ctx, 3, 2) == 0
    eng.step(5, 0)
    assert eng.error() == T.TINFER_ERR_TIMEOUT
    # the same step again, now without the fault, matches a fresh engine
    eng.step(5, 0)
    torch.cuda.synchronize()
    got = eng.logits.cpu().numpy().copy()
    assert eng.error() == T.TINFER_OK
    eng.close()
    ref = T.Engine(c, w)
    ref.step(5, 0)
    assert np.array_equal(ref.logits.cpu().numpy(), got)
    ref.close()


def test_create_destroy_cycles():
    c = synth.config("tiny", max_ctx=8)
    w = synth.make_model(c)
    for mode in MODES * 3:
        eng = T.Engine(c, w, mode)
        eng.step(1, 0)
        assert eng.error() == T.TINFER_OK
        eng.close()


def test_grid_barrier_schedule_matches_oracle_and_stamped_schedule():
    """The grid-barrier schedule (TINFER_SYNC_GRID_BARRIER) computes the same step as the stamped
    hand-off: teacher-forced against the oracle, and bitwise equal to the default schedule."""
    c = synth.config("tiny", max_ctx=300)
    w = synth.make_model(c, seed=6)
    outs = []
    for sync in (T.TINFER_SYNC_GRID_BARRIER, T.TINFER_SYNC_STAMPS):
        K, V = synth.make_kv(c, 270, seed=6)
        eng = T.Engine(c, w, kv=(K, V))
        assert T.tinfer_set_schedule(eng.ctx, T.TINFER_S_SYNC, sync) == 0
        assert T.tinfer_get_schedule(eng.ctx, T.TINFER_S_SYNC) == sync
        om = ORC.model(c, w)
        toks = synth.make_tokens(c, 6, seed=6)
        seq = []
        for k, t in enumerate(toks.tolist()):
            eng.step(t, 270 + k)
            torch.cuda.synchronize()
            got = eng.logits.cpu().numpy().copy()
            ref, _, rc = ORC.decode_step(om, t, 270 + k, K, V)
            err, rel, _ = compare_logits(got, ref)
            assert err <= LOGIT_MAX_ABS and rel <= LOGIT_REL_L2, (sync, k, err, rel)
            seq.append(got)
        assert eng.error() == T.TINFER_OK
        outs.append(np.stack(seq))
        eng.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_grid_barrier_schedule_reports_a_withheld_result():
    c = synth.config("tiny", max_ctx=8)
    w = synth.make_model(c)
    eng = T.Engine(c, w)
    assert T.tinfer_set_schedule(eng.ctx, T.TINFER_S_SYNC, T.TINFER_SYNC_GRID_BARRIER) == 0
    assert T.tinfer_set_timeout_ns(eng.ctx, 20_000_000) == 0
    assert T.tinfer_debug_withhold_results(eng.ctx, 3, 2) == 0
    eng.step(5, 0)
    assert eng.error() == T.TINFER_ERR_TIMEOUT
    eng.step(5, 0)  # the context recovers, counter included
    assert eng.error() == T.TINFER_OK
    eng.close()
    eng = T.Engine(c, w, T.TINFER_GRAPH)
    assert T.tinfer_set_schedule(eng.ctx, T.TINFER_S_SYNC, T.TINFER_SYNC_GRID_BARRIER) == T.TINFER_ERR_UNSUPPORTED
    eng.close()


@pytest.mark.parametrize("mode", MODES)
def test_fixed_attention_chunk_counts_match_oracle(mode):
    """TINFER_S_ATTN_CHUNKS: a fixed number of split-K chunks per KV head (empty chunks at short
    contexts included) gives the oracle's step; values that would overflow a ring slot at max_ctx or
    the partial buffers are rejected on the host."""
    c = synth.config("tiny", max_ctx=300)
    w = synth.make_model(c, seed=7)
    K, V = synth.make_kv(c, 270, seed=7)
    eng = T.Engine(c, w, mode, kv=(K, V))
    auto = T.tinfer_get_schedule(eng.ctx, T.TINFER_S_ATTN_CHUNKS)
    assert auto == 0
    assert T.tinfer_set_schedule(eng.ctx, T.TINFER_S_ATTN_CHUNKS, 1) == T.TINFER_ERR_INVALID_ARG
    assert T.tinfer_set_schedule(eng.ctx, T.TINFER_S_ATTN_CHUNKS, 100000) == T.TINFER_ERR_INVALID_ARG
    om = ORC.model(c, w)
    toks = synth.make_tokens(c, 6, seed=7)
    for k, (n, t) in enumerate(zip([2, 5, 33, 2, 76, 0], toks.tolist())):
        assert T.tinfer_set_schedule(eng.ctx, T.TINFER_S_ATTN_CHUNKS, n) == 0
        assert T.tinfer_get_schedule(eng.ctx, T.TINFER_S_ATTN_CHUNKS) == n
        eng.step(t, 270 + k)
        torch.cuda.synchronize()
        ref, am, rc = ORC.decode_step(om, t, 270 + k, K, V)
        err, rel, margin = compare_logits(eng.logits.cpu().numpy(), ref)
        assert err <= LOGIT_MAX_ABS and rel <= LOGIT_REL_L2, (n, k, err, rel)
        if margin > ARGMAX_MARGIN:
            assert int(eng.argmax.item()) == am
    assert eng.error() == T.TINFER_OK
    eng.close()

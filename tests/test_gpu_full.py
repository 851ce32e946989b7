"""Parity at the benchmark's full sizes, in the launch configurations the benchmark times (the
persistent megakernel on all SMs and the CUDA graph of per-phase kernels, the engine's own attention
chunking): decode steps after the prefilled context of each workload, every logit against the fp64
oracle; both modes bitwise equal to each other; and one teacher-forced run over the whole window of
positions the benchmark times on the Llama-shaped workload."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402
from util import ARGMAX_MARGIN, LOGIT_MAX_ABS, LOGIT_REL_L2, compare_logits, kv_close, kv_deviation  # noqa: E402

pytestmark = pytest.mark.gpu
MODES = {"mega": T.TINFER_MEGAKERNEL, "graph": T.TINFER_GRAPH}


def teacher_forced(name, mode, steps, report=None):
    c = synth.config(name)
    w = synth.make_model(c, seed=0)
    P = c["prefill"]
    K, V = synth.make_kv(c, P, seed=0)
    eng = T.Engine(c, w, mode, kv=(K, V))
    orc = Oracle("f64")
    om = orc.model(c, w)
    tok = int(synth.make_tokens(c, 1, seed=0)[0])
    worst = dict(err=0.0, rel=0.0, kv_steps=0.0, kv_rms=0.0)
    for k in range(steps):
        pos = P + k
        eng.step(tok, pos)
        torch.cuda.synchronize()
        ref, am_ref, rc = orc.decode_step(om, tok, pos, K, V)
        assert rc == 0
        got = eng.logits.cpu().numpy()
        err, rel, margin = compare_logits(got, ref)
        assert err <= LOGIT_MAX_ABS and rel <= LOGIT_REL_L2, (name, k, err, rel)
        if margin > ARGMAX_MARGIN:
            assert int(eng.argmax.item()) == am_ref, (name, k, int(eng.argmax.item()), am_ref, margin)
        Kg = eng.k[:, :, pos].cpu().numpy().view(np.uint16)
        Vg = eng.v[:, :, pos].cpu().numpy().view(np.uint16)
        assert kv_close(Kg, K[:, :, pos]) <= 0 and kv_close(Vg, V[:, :, pos]) <= 0, (name, k)
        for g, r in ((Kg, K[:, :, pos]), (Vg, V[:, :, pos])):
            st, rr = kv_deviation(g, r)
            worst["kv_steps"] = max(worst["kv_steps"], st)
            worst["kv_rms"] = max(worst["kv_rms"], rr)
        worst["err"] = max(worst["err"], err)
        worst["rel"] = max(worst["rel"], rel)
        tok = am_ref
    # slots other than [P, P + steps) are untouched
    Kall = eng.k.cpu().numpy().view(np.uint16)
    assert np.array_equal(Kall[:, :, :P], K[:, :, :P])
    assert np.array_equal(Kall[:, :, P + steps:], K[:, :, P + steps:])
    assert eng.error() == T.TINFER_OK
    eng.close()
    if report is not None:
        report[(name, mode)] = worst
    print(f"\n{name} mode {mode}: {steps} steps, logits max|d| {worst['err']:.3g}, rel L2 {worst['rel']:.3g}; "
          f"KV: at most {worst['kv_steps']:.2f} bf16 steps (|v| >= RMS/16), near zero at most "
          f"{worst['kv_rms']:.3g} x RMS")
    return worst


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("name,steps", [("llama1b", 3), ("tinyllama_int4", 2), ("qwen1.5b", 2),
                                        ("int4_3b", 2)])
def test_full_size_first_steps_match_oracle(name, steps, mode):
    teacher_forced(name, MODES[mode], steps)


@pytest.mark.parametrize("name,steps", [("llama1b", 4), ("qwen1.5b", 3), ("int4_3b", 2)])
def test_full_size_megakernel_and_graph_bitwise_equal(name, steps):
    """The persistent kernel (sliced attention merge over stamped partials, 5-stage ring) and the
    graph of per-phase kernels (ticket merge, 4-stage ring) at the real context lengths, where the
    attention runs 19-152 chunks per KV head: the same logits and the same cache, bit for bit."""
    c = synth.config(name)
    w = synth.make_model(c, seed=0)
    P = c["prefill"]
    toks = synth.make_tokens(c, steps, seed=5)
    outs = []
    for mode in (T.TINFER_MEGAKERNEL, T.TINFER_GRAPH):
        K, V = synth.make_kv(c, P, seed=0)
        eng = T.Engine(c, w, mode, kv=(K, V))
        seq = []
        for k, t in enumerate(toks.tolist()):
            eng.step(int(t), P + k)
            seq.append(eng.logits.cpu().numpy().copy())
        outs.append((np.stack(seq), eng.k.cpu().numpy().copy(), eng.v.cpu().numpy().copy()))
        assert eng.error() == T.TINFER_OK
        eng.close()
    assert np.array_equal(outs[0][0].view(np.uint32), outs[1][0].view(np.uint32))
    assert np.array_equal(outs[0][1], outs[1][1]) and np.array_equal(outs[0][2], outs[1][2])


def test_llama1b_whole_benchmark_window_teacher_forced():
    """Every position the benchmark times on the Llama-shaped workload (1024..1151): the attention
    split changes with the position, so each step is a different chunking."""
    c = synth.config("llama1b")
    teacher_forced("llama1b", T.TINFER_MEGAKERNEL, c["steps"])

"""Parity at the benchmark's full sizes, in the launch configuration the benchmark times (the
persistent megakernel on all SMs, the engine's own attention chunking): the first decode steps after
the prefilled context of each workload, every logit against the fp64 oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import decode_persistent_megakernel_gb300 as T  # noqa: E402
import synth  # noqa: E402
from oracle import Oracle  # noqa: E402
from util import ARGMAX_MARGIN, LOGIT_MAX_ABS, LOGIT_REL_L2, compare_logits, kv_close  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,steps", [("llama1b", 3), ("tinyllama_int4", 2), ("qwen1.5b", 2),
                                        ("int4_3b", 2)])
def test_full_size_first_steps_match_oracle(name, steps):
    c = synth.config(name)
    w = synth.make_model(c, seed=0)
    P = c["prefill"]
    K, V = synth.make_kv(c, P, seed=0)
    eng = T.Engine(c, w, T.TINFER_MEGAKERNEL, kv=(K, V))
    orc = Oracle("f64")
    om = orc.model(c, w)
    tok = int(synth.make_tokens(c, 1, seed=0)[0])
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
            assert int(eng.argmax.item()) == am_ref
        Kg = eng.k[:, :, pos].cpu().numpy().view(np.uint16)
        Vg = eng.v[:, :, pos].cpu().numpy().view(np.uint16)
        assert kv_close(Kg, K[:, :, pos]) <= 0 and kv_close(Vg, V[:, :, pos]) <= 0
        tok = am_ref
    assert eng.error() == T.TINFER_OK
    eng.close()

"""Host logic of the timeline report (decode_persistent_megakernel_gb300.timeline): the per-phase
quantities from a hand-made stamp array of one layer and the LM head on two CTAs."""
import numpy as np

from decode_persistent_megakernel_gb300.timeline import phase_table


def test_phase_table_from_hand_made_stamps():
    L, nph, F = 1, 6, 10
    t = np.zeros((2, nph, F))
    # CTA c, phase k: start 1000 k + 10 c, end start + 900 (CTA 1 ends 100 later)
    for c in range(2):
        for k in range(nph):
            s = 1000.0 * k + 10 * c + 1
            t[c, k, 0] = s
            t[c, k, 2] = s + 900 + 100 * c
            if k != 1:  # GEMV phases: entry, fetched, ready, first stage, last stage
                t[c, k, 6] = s + 50
                t[c, k, 7] = s + 250
                t[c, k, 1] = s + 300
                t[c, k, 8] = s + 320
                t[c, k, 9] = s + 800
            else:  # attention: keys, queries rotated, scores, partials, values, merge seen
                for f, off in ((1, 100), (5, 90), (6, 300), (7, 500), (8, 400), (9, 700)):
                    t[c, k, f] = s + off
    tab = phase_table(t, L)
    assert set(tab) == {"QKV", "ATT", "O", "GU", "DN", "LM"}
    q = tab["QKV"][0]
    # the first phase's critical share runs from the earliest start to the latest end
    assert q["crit"] == (1 + 10 + 1000) - 1
    assert q["plan"] == 50 and q["fetch"] == 200 and q["act"] == 50
    assert q["stage0"] == 20 and q["stream"] == 480 and q["epi"] == 150  # 100 and 200 on the two CTAs
    o = tab["O"][0]
    # phase 2 ends latest at 2000 + 10 + 1 + 1000; phase 1 latest at 1000 + 10 + 1 + 1000
    assert o["crit"] == 1000
    assert o["skew_prev"] == 55  # latest (2011) minus median (1956) end of the previous phase
    assert o["fetch_end_max"] == (2000 + 10 + 1 + 250) - (1000 + 10 + 1 + 1000)
    a = tab["ATT"][0]
    assert a["keys"] == 100 and a["scores"] == 300 and a["merge_seen"] == 700


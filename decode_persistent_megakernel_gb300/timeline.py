"""Per-phase timeline of the persistent decode kernel ("Decoding in tiles", section 5, Figure 9: each
worker's time split into streaming, waiting and small work), from the %globaltimer stamps that
tinfer_set_trace records for every CTA and phase.

  python -m decode_persistent_megakernel_gb300.timeline [WORKLOAD] [N_TRACED]

builds the engine on the seeded synthetic workload (persistent kernel), times untraced steps with
CUDA events, then records N_TRACED traced steps from the first decode position and prints, per
phase kind (QKV, attention, O, gate/up, down, LM head), medians over layers and steps of:
  crit       latest end of the phase minus latest end of the one before (its share of the step)
  skew_prev  latest minus median end of the previous phase
  dur        median over CTAs of the phase's own duration
GEMV phases: plan (start -> GEMV code), fetch (-> input vector in shared memory), act (-> input
segment in registers), stage0 (-> first weight stage), stream (first -> last stage), epi (last stage
-> end), fetch_end_max (latest input arrival minus latest end of the previous phase);
attention: keys, qrot, scores, vals, parts, merge_seen, each from the phase start.
Stamps have 32 ns resolution; medians over 152 CTAs resolve finer differences.
"""
from __future__ import annotations

import sys

import numpy as np

PHASE_NAMES = ["QKV", "ATT", "O", "GU", "DN"]


def phase_table(t: np.ndarray, n_layers: int) -> dict:
    """t: stamps [grid][phases][TRACE_FIELDS] (ns, 0 = not recorded) of one traced step. Returns
    {phase kind: [per-layer dict of the quantities above, in ns]}."""
    nph = n_layers * 5 + 1
    end, start = t[:, :, 2], t[:, :, 0]
    out: dict = {}
    for k in range(nph):
        ph = "LM" if k == nph - 1 else PHASE_NAMES[k % 5]
        prev_end = end[:, k - 1].max() if k > 0 else start[:, 0].min()
        prev_med = np.median(end[:, k - 1]) if k > 0 else prev_end
        d = {"crit": end[:, k].max() - prev_end, "skew_prev": prev_end - prev_med}
        act = t[:, k, 2] > 0
        d["dur"] = np.median(t[act, k, 2] - t[act, k, 0])
        if ph != "ATT":
            m = act & (t[:, k, 6] > 0) & (t[:, k, 7] > 0)
            if m.any():
                d["plan"] = np.median(t[m, k, 6] - t[m, k, 0])
                d["fetch"] = np.median(t[m, k, 7] - t[m, k, 6])
                d["act"] = np.median(t[m, k, 1] - t[m, k, 7])
                m2 = m & (t[:, k, 8] > 0) & (t[:, k, 9] > 0)
                if m2.any():
                    d["stage0"] = np.median(t[m2, k, 8] - t[m2, k, 1])
                    d["stream"] = np.median(t[m2, k, 9] - t[m2, k, 8])
                    d["epi"] = np.median(t[m2, k, 2] - t[m2, k, 9])
                d["fetch_end_max"] = t[m, k, 7].max() - prev_end
        else:
            for f, nm in ((1, "keys"), (5, "qrot"), (6, "scores"), (8, "vals"), (7, "parts"), (9, "merge_seen")):
                mm = act & (t[:, k, f] > 0)
                if mm.any():
                    d[nm] = np.median(t[mm, k, f] - t[mm, k, 0])
        out.setdefault(ph, []).append(d)
    return out


def main(argv: list[str]) -> None:
    import torch

    import synth
    import decode_persistent_megakernel_gb300 as T

    name = argv[0] if argv else "llama1b"
    n_traced = int(argv[1]) if len(argv) > 1 else 5
    c = synth.config(name)
    w = synth.make_model(c, seed=0)
    P = c["prefill"] + c["prompt"]
    K, V = synth.make_kv(c, P, seed=0)
    eng = T.Engine(c, w, T.TINFER_MEGAKERNEL, kv=(K, V))
    tok = int(synth.make_tokens(c, 1, seed=0)[0])
    for i in range(10):
        eng.step(tok, P + i, logits=False)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = 200
    e0.record()
    for i in range(n):
        eng.step(tok, P + (i % c["steps"]), logits=False)
    e1.record()
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / n
    acc: dict = {}
    totals = []
    for r in range(n_traced):
        t = eng.trace_step(tok, P + r).astype(np.float64)
        totals.append(t[:, :, 2].max() - t[:, 0, 0][t[:, 0, 0] > 0].min())
        for ph, rows in phase_table(t, c["n_layers"]).items():
            acc.setdefault(ph, []).extend(rows)
    assert eng.error() == T.TINFER_OK
    eng.close()
    print(f"{name}: {us:.1f} us per step untraced (CUDA events, {n} steps); traced step {np.median(totals) / 1e3:.1f} us")
    crit = {}
    for ph in PHASE_NAMES + ["LM"]:
        rows = acc[ph]
        keys = list(rows[0].keys())
        cells = "  ".join(f"{k} {np.median([r[k] for r in rows if k in r]) / 1e3:.2f}" for k in keys)
        crit[ph] = np.median([r["crit"] for r in rows]) / 1e3
        print(f"{ph:4s} {cells}")
    print(f"per layer (sum of crit medians) {sum(crit[p] for p in PHASE_NAMES):.2f} us; LM head {crit['LM']:.2f} us")


if __name__ == "__main__":
    main(sys.argv[1:])

"""Writes lm760m_drift.json: how far the fp64 oracle's own chunk scan moves,
chunk by chunk, on the 760M-scale layer workload (B2 H4 d=m=384, N 32768,
chunk 2048, momentum 0.9, Muon 5, L2-Normalize) when its fast-weight state
is rounded to bf16 at every chunk boundary.

Why: the update of every chunk (momentum, Newton-Schulz orthogonalisation,
row normalisation; "5.2.1 LaCT and TTT-E2E", eqs (5), (6) and the momentum
sentence after eq (6)) feeds the next chunk, and the scan is strictly
sequential ("Test-Time Training with KV Binding Is Secretly Linear
Attention", App. I), so a small difference in the state grows from chunk to
chunk.  Any implementation that computes with bf16 operands injects a
difference of about bf16 rounding into the state every chunk; this file
records what that injection alone does to the exact scan.  The full-length
GPU parity test bounds its own per-chunk error by a multiple of these values.

Only the oracle computes here: the reference run is the oracle's single pass;
the perturbed run is the same oracle called one chunk at a time, its final
weights rounded to bf16 (round to nearest even, by torch) before they start
the next chunk, the momentum carried unrounded.  Inputs come from the seeded
workload generator.  Run from the repository root:

    python tests/golden/make_lm760m_drift.py
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402
from oracle import ttt_oracle as O  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lm760m_drift.json")


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def sequence_runs(wl, inputs, b, h):
    """(reference outputs, reference weights, perturbed outputs, perturbed
    weights) of one (batch, head) sequence; outputs [N, d]."""
    q, k, v, eta, W1, W2, W3 = inputs
    sl = lambda t: t[b:b + 1, h:h + 1].double().numpy()
    Q, K, V, E = sl(q), sl(k), sl(v), sl(eta)
    Ws = [t[h:h + 1].double().numpy() for t in (W1, W2, W3)]
    kw = dict(l2norm=wl.l2norm, muon_steps=wl.muon_steps, momentum_beta=wl.momentum_beta)
    ref = O.ttt_layer_forward(Q, K, V, E, *Ws, wl.chunk, wl.mode, **kw)
    cur = [bf16_round(w)[None] for w in Ws]   # [1, 1, rows, cols]: per-batch weights
    mom, outs = None, []
    for c in range(wl.N // wl.chunk):
        s = slice(c * wl.chunk, (c + 1) * wl.chunk)
        o, a1, a2, a3, mom = O.ttt_layer_forward(Q[..., s, :], K[..., s, :], V[..., s, :],
                                                 E[..., s], *cur, wl.chunk, wl.mode,
                                                 momentum=mom, **kw)
        outs.append(o[0, 0])
        cur = [bf16_round(a1), bf16_round(a2), bf16_round(a3)]
    return ref[0][0, 0], [r[0, 0] for r in ref[1:4]], np.concatenate(outs), \
        [c[0, 0] for c in cur]


def main():
    wl = W.LM_760M
    inputs = W.layer_inputs(wl)
    nc = wl.N // wl.chunk
    num = np.zeros(nc)
    den = np.zeros(nc)
    wnum = np.zeros(3)
    wden = np.zeros(3)
    per_seq = {}
    for b in range(wl.B):
        for h in range(wl.H):
            ro, rw, po, pw = sequence_runs(wl, inputs, b, h)
            seq = []
            for c in range(nc):
                s = slice(c * wl.chunk, (c + 1) * wl.chunk)
                dn, rn = np.sum((ro[s] - po[s]) ** 2), np.sum(ro[s] ** 2)
                num[c] += dn
                den[c] += rn
                seq.append(float(np.sqrt(dn / rn)))
            for i in range(3):
                wnum[i] += np.sum((rw[i] - pw[i]) ** 2)
                wden[i] += np.sum(rw[i] ** 2)
            per_seq[f"{b},{h}"] = seq
            print(f"sequence ({b}, {h}): chunk 0 {seq[0]:.2e}, chunk {nc - 1} {seq[-1]:.2e}")
    res = {
        "what": "relative L2 difference, per chunk of the output over all (batch, head) "
                "sequences, between the fp64 oracle and the same oracle with its fast-weight "
                "state rounded to bf16 at every chunk boundary",
        "workload": wl.name,
        "source": "5.2.1 LaCT and TTT-E2E, eqs (5)-(6) and the momentum sentence; Test-Time "
                  "Training with KV Binding Is Secretly Linear Attention, App. I",
        "written_by": "tests/golden/make_lm760m_drift.py (oracle only)",
        "per_chunk": [float(np.sqrt(n / d)) for n, d in zip(num, den)],
        "final_weights": {"W1": float(np.sqrt(wnum[0] / wden[0])),
                          "W2": float(np.sqrt(wnum[1] / wden[1])),
                          "W3": float(np.sqrt(wnum[2] / wden[2]))},
        "per_sequence": per_seq,
    }
    with open(OUT, "w") as f:
        json.dump(res, f, indent=1)
    print("wrote", OUT)


if __name__ == "__main__":
    main()

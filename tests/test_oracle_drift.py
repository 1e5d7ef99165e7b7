"""How far the fp64 oracle's own chunk scan moves under bf16-sized
perturbations on the 760M-scale layer workload (CPU only).

The scan is strictly sequential ("Test-Time Training with KV Binding Is
Secretly Linear Attention", App. I), and every chunk's update (momentum,
Newton-Schulz, row normalisation; "5.2.1 LaCT and TTT-E2E", eqs (5), (6) and
the momentum sentence) starts from the previous state, so a difference in
the state grows from chunk to chunk.  These tests show, with the oracle
alone, that bf16 rounding of the initial weights (once), or of the state
(every chunk), moves the outputs of the last chunks and the final weights by
more than the 3e-2 tolerance: the full-length comparison of a bf16 path needs
a per-chunk bound, recorded in tests/golden/lm760m_drift.json.
"""
import importlib.util
import json
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ttt_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "lm760m_drift.json")
TOL = 3e-2   # the bf16-with-Muon tolerance of the workload table


def _gen_module():
    spec = importlib.util.spec_from_file_location(
        "make_lm760m_drift", os.path.join(HERE, "golden", "make_lm760m_drift.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.fixture(scope="module")
def lm_inputs():
    return W.layer_inputs(W.LM_760M)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_initial_weights_rounded_once(lm_inputs):
    """Rounding only W1, W2, W3 at the start to bf16 (relative change ~2e-3):
    chunk 0 moves by about that much, chunk 15 and the final weights by more
    than the tolerance, and the difference grows every chunk."""
    wl = W.LM_760M
    q, k, v, eta, W1, W2, W3 = lm_inputs
    sl = lambda t: t[:1, :1].double().numpy()
    Q, K, V, E = sl(q), sl(k), sl(v), sl(eta)
    Ws = [t[:1].double().numpy() for t in (W1, W2, W3)]
    Wb = [t[:1].to(torch.bfloat16).double().numpy() for t in (W1, W2, W3)]
    kw = dict(muon_steps=wl.muon_steps, momentum_beta=wl.momentum_beta)
    r = O.ttt_layer_forward(Q, K, V, E, *Ws, wl.chunk, wl.mode, **kw)
    p = O.ttt_layer_forward(Q, K, V, E, *Wb, wl.chunk, wl.mode, **kw)
    per = [_rel(p[0][0, 0, c * wl.chunk:(c + 1) * wl.chunk], r[0][0, 0, c * wl.chunk:(c + 1) *
                                                                     wl.chunk])
           for c in range(wl.N // wl.chunk)]
    assert 1e-3 < per[0] < 5e-3
    assert all(b > a for a, b in zip(per, per[1:]))
    assert per[-1] > 3 * TOL
    for i in (1, 2, 3):
        assert _rel(p[i], r[i]) > 2 * TOL


def test_golden_drift_file_is_what_its_script_writes(lm_inputs):
    """The committed per-chunk bound: rounding the state at every chunk keeps
    chunk 0 at bf16 level and exceeds the tolerance well before the end; the
    file's first sequence is reproduced by its generator."""
    with open(GOLDEN) as f:
        g = json.load(f)
    per = g["per_chunk"]
    assert len(per) == W.LM_760M.N // W.LM_760M.chunk
    assert 1e-3 < per[0] < 5e-3
    assert all(b > a for a, b in zip(per, per[1:]))
    assert per[-1] > 3 * TOL
    assert min(g["final_weights"].values()) > 2 * TOL
    mod = _gen_module()
    ro, _, po, _ = mod.sequence_runs(W.LM_760M, lm_inputs, 0, 0)
    b = W.LM_760M.chunk
    again = [_rel(po[c * b:(c + 1) * b], ro[c * b:(c + 1) * b]) for c in range(len(per))]
    np.testing.assert_allclose(again, g["per_sequence"]["0,0"], rtol=1e-6)

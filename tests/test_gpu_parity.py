"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances are the ones the method's benchmark table states: max relative
error (max|x - r| / max|r|) <= 1e-4 for the fp32 path; relative L2 error
<= 2e-2 for bf16 (<= 3e-2 with Muon), per output tensor (out and each final
fast-weight matrix).
"""
import dataclasses
import json
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ttt_oracle as O
from tests.gpu_util import assert_status_ok, f64, lib, max_rel, rel_l2

pytestmark = pytest.mark.gpu

F32_MAX_REL = 1e-4
BF16_REL_L2 = 2e-2
BF16_MUON_REL_L2 = 3e-2
DEV = "cuda:0"


# ---------------------------------------------------------------------------
# the GEMM building block against a plain fp32 product

@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("tile_n", [64, 128, 192, 256])
def test_selftest_gemm_bf16(a_mn, b_mn, tile_n):
    cla = lib()
    g = torch.Generator(device="cpu").manual_seed(7)
    Z, M, N, K = 2, 256, 384, 192
    A = torch.randn((Z, K, M) if a_mn else (Z, M, K), generator=g).to(torch.bfloat16)
    B = torch.randn((Z, K, N) if b_mn else (Z, N, K), generator=g).to(torch.bfloat16)
    D = cla.selftest_gemm(A.to(DEV), B.to(DEV), bool(a_mn), bool(b_mn), tile_n)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    Af = A.double().transpose(1, 2) if a_mn else A.double()
    Bf = B.double() if b_mn else B.double().transpose(1, 2)
    ref = torch.bmm(Af, Bf).numpy()
    assert rel_l2(f64(D), ref) < 1e-5


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1)])
def test_selftest_gemm_f32(a_mn, b_mn):
    cla = lib()
    g = torch.Generator(device="cpu").manual_seed(8)
    Z, M, N, K = 3, 70, 45, 33
    A = torch.randn((Z, K, M) if a_mn else (Z, M, K), generator=g)
    B = torch.randn((Z, K, N) if b_mn else (Z, N, K), generator=g)
    D = cla.selftest_gemm(A.to(DEV), B.to(DEV), bool(a_mn), bool(b_mn))
    torch.cuda.synchronize()
    Af = A.double().transpose(1, 2) if a_mn else A.double()
    Bf = B.double() if b_mn else B.double().transpose(1, 2)
    assert max_rel(f64(D), torch.bmm(Af, Bf).numpy()) < 1e-5


# ---------------------------------------------------------------------------
# TTT layer

def run_layer(cla, wl, q, k, v, eta, W1, W2, W3, momentum=None):
    rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                           momentum_beta=wl.momentum_beta)
    res = cla.ttt_layer_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), W1.to(DEV),
                                W2.to(DEV), W3.to(DEV), wl.chunk, wl.mode, rule,
                                update_chunks=wl.update_chunks, momentum=momentum)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    return [f64(t) for t in res]


def run_oracle(wl, q, k, v, eta, W1, W2, W3, n_chunks=None, momentum=None):
    return O.ttt_layer_forward(f64(q), f64(k), f64(v), f64(eta), f64(W1), f64(W2), f64(W3),
                               wl.chunk, wl.mode, update_chunks=wl.update_chunks,
                               l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                               momentum_beta=wl.momentum_beta, momentum=momentum,
                               n_chunks=n_chunks)


def test_layer_tiny_fp32():
    """The tiny fp32 workload exactly as specified: max rel error <= 1e-4."""
    cla = lib()
    wl = W.TINY_F32
    inp = W.layer_inputs(wl)
    got = run_layer(cla, wl, *inp)
    ref = run_oracle(wl, *inp)
    for g_, r_ in zip(got, ref[:4]):
        assert max_rel(g_, r_) <= F32_MAX_REL


FP32_CASES = [
    dict(mode=W.APPLY_THEN_UPDATE, chunk=16, N=64, d_h=24, m_h=40, muon_steps=3, momentum_beta=0.9),
    dict(mode=W.BLOCK_CAUSAL, chunk=32, N=128, d_h=33, m_h=17, muon_steps=0, momentum_beta=0.5),
    dict(mode=W.BIDIRECTIONAL, chunk=96, N=96, d_h=16, m_h=16, muon_steps=2, momentum_beta=0.0),
    dict(mode=W.STRIDED, chunk=16, N=96, d_h=20, m_h=36, muon_steps=1, momentum_beta=0.0,
         update_chunks=(1, 0, 1, 0, 0, 1)),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=8, N=40, d_h=8, m_h=8, l2norm=False),
]


@pytest.mark.parametrize("case", FP32_CASES)
def test_layer_fp32_variants(case):
    cla = lib()
    wl = dataclasses.replace(W.TINY_F32, B=2, H=2, **case)
    inp = W.layer_inputs(wl)
    got = run_layer(cla, wl, *inp)
    ref = run_oracle(wl, *inp)
    for g_, r_ in zip(got, ref[:4]):
        assert max_rel(g_, r_) <= F32_MAX_REL


BF16_CASES = [
    dict(mode=W.APPLY_THEN_UPDATE, chunk=128, N=512, d_h=128, m_h=128),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=128, N=512, d_h=128, m_h=128, muon_steps=3,
         momentum_beta=0.9),
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=1024, d_h=128, m_h=192, momentum_beta=0.5),
    dict(mode=W.BLOCK_CAUSAL, chunk=128, N=512, d_h=192, m_h=128, muon_steps=2),
    dict(mode=W.BLOCK_CAUSAL, chunk=128, N=384, d_h=128, m_h=320, muon_steps=2,
         momentum_beta=0.9),
    dict(mode=W.BIDIRECTIONAL, chunk=512, N=512, d_h=128, m_h=128, muon_steps=1),
    dict(mode=W.STRIDED, chunk=128, N=1024, d_h=128, m_h=256,
         update_chunks=(1, 0, 1, 1, 0, 0, 0, 0)),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=128, N=512, d_h=64, m_h=64, l2norm=False),
    # square orders that are multiples of 128: the row-panel Newton-Schulz kernel
    # with clusters of 2, 3 and 4 CTAs, one step without normalisation
    dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=768, d_h=256, m_h=256, muon_steps=3,
         momentum_beta=0.9),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=384, N=768, d_h=384, m_h=384, muon_steps=5,
         momentum_beta=0.9, l2_normed_k=True),
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=512, d_h=512, m_h=512, muon_steps=2),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=128, N=384, d_h=384, m_h=384, muon_steps=1,
         l2norm=False),
    # square orders that are not multiples of 128: the tile-cluster Newton-Schulz
    # kernel (clusters of 2, 6 and 8 CTAs).  With Muon, chunk >= d: a chunk
    # shorter than d leaves the momentum rank-deficient, and each Newton-Schulz
    # step multiplies its near-zero singular values by about a = 3.44, so bf16
    # rounding noise there grows ~3.44^steps (rounding M alone to bf16 moves the
    # oracle by 5e-2 at d = 320, chunk 128, 5 steps)
    dict(mode=W.APPLY_THEN_UPDATE, chunk=128, N=512, d_h=192, m_h=192, muon_steps=3,
         momentum_beta=0.9),
    dict(mode=W.BLOCK_CAUSAL, chunk=384, N=768, d_h=320, m_h=320, muon_steps=3,
         momentum_beta=0.9, l2_normed_k=True),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=512, d_h=448, m_h=448, muon_steps=2),
]


@pytest.mark.parametrize("case", BF16_CASES)
def test_layer_bf16_variants(case):
    cla = lib()
    base = dict(B=2, H=2, muon_steps=0, momentum_beta=0.0, l2_normed_k=False)
    base.update(case)
    wl = dataclasses.replace(W.LM_760M, **base)
    inp = W.layer_inputs(wl)
    got = run_layer(cla, wl, *inp)
    ref = run_oracle(wl, *inp)
    tol = BF16_MUON_REL_L2 if wl.muon_steps else BF16_REL_L2
    errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref[:4])]
    assert max(errs) <= tol, errs


def test_layer_bf16_per_batch_weights_and_momentum_carry():
    """Per-batch initial weights, and a sequence split in two calls with the
    final weights and momentum fed back equals the oracle's single pass."""
    cla = lib()
    wl = dataclasses.replace(W.LM_760M, B=2, H=2, N=512, d_h=128, m_h=128, chunk=128,
                             muon_steps=2, momentum_beta=0.9)
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wl)
    W1b, W2b, W3b = (x.unsqueeze(0).repeat(2, 1, 1, 1).contiguous() for x in (W1, W2, W3))
    W1b[1] *= 1.5
    ref = run_oracle(wl, q, k, v, eta, W1b, W2b, W3b)
    half = wl.N // 2
    wh = dataclasses.replace(wl, N=half)
    mom = torch.zeros(3 * 2 * 2 * 128 * 128, device=DEV)
    sl = lambda t: t[..., :half, :].contiguous()
    o1, A1, A2, A3 = run_layer(cla, wh, sl(q), sl(k), sl(v), eta[..., :half].contiguous(),
                               W1b, W2b, W3b, momentum=mom)
    sr = lambda t: t[..., half:, :].contiguous()
    o2, B1, B2, B3 = run_layer(cla, wh, sr(q), sr(k), sr(v), eta[..., half:].contiguous(),
                               torch.from_numpy(A1).float(), torch.from_numpy(A2).float(),
                               torch.from_numpy(A3).float(), momentum=mom)
    out = np.concatenate([o1, o2], axis=2)
    errs = [rel_l2(out, ref[0]), rel_l2(B1, ref[1]), rel_l2(B2, ref[2]), rel_l2(B3, ref[3])]
    assert max(errs) <= BF16_MUON_REL_L2, errs


def test_layer_replace_q_with_k_and_gradient_ascent():
    cla = lib()
    wl = dataclasses.replace(W.LM_760M, B=1, H=2, N=512, d_h=128, m_h=128, chunk=128,
                             muon_steps=0, momentum_beta=0.0)
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wl)
    for qq, ee in ((k, eta), (q, -eta)):
        got = run_layer(cla, wl, qq, k, v, ee.contiguous(), W1, W2, W3)
        ref = run_oracle(wl, qq, k, v, ee, W1, W2, W3)
        errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref[:4])]
        assert max(errs) <= BF16_REL_L2, errs


# ---------------------------------------------------------------------------
# chunked linear attention

LIN_CASES = [
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=1024),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=128, N=1024),
    dict(mode=W.BIDIRECTIONAL, chunk=1024, N=1024),
    dict(mode=W.STRIDED, chunk=128, N=1024, update_chunks=(0, 1, 1, 0, 1, 0, 0, 1)),
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=768, d_k=64, d_v=192),
    dict(mode=W.APPLY_THEN_UPDATE, chunk=512, N=2048, d_k=64, d_v=128),
    # 32 chunks of one-launch shape: each prefix item takes its 32 partial
    # slices through four ring stages (eight per stage at d_k = d_v = 128)
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=8192),
    dict(mode=W.STRIDED, chunk=256, N=8192,
         update_chunks=tuple(int(c % 3 != 1 and c < 29) for c in range(32))),
]


@pytest.mark.parametrize("case", LIN_CASES)
@pytest.mark.parametrize("with_state", [False, True])
def test_linattn_bf16(case, with_state):
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, **case)
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=with_state)
    o, S = cla.linattn_chunked_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), wl.chunk,
                                       wl.mode, S0=None if S0 is None else S0.to(DEV),
                                       update_chunks=wl.update_chunks)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    ro, rS = O.linattn_chunked_forward(f64(q), f64(k), f64(v), f64(eta),
                                       None if S0 is None else f64(S0), wl.chunk, wl.mode,
                                       wl.update_chunks)
    assert rel_l2(f64(o), ro) <= BF16_REL_L2
    assert rel_l2(f64(S), rS) <= BF16_REL_L2


@pytest.mark.parametrize("mode", [W.APPLY_THEN_UPDATE, W.BLOCK_CAUSAL])
def test_linattn_fp32(mode):
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=3, N=200, d_k=24, d_v=40, chunk=40, mode=mode,
                             io_dtype="f32")
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=True)
    o, S = cla.linattn_chunked_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), wl.chunk,
                                       wl.mode, S0=S0.to(DEV))
    torch.cuda.synchronize()
    ro, rS = O.linattn_chunked_forward(f64(q), f64(k), f64(v), f64(eta), f64(S0), wl.chunk,
                                       wl.mode)
    assert max_rel(f64(o), ro) <= F32_MAX_REL
    assert max_rel(f64(S), rS) <= F32_MAX_REL


# ---------------------------------------------------------------------------
# full-size workloads

def test_linattn_full_size():
    """Linear-attention workload at full size (B4 H4 N8192 d128, chunk 2048)."""
    cla = lib()
    wl = W.LINATTN_C2
    q, k, v, eta, _ = W.linattn_inputs(wl)
    o, S = cla.linattn_chunked_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), wl.chunk,
                                       wl.mode)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    ro, rS = O.linattn_chunked_forward(f64(q), f64(k), f64(v), f64(eta), None, wl.chunk, wl.mode)
    assert rel_l2(f64(o), ro) <= BF16_REL_L2
    assert rel_l2(f64(S), rS) <= BF16_REL_L2


GOLDEN_DRIFT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                            "lm760m_drift.json")
# The full-length bound: a chunk's error may be at most this multiple of what
# rounding the oracle's own state to bf16 at every chunk boundary does to it
# (tests/golden/lm760m_drift.json).  The bf16 path rounds more than the state
# (GEMM operands, Newton-Schulz iterates, activations); it has measured about
# 2-2.6 times that per-chunk injection.
DRIFT_FACTOR = 4.0


def test_layer_lm_full_size():
    """LM-style workload at full size (B2 H4 d=m=384 N32768 chunk 2048, Muon 5,
    beta 0.9), every chunk against the oracle's full scan: chunks 0 and 1
    within the bf16-with-Muon tolerance, every chunk and the final weights
    within DRIFT_FACTOR times the oracle's own per-chunk sensitivity to bf16
    rounding of its state (the scan amplifies any difference about 1.25x per
    chunk, so the tolerance cannot hold at the end for a bf16 path); the
    weights after two chunks from a prefix call within the tolerance; unit
    row norms of the final weights."""
    cla = lib()
    wl = W.LM_760M
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wl)
    got = run_layer(cla, wl, q, k, v, eta, W1, W2, W3)
    ref = run_oracle(wl, q, k, v, eta, W1, W2, W3)
    with open(GOLDEN_DRIFT) as f:
        drift = json.load(f)
    b = wl.chunk
    per = [rel_l2(got[0][..., c * b:(c + 1) * b, :], ref[0][..., c * b:(c + 1) * b, :])
           for c in range(wl.N // b)]
    wf = [rel_l2(got[i], ref[i]) for i in (1, 2, 3)]
    print("per-chunk rel L2 vs oracle:", " ".join(f"{e:.2e}" for e in per))
    print("per-chunk ratio to the state-rounding drift:",
          " ".join(f"{e / d:.2f}" for e, d in zip(per, drift["per_chunk"])))
    print("final weights rel L2:", wf)
    assert per[0] <= BF16_MUON_REL_L2 and per[1] <= BF16_MUON_REL_L2, per
    for c, (e, dr) in enumerate(zip(per, drift["per_chunk"])):
        assert e <= DRIFT_FACTOR * dr, (c, e, dr)
    for e, name in zip(wf, ("W1", "W2", "W3")):
        assert e <= DRIFT_FACTOR * drift["final_weights"][name], (name, e)
    for Wf in got[1:]:
        np.testing.assert_allclose(np.linalg.norm(Wf, axis=-1), 1.0, atol=1e-3)
    nc = 2
    pre = wl.chunk * nc
    refp = run_oracle(wl, q, k, v, eta, W1, W2, W3, n_chunks=nc)
    wp = dataclasses.replace(wl, N=pre)
    sl = lambda t: t[..., :pre, :].contiguous()
    gp = run_layer(cla, wp, sl(q), sl(k), sl(v), eta[..., :pre].contiguous(), W1, W2, W3)
    errs = [rel_l2(g_, r_) for g_, r_ in zip(gp[1:], refp[1:4])]
    assert max(errs) <= BF16_MUON_REL_L2, errs


def test_layer_long_context_prefix_and_full_length():
    """Million-token workload (B1 H4 d=m=512, chunk 8192, Muon 5, beta 0.9):
    a prefix call of its first three chunks (all four heads) against the
    oracle, outputs and weights within the bf16-with-Muon tolerance; then the
    full 1,048,576-token call, whose first three chunks hold the same inputs,
    gives the same first-chunk outputs as the prefix call (the scan is causal)
    and ends with unit-norm, finite weights."""
    cla = lib()
    wl = W.LONG_1M
    nc = 3
    pre = nc * wl.chunk
    wp = dataclasses.replace(wl, N=pre)
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wp)
    gp = run_layer(cla, wp, q, k, v, eta, W1, W2, W3)
    ref = run_oracle(wp, q, k, v, eta, W1, W2, W3)
    errs = [rel_l2(g_, r_) for g_, r_ in zip(gp, ref[:4])]
    print("long-context prefix rel L2 (out, W1, W2, W3):", errs)
    assert max(errs) <= BF16_MUON_REL_L2, errs
    fq, fk, fv, feta, _, _, _ = W.layer_inputs_on_device(wl, DEV, seed=1)
    for dst, src in ((fq, q), (fk, k), (fv, v)):
        dst[..., :pre, :] = src.to(DEV)
    feta[..., :pre] = eta.to(DEV)
    rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                           momentum_beta=wl.momentum_beta)
    out, F1, F2, F3 = cla.ttt_layer_forward(fq, fk, fv, feta, W1.to(DEV), W2.to(DEV), W3.to(DEV),
                                            wl.chunk, wl.mode, rule)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    head = f64(out[..., :pre, :])
    assert rel_l2(head, ref[0]) <= BF16_MUON_REL_L2
    assert np.array_equal(head, gp[0])
    for Wf in (F1, F2, F3):
        n = torch.linalg.vector_norm(Wf, dim=-1)
        assert bool(torch.isfinite(Wf).all())
        assert float((n - 1).abs().max()) < 1e-3


def test_layer_strided_full_size():
    """View-synthesis strided workload at full size (B1 H2 d384 m768, 8 x 8192,
    update on chunks 0-3): every output and final weight."""
    cla = lib()
    wl = W.NVS_STRIDED
    inp = W.layer_inputs(wl)
    got = run_layer(cla, wl, *inp)
    ref = run_oracle(wl, *inp)
    errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref[:4])]
    assert max(errs) <= BF16_REL_L2, errs


def test_layer_bitwise_repeatable():
    """Two calls on the same inputs give bit-identical outputs and final weights:
    the gradient's squared norm (the Newton-Schulz scale) is reduced from
    per-tile partials in a fixed order, with no floating-point atomics."""
    cla = lib()
    wl = dataclasses.replace(W.LM_760M, B=2, H=2, N=2048, chunk=512, muon_steps=5,
                             momentum_beta=0.9)
    inp = W.layer_inputs(wl)
    runs = [run_layer(cla, wl, *inp) for _ in range(2)]
    for a_, b_ in zip(*runs):
        assert np.array_equal(a_, b_)


# Workloads that exercise every update path: the fused Newton-Schulz launch
# (Muon, apply and update of the same chunk every step), the per-product
# Newton-Schulz launches and the normalisation launch (non-square weights,
# strided update flags: steps that only apply or only update), and the
# normalisation alone (no Muon).
SCHED_WORKLOADS = [
    dict(B=2, H=2, N=2048, d_h=256, m_h=256, chunk=256, muon_steps=5, momentum_beta=0.9),
    dict(B=1, H=2, N=1024, d_h=128, m_h=256, chunk=128, muon_steps=2, momentum_beta=0.5,
         mode=W.STRIDED, update_chunks=(1, 0, 0, 1, 0, 1, 1, 0)),
    dict(B=1, H=3, N=1024, d_h=128, m_h=256, chunk=128, muon_steps=0, momentum_beta=0.5,
         mode=W.STRIDED, update_chunks=(1, 0, 0, 1, 0, 1, 1, 0)),
]

_SCHED_CHILD = r"""
import dataclasses, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import workloads as W
from tests.test_gpu_parity import SCHED_WORKLOADS, run_layer
from tests.gpu_util import lib
cla = lib()
res = {}
for i, kw in enumerate(SCHED_WORKLOADS):
    wl = dataclasses.replace(W.LM_760M, **kw)
    for j, t in enumerate(run_layer(cla, wl, *W.layer_inputs(wl))):
        res[f"w{i}_{j}"] = t
np.savez(sys.argv[2], **res)
"""


@pytest.mark.parametrize("env", [
    {"TTT_SPLIT_APPLY": "0", "TTT_SEQUENCE_GROUPS": "1"},
    {"TTT_SPLIT_APPLY": "0", "TTT_SEQUENCE_GROUPS": "3"},
    {"TTT_SEQUENCE_GROUPS": "1"},
    # one CTA per sequence and apply launch: the apply side lags far behind the
    # update chain, so every update has to wait for the applies still reading
    # its bf16 copy
    {"TTT_SEQUENCE_GROUPS": "4", "TTT_APPLY_CTAS": "1"},
    {"TTT_DISABLE_GRAPHS": "1", "TTT_APPLY_CTAS": "2"},
])
def test_layer_schedules_bitwise_equal(env, tmp_path):
    """Every launch schedule of the layer (apply side on its own streams or
    inside the update launches, 1 to 4 stream groups, graphs or eager launches,
    a starved apply side) gives bit-identical outputs and final weights: each
    output tile is computed by the same code in the same order wherever it is
    launched, and the double-buffered bf16 weights are never overwritten while
    an apply still reads them."""
    import os
    import subprocess
    import sys
    cla = lib()
    here = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    ref = {}
    for i, kw in enumerate(SCHED_WORKLOADS):
        wl = dataclasses.replace(W.LM_760M, **kw)
        for j, t in enumerate(run_layer(cla, wl, *W.layer_inputs(wl))):
            ref[f"w{i}_{j}"] = t
    out = str(tmp_path / "sched.npz")
    subprocess.run([sys.executable, "-c", _SCHED_CHILD, here, out], check=True, cwd=here,
                   env=dict(os.environ, **env), timeout=600)
    got = np.load(out)
    for key, r in ref.items():
        assert np.array_equal(got[key], r), key


def test_layer_output_16_byte_aligned_matches_32():
    """An output buffer that is 16- but not 32-byte aligned takes the staged
    epilogue row path (shared-memory transpose, 16-byte stores) instead of the
    lane-per-row 32-byte stores; the results are bit-identical."""
    cla = lib()
    wl = dataclasses.replace(W.LM_760M, B=1, H=2, N=1024, d_h=256, m_h=256, chunk=256,
                             muon_steps=2, momentum_beta=0.5)
    q, k, v, eta, W1, W2, W3 = [t.to(DEV) for t in W.layer_inputs(wl)]
    rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                           momentum_beta=wl.momentum_beta)
    outs = []
    for shift in (0, 8):   # bf16 elements: 0 or 16 bytes past a 256-byte aligned base
        buf = torch.empty(q.numel() + 16, dtype=torch.bfloat16, device=DEV)
        out = buf[shift:shift + q.numel()].view(q.shape)
        assert (out.data_ptr() % 32 == 0) == (shift == 0)
        cla.ttt_layer_forward(q, k, v, eta, W1, W2, W3, wl.chunk, wl.mode, rule, out=out)
        torch.cuda.synchronize()
        assert_status_ok(cla)
        outs.append(out.float().cpu().numpy())
    assert np.array_equal(outs[0], outs[1])


HOST_CASES = [
    # two stream groups, Muon, momentum; k is the same tensor as q
    dict(wl=dict(B=2, H=2, N=2048, d_h=256, m_h=256, chunk=512, muon_steps=5,
                 momentum_beta=0.9), k_is_q=True, momentum=False, per_batch=False),
    # strided update flags, carried momentum, per-batch initial weights
    dict(wl=dict(B=1, H=2, N=1024, d_h=128, m_h=256, chunk=128, muon_steps=0,
                 momentum_beta=0.5, mode=W.STRIDED,
                 update_chunks=(1, 0, 0, 1, 0, 1, 1, 0)), k_is_q=False, momentum=True,
         per_batch=True),
]


@pytest.mark.parametrize("case", HOST_CASES)
def test_layer_host_buffers_match_device_call(case):
    """The host-buffer call (chunk copies overlapped with the kernels) returns
    exactly what the device call returns on the same inputs."""
    cla = lib()
    wl = dataclasses.replace(W.LM_760M, **case["wl"])
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wl)
    if case["k_is_q"]:
        k = q
    if case["per_batch"]:
        W1, W2, W3 = [w.unsqueeze(0).expand(wl.B, *w.shape).contiguous() for w in (W1, W2, W3)]
    B, H, d, m = wl.B, wl.H, wl.d_h, wl.m_h
    mom = torch.randn(3, B, H, m * d, generator=torch.Generator().manual_seed(3)) * 0.01
    rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                           momentum_beta=wl.momentum_beta)
    # device call
    dmom = mom.to(DEV) if case["momentum"] else None
    dk = None if case["k_is_q"] else k.to(DEV)
    dq = q.to(DEV)
    ref = cla.ttt_layer_forward(dq, dq if dk is None else dk, v.to(DEV), eta.to(DEV), W1.to(DEV),
                                W2.to(DEV), W3.to(DEV), wl.chunk, wl.mode, rule,
                                update_chunks=wl.update_chunks, momentum=dmom)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    ref = [t.cpu() for t in ref]
    # host call on page-locked copies
    hq, hv, heta = q.pin_memory(), v.pin_memory(), eta.pin_memory()
    hk = hq if case["k_is_q"] else k.pin_memory()
    hW = [w.pin_memory() for w in (W1, W2, W3)]
    hmom = mom.clone().pin_memory() if case["momentum"] else None
    got = cla.ttt_layer_forward_host(hq, hk, hv, heta, *hW, wl.chunk, wl.mode, rule,
                                     update_chunks=wl.update_chunks, momentum=hmom)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    for g_, r_ in zip(got, ref):
        assert torch.equal(g_, r_)
    if case["momentum"]:
        assert torch.equal(hmom, dmom.cpu())


def test_linattn_output_16_byte_aligned():
    """An output buffer that is 16- but not 32-byte aligned takes the
    multi-launch path instead of the one-launch kernel; both match the oracle."""
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, N=1024, chunk=256)
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=True)
    ro, rS = O.linattn_chunked_forward(f64(q), f64(k), f64(v), f64(eta), f64(S0), wl.chunk,
                                       wl.mode, wl.update_chunks)
    for shift in (0, 8):
        buf = torch.empty(q.numel() + 16, dtype=torch.bfloat16, device=DEV)
        out = buf[shift:shift + q.numel()].view(q.shape)
        o, S = cla.linattn_chunked_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV),
                                           wl.chunk, wl.mode, S0=S0.to(DEV), out=out)
        torch.cuda.synchronize()
        assert_status_ok(cla)
        assert rel_l2(f64(o), ro) <= BF16_REL_L2
        assert rel_l2(f64(S), rS) <= BF16_REL_L2

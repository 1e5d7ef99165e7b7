"""GPU parity of degenerate and boundary cases against the oracle: a strided
mask with no updating chunk, zero learning rates, a single apply-then-update
chunk, and the largest fast-weight order the library accepts (1024), for the
TTT layer ("Test-Time Training with KV Binding Is Secretly Linear Attention",
sec. 4; LaCT notes eqs (2)-(6), (10)) and for chunked linear attention
(Thm 5.2, App. H).

Where no update happens, the final fast weights (or state) are the initial
ones bit for bit: no arithmetic touches them.  Tolerances as everywhere:
max relative error <= 1e-4 for fp32, relative L2 <= 2e-2 for bf16 (3e-2 with
Muon), per output tensor.
"""
import dataclasses

import pytest
import torch

import workloads as W
from oracle import ttt_oracle as O
from tests.gpu_util import assert_status_ok, f64, lib, max_rel, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F32_MAX_REL = 1e-4
BF16 = 2e-2
BF16_MUON = 3e-2


def _layer(cla, wl, q, k, v, eta, W1, W2, W3):
    rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                           momentum_beta=wl.momentum_beta)
    res = cla.ttt_layer_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), W1.to(DEV),
                                W2.to(DEV), W3.to(DEV), wl.chunk, wl.mode, rule,
                                update_chunks=wl.update_chunks)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    return [t.cpu() for t in res]


def _oracle(wl, q, k, v, eta, W1, W2, W3):
    return O.ttt_layer_forward(f64(q), f64(k), f64(v), f64(eta), f64(W1), f64(W2), f64(W3),
                               wl.chunk, wl.mode, update_chunks=wl.update_chunks,
                               l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                               momentum_beta=wl.momentum_beta)[:4]


def _check(wl, got, ref):
    if wl.io_dtype == "f32":
        for g_, r_ in zip(got, ref):
            assert max_rel(f64(g_), r_) <= F32_MAX_REL
    else:
        tol = BF16_MUON if wl.muon_steps else BF16
        errs = [rel_l2(f64(g_), r_) for g_, r_ in zip(got, ref)]
        assert max(errs) <= tol, errs


NO_UPDATE_CASES = [
    dict(base="bf16", B=2, H=2, N=512, chunk=128, d_h=128, m_h=128, muon_steps=2,
         momentum_beta=0.9),
    dict(base="f32", B=2, H=2, N=96, chunk=16, d_h=24, m_h=40, muon_steps=1, momentum_beta=0.5),
]


def _workload(case):
    case = dict(case)
    base = W.LM_760M if case.pop("base") == "bf16" else W.TINY_F32
    return dataclasses.replace(base, **case)


@pytest.mark.parametrize("case", NO_UPDATE_CASES, ids=["bf16", "f32"])
def test_layer_strided_mask_without_updates(case):
    """Strided mask whose flags are all 0: every chunk applies the initial
    weights, and the final weights are the initial ones bit for bit."""
    cla = lib()
    wl = _workload(case)
    nc = wl.N // wl.chunk
    wl = dataclasses.replace(wl, mode=W.STRIDED, update_chunks=(0,) * nc)
    inp = W.layer_inputs(wl)
    got = _layer(cla, wl, *inp)
    for g_, w0 in zip(got[1:], inp[4:]):
        assert torch.equal(g_, w0.unsqueeze(0).expand_as(g_))
    _check(wl, got, _oracle(wl, *inp))


def test_layer_zero_learning_rates():
    """eta = 0: every gradient (and momentum, and Muon of it) is zero; each
    update only renormalises the rows."""
    cla = lib()
    wl = dataclasses.replace(W.LM_760M, B=2, H=2, N=512, chunk=128, d_h=128, m_h=128,
                             mode=W.BLOCK_CAUSAL, muon_steps=2, momentum_beta=0.9)
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wl)
    eta = torch.zeros_like(eta)
    got = _layer(cla, wl, q, k, v, eta, W1, W2, W3)
    _check(wl, got, _oracle(wl, q, k, v, eta, W1, W2, W3))


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_layer_single_apply_then_update_chunk(io):
    """One chunk, apply first: the outputs use the initial weights only; the
    final weights are one update."""
    cla = lib()
    if io == "bf16":
        wl = dataclasses.replace(W.LM_760M, B=1, H=2, N=256, chunk=256, d_h=128, m_h=128,
                                 muon_steps=3, momentum_beta=0.9)
    else:
        wl = dataclasses.replace(W.TINY_F32, B=1, H=2, N=64, chunk=64)
    inp = W.layer_inputs(wl)
    _check(wl, _layer(cla, wl, *inp), _oracle(wl, *inp))


def test_layer_bf16_largest_order():
    """d = m = 1024, the largest order accepted: Muon runs through the
    per-product Newton-Schulz launches (chunk >= d keeps the momentum full
    rank)."""
    cla = lib()
    wl = dataclasses.replace(W.LM_760M, B=1, H=1, N=2048, chunk=1024, d_h=1024, m_h=1024,
                             mode=W.BLOCK_CAUSAL, muon_steps=2, momentum_beta=0.9)
    inp = W.layer_inputs(wl)
    _check(wl, _layer(cla, wl, *inp), _oracle(wl, *inp))


def test_layer_f32_largest_order():
    """d = m = 1024 in fp32 (no tensor cores), with momentum."""
    cla = lib()
    wl = dataclasses.replace(W.TINY_F32, B=1, H=1, N=128, chunk=64, d_h=1024, m_h=1024,
                             momentum_beta=0.9)
    inp = W.layer_inputs(wl)
    _check(wl, _layer(cla, wl, *inp), _oracle(wl, *inp))


def _linattn(cla, wl, q, k, v, eta, S0):
    o, S = cla.linattn_chunked_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), wl.chunk,
                                       wl.mode, S0=S0.to(DEV), update_chunks=wl.update_chunks)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    return o.cpu(), S.cpu()


def test_linattn_without_updates_keeps_the_state():
    """A strided mask with no updating chunk, and zero learning rates under
    the block-causal mask: the state stays S0 bit for bit and every output
    is Q S0^T."""
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, N=1024, chunk=256)
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=True)
    ws = dataclasses.replace(wl, mode=W.STRIDED, update_chunks=(0, 0, 0, 0))
    wz = dataclasses.replace(wl, mode=W.BLOCK_CAUSAL)
    for wcase, e in ((ws, eta), (wz, torch.zeros_like(eta))):
        o, S = _linattn(cla, wcase, q, k, v, e, S0)
        assert torch.equal(S, S0)
        ro, rS = O.linattn_chunked_forward(f64(q), f64(k), f64(v), f64(e), f64(S0), wcase.chunk,
                                           wcase.mode, wcase.update_chunks)
        assert rel_l2(f64(o), ro) <= BF16

"""GPU parity of the layer's reduction variants and of more inner steps
against the oracle ("Test-Time Training with KV Binding Is Secretly Linear
Attention", sec. 6.1 Steps 1-2 / Variants 1-2, sec. 6.2 and App. H for the
parallel form, sec. 4.1 for inner-loop steps):

* Variant 1: only W2 updates (W1, W3 static, so phi is a static feature map),
  with L2-Normalize: the recurrent form.
* Variant 2: Variant 1 without normalisation: the parallel form (features,
  then chunked linear attention with momentum and Muon) and, on request, the
  recurrent form; both against the oracle.
* inner_steps > 1 on the full LaCT layer.

Tolerances as in test_gpu_parity: rel L2 <= 2e-2 for bf16 (3e-2 with Muon),
max relative error <= 1e-4 for fp32.  Muon cases keep chunk >= min(d, m)
(full-rank momentum).
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from oracle import ttt_oracle as O
from tests.gpu_util import assert_status_ok, f64, lib, max_rel, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
BF16 = 2e-2
BF16_MUON = 3e-2
F32 = 1e-4


def _wl(**kw):
    base = dict(B=2, H=2, muon_steps=0, momentum_beta=0.0, l2_normed_k=False)
    base.update(kw)
    return dataclasses.replace(W.LM_760M, **base)


def _gpu(cla, wl, inp, momentum=None, **rule_kw):
    q, k, v, eta, W1, W2, W3 = inp
    rule = cla.update_rule(l2norm=wl.l2norm, muon_steps=wl.muon_steps,
                           momentum_beta=wl.momentum_beta, **rule_kw)
    res = cla.ttt_layer_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), W1.to(DEV),
                                W2.to(DEV), W3.to(DEV), wl.chunk, wl.mode, rule,
                                update_chunks=wl.update_chunks, momentum=momentum)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    return [f64(t) for t in res]


def _oracle(wl, inp, momentum=None, **kw):
    return O.ttt_layer_forward(*[f64(t) for t in inp], wl.chunk, wl.mode,
                               update_chunks=wl.update_chunks, l2norm=wl.l2norm,
                               muon_steps=wl.muon_steps, momentum_beta=wl.momentum_beta,
                               momentum=momentum, **kw)


def _check(got, ref, tol, fp32=False):
    if fp32:
        errs = [max_rel(g_, r_) for g_, r_ in zip(got, ref[:4])]
    else:
        errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref[:4])]
    assert max(errs) <= tol, errs


V1_CASES = [
    # half-panel Newton-Schulz kernel on W2 alone
    dict(mode=W.APPLY_THEN_UPDATE, chunk=384, N=768, d_h=384, m_h=384, muon_steps=5,
         momentum_beta=0.9, l2_normed_k=True),
    # tile-cluster kernel on W2 alone
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=512, d_h=192, m_h=192, muon_steps=3,
         momentum_beta=0.9),
    # non-square W2: the per-product Newton-Schulz launches on one group
    dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=768, d_h=128, m_h=256, muon_steps=2),
    # no Muon: the normalisation launch on W2 alone
    dict(mode=W.APPLY_THEN_UPDATE, chunk=128, N=512, d_h=128, m_h=128, momentum_beta=0.5),
    dict(mode=W.STRIDED, chunk=128, N=1024, d_h=128, m_h=128, muon_steps=2,
         update_chunks=(1, 0, 1, 1, 0, 0, 0, 0)),
]


@pytest.mark.parametrize("case", V1_CASES)
def test_variant1_last_layer_only_recurrent(case):
    cla = lib()
    wl = _wl(**case)
    inp = W.layer_inputs(wl)
    got = _gpu(cla, wl, inp, last_layer_only=True)
    ref = _oracle(wl, inp, last_layer_only=True)
    _check(got, ref, BF16_MUON if wl.muon_steps else BF16)
    # W1 and W3 stay at their initial values
    for i, w in ((1, inp[4]), (3, inp[6])):
        assert np.array_equal(got[i], np.broadcast_to(f64(w), got[i].shape))


def test_variant1_fp32():
    cla = lib()
    wl = dataclasses.replace(W.TINY_F32, B=2, H=2, N=96, d_h=24, m_h=40, chunk=16,
                             muon_steps=2, momentum_beta=0.9)
    inp = W.layer_inputs(wl)
    _check(_gpu(cla, wl, inp, last_layer_only=True), _oracle(wl, inp, last_layer_only=True),
           F32, fp32=True)


V2_CASES = [
    # one-launch linear attention (d_v = d = 128, d_k = m = 128), momentum
    dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=1024, d_h=128, m_h=128, momentum_beta=0.9),
    # Muon of the momentum over 384 x 384 matrices (multi-launch flow)
    dict(mode=W.APPLY_THEN_UPDATE, chunk=384, N=1536, d_h=384, m_h=384, muon_steps=5,
         momentum_beta=0.9, l2_normed_k=True),
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=1024, d_h=128, m_h=256, muon_steps=2,
         momentum_beta=0.5),
    dict(mode=W.BIDIRECTIONAL, chunk=512, N=512, d_h=128, m_h=128, muon_steps=1),
    dict(mode=W.STRIDED, chunk=256, N=2048, d_h=128, m_h=192, momentum_beta=0.9,
         update_chunks=(1, 1, 0, 1, 0, 0, 1, 0)),
]


@pytest.mark.parametrize("case", V2_CASES)
@pytest.mark.parametrize("form", ["parallel", "recurrent"])
def test_variant2_no_norm_both_forms(case, form):
    cla = lib()
    wl = _wl(l2norm=False, **case)
    inp = W.layer_inputs(wl)
    f = cla.FORM_PARALLEL if form == "parallel" else cla.FORM_RECURRENT
    got = _gpu(cla, wl, inp, last_layer_only=True, form=f)
    ref = _oracle(wl, inp, last_layer_only=True)
    _check(got, ref, BF16_MUON if wl.muon_steps else BF16)


def test_variant2_parallel_momentum_carry():
    """The parallel form reads and writes the W2 momentum (M2 of the
    momentum buffer) and leaves M1, M3 alone; a sequence split in two calls
    matches the oracle's single pass."""
    cla = lib()
    wl = _wl(l2norm=False, mode=W.APPLY_THEN_UPDATE, chunk=256, N=1024, d_h=128, m_h=128,
             muon_steps=2, momentum_beta=0.9)
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wl)
    ref = _oracle(wl, (q, k, v, eta, W1, W2, W3), last_layer_only=True)
    BH, dm = wl.B * wl.H, wl.d_h * wl.m_h
    mom = torch.zeros(3 * BH * dm, device=DEV)
    mom[:BH * dm] = 7.0        # M1 and M3 are not touched
    mom[2 * BH * dm:] = -3.0
    half = wl.N // 2
    wh = dataclasses.replace(wl, N=half)
    a = [t[..., :half, :].contiguous() if t.dim() == 4 else t[..., :half].contiguous()
         for t in (q, k, v, eta)]
    r1 = _gpu(cla, wh, (*a, W1, W2, W3), momentum=mom, last_layer_only=True)
    b = [t[..., half:, :].contiguous() if t.dim() == 4 else t[..., half:].contiguous()
         for t in (q, k, v, eta)]
    W1b = torch.from_numpy(r1[1]).float()
    W2b = torch.from_numpy(r1[2]).float()
    W3b = torch.from_numpy(r1[3]).float()
    r2 = _gpu(cla, wh, (*b, W1b, W2b, W3b), momentum=mom, last_layer_only=True)
    out = np.concatenate([r1[0], r2[0]], axis=2)
    errs = [rel_l2(out, ref[0]), rel_l2(r2[2], ref[2])]
    assert max(errs) <= BF16_MUON, errs
    m = mom.view(3, wl.B, wl.H, dm).cpu().double().numpy()
    assert rel_l2(m[1].reshape(ref[4][1].shape), ref[4][1]) <= BF16_MUON
    assert np.all(m[0] == 7.0) and np.all(m[2] == -3.0)


def test_variant2_parallel_fp32():
    cla = lib()
    wl = dataclasses.replace(W.TINY_F32, B=2, H=2, N=96, d_h=24, m_h=40, chunk=32,
                             l2norm=False, muon_steps=2, momentum_beta=0.9,
                             mode=W.BLOCK_CAUSAL)
    inp = W.layer_inputs(wl)
    got = _gpu(cla, wl, inp, last_layer_only=True, form=cla.FORM_PARALLEL)
    _check(got, _oracle(wl, inp, last_layer_only=True), F32, fp32=True)


def test_variant2_parallel_host_buffers_match_device_call():
    cla = lib()
    wl = _wl(l2norm=False, mode=W.BLOCK_CAUSAL, chunk=256, N=1024, d_h=128, m_h=128,
             muon_steps=2, momentum_beta=0.9)
    q, k, v, eta, W1, W2, W3 = W.layer_inputs(wl)
    rule = cla.update_rule(l2norm=False, muon_steps=2, momentum_beta=0.9, last_layer_only=True)
    ref = cla.ttt_layer_forward(q.to(DEV), k.to(DEV), v.to(DEV), eta.to(DEV), W1.to(DEV),
                                W2.to(DEV), W3.to(DEV), wl.chunk, wl.mode, rule)
    torch.cuda.synchronize()
    ref = [t.cpu() for t in ref]
    got = cla.ttt_layer_forward_host(q.pin_memory(), k.pin_memory(), v.pin_memory(),
                                     eta.pin_memory(), W1.pin_memory(), W2.pin_memory(),
                                     W3.pin_memory(), wl.chunk, wl.mode, rule)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    for g_, r_ in zip(got, ref):
        assert torch.equal(g_, r_)


INNER_CASES = [
    dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=768, d_h=256, m_h=256, muon_steps=2,
         momentum_beta=0.9, inner=2),
    dict(mode=W.BLOCK_CAUSAL, chunk=128, N=512, d_h=128, m_h=192, momentum_beta=0.5, inner=3),
    dict(mode=W.STRIDED, chunk=128, N=768, d_h=128, m_h=128, muon_steps=1, inner=2,
         update_chunks=(1, 0, 0, 1, 1, 0)),
]


@pytest.mark.parametrize("case", INNER_CASES)
def test_inner_steps(case):
    cla = lib()
    case = dict(case)
    inner = case.pop("inner")
    wl = _wl(**case)
    inp = W.layer_inputs(wl)
    got = _gpu(cla, wl, inp, inner_steps=inner)
    ref = _oracle(wl, inp, inner_steps=inner)
    _check(got, ref, BF16_MUON if wl.muon_steps else BF16)


def test_inner_steps_fp32_and_last_layer_only():
    cla = lib()
    wl = dataclasses.replace(W.TINY_F32, B=1, H=2, N=64, d_h=16, m_h=24, chunk=16,
                             muon_steps=2, momentum_beta=0.9)
    inp = W.layer_inputs(wl)
    _check(_gpu(cla, wl, inp, inner_steps=2), _oracle(wl, inp, inner_steps=2), F32, fp32=True)
    _check(_gpu(cla, wl, inp, inner_steps=3, last_layer_only=True),
           _oracle(wl, inp, inner_steps=3, last_layer_only=True), F32, fp32=True)


def test_parallel_form_is_refused_where_not_exact():
    cla = lib()
    wl = _wl(mode=W.APPLY_THEN_UPDATE, chunk=128, N=256, d_h=128, m_h=128)
    inp = [t.to(DEV) for t in W.layer_inputs(wl)]
    for kw in (dict(l2norm=True, last_layer_only=True), dict(l2norm=False),
               dict(l2norm=False, last_layer_only=True, inner_steps=2)):
        rule = cla.update_rule(form=cla.FORM_PARALLEL, **kw)
        with pytest.raises(cla.TTTError) as e:
            cla.ttt_layer_forward(*inp, wl.chunk, wl.mode, rule)
        assert e.value.code == -8   # TTT_ERR_ARG

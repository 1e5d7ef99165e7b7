"""GPU parity of chunked linear attention with momentum, per-chunk learning
rates and Muon of the momentum (linattn_chunked_forward_rule) against the
oracle's ``linattn_momentum_forward`` ("Test-Time Training with KV Binding Is
Secretly Linear Attention", Thm 5.3, App. E.3, App. H; sec. 6.1 Variants
3-5: a single linear fast weight with Muon, with or without momentum, with a
per-token or a constant learning rate).

Tolerances: relative L2 <= 2e-2 for bf16 (3e-2 with Muon), max relative
error <= 1e-4 for fp32, per output tensor (out, S_final, M_final).
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


def _rule_inputs(wl, seed=5, momentum=True, rate=True, state=True):
    """alpha in (0.5, 0.95), lr in (0.5, 1.5) per (batch, head, chunk); an
    initial state and momentum ~ N(0, 1/d_k)."""
    g = torch.Generator().manual_seed(seed)
    n = wl.N // wl.chunk
    alpha = (0.5 + 0.45 * torch.rand((wl.B, wl.H, n), generator=g)) if momentum else None
    lr = (0.5 + torch.rand((wl.B, wl.H, n), generator=g)) if rate else None
    std = 1.0 / wl.d_k ** 0.5
    M0 = torch.randn((wl.B, wl.H, wl.d_v, wl.d_k), generator=g) * std if state else None
    return alpha, lr, M0


def _run(cla, wl, q, k, v, eta, S0, alpha, lr, M0, muon_steps=0, out=None):
    d = lambda t: None if t is None else t.to(DEV).contiguous()
    o, S, M = cla.linattn_chunked_forward_rule(
        d(q), d(k), d(v), d(eta), wl.chunk, wl.mode, S0=d(S0), update_chunks=wl.update_chunks,
        alpha=d(alpha), lr=d(lr), M0=d(M0), M_final=True, muon_steps=muon_steps, out=out)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    return f64(o), f64(S), f64(M)


def _oracle(wl, q, k, v, eta, S0, alpha, lr, M0, muon_steps=0):
    n = lambda t: None if t is None else f64(t)
    return O.linattn_momentum_forward(f64(q), f64(k), f64(v), f64(eta), n(S0), wl.chunk, wl.mode,
                                      wl.update_chunks, n(alpha), n(lr), n(M0),
                                      muon_steps=muon_steps)


# one-launch kernel shapes (d_v = 128, d_k 64 / 128) and multi-launch shapes
MOM_CASES = [
    dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=1024),
    dict(mode=W.BLOCK_CAUSAL, chunk=512, N=2048, d_k=64),
    dict(mode=W.BIDIRECTIONAL, chunk=1024, N=1024),
    dict(mode=W.STRIDED, chunk=128, N=1024, update_chunks=(1, 0, 1, 1, 0, 0, 1, 0)),
    dict(mode=W.BLOCK_CAUSAL, chunk=256, N=768, d_k=64, d_v=192),
    dict(mode=W.STRIDED, chunk=128, N=768, d_k=128, d_v=64, update_chunks=(0, 1, 1, 0, 1, 0)),
    # 32 chunks: the prefix items' partial slices cross four ring stages
    dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=8192),
    dict(mode=W.STRIDED, chunk=256, N=8192,
         update_chunks=tuple(int(c % 4 != 3 and c > 1) for c in range(32))),
]


@pytest.mark.parametrize("case", MOM_CASES)
@pytest.mark.parametrize("state", [False, True])
def test_momentum_and_rates_bf16(case, state):
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, **case)
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=state)
    alpha, lr, M0 = _rule_inputs(wl, state=state)
    got = _run(cla, wl, q, k, v, eta, S0, alpha, lr, M0)
    ref = _oracle(wl, q, k, v, eta, S0, alpha, lr, M0)
    errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref)]
    assert max(errs) <= BF16, errs


def test_momentum_multi_launch_path_matches_one_launch():
    """An output buffer that is 16- but not 32-byte aligned takes the
    multi-launch path; both paths match the oracle."""
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, N=1024, chunk=256)
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=True)
    alpha, lr, M0 = _rule_inputs(wl)
    ref = _oracle(wl, q, k, v, eta, S0, alpha, lr, M0)
    for shift in (0, 8):
        buf = torch.empty(q.numel() + 16, dtype=torch.bfloat16, device=DEV)
        out = buf[shift:shift + q.numel()].view(q.shape)
        got = _run(cla, wl, q, k, v, eta, S0, alpha, lr, M0, out=out)
        errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref)]
        assert max(errs) <= BF16, (shift, errs)


@pytest.mark.parametrize("mode", [W.APPLY_THEN_UPDATE, W.BLOCK_CAUSAL])
def test_momentum_and_rates_fp32(mode):
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=3, N=200, d_k=24, d_v=40, chunk=40, mode=mode,
                             io_dtype="f32")
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=True)
    alpha, lr, M0 = _rule_inputs(wl)
    got = _run(cla, wl, q, k, v, eta, S0, alpha, lr, M0)
    ref = _oracle(wl, q, k, v, eta, S0, alpha, lr, M0)
    for g_, r_ in zip(got, ref):
        assert max_rel(g_, r_) <= F32


# Variants 3-5 of the reduction: a single linear fast weight with Muon
# (chunk >= d, so every momentum has full rank)
MUON_CASES = [
    # Variant 3: Muon + momentum + per-token eta
    dict(case=dict(mode=W.APPLY_THEN_UPDATE, chunk=256, N=1024), momentum=True, steps=5),
    dict(case=dict(mode=W.BLOCK_CAUSAL, chunk=256, N=1024, d_k=64, d_v=64), momentum=True,
         steps=3),
    # Variant 5: Muon, no momentum
    dict(case=dict(mode=W.BLOCK_CAUSAL, chunk=256, N=1024), momentum=False, steps=5),
    dict(case=dict(mode=W.STRIDED, chunk=256, N=2048, update_chunks=(1, 1, 0, 1, 0, 0, 1, 0)),
         momentum=True, steps=2),
]


@pytest.mark.parametrize("mc", MUON_CASES)
def test_muon_of_momentum_bf16(mc):
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, **mc["case"])
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=True)
    alpha, lr, M0 = _rule_inputs(wl, momentum=mc["momentum"], state=mc["momentum"])
    got = _run(cla, wl, q, k, v, eta, S0, alpha, lr, M0, muon_steps=mc["steps"])
    ref = _oracle(wl, q, k, v, eta, S0, alpha, lr, M0, muon_steps=mc["steps"])
    errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref)]
    assert max(errs) <= BF16_MUON, errs


def test_muon_constant_rate_variant4():
    """Variant 4: a constant learning rate in place of the per-token one."""
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=1, H=4, N=1024, chunk=256, mode=W.APPLY_THEN_UPDATE)
    q, k, v, _, S0 = W.linattn_inputs(wl, with_state=True)
    eta = torch.full((wl.B, wl.H, wl.N), 1.0 / wl.chunk)
    alpha = torch.full((wl.B, wl.H, wl.N // wl.chunk), 0.9)
    got = _run(cla, wl, q, k, v, eta, S0, alpha, None, None, muon_steps=5)
    ref = _oracle(wl, q, k, v, eta, S0, alpha, None, None, muon_steps=5)
    errs = [rel_l2(g_, r_) for g_, r_ in zip(got, ref)]
    assert max(errs) <= BF16_MUON, errs


def test_muon_fp32():
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, N=240, d_k=24, d_v=40, chunk=48,
                             mode=W.BLOCK_CAUSAL, io_dtype="f32")
    q, k, v, eta, S0 = W.linattn_inputs(wl, with_state=True)
    alpha, lr, M0 = _rule_inputs(wl)
    got = _run(cla, wl, q, k, v, eta, S0, alpha, lr, M0, muon_steps=3)
    ref = _oracle(wl, q, k, v, eta, S0, alpha, lr, M0, muon_steps=3)
    for g_, r_ in zip(got, ref):
        assert max_rel(g_, r_) <= F32


def test_no_rule_is_bitwise_the_plain_call():
    """No momentum, unit rates and no Muon compute exactly what
    linattn_chunked_forward computes."""
    cla = lib()
    wl = dataclasses.replace(W.LINATTN_C2, B=2, H=2, N=1024, chunk=256)
    q, k, v, eta, S0 = [t.to(DEV) for t in W.linattn_inputs(wl, with_state=True)]
    o1, S1 = cla.linattn_chunked_forward(q, k, v, eta, wl.chunk, wl.mode, S0=S0)
    o2, S2, M2 = cla.linattn_chunked_forward_rule(q, k, v, eta, wl.chunk, wl.mode, S0=S0)
    torch.cuda.synchronize()
    assert_status_ok(cla)
    assert M2 is None
    assert torch.equal(o1, o2) and torch.equal(S1, S2)

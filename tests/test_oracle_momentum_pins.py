"""Pins of the oracle's chunked linear attention with momentum, a per-chunk
learning rate and Muon of the momentum (``linattn_momentum_forward``) against
what "Test-Time Training with KV Binding Is Secretly Linear Attention" fixes
independently of the recurrence:

* App. H (H.1, H.2): the parallel form.  With per-chunk learning rates lr
  and momentum factors alpha the state after chunk t is
  S0 + sum_{i<=t} C_ti (eta*V_i)^T K_i with the accumulation mask
  C_ti = sum_{j=i}^{t} lr_j prod_{s=i+1}^{j} alpha_s (per-token eta folded
  into the values), evaluated here token by token as a brute-force sum over
  visible keys; an initial momentum M0 adds
  sum_{j<=t} lr_j prod_{s<=j} alpha_s M0 (Thm 5.3's unrolling with
  M_{-1} = M0).
* App. E.3: with Muon, S_{t+1} = S0 + sum_j lr_j Muon(M_j), M_j the unrolled
  momentum; Muon evaluated from the singular value decomposition of M_j.
* Thm 5.2 / the plain chunk form: alpha = 0, lr = 1 is the existing chunked
  linear attention.
* The TTT view: a single linear fast weight updated by W <- W - Muon(M),
  M <- beta M + g (the layer oracle's own update code) gives the same
  outputs for constant alpha = beta.
"""
import numpy as np
import pytest

from oracle import ttt_oracle as O

RNG = np.random.default_rng(1234)


def _inputs(B=1, H=2, N=48, dk=5, dv=4, chunk=8, state=True):
    q = RNG.normal(size=(B, H, N, dk))
    k = RNG.normal(size=(B, H, N, dk))
    v = RNG.normal(size=(B, H, N, dv))
    eta = RNG.uniform(0.1, 1.0, size=(B, H, N))
    n = N // chunk
    alpha = RNG.uniform(0.2, 0.95, size=(B, H, n))
    lr = RNG.uniform(0.3, 1.5, size=(B, H, n))
    S0 = RNG.normal(size=(B, H, dv, dk)) if state else None
    M0 = RNG.normal(size=(B, H, dv, dk)) * 0.3 if state else None
    return q, k, v, eta, alpha, lr, S0, M0


def _visible(mode, t, upd):
    """Updating chunks whose update a query of chunk t sees."""
    return [j for j in upd if (j < t if mode == O.APPLY_THEN_UPDATE else j <= t)]


def _closed_form(q, k, v, eta, alpha, lr, S0, M0, chunk, mode, flags):
    """App. H token by token: o_p = S0 q_p + (momentum carry-in) + sum over
    visible keys r of C_{t, chunk(r)} eta_r (q_p . k_r) v_r."""
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    n = N // chunk
    upd = [c for c in range(n) if flags[c]]
    out = np.zeros((B, H, N, dv))
    for b in range(B):
        for h in range(H):
            a, l = alpha[b, h], lr[b, h]

            def decay(i, j):   # prod of alpha_s over updating s in (i, j]
                return np.prod([a[s] for s in upd if i < s <= j])

            for p in range(N):
                t = p // chunk
                T = _visible(mode, t, upd)
                o = S0[b, h] @ q[b, h, p] if S0 is not None else np.zeros(dv)
                if M0 is not None:
                    carry = sum(l[j] * decay(-1, j) for j in T)
                    o = o + carry * (M0[b, h] @ q[b, h, p])
                for r in range(N):
                    i = r // chunk
                    if i not in upd or not T or i > max(T):
                        continue
                    C = sum(l[j] * decay(i, j) for j in T if j >= i)
                    o = o + C * eta[b, h, r] * (q[b, h, p] @ k[b, h, r]) * v[b, h, r]
                out[b, h, p] = o
    return out


CASES = [
    (O.APPLY_THEN_UPDATE, None),
    (O.BLOCK_CAUSAL, None),
    (O.STRIDED, (1, 0, 1, 1, 0, 1)),
]


@pytest.mark.parametrize("mode,flags", CASES)
@pytest.mark.parametrize("state", [False, True])
def test_momentum_mask_closed_form(mode, flags, state):
    q, k, v, eta, alpha, lr, S0, M0 = _inputs(state=state)
    chunk = 8
    n = q.shape[2] // chunk
    fl = [True] * n if flags is None else [bool(x) for x in flags]
    got, Sf, Mf = O.linattn_momentum_forward(q, k, v, eta, S0, chunk, mode, flags, alpha, lr, M0)
    ref = _closed_form(q, k, v, eta, alpha, lr, S0, M0, chunk, mode, fl)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)
    # the final state is what a query after the last chunk would read
    upd = [c for c in range(n) if fl[c]]
    qe = q[:, :, :1]
    last = np.einsum("bhij,bhj->bhi", Sf, qe[:, :, 0])
    probe = _closed_form(np.concatenate([q, np.repeat(qe, chunk, axis=2)], axis=2),
                         np.concatenate([k, np.zeros_like(k[:, :, :chunk])], axis=2),
                         np.concatenate([v, np.zeros_like(v[:, :, :chunk])], axis=2),
                         np.concatenate([eta, np.zeros_like(eta[:, :, :chunk])], axis=2),
                         np.concatenate([alpha, np.zeros_like(alpha[:, :, :1])], axis=2),
                         np.concatenate([lr, np.zeros_like(lr[:, :, :1])], axis=2),
                         S0, M0, chunk, O.BLOCK_CAUSAL, fl + [False])
    np.testing.assert_allclose(last, probe[:, :, -1], rtol=1e-10, atol=1e-10)
    assert upd   # every case updates somewhere


def test_bidirectional_is_one_scaled_update():
    q, k, v, eta, alpha, lr, S0, M0 = _inputs(N=16, chunk=16)
    got, Sf, Mf = O.linattn_momentum_forward(q, k, v, eta, S0, 16, O.BIDIRECTIONAL, None,
                                             alpha, lr, M0)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            G = (eta[b, h, :, None] * v[b, h]).T @ k[b, h]
            M = alpha[b, h, 0] * M0[b, h] + G
            S = S0[b, h] + lr[b, h, 0] * M
            np.testing.assert_allclose(got[b, h], q[b, h] @ S.T, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(Mf[b, h], M, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", [O.APPLY_THEN_UPDATE, O.BLOCK_CAUSAL])
def test_no_momentum_unit_rate_is_plain_linear_attention(mode):
    q, k, v, eta, _, _, S0, _ = _inputs()
    got, Sf, _ = O.linattn_momentum_forward(q, k, v, eta, S0, 8, mode)
    ref, rS = O.linattn_chunked_forward(q, k, v, eta, S0, 8, mode)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Sf, rS, rtol=1e-12, atol=1e-12)


def _muon_svd(M, steps, coef):
    """Muon of M from its SVD: X = M / (|M|_F + eps) has singular values
    sigma / (|M|_F + eps); every Newton-Schulz step maps a singular value x to
    a x + b x^3 + c x^5 and keeps the singular vectors."""
    a, b, c = coef
    U, sig, Vt = np.linalg.svd(M, full_matrices=False)
    x = sig / (np.linalg.norm(M) + O.NS_EPS)
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return (U * x) @ Vt


@pytest.mark.parametrize("mode,flags", CASES)
def test_muon_of_momentum_closed_form(mode, flags):
    """App. E.3: S_{t+1} = S0 + sum_j lr_j Muon(M_j) with the unrolled
    momentum M_j = prod alpha M0 + sum_{i<=j} beta_i^j G_i."""
    q, k, v, eta, alpha, lr, S0, M0 = _inputs(dk=6, dv=4)
    chunk, steps = 8, 3
    n = q.shape[2] // chunk
    fl = [True] * n if flags is None else [bool(x) for x in flags]
    got, Sf, Mf = O.linattn_momentum_forward(q, k, v, eta, S0, chunk, mode, flags, alpha, lr, M0,
                                             muon_steps=steps)
    upd = [c for c in range(n) if fl[c]]
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            a = alpha[b, h]
            G = {i: (eta[b, h, i * chunk:(i + 1) * chunk, None] *
                     v[b, h, i * chunk:(i + 1) * chunk]).T @ k[b, h, i * chunk:(i + 1) * chunk]
                 for i in upd}
            Mj = {}
            for j in upd:
                m = np.prod([a[s] for s in upd if s <= j]) * M0[b, h]
                for i in upd:
                    if i <= j:
                        m = m + np.prod([a[s] for s in upd if i < s <= j]) * G[i]
                Mj[j] = m
            for t in range(n):
                T = _visible(mode, t, upd)
                S = S0[b, h] + sum((lr[b, h, j] * _muon_svd(Mj[j], steps, O.MUON_COEF)
                                    for j in T), np.zeros_like(S0[b, h]))
                np.testing.assert_allclose(got[b, h, t * chunk:(t + 1) * chunk],
                                           q[b, h, t * chunk:(t + 1) * chunk] @ S.T,
                                           rtol=1e-9, atol=1e-9)
            np.testing.assert_allclose(Mf[b, h], Mj[upd[-1]], rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("steps", [0, 2])
def test_constant_momentum_matches_linear_fast_weight_scan(steps):
    """The TTT view: W <- W - U(M), M <- beta M + g with g = -(eta V)^T K
    (the chunk-scan code of the layer oracle) equals the linear-attention
    form with alpha = beta, lr = 1 (Muon is odd: Muon(-M) = -Muon(M))."""
    q, k, v, eta, _, _, S0, _ = _inputs(B=2, H=1, dk=5, dv=5)
    beta = 0.7
    n = q.shape[2] // 8
    for mode in (O.APPLY_THEN_UPDATE, O.BLOCK_CAUSAL):
        ref, Wf = O.ttt_linear_forward(q, k, v, eta, S0, 8, mode, l2norm=False,
                                       muon_steps=steps, momentum_beta=beta)
        got, Sf, _ = O.linattn_momentum_forward(q, k, v, eta, S0, 8, mode,
                                                alpha=np.full((2, 1, n), beta),
                                                muon_steps=steps)
        np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(Sf, Wf, rtol=1e-10, atol=1e-10)


def test_split_call_carries_state_and_momentum():
    q, k, v, eta, alpha, lr, S0, M0 = _inputs()
    full = O.linattn_momentum_forward(q, k, v, eta, S0, 8, O.APPLY_THEN_UPDATE, None, alpha, lr,
                                      M0, muon_steps=2)
    h = 24
    a = O.linattn_momentum_forward(q[:, :, :h], k[:, :, :h], v[:, :, :h], eta[:, :, :h], S0, 8,
                                   O.APPLY_THEN_UPDATE, None, alpha[..., :3], lr[..., :3], M0,
                                   muon_steps=2)
    b = O.linattn_momentum_forward(q[:, :, h:], k[:, :, h:], v[:, :, h:], eta[:, :, h:], a[1], 8,
                                   O.APPLY_THEN_UPDATE, None, alpha[..., 3:], lr[..., 3:], a[2],
                                   muon_steps=2)
    np.testing.assert_allclose(np.concatenate([a[0], b[0]], axis=2), full[0], rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(b[1], full[1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b[2], full[2], rtol=1e-12, atol=1e-12)

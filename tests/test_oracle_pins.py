"""Pins of the fp64 oracle to things other than itself.

Each test checks an oracle function against what the pages and the
mathematics fix: finite differences, brute-force element loops on tiny
inputs, closed forms (Thm 5.2 / 5.3, App. H of "Test-Time Training with KV
Binding Is Secretly Linear Attention"; the causal and full-sequence linear
attention of "From Linear Attention to Test-Time Training"), SVD of the
Newton-Schulz iterate, and invariants of the row normalisation.
"""
import itertools

import numpy as np
import pytest

from oracle import ttt_oracle as O

RNG = np.random.default_rng(1234)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ---------------------------------------------------------------------------
# SiLU pieces: special values and identities, derivative by central differences

def test_silu_identities():
    x = np.linspace(-12, 12, 97)
    assert O.silu(np.array(0.0)) == 0.0
    assert O.sigmoid(np.array(0.0)) == 0.5
    # silu(-x) = -x sigmoid(-x) = -x (1 - sigmoid(x)) = silu(x) - x
    np.testing.assert_allclose(O.silu(-x), O.silu(x) - x, atol=1e-14)
    # silu(x) -> x for large x, -> 0 for very negative x
    assert abs(O.silu(np.array(40.0)) - 40.0) < 1e-12
    assert abs(O.silu(np.array(-40.0))) < 1e-12
    assert O.silu_prime(np.array(0.0)) == 0.5


def test_silu_prime_finite_difference():
    x = np.linspace(-8, 8, 161)
    h = 1e-6
    fd = (O.silu(x + h) - O.silu(x - h)) / (2 * h)
    np.testing.assert_allclose(O.silu_prime(x), fd, rtol=0, atol=1e-9)


# ---------------------------------------------------------------------------
# eq (3): the SwiGLU apply against an element-by-element loop

def brute_swiglu(W1, W2, W3, x):
    d = x.shape[0]
    m = W1.shape[0]
    hidden = []
    for j in range(m):
        a = sum(W1[j, l] * x[l] for l in range(d))
        b = sum(W3[j, l] * x[l] for l in range(d))
        hidden.append(a / (1.0 + np.exp(-a)) * b)
    return np.array([sum(W2[i, j] * hidden[j] for j in range(m)) for i in range(d)])


@pytest.mark.parametrize("d,m", [(3, 5), (4, 4), (6, 2)])
def test_swiglu_apply_brute_force(d, m):
    W1, W3, W2 = rand(m, d), rand(m, d), rand(d, m)
    X = rand(4, d)
    F = O.swiglu_apply(W1, W2, W3, X)
    for r in range(X.shape[0]):
        np.testing.assert_allclose(F[r], brute_swiglu(W1, W2, W3, X[r]), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# eq (2) + (4): hand-derived gradient against central finite differences

def fd_grad(fn, W, h=1e-6):
    g = np.zeros_like(W)
    for idx in itertools.product(*[range(s) for s in W.shape]):
        Wp = W.copy(); Wp[idx] += h
        Wm = W.copy(); Wm[idx] -= h
        g[idx] = (fn(Wp) - fn(Wm)) / (2 * h)
    return g


def brute_loss(W1, W2, W3, K, V, eta):
    return sum(eta[i] * -float(brute_swiglu(W1, W2, W3, K[i]) @ V[i]) for i in range(K.shape[0]))


@pytest.mark.parametrize("d,m,b", [(3, 4, 2), (5, 3, 5), (8, 8, 3), (4, 7, 4)])
def test_swiglu_gradients_finite_difference(d, m, b):
    W1, W3, W2 = rand(m, d), rand(m, d), rand(d, m)
    K, V = rand(b, d), rand(b, d)
    eta = np.abs(rand(b)) + 0.1
    g1, g2, g3 = O.swiglu_chunk_gradients(W1, W2, W3, K, V, eta)
    # the loss itself against the element loop
    assert abs(O.dot_product_loss(W1, W2, W3, K, V, eta) - brute_loss(W1, W2, W3, K, V, eta)) < 1e-10
    f1 = fd_grad(lambda W: O.dot_product_loss(W, W2, W3, K, V, eta), W1)
    f2 = fd_grad(lambda W: O.dot_product_loss(W1, W, W3, K, V, eta), W2)
    f3 = fd_grad(lambda W: O.dot_product_loss(W1, W2, W, K, V, eta), W3)
    for g, f in ((g1, f1), (g2, f2), (g3, f3)):
        assert np.linalg.norm(g - f) <= 1e-7 * max(np.linalg.norm(f), 1e-12)


def test_linear_gradient_finite_difference():
    W, K, V = rand(3, 4), rand(5, 4), rand(5, 3)
    eta = rand(5)

    def loss(W_):
        return float(np.sum(eta * -np.sum((K @ W_.T) * V, axis=1)))

    np.testing.assert_allclose(O.linear_chunk_gradient(W, K, V, eta), fd_grad(loss, W), atol=1e-8)


def test_gradient_ascent_flips_sign():
    # eta -> -eta flips every gradient: the gradient-ascent variant
    d, m, b = 4, 6, 5
    W1, W3, W2 = rand(m, d), rand(m, d), rand(d, m)
    K, V, eta = rand(b, d), rand(b, d), rand(b)
    gp = O.swiglu_chunk_gradients(W1, W2, W3, K, V, eta)
    gm = O.swiglu_chunk_gradients(W1, W2, W3, K, V, -eta)
    for a, b_ in zip(gp, gm):
        np.testing.assert_allclose(a, -b_, atol=1e-14)


# ---------------------------------------------------------------------------
# eq (6): Newton-Schulz equals the scalar polynomial on the singular values

def ns_by_svd(G, steps, coef, eps=O.NS_EPS):
    a, b, c = coef
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    s = s / (np.linalg.norm(G) + eps)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return (U * s) @ Vt


@pytest.mark.parametrize("shape", [(6, 6), (4, 9), (9, 4), (16, 16)])
@pytest.mark.parametrize("steps", [0, 1, 3, 5])
@pytest.mark.parametrize("coef", [O.MUON_COEF, (1.5, -0.5, 0.0)])
def test_newton_schulz_matches_svd(shape, steps, coef):
    G = rand(*shape)
    np.testing.assert_allclose(O.newton_schulz(G, steps, coef), ns_by_svd(G, steps, coef),
                               rtol=0, atol=1e-10)


def test_newton_schulz_orthogonalises():
    # "sets all singular values to 1": the cubic iteration converges to U V^T
    G = rand(12, 20)
    X = O.newton_schulz(G, 40, (1.5, -0.5, 0.0))
    U, _, Vt = np.linalg.svd(G, full_matrices=False)
    np.testing.assert_allclose(X, U @ Vt, atol=1e-8)
    np.testing.assert_allclose(X @ X.T, np.eye(12), atol=1e-8)
    # the quintic Muon iteration leaves singular values near 1 after 5 steps
    Y = O.newton_schulz(rand(32, 32), 5, O.MUON_COEF)
    sv = np.linalg.svd(Y, compute_uv=False)
    assert sv.max() < 1.25 and np.median(sv) > 0.6


def test_newton_schulz_odd_and_scale_free():
    G = rand(7, 11)
    np.testing.assert_allclose(O.newton_schulz(-G, 5), -O.newton_schulz(G, 5), atol=1e-12)
    np.testing.assert_allclose(O.newton_schulz(37.0 * G, 5), O.newton_schulz(G, 5), atol=1e-6)


# ---------------------------------------------------------------------------
# eq (5): L2-Normalize along the input dimension

def test_l2_normalize_rows_invariants():
    W = rand(9, 5, scale=3.0)
    Nw = O.l2_normalize_rows(W)
    np.testing.assert_allclose(np.linalg.norm(Nw, axis=1), 1.0, atol=1e-14)
    np.testing.assert_allclose(O.l2_normalize_rows(4.5 * W), Nw, atol=1e-14)
    # each row keeps its direction
    cos = np.sum(Nw * W, axis=1) / np.linalg.norm(W, axis=1)
    np.testing.assert_allclose(cos, 1.0, atol=1e-14)
    Z = np.zeros((2, 3))
    assert np.all(O.l2_normalize_rows(Z) == 0)


# ---------------------------------------------------------------------------
# chunked linear attention and the linear fast weight against closed forms

def visible_mask(N, chunk, mode, flags=None):
    """M[i, j] = 1 when token j's update is in the state token i reads."""
    c = np.arange(N) // chunk
    n = N // chunk
    flags = np.ones(n, bool) if flags is None else np.asarray(flags, bool)
    upd = flags[c][None, :]
    if mode == O.APPLY_THEN_UPDATE:
        return (c[None, :] < c[:, None]) & upd
    return (c[None, :] <= c[:, None]) & upd


def closed_form_linattn(q, k, v, eta, S0, chunk, mode, flags=None):
    """o_i = S0 q_i + sum_{visible j} eta_j (q_i . k_j) v_j (Thm 5.2, App. H, alpha = 0)."""
    B, H, N, _ = q.shape
    out = np.zeros(v.shape)
    M = visible_mask(N, chunk, mode, flags)
    for b in range(B):
        for h in range(H):
            A = (q[b, h] @ k[b, h].T) * M
            out[b, h] = A @ (eta[b, h, :, None] * v[b, h])
            if S0 is not None:
                out[b, h] += q[b, h] @ S0[b, h].T
    return out


CASES = [
    (O.APPLY_THEN_UPDATE, 16, None), (O.BLOCK_CAUSAL, 16, None), (O.BLOCK_CAUSAL, 1, None),
    (O.APPLY_THEN_UPDATE, 1, None), (O.BIDIRECTIONAL, 64, None),
    (O.STRIDED, 8, [1, 0, 1, 1, 0, 0, 1, 0]),
]


@pytest.mark.parametrize("mode,chunk,flags", CASES)
@pytest.mark.parametrize("with_state", [False, True])
def test_linattn_matches_closed_form(mode, chunk, flags, with_state):
    B, H, N, dk, dv = 2, 2, 64, 5, 3
    q, k, v = rand(B, H, N, dk), rand(B, H, N, dk), rand(B, H, N, dv)
    eta = rand(B, H, N)
    S0 = rand(B, H, dv, dk) if with_state else None
    out, Sf = O.linattn_chunked_forward(q, k, v, eta, S0, chunk, mode, flags)
    np.testing.assert_allclose(out, closed_form_linattn(q, k, v, eta, S0, chunk, mode, flags),
                               rtol=1e-10, atol=1e-10)
    # final state: S0 + sum over updated tokens of eta_j v_j k_j^T
    fl = np.ones(N // chunk, bool) if flags is None else np.asarray(flags, bool)
    sel = fl[np.arange(N) // chunk]
    expect = np.einsum("bhn,bhnv,bhnk->bhvk", eta * sel, v, k)
    if S0 is not None:
        expect += S0
    np.testing.assert_allclose(Sf, expect, atol=1e-10)


def test_linattn_token_causal_and_full_sequence():
    # chunk = 1, update then apply: S_t = S_{t-1} + eta_t v_t k_t^T, o_t = S_t q_t
    N, dk, dv = 12, 4, 3
    q, k, v = rand(1, 1, N, dk), rand(1, 1, N, dk), rand(1, 1, N, dv)
    eta = rand(1, 1, N)
    out, _ = O.linattn_chunked_forward(q, k, v, eta, None, 1, O.BLOCK_CAUSAL)
    S = np.zeros((dv, dk))
    for t in range(N):
        S += eta[0, 0, t] * np.outer(v[0, 0, t], k[0, 0, t])
        np.testing.assert_allclose(out[0, 0, t], S @ q[0, 0, t], atol=1e-12)
    # chunk = N: O = Q (K^T (eta V)) in the row form
    out, _ = O.linattn_chunked_forward(q, k, v, eta, None, N, O.BIDIRECTIONAL)
    full = q[0, 0] @ (k[0, 0].T @ (eta[0, 0, :, None] * v[0, 0]))
    np.testing.assert_allclose(out[0, 0], full, atol=1e-12)


@pytest.mark.parametrize("mode,chunk,flags", CASES)
def test_linear_fast_weight_is_linear_attention(mode, chunk, flags):
    # Thm 5.2 / section 6.1 step 6: linear f_W, W0 = 0, dot-product loss,
    # no normalisation -> block-causal linear attention
    B, H, N, dk, dv = 1, 2, 64, 4, 6
    q, k, v = rand(B, H, N, dk), rand(B, H, N, dk), rand(B, H, N, dv)
    eta = rand(B, H, N)
    out, Wf = O.ttt_linear_forward(q, k, v, eta, np.zeros((H, dv, dk)), chunk, mode, flags)
    np.testing.assert_allclose(out, closed_form_linattn(q, k, v, eta, None, chunk, mode, flags),
                               atol=1e-10)
    # gradient ascent: o(-eta) = -o(eta) when W0 = 0
    out_neg, _ = O.ttt_linear_forward(q, k, v, -eta, np.zeros((H, dv, dk)), chunk, mode, flags)
    np.testing.assert_allclose(out_neg, -out, atol=1e-12)


def momentum_mask(N, chunk, mode, beta):
    """C^{up L} of App. H with per-chunk alpha = beta and eta folded into V."""
    n = N // chunk
    C = np.zeros((n, n))
    for t in range(n):
        last = t - 1 if mode == O.APPLY_THEN_UPDATE else t
        for i in range(0, last + 1):
            C[t, i] = sum(beta ** (j - i) for j in range(i, last + 1))
    return np.kron(C, np.ones((chunk, chunk)))


@pytest.mark.parametrize("mode", [O.APPLY_THEN_UPDATE, O.BLOCK_CAUSAL])
def test_momentum_unrolling_linear(mode):
    # Thm 5.3 / App. H: momentum only re-weights the values by sum_j beta^(j-i)
    H, N, dk, dv, chunk, beta = 2, 48, 5, 4, 8, 0.7
    q, k, v = rand(1, H, N, dk), rand(1, H, N, dk), rand(1, H, N, dv)
    eta = rand(1, H, N)
    W0 = rand(H, dv, dk)
    out, _ = O.ttt_linear_forward(q, k, v, eta, W0, chunk, mode, momentum_beta=beta)
    C = momentum_mask(N, chunk, mode, beta)
    for h in range(H):
        ref = q[0, h] @ W0[h].T + ((q[0, h] @ k[0, h].T) * C) @ (eta[0, h, :, None] * v[0, h])
        np.testing.assert_allclose(out[0, h], ref, atol=1e-10)


@pytest.mark.parametrize("mode", [O.APPLY_THEN_UPDATE, O.BLOCK_CAUSAL])
@pytest.mark.parametrize("beta", [0.0, 0.6])
def test_parallel_form_static_kernel(mode, beta):
    # App. H: only the output matrix (W2 here) is dynamic, no normalisation ->
    # O = Phi(Q) W2_0^T + ((Phi(Q) Phi(K)^T) * C) (eta V)
    H, N, d, m, chunk = 2, 40, 4, 6, 8
    q, k, v = rand(1, H, N, d), rand(1, H, N, d), rand(1, H, N, d)
    eta = rand(1, H, N)
    W1, W2, W3 = rand(H, m, d), rand(H, d, m), rand(H, m, d)
    out, W1f, W2f, W3f, _ = O.ttt_layer_forward(q, k, v, eta, W1, W2, W3, chunk, mode,
                                                l2norm=False, momentum_beta=beta,
                                                last_layer_only=True)
    C = momentum_mask(N, chunk, mode, beta)
    for h in range(H):
        def phi(X):
            A1 = X @ W1[h].T
            return A1 / (1 + np.exp(-A1)) * (X @ W3[h].T)
        PQ, PK = phi(q[0, h]), phi(k[0, h])
        ref = PQ @ W2[h].T + ((PQ @ PK.T) * C) @ (eta[0, h, :, None] * v[0, h])
        np.testing.assert_allclose(out[0, h], ref, atol=1e-10)
        np.testing.assert_allclose(W1f[0, h], W1[h])
        np.testing.assert_allclose(W3f[0, h], W3[h])


# ---------------------------------------------------------------------------
# the full nonlinear update, composed from independently computed pieces

@pytest.mark.parametrize("mode", [O.APPLY_THEN_UPDATE, O.BLOCK_CAUSAL])
@pytest.mark.parametrize("muon_steps,beta", [(0, 0.0), (2, 0.5)])
def test_full_update_from_independent_pieces(mode, muon_steps, beta):
    """Two chunks of the SwiGLU layer rebuilt from finite-difference gradients,
    SVD-based Muon and a library row norm; the oracle's rows must match."""
    d, m, chunk = 3, 4, 3
    N = 2 * chunk
    q, k, v = rand(1, 1, N, d), rand(1, 1, N, d), rand(1, 1, N, d)
    eta = np.abs(rand(1, 1, N)) * 0.5
    W = [rand(1, m, d), rand(1, d, m), rand(1, m, d)]
    out, W1f, W2f, W3f, _ = O.ttt_layer_forward(q, k, v, eta, *W, chunk, mode,
                                                muon_steps=muon_steps, momentum_beta=beta)
    Ws = [W[0][0].copy(), W[1][0].copy(), W[2][0].copy()]
    Ms = [np.zeros_like(x) for x in Ws]
    outs = np.zeros((N, d))
    for c in range(2):
        sl = slice(c * chunk, (c + 1) * chunk)
        if mode == O.APPLY_THEN_UPDATE:
            outs[sl] = [brute_swiglu(*Ws, x) for x in q[0, 0, sl]]
        K, V, e = k[0, 0, sl], v[0, 0, sl], eta[0, 0, sl]
        grads = []
        for i in range(3):
            def loss(Wi, i=i):
                ws = list(Ws); ws[i] = Wi
                return brute_loss(*ws, K, V, e)
            grads.append(fd_grad(loss, Ws[i]))
        for i in range(3):
            Ms[i] = beta * Ms[i] + grads[i]
            U = ns_by_svd(Ms[i], muon_steps, O.MUON_COEF) if muon_steps else Ms[i]
            Wn = Ws[i] - U
            Ws[i] = Wn / np.linalg.norm(Wn, axis=1, keepdims=True)
        if mode != O.APPLY_THEN_UPDATE:
            outs[sl] = [brute_swiglu(*Ws, x) for x in q[0, 0, sl]]
    for got, ref in ((W1f[0, 0], Ws[0]), (W2f[0, 0], Ws[1]), (W3f[0, 0], Ws[2])):
        np.testing.assert_allclose(got, ref, atol=1e-6)
    np.testing.assert_allclose(out[0, 0], outs, atol=1e-6)


# ---------------------------------------------------------------------------
# composite invariants of the scan

def _layer_args(H=2, N=32, d=4, m=6):
    return (rand(1, H, N, d), rand(1, H, N, d), rand(1, H, N, d), np.abs(rand(1, H, N)) * 0.1,
            rand(H, m, d), rand(H, d, m), rand(H, m, d))


def test_strided_all_flags_is_block_causal():
    args = _layer_args()
    a = O.ttt_layer_forward(*args, 8, O.BLOCK_CAUSAL, muon_steps=2, momentum_beta=0.3)
    b = O.ttt_layer_forward(*args, 8, O.STRIDED, update_chunks=[1, 1, 1, 1],
                            muon_steps=2, momentum_beta=0.3)
    for x, y in zip(a[:4], b[:4]):
        np.testing.assert_allclose(x, y, atol=0)


def test_strided_apply_only_chunks_keep_state():
    args = _layer_args()
    out, W1f, W2f, W3f, _ = O.ttt_layer_forward(*args, 8, O.STRIDED, update_chunks=[1, 0, 0, 0])
    # after the single update, chunks 1..3 are read with the same weights
    ref = O.swiglu_apply(W1f[0, 0], W2f[0, 0], W3f[0, 0], args[0][0, 0])
    np.testing.assert_allclose(out[0, 0], ref, atol=1e-12)


@pytest.mark.parametrize("mode", [O.APPLY_THEN_UPDATE, O.BLOCK_CAUSAL])
def test_split_call_carry(mode):
    q, k, v, eta, W1, W2, W3 = _layer_args(N=48)
    full = O.ttt_layer_forward(q, k, v, eta, W1, W2, W3, 8, mode, muon_steps=3, momentum_beta=0.9)
    s = 24
    a = O.ttt_layer_forward(q[..., :s, :], k[..., :s, :], v[..., :s, :], eta[..., :s],
                            W1, W2, W3, 8, mode, muon_steps=3, momentum_beta=0.9)
    b = O.ttt_layer_forward(q[..., s:, :], k[..., s:, :], v[..., s:, :], eta[..., s:],
                            a[1], a[2], a[3], 8, mode, muon_steps=3, momentum_beta=0.9,
                            momentum=a[4])
    np.testing.assert_allclose(np.concatenate([a[0], b[0]], axis=2), full[0], atol=1e-12)
    for x, y in zip(b[1:4], full[1:4]):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_prefix_scan_matches_full():
    args = _layer_args(N=40)
    full = O.ttt_layer_forward(*args, 8, O.APPLY_THEN_UPDATE, muon_steps=1)
    pre = O.ttt_layer_forward(*args, 8, O.APPLY_THEN_UPDATE, muon_steps=1, n_chunks=3)
    np.testing.assert_allclose(pre[0][..., :24, :], full[0][..., :24, :], atol=0)
    assert np.all(pre[0][..., 24:, :] == 0)


def test_replace_q_with_k_runs():
    q, k, v, eta, W1, W2, W3 = _layer_args()
    out, *_ = O.ttt_layer_forward(k, k, v, eta, W1, W2, W3, 8, O.APPLY_THEN_UPDATE)
    assert np.all(np.isfinite(out))


# ---------------------------------------------------------------------------
# more inner-loop steps ("Test-Time Training with KV Binding Is Secretly
# Linear Attention", sec. 4.1): r update steps on a chunk are r single-step
# updates on r copies of that chunk

def _repeat_chunks(x, chunk, r):
    """Every chunk of the sequence axis (axis 2) repeated r times in place."""
    B, H, N = x.shape[:3]
    n = N // chunk
    parts = np.split(x, n, axis=2)
    return np.concatenate([p for p in parts for _ in range(r)], axis=2)


@pytest.mark.parametrize("mode,flags", [(O.APPLY_THEN_UPDATE, None), (O.BLOCK_CAUSAL, None),
                                        (O.STRIDED, (1, 0, 1))])
@pytest.mark.parametrize("muon", [0, 2])
def test_inner_steps_are_repeated_chunks(mode, flags, muon):
    rng = np.random.default_rng(77)
    B, H, N, d, m, chunk, r = 1, 2, 12, 4, 6, 4, 3
    q, k, v = (rng.normal(size=(B, H, N, d)) * 0.5 for _ in range(3))
    eta = rng.uniform(0.05, 0.3, size=(B, H, N))
    W1, W3 = (rng.normal(size=(H, m, d)) * 0.5 for _ in range(2))
    W2 = rng.normal(size=(H, d, m)) * 0.5
    kw = dict(l2norm=True, muon_steps=muon, momentum_beta=0.6)
    got = O.ttt_layer_forward(q, k, v, eta, W1, W2, W3, chunk, mode, flags, inner_steps=r,
                              **kw)
    rep = [_repeat_chunks(x, chunk, r) for x in (q, k, v, eta[..., None])]
    # copies of a chunk that the strided mask does not update still only apply
    rflags = None if flags is None else [f for f in flags for _ in range(r)]
    ref = O.ttt_layer_forward(rep[0], rep[1], rep[2], rep[3][..., 0], W1, W2, W3, chunk, mode,
                              rflags, **kw)
    n = N // chunk
    # the output of chunk c: the first copy's (apply before the update) or
    # the last copy's (apply after the updates; a chunk without update
    # applies the same weights in every copy)
    pick = 0 if mode == O.APPLY_THEN_UPDATE else r - 1
    want = np.concatenate([ref[0][:, :, (c * r + pick) * chunk:(c * r + pick + 1) * chunk]
                           for c in range(n)], axis=2)
    np.testing.assert_allclose(got[0], want, rtol=1e-10, atol=1e-12)
    for i in (1, 2, 3):
        np.testing.assert_allclose(got[i], ref[i], rtol=1e-10, atol=1e-12)
    # one step is the default
    one = O.ttt_layer_forward(q, k, v, eta, W1, W2, W3, chunk, mode, flags, inner_steps=1, **kw)
    base = O.ttt_layer_forward(q, k, v, eta, W1, W2, W3, chunk, mode, flags, **kw)
    np.testing.assert_array_equal(one[0], base[0])

"""Plain fp64 CPU oracle for the large-chunk TTT-KVB (LaCT) layer and its
chunked linear-attention reduction.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  It shares
no code with the CUDA path; both sides receive the same arrays from the seeded
generators in ``workloads.py`` and nothing else.

Everything here is float64 numpy.  Matrix products (``@``) are the only library
primitive used; there is no blocking, fusion or reordering beyond what the
definitions below state.  Column-vector math on the pages becomes row-major
tensor math here: a chunk holds its tokens as rows, so ``f_W(x)`` for all rows
``X`` is ``F = (SiLU(X W1^T) * (X W3^T)) W2^T``.

Sources (page title, then section / equation):
  * "5.2.1 LaCT and TTT-E2E" notes page: eq (2) large-chunk gradient with a
    per-token learning rate, eq (3) bias-free SwiGLU fast weight, eq (4)
    dot-product loss, eq (5) L2-Normalize update, eq (6) Muon update and the
    momentum sentence after it, the mask list of section 1.1, eq (10)
    apply-then-update.
  * "Test-Time Training with KV Binding Is Secretly Linear Attention":
    Thm 5.2 / 5.3 (unrolled updates), App. E.2 (upstream gradient -v),
    App. E.4 (channel-wise l2 normalisation), App. H (parallel form),
    App. I.1 (silu' term of the W1 gradient).
  * "From Linear Attention to Test-Time Training": causal linear attention
    state update and the full-sequence (bidirectional) form.

Readings where the pages are silent or garbled (each is listed with its reason
in the design notes of the repository):
  * matrix names follow eq (3): W1, W3 are [m_h x d_h], W2 is [d_h x m_h];
  * the loss is summed over the chunk with no 1/b (eq 2);
  * L2-Normalize makes every output row of a matrix unit-norm over its input
    entries (eq 5 "along the input dimension"; App. E.4 "channel-wise"), eps
    1e-12, target norm 1;
  * momentum is ``M <- beta*M + g`` with M0 = 0, then Muon on M; the update has
    no outer learning rate (eq 6 and the momentum sentence after it);
  * Muon is the Newton-Schulz quintic of the Muon write-up the paper cites,
    ``X <- aX + b(XX^T)X + c(XX^T)^2 X`` after ``X = G/(||G||_F + 1e-7)``, with
    the matrix transposed so that the Gram product is on the smaller side;
  * "bidirectional" is one chunk covering the sequence, update then apply;
  * strided mode updates only on flagged chunks, update then apply, and
    applies on every chunk.

Parity is pinned for every function here by tests under ``tests/``
(finite differences, closed forms, SVD, invariants); see the test module
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

APPLY_THEN_UPDATE = 0
BLOCK_CAUSAL = 1
BIDIRECTIONAL = 2
STRIDED = 3

# Quintic Newton-Schulz coefficients of the Muon write-up (Jordan et al.,
# 2024) that the paper cites for its gradient orthogonalisation.
MUON_COEF = (3.4445, -4.7750, 2.0315)
NS_EPS = 1e-7
NORM_EPS = 1e-12


# ---------------------------------------------------------------------------
# elementwise pieces of eq (3)

def sigmoid(x):
    """Logistic function; tanh form avoids overflow for large |x|."""
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def silu(x):
    """SiLU(x) = x * sigmoid(x) (eq 3 gate)."""
    return x * sigmoid(x)


def silu_prime(x):
    """Derivative of SiLU, the silu' factor of the W1 gradient (App. I.1)."""
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


# ---------------------------------------------------------------------------
# the fast-weight net and its chunk gradient

def swiglu_apply(W1, W2, W3, X):
    """Apply the bias-free SwiGLU fast weight to every row of X (eq 3).

    W1, W3: [m, d]; W2: [d, m]; X: [rows, d] -> [rows, d].
    """
    return (silu(X @ W1.T) * (X @ W3.T)) @ W2.T


def dot_product_loss(W1, W2, W3, K, V, eta):
    """Chunk loss sum_i eta_i * L_i with L_i = -f_W(k_i)^T v_i (eqs 2, 4)."""
    F = swiglu_apply(W1, W2, W3, K)
    return float(np.sum(eta * -np.sum(F * V, axis=1)))


def swiglu_chunk_gradients(W1, W2, W3, K, V, eta):
    """Gradient of the eta-weighted dot-product loss over one chunk (eq 2).

    Hand-derived backward pass of eq (3) under eq (4):
      dL/dF   = -eta * V                      (App. E.2: upstream gradient -v)
      g2      = (dL/dF)^T (SiLU(H1) * H3)
      dA      = (dL/dF) W2
      dH1     = dA * H3 * SiLU'(H1)           (App. I.1)
      dH3     = dA * SiLU(H1)
      g1, g3  = dH1^T K, dH3^T K
    with H1 = K W1^T, H3 = K W3^T.  Returns (g1 [m,d], g2 [d,m], g3 [m,d]).
    """
    H1 = K @ W1.T
    H3 = K @ W3.T
    A = silu(H1) * H3
    dF = -(eta[:, None] * V)
    g2 = dF.T @ A
    dA = dF @ W2
    dH1 = dA * H3 * silu_prime(H1)
    dH3 = dA * silu(H1)
    g1 = dH1.T @ K
    g3 = dH3.T @ K
    return g1, g2, g3


def linear_apply(W, X):
    """Linear fast weight f_W(x) = W x for every row of X (W: [d_v, d_k])."""
    return X @ W.T


def linear_chunk_gradient(W, K, V, eta):
    """Gradient of sum_i eta_i * (-(W k_i)^T v_i) with respect to W."""
    return -(eta[:, None] * V).T @ K


# ---------------------------------------------------------------------------
# update rule pieces (eqs 5, 6 and the momentum sentence)

def newton_schulz(G, steps, coef=MUON_COEF, eps=NS_EPS):
    """Muon orthogonalisation of one matrix by ``steps`` Newton-Schulz steps.

    X = G / (||G||_F + eps); if X has more rows than columns it is transposed
    so that A = X X^T is the smaller Gram matrix; each step does
    A = X X^T, B = b A + c A A, X = a X + B X; the result is transposed back.
    """
    a, b, c = coef
    X = np.array(G, dtype=np.float64) / (np.linalg.norm(G) + eps)
    tall = X.shape[0] > X.shape[1]
    if tall:
        X = X.T
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tall else X


def l2_normalize_rows(W, eps=NORM_EPS):
    """Scale every row of W to unit L2 norm over its input entries (eq 5)."""
    n = np.sqrt(np.sum(W * W, axis=1, keepdims=True))
    return W / np.maximum(n, eps)


def update_one_matrix(W, g, M, l2norm, muon_steps, beta, coef):
    """One weight-update of eq (5)/(6) with optional momentum.

    M <- beta M + g;  U = Muon(M) if muon_steps else M;
    W <- L2-Normalize(W - U) if l2norm else W - U.   Returns (W, M).
    """
    M = beta * M + g
    U = newton_schulz(M, muon_steps, coef) if muon_steps > 0 else M
    W = W - U
    if l2norm:
        W = l2_normalize_rows(W)
    return W, M


# ---------------------------------------------------------------------------
# the chunk scan (section 1.1 masks, eq 10)

def _update_flags(n_chunks, mode, update_chunks):
    if mode == STRIDED:
        if update_chunks is None:
            raise ValueError("strided mode needs update_chunks")
        flags = [bool(x) for x in update_chunks]
        if len(flags) != n_chunks:
            raise ValueError("update_chunks must have one flag per chunk")
        return flags
    return [True] * n_chunks


def chunk_scan(Q, K, V, eta, Ws, chunk, mode, update_chunks, apply_fn, grad_fn,
               dynamic, l2norm, muon_steps, beta, coef, Ms, n_chunks=None, inner_steps=1):
    """Sequential chunk recurrence for one (batch, head).

    Q, K, V: [N, d]; eta: [N]; Ws: list of fast-weight matrices; Ms: list of
    momentum matrices (same shapes).  ``dynamic[i]`` says whether Ws[i] is
    updated.  Apply-then-update uses the state from before the chunk (eq 10);
    the other masks update first, then apply.  Strided mode only updates on
    flagged chunks.  ``inner_steps`` updates are taken on each updating
    chunk, each from the gradient at the current weights ("Test-Time
    Training with KV Binding Is Secretly Linear Attention", sec. 4.1: more
    inner-loop steps at test time); the apply reads the weights before the
    first or after the last of them.  ``n_chunks`` limits the scan to a
    prefix of the sequence (outputs past the prefix stay zero).
    Returns (O, Ws, Ms).
    """
    N = Q.shape[0]
    if N % chunk != 0:
        raise ValueError("sequence length must be a multiple of the chunk")
    total = N // chunk
    if mode == BIDIRECTIONAL and total != 1:
        raise ValueError("bidirectional mode is a single chunk covering the sequence")
    flags = _update_flags(total, mode, update_chunks)
    steps = total if n_chunks is None else min(n_chunks, total)
    Ws = [np.array(W, dtype=np.float64) for W in Ws]
    Ms = [np.array(M, dtype=np.float64) for M in Ms]
    O = np.zeros((N, apply_fn(Ws, Q[:1]).shape[1]), dtype=np.float64)
    for c in range(steps):
        sl = slice(c * chunk, (c + 1) * chunk)
        if mode == APPLY_THEN_UPDATE:
            O[sl] = apply_fn(Ws, Q[sl])
        if flags[c]:
            for _ in range(max(1, inner_steps)):
                gs = grad_fn(Ws, K[sl], V[sl], eta[sl])
                for i, g in enumerate(gs):
                    if dynamic[i]:
                        Ws[i], Ms[i] = update_one_matrix(Ws[i], g, Ms[i], l2norm,
                                                         muon_steps, beta, coef)
        if mode != APPLY_THEN_UPDATE:
            O[sl] = apply_fn(Ws, Q[sl])
    return O, Ws, Ms


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _per_batch(W, B):
    """Weights given as [H,...] are shared over the batch; [B,H,...] are not."""
    W = _f64(W)
    return (lambda b, h: W[h]) if W.ndim == 3 else (lambda b, h: W[b, h])


def ttt_layer_forward(q, k, v, eta, W1, W2, W3, chunk, mode, update_chunks=None,
                      l2norm=True, muon_steps=0, momentum_beta=0.0,
                      ns_coef=MUON_COEF, momentum=None, last_layer_only=False,
                      n_chunks=None, inner_steps=1):
    """LaCT TTT layer forward over [B, H, N, d] inputs.

    W1, W3: [H, m, d] or [B, H, m, d]; W2: [H, d, m] or [B, H, d, m].
    momentum: optional (M1, M2, M3) with shapes [B, H, ...] carried in; zero
    otherwise.  ``last_layer_only`` keeps W1, W3 static (only W2 updates).
    ``inner_steps``: update steps per updating chunk (see chunk_scan).
    Returns (out [B,H,N,d], W1f, W2f, W3f, (M1, M2, M3)), all float64.
    """
    q, k, v, eta = _f64(q), _f64(k), _f64(v), _f64(eta)
    B, H, N, d = q.shape
    g1w, g2w, g3w = _per_batch(W1, B), _per_batch(W2, B), _per_batch(W3, B)
    m = g1w(0, 0).shape[0]
    out = np.zeros((B, H, N, d))
    W1f = np.zeros((B, H, m, d)); W3f = np.zeros((B, H, m, d)); W2f = np.zeros((B, H, d, m))
    M1f = np.zeros((B, H, m, d)); M3f = np.zeros((B, H, m, d)); M2f = np.zeros((B, H, d, m))

    def apply_fn(Ws, X):
        return swiglu_apply(Ws[0], Ws[1], Ws[2], X)

    def grad_fn(Ws, K, V, e):
        return swiglu_chunk_gradients(Ws[0], Ws[1], Ws[2], K, V, e)

    dynamic = (not last_layer_only, True, not last_layer_only)
    for b in range(B):
        for h in range(H):
            Ws = [g1w(b, h), g2w(b, h), g3w(b, h)]
            if momentum is None:
                Ms = [np.zeros_like(W) for W in Ws]
            else:
                Ms = [_f64(momentum[0])[b, h], _f64(momentum[1])[b, h], _f64(momentum[2])[b, h]]
            O, Ws, Ms = chunk_scan(q[b, h], k[b, h], v[b, h], eta[b, h], Ws, chunk, mode,
                                   update_chunks, apply_fn, grad_fn, dynamic, l2norm,
                                   muon_steps, momentum_beta, ns_coef, Ms, n_chunks,
                                   inner_steps)
            out[b, h] = O
            W1f[b, h], W2f[b, h], W3f[b, h] = Ws
            M1f[b, h], M2f[b, h], M3f[b, h] = Ms
    return out, W1f, W2f, W3f, (M1f, M2f, M3f)


def ttt_linear_forward(q, k, v, eta, W0, chunk, mode, update_chunks=None,
                       l2norm=False, muon_steps=0, momentum_beta=0.0,
                       ns_coef=MUON_COEF):
    """The same chunk scan with a single linear fast weight f_W(x) = W x.

    W0: [H, d_v, d_k] or [B, H, d_v, d_k].  Returns (out, W_final).
    """
    q, k, v, eta = _f64(q), _f64(k), _f64(v), _f64(eta)
    B, H, N, _ = q.shape
    getw = _per_batch(W0, B)
    dv = getw(0, 0).shape[0]
    out = np.zeros((B, H, N, dv))
    Wf = np.zeros((B, H) + getw(0, 0).shape)
    for b in range(B):
        for h in range(H):
            W = getw(b, h)
            O, Ws, _ = chunk_scan(q[b, h], k[b, h], v[b, h], eta[b, h], [W], chunk, mode,
                                  update_chunks, lambda Ws, X: linear_apply(Ws[0], X),
                                  lambda Ws, K, V, e: (linear_chunk_gradient(Ws[0], K, V, e),),
                                  (True,), l2norm, muon_steps, momentum_beta, ns_coef,
                                  [np.zeros_like(W)])
            out[b, h] = O
            Wf[b, h] = Ws[0]
    return out, Wf


# ---------------------------------------------------------------------------
# chunked linear attention (the linear-final-layer reduction)

def linattn_chunked_forward(q, k, v, eta, S0, chunk, mode, update_chunks=None):
    """Chunked linear attention with state S [d_v, d_k] per (batch, head).

    Per chunk: S <- S + (eta * V)^T K, and O = Q S^T, in the order the mask
    sets (apply-then-update reads S before the chunk's update).  S0 may be
    None (zeros).  Returns (out [B,H,N,d_v], S_final [B,H,d_v,d_k]).
    """
    q, k, v, eta = _f64(q), _f64(k), _f64(v), _f64(eta)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if N % chunk != 0:
        raise ValueError("sequence length must be a multiple of the chunk")
    n = N // chunk
    if mode == BIDIRECTIONAL and n != 1:
        raise ValueError("bidirectional mode is a single chunk covering the sequence")
    flags = _update_flags(n, mode, update_chunks)
    out = np.zeros((B, H, N, dv))
    Sf = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else _f64(S0)[b, h].copy()
            for c in range(n):
                sl = slice(c * chunk, (c + 1) * chunk)
                if mode == APPLY_THEN_UPDATE:
                    out[b, h, sl] = q[b, h, sl] @ S.T
                if flags[c]:
                    S = S + (eta[b, h, sl, None] * v[b, h, sl]).T @ k[b, h, sl]
                if mode != APPLY_THEN_UPDATE:
                    out[b, h, sl] = q[b, h, sl] @ S.T
            Sf[b, h] = S
    return out, Sf


# ---------------------------------------------------------------------------
# chunked linear attention with momentum, a per-chunk learning rate and an
# optional Muon of the momentum (the reducible TTT variants)

def linattn_momentum_forward(q, k, v, eta, S0, chunk, mode, update_chunks=None,
                             alpha=None, lr=None, M0=None, muon_steps=0,
                             ns_coef=MUON_COEF):
    """Chunked linear attention whose state is updated through a momentum
    accumulator, with a per-chunk momentum coefficient and learning rate.

    Follows the sequential recurrence of "Test-Time Training with KV Binding
    Is Secretly Linear Attention": Thm 5.3 / App. D (gradient descent with a
    per-step momentum factor alpha_t), App. H.2 (its chunk form with a
    per-chunk learning rate), and App. E.3 (Muon applied to the momentum
    accumulator).  With a linear fast weight f_S(x) = S x and the dot-product
    loss the chunk's negative gradient is G_t = (eta * V_t)^T K_t (per-token
    eta folded into the values), and per updating chunk t

        M_t = alpha_t M_{t-1} + G_t          (M_{-1} = M0, zeros if None)
        U_t = Muon(M_t) if muon_steps else M_t
        S  <- S + lr_t U_t

    Chunks that do not update (strided mask) leave M and S unchanged.  The
    outputs O_t = Q_t S^T read S before (apply-then-update) or after the
    chunk's update, as in linattn_chunked_forward.

    q, k: [B, H, N, d_k]; v: [B, H, N, d_v]; eta: [B, H, N];
    S0, M0: [B, H, d_v, d_k] or None; alpha, lr: [B, H, N / chunk] or None
    (None: alpha = 0, i.e. no momentum; lr = 1).
    Returns (out [B, H, N, d_v], S_final, M_final).
    """
    q, k, v, eta = _f64(q), _f64(k), _f64(v), _f64(eta)
    B, H, N, dk = q.shape
    dv = v.shape[-1]
    if N % chunk != 0:
        raise ValueError("sequence length must be a multiple of the chunk")
    n = N // chunk
    if mode == BIDIRECTIONAL and n != 1:
        raise ValueError("bidirectional mode is a single chunk covering the sequence")
    flags = _update_flags(n, mode, update_chunks)
    al = np.zeros((B, H, n)) if alpha is None else _f64(alpha)
    lrs = np.ones((B, H, n)) if lr is None else _f64(lr)
    out = np.zeros((B, H, N, dv))
    Sf = np.zeros((B, H, dv, dk))
    Mf = np.zeros((B, H, dv, dk))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else _f64(S0)[b, h].copy()
            M = np.zeros((dv, dk)) if M0 is None else _f64(M0)[b, h].copy()
            for c in range(n):
                sl = slice(c * chunk, (c + 1) * chunk)
                if mode == APPLY_THEN_UPDATE:
                    out[b, h, sl] = q[b, h, sl] @ S.T
                if flags[c]:
                    G = (eta[b, h, sl, None] * v[b, h, sl]).T @ k[b, h, sl]
                    M = al[b, h, c] * M + G
                    U = newton_schulz(M, muon_steps, ns_coef) if muon_steps > 0 else M
                    S = S + lrs[b, h, c] * U
                if mode != APPLY_THEN_UPDATE:
                    out[b, h, sl] = q[b, h, sl] @ S.T
            Sf[b, h] = S
            Mf[b, h] = M
    return out, Sf, Mf

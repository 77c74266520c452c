"""Plain fp64 CPU oracle of the LaCT fast-weight chunk step.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline and its ``--impl reference`` arm) may call it. It shares no code
with the CUDA path; both take their inputs from ``lact_inputs``.

What it computes, for one (batch, head) at a time, following

* "Test-Time Training Done Right" (arXiv 2505.23884), abstract: fast weights
  adapted at inference; chunks of 2K to ~1M tokens; Muon as the optimiser.
* The LaCT review page (iplexlaw), section "Fast weights are temporary
  context memory": the key-value relation is stored in the weights W of a
  small network and read with a query.
* Same page, section "Local attention and nonlinear memory work together":
  the memory is a three-matrix SwiGLU MLP; a negative inner-product loss
  aligns the outputs for keys with the values; the chunk gradient carries
  token-specific learning rates; the update is gradient descent or Muon (a
  Newton-Schulz transform of each matrix gradient); the updated fast weights
  are L2-normalised.
* Same page, section "Update order must respect the task": language chunks
  read the memory of earlier chunks, then update it; posed image sets first
  absorb all inputs, then answer the queries.

The pages print no equations. The formulas below are the plain reading of
that prose (each choice is listed in the design notes):

  f_W(x) = W2 (silu(W1 x) * (W3 x)),   W1, W3: [dh, d],  W2: [d, dh]
  L      = - sum_i eta_i <f_W(k_i), v_i>            (one chunk)
  GD:    W <- W - dL/dW                              (step size lives in eta)
  momentum: M <- beta M + dL/dW (M starts at 0 and carries across chunks),
         W <- W - M, per matrix (beta = 0.9)
  Muon:  W <- W - lr * NS5(dL/dW)   per matrix,  NS5 = five quintic
         Newton-Schulz steps with (a, b, c) = (3.4445, -4.7750, 2.0315) on
         the Frobenius-normalised gradient (eps 1e-7), on the orientation
         with rows <= cols
  renorm: every row of every matrix is scaled back to its pre-update L2 norm.

Every floating-point step is fp64, except the points where the Muon step's
GEMM operands are, by the problem statement, bf16: there the value is rounded
to bf16 (round to nearest even) exactly as the kernel does, then the product
is formed in fp64.
"""
from __future__ import annotations

import numpy as np

NS_A, NS_B, NS_C = 3.4445, -4.7750, 2.0315
NS_EPS = 1e-7
MUON_LR = 0.02
MOMENTUM_BETA = 0.9


# --------------------------------------------------------------------------
# Elementwise pieces of the SwiGLU memory (review page, "Local attention and
# nonlinear memory work together": the three-matrix SwiGLU MLP).
# --------------------------------------------------------------------------
def sigmoid(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def silu(x: np.ndarray) -> np.ndarray:
    return x * sigmoid(x)


def silu_grad(x: np.ndarray) -> np.ndarray:
    """d/dx [x * sigmoid(x)] = sigmoid(x) * (1 + x * (1 - sigmoid(x)))."""
    s = sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


# --------------------------------------------------------------------------
# Readout: queries read the fast weights (review page, "Fast weights are
# temporary context memory").
# --------------------------------------------------------------------------
def fast_weight_apply(W1, W2, W3, X):
    """o_i = W2 (silu(W1 x_i) * (W3 x_i)) for every row x_i of X [n, d]."""
    H1 = X @ W1.T                 # [n, dh]
    H3 = X @ W3.T                 # [n, dh]
    U = silu(H1) * H3             # [n, dh]
    return U @ W2.T               # [n, d]


def chunk_loss(W1, W2, W3, K, V, eta):
    """L = -sum_i eta_i <f_W(k_i), v_i> (the negative inner-product loss)."""
    F = fast_weight_apply(W1, W2, W3, K)
    return -float(np.sum(eta * np.sum(F * V, axis=1)))


# --------------------------------------------------------------------------
# Chunk-wide gradient of the loss above, by the chain rule through the MLP.
# --------------------------------------------------------------------------
def chunk_gradient(W1, W2, W3, K, V, eta):
    """Return (dL/dW1, dL/dW2, dL/dW3) summed over every token of the chunk."""
    H1 = K @ W1.T                        # [n, dh]
    H3 = K @ W3.T                        # [n, dh]
    U = silu(H1) * H3                    # hidden activation, [n, dh]
    G = -eta[:, None] * V                # dL/df(k_i) = -eta_i v_i, [n, d]
    dW2 = G.T @ U                        # [d, dh]
    DU = G @ W2                          # dL/du_i = W2^T g_i, [n, dh]
    DH1 = DU * H3 * silu_grad(H1)        # dL/dh1_i
    DH3 = DU * silu(H1)                  # dL/dh3_i
    dW1 = DH1.T @ K                      # [dh, d]
    dW3 = DH3.T @ K                      # [dh, d]
    return dW1, dW2, dW3


# --------------------------------------------------------------------------
# Linear fast-weight memory: one d x d matrix W, o = W q (review page,
# "Local attention and nonlinear memory work together" and Fig. 8: the
# larger linear state that the smaller SwiGLU state is compared against).
# --------------------------------------------------------------------------
def linear_apply(W, X):
    """o_i = W x_i for every row x_i of X [n, d]."""
    return X @ W.T


def linear_chunk_loss(W, K, V, eta):
    """L = -sum_i eta_i <W k_i, v_i>."""
    return -float(np.sum(eta * np.sum(linear_apply(W, K) * V, axis=1)))


def linear_chunk_gradient(W, K, V, eta):
    """dL/dW = -sum_i eta_i v_i k_i^T, as one GEMM over the chunk: [d, d]."""
    return -(eta[:, None] * V).T @ K


# --------------------------------------------------------------------------
# Muon: Newton-Schulz orthogonalisation of a matrix gradient (review page,
# "Local attention and nonlinear memory work together").
# --------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round each value to the nearest bf16 number (8 significant bits, ties to
    even), returned as fp64. Values stay in the normal range here."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                   # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def newton_schulz5(G, steps: int = 5, a: float = NS_A, b: float = NS_B, c: float = NS_C,
                   eps: float = NS_EPS, bf16_points: bool = True):
    """Quintic Newton-Schulz iteration on G (any m x n), returned in G's shape.

    X = G / (||G||_F + eps), on the orientation with rows <= cols; then `steps`
    times: A = X X^T; B = b A + c A A; X = a X + B X. With bf16_points the GEMM
    operands are rounded to bf16 where the kernel rounds them: X for X X^T, A
    for A A, B and X for B X (A, A A, B and X themselves stay unrounded).
    """
    r = bf16_round if bf16_points else (lambda t: t)
    X = np.asarray(G, dtype=np.float64)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    X = X / (np.linalg.norm(X) + eps)
    for _ in range(steps):
        Xr = r(X)
        A = Xr @ Xr.T
        Ar = r(A)
        AA = Ar @ Ar
        Bm = b * A + c * AA
        X = a * X + r(Bm) @ Xr
    return X.T if transposed else X


def optimizer_delta(dW, opt: str, lr: float = MUON_LR, ns_steps: int = 5,
                    a: float = NS_A, b: float = NS_B, c: float = NS_C):
    """Weight change of one update: -dW (gradient descent) or -lr NS5(dW) (Muon)."""
    if opt == "gd":
        return -dW
    if opt == "muon":
        return -lr * newton_schulz5(dW, steps=ns_steps, a=a, b=b, c=c)
    raise ValueError(opt)


# --------------------------------------------------------------------------
# L2 renormalisation of the updated fast weights, row by row, back to the
# norm each row had before the update.
# --------------------------------------------------------------------------
def renorm_update(W, delta):
    n0 = np.linalg.norm(W, axis=1)
    Wt = W + delta
    n1 = np.linalg.norm(Wt, axis=1)
    scale = np.where(n1 > 0.0, n0 / np.where(n1 > 0.0, n1, 1.0), 1.0)
    return Wt * scale[:, None]


def momentum_velocity(M, g, beta: float = MOMENTUM_BETA):
    """Heavy-ball momentum (review page, "Local attention and nonlinear memory
    work together": gradient descent, momentum and Muon are the update rules
    compared): the velocity after this chunk, beta M + g."""
    return beta * M + g


def memory_gradient(W, K, V, eta):
    """Chunk gradient of the memory W: (W1, W2, W3) SwiGLU or (W,) linear."""
    if len(W) == 1:
        return (linear_chunk_gradient(W[0], K, V, eta),)
    return chunk_gradient(W[0], W[1], W[2], K, V, eta)


def memory_apply(W, X):
    """Readout of the memory W: (W1, W2, W3) SwiGLU or (W,) linear."""
    return linear_apply(W[0], X) if len(W) == 1 else fast_weight_apply(W[0], W[1], W[2], X)


def chunk_update(W, K, V, eta, opt: str, lr: float = MUON_LR, ns_steps: int = 5,
                 a: float = NS_A, b: float = NS_B, c: float = NS_C, token_slice: int | None = None,
                 mom=None, beta: float = MOMENTUM_BETA):
    """One update of the fast weights W = (W1, W2, W3), or (W,) for the
    linear memory, on one chunk.

    token_slice only bounds memory: the chunk gradient is the sum over tokens,
    so it is taken slice by slice and added up before the single optimiser step.
    For opt == "momentum", `mom` is the list of the three velocities; it is
    replaced in place by the new ones and the step is -velocity.
    """
    n = K.shape[0]
    step = n if not token_slice else token_slice
    grads = [np.zeros_like(Wm) for Wm in W]
    for s in range(0, max(n, 1), max(step, 1)):
        if n == 0:
            break
        e = min(n, s + step)
        for g, d in zip(grads, memory_gradient(W, K[s:e], V[s:e], eta[s:e])):
            g += d
    if opt == "momentum":
        for m, g in enumerate(grads):
            mom[m] = momentum_velocity(mom[m], g, beta)
        return tuple(renorm_update(Wm, -Mm) for Wm, Mm in zip(W, mom))
    return tuple(renorm_update(Wm, optimizer_delta(g, opt, lr, ns_steps, a, b, c)) for Wm, g in zip(W, grads))


def zero_velocity(W):
    return [np.zeros_like(Wm) for Wm in W]


# --------------------------------------------------------------------------
# Orders (review page, "Update order must respect the task").
# --------------------------------------------------------------------------
def sequence_causal(W, Q, K, V, eta, chunk: int, opt: str, **kw):
    """Apply-then-update per chunk. The last chunk updates W too.
    Returns (O [n, d], final W)."""
    n = Q.shape[0]
    O = np.zeros_like(Q)
    if opt == "momentum":
        kw = dict(kw, mom=zero_velocity(W))
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        O[s:e] = memory_apply(W, Q[s:e])
        W = chunk_update(W, K[s:e], V[s:e], eta[s:e], opt, **kw)
    return O, W


def sequence_set(W, Q, K, V, eta, opt: str, **kw):
    """Update-then-apply: one update on all input tokens, then read the queries."""
    if opt == "momentum":
        kw = dict(kw, mom=zero_velocity(W))
    W = chunk_update(W, K, V, eta, opt, **kw)
    return memory_apply(W, Q), W


def run_workload(w, inp, heads=None, token_slice: int | None = None):
    """Run a whole workload (lact_inputs.Workload + Inputs) head by head.

    Returns O [B,H,n_q,d] and W1, W2, W3 [B,H,...] in fp64 (heads not listed
    in `heads`, a list of (b, h), stay zero). For the linear memory W1 is the
    memory [B,H,d,d] and W2, W3 are None."""
    from lact_inputs import as_f64  # input widening only (bf16 bits -> fp64)
    B, H = w.B, w.H
    heads = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    O = np.zeros((B, H, w.n_q, w.d))
    linear = w.memory == "linear"
    W1 = np.zeros((B, H, w.d, w.d) if linear else (B, H, w.dh, w.d))
    W2 = None if linear else np.zeros((B, H, w.d, w.dh))
    W3 = None if linear else np.zeros((B, H, w.dh, w.d))
    kw = dict(lr=w.muon_lr, ns_steps=w.ns_steps, a=w.ns_a, b=w.ns_b, c=w.ns_c, beta=w.momentum)
    for (b, h) in heads:
        if linear:
            W0 = (inp.W1[h].astype(np.float64),)
        else:
            W0 = (inp.W1[h].astype(np.float64), inp.W2[h].astype(np.float64), inp.W3[h].astype(np.float64))
        Q, K, V = as_f64(inp.q[b, h]), as_f64(inp.k[b, h]), as_f64(inp.v[b, h])
        e = inp.eta[b, h].astype(np.float64)
        if w.order == "causal":
            o, Wf = sequence_causal(W0, Q, K, V, e, w.chunk, w.opt, **kw)
        else:
            o, Wf = sequence_set(W0, Q, K, V, e, w.opt, token_slice=token_slice, **kw)
        O[b, h] = o
        W1[b, h] = Wf[0]
        if not linear:
            W2[b, h], W3[b, h] = Wf[1], Wf[2]
    return O, W1, W2, W3

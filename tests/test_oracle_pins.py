"""Pins of the fp64 oracle against facts fixed outside of it.

Each test ties one oracle function to something other than its own formula:
finite differences of the loss, a textbook or library routine, a closed form
of the Newton-Schulz iteration on a matrix of known SVD, invariants of the
renormalisation, and special cases of the two update orders. They run on the
CPU only.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from oracle import lact_oracle as O

RNG = np.random.default_rng(20250529)


def _tiny(d=4, dh=8, n=7, seed=0):
    g = np.random.default_rng(seed)
    W1 = g.normal(size=(dh, d)) / math.sqrt(d)
    W2 = g.normal(size=(d, dh)) / math.sqrt(dh)
    W3 = g.normal(size=(dh, d)) / math.sqrt(d)
    K = g.normal(size=(n, d))
    V = g.normal(size=(n, d))
    eta = 0.01 * np.log1p(np.exp(g.normal(size=n))) + 0.05
    return W1, W2, W3, K, V, eta


# ---------------------------------------------------------------- silu pieces
def test_silu_matches_library_sigmoid():
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(O.silu(x), x * scipy.special.expit(x), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(O.sigmoid(x), scipy.special.expit(x), rtol=1e-14, atol=1e-300)


def test_silu_grad_is_derivative_of_silu():
    x = np.linspace(-8, 8, 321)
    h = 1e-6
    fd = (x + h) * scipy.special.expit(x + h) - (x - h) * scipy.special.expit(x - h)
    np.testing.assert_allclose(O.silu_grad(x), fd / (2 * h), rtol=1e-8, atol=1e-9)


# ------------------------------------------------------------------ readout
def test_apply_matches_elementwise_loops():
    W1, W2, W3, K, _, _ = _tiny(d=3, dh=5, n=4, seed=1)
    out = O.fast_weight_apply(W1, W2, W3, K)
    for i in range(K.shape[0]):
        for j in range(W2.shape[0]):
            acc = 0.0
            for r in range(W1.shape[0]):
                h1 = sum(W1[r, c] * K[i, c] for c in range(K.shape[1]))
                h3 = sum(W3[r, c] * K[i, c] for c in range(K.shape[1]))
                acc += W2[j, r] * (h1 / (1.0 + math.exp(-h1))) * h3
            assert abs(out[i, j] - acc) < 1e-12


def test_apply_permutation_case_by_hand():
    # W1 = diag(s) P, W3 = R (permutation), W2 = T (permutation), d = dh = 3:
    # o_j = silu(s_r q_{P(r)}) q_{R(r)} with r = T^{-1}(j).
    q = np.array([0.3, -1.2, 2.0])
    s = np.array([1.5, -0.5, 2.0])
    P = np.eye(3)[[2, 0, 1]]
    R = np.eye(3)[[1, 2, 0]]
    T = np.eye(3)[[1, 0, 2]]
    o = O.fast_weight_apply(np.diag(s) @ P, T, R, q[None, :])[0]
    h1 = s * q[[2, 0, 1]]
    u = h1 * scipy.special.expit(h1) * q[[1, 2, 0]]
    np.testing.assert_allclose(o, u[[1, 0, 2]], rtol=1e-14)


def test_apply_zero_gate_matrix_gives_zero():
    W1, W2, W3, K, _, _ = _tiny(seed=2)
    assert np.all(O.fast_weight_apply(W1, W2, np.zeros_like(W3), K) == 0.0)


# ----------------------------------------------------------------- gradient
@pytest.mark.parametrize("seed", [3, 4])
def test_gradient_matches_central_differences(seed):
    W1, W2, W3, K, V, eta = _tiny(seed=seed)
    g = O.chunk_gradient(W1, W2, W3, K, V, eta)
    Ws = [W1, W2, W3]
    h = 1e-6
    for m in range(3):
        fd = np.zeros_like(Ws[m])
        for idx in np.ndindex(Ws[m].shape):
            plus = [w.copy() for w in Ws]
            minus = [w.copy() for w in Ws]
            plus[m][idx] += h
            minus[m][idx] -= h
            fd[idx] = (O.chunk_loss(*plus, K, V, eta) - O.chunk_loss(*minus, K, V, eta)) / (2 * h)
        err = np.max(np.abs(fd - g[m])) / np.max(np.abs(g[m]))
        assert err < 1e-7, (m, err)


def test_gradient_single_token_closed_form():
    W1, W2, W3, K, V, eta = _tiny(n=1, seed=5)
    k, v, e = K[0], V[0], eta[0]
    h1, h3 = W1 @ k, W3 @ k
    sg = scipy.special.expit(h1)
    u = h1 * sg * h3
    back = W2.T @ v                        # W2^T v
    dW2 = -e * np.outer(v, u)
    dW1 = -e * np.outer(back * h3 * sg * (1 + h1 * (1 - sg)), k)
    dW3 = -e * np.outer(back * h1 * sg, k)
    g = O.chunk_gradient(W1, W2, W3, K, V, eta)
    for a, b in zip(g, (dW1, dW2, dW3)):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)


def test_gradient_is_sum_over_tokens_and_linear_in_eta():
    W1, W2, W3, K, V, eta = _tiny(n=9, seed=6)
    g = O.chunk_gradient(W1, W2, W3, K, V, eta)
    parts = [O.chunk_gradient(W1, W2, W3, K[i:i + 1], V[i:i + 1], eta[i:i + 1]) for i in range(9)]
    for m in range(3):
        np.testing.assert_allclose(g[m], sum(p[m] for p in parts), rtol=1e-12, atol=1e-15)
    g3 = O.chunk_gradient(W1, W2, W3, K, V, 3.0 * eta)
    for m in range(3):
        np.testing.assert_allclose(g3[m], 3.0 * g[m], rtol=1e-12, atol=1e-15)
    g0 = O.chunk_gradient(W1, W2, W3, K, np.zeros_like(V), eta)
    assert all(np.all(x == 0.0) for x in g0)


# ------------------------------------------------------------- bf16 rounding
def test_bf16_round_matches_torch_conversion():
    x = RNG.normal(size=20000).astype(np.float32) * np.float32(3.0)
    # exact ties: an 8-bit significand plus half a unit in the last place,
    # in [1, 2) (ulp 2**-7) and in [0.25, 0.5)
    sig = np.arange(128, 256, dtype=np.float32)
    ties = np.concatenate([(sig + np.float32(0.5)) / np.float32(128.0),
                           (sig + np.float32(0.5)) / np.float32(512.0)])
    x = np.concatenate([x, ties, -ties, np.float32([0.0, 1.0, -2.5])])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(x.astype(np.float64)), want)


# ------------------------------------------------------------ Newton-Schulz
def _scalar_ns(x, steps=5, a=O.NS_A, b=O.NS_B, c=O.NS_C):
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def _orth(n, g):
    q, r = np.linalg.qr(g.normal(size=(n, n)))
    return q * np.sign(np.diag(r))


@pytest.mark.parametrize("shape", [(6, 10), (10, 6), (8, 8)])
def test_newton_schulz_closed_form_on_known_svd(shape):
    g = np.random.default_rng(7)
    m, n = shape
    k = min(m, n)
    U, V = _orth(m, g), _orth(n, g)
    s = np.sort(g.uniform(0.2, 3.0, size=k))[::-1]
    G = U[:, :k] @ np.diag(s) @ V[:, :k].T
    want = U[:, :k] @ np.diag(_scalar_ns(s / (np.linalg.norm(s) + O.NS_EPS))) @ V[:, :k].T
    got = O.newton_schulz5(G, bf16_points=False)
    np.testing.assert_allclose(got, want, atol=1e-11)
    # with the bf16 rounding points the iteration drifts from the exact one
    # by a few percent on small matrices (rounding of X amplified by p'(x))
    got16 = O.newton_schulz5(G, bf16_points=True)
    assert np.linalg.norm(got16 - want) / np.linalg.norm(want) < 8e-2


def test_newton_schulz_diagonal_reduces_to_scalar_iteration_with_rounding():
    s = np.array([0.9, 0.5, 0.31, 0.07, 0.02])
    G = np.zeros((5, 7))
    G[np.arange(5), np.arange(5)] = s
    x = s / (np.linalg.norm(s) + O.NS_EPS)
    r = O.bf16_round
    for _ in range(5):
        xr = r(x)
        A = xr * xr
        Bm = O.NS_B * A + O.NS_C * r(A) * r(A)
        x = O.NS_A * x + r(Bm) * xr
    want = np.zeros((5, 7))
    want[np.arange(5), np.arange(5)] = x
    np.testing.assert_array_equal(O.newton_schulz5(G, bf16_points=True), want)


def test_newton_schulz_invariances():
    g = np.random.default_rng(8)
    G = g.normal(size=(5, 9))
    P, R = _orth(5, g), _orth(9, g)
    base = O.newton_schulz5(G, bf16_points=False)
    np.testing.assert_allclose(O.newton_schulz5(G.T, bf16_points=False), base.T, atol=1e-12)
    np.testing.assert_allclose(O.newton_schulz5(P @ G @ R, bf16_points=False), P @ base @ R, atol=1e-11)
    np.testing.assert_array_equal(O.newton_schulz5(G.T), O.newton_schulz5(G).T)


def test_newton_schulz_singular_values_in_band():
    # The published property of these quintic coefficients: after five steps
    # the singular values land roughly in [0.5, 1.5] rather than exactly at 1,
    # for every normalised input singular value not too close to zero.
    g = np.random.default_rng(9)
    for _ in range(5):
        G = g.normal(size=(16, 48))
        sv_in = np.linalg.svd(G / np.linalg.norm(G), compute_uv=False)
        assert sv_in.min() > 2e-3
        for pts in (False, True):
            sv = np.linalg.svd(O.newton_schulz5(G, bf16_points=pts), compute_uv=False)
            assert sv.min() > 0.5 and sv.max() < 1.5


# ----------------------------------------------------------- renormalisation
def test_renorm_preserves_row_norms_and_direction():
    g = np.random.default_rng(10)
    W = g.normal(size=(12, 7))
    D = 0.3 * g.normal(size=(12, 7))
    W[3] = 0.0
    D[3] = 0.0
    out = O.renorm_update(W, D)
    np.testing.assert_allclose(np.linalg.norm(out, axis=1), np.linalg.norm(W, axis=1), rtol=1e-14)
    Wt = W + D
    for j in range(12):
        if j == 3:
            assert np.all(out[j] == 0.0)
            continue
        cos = out[j] @ Wt[j] / (np.linalg.norm(out[j]) * np.linalg.norm(Wt[j]))
        assert abs(cos - 1.0) < 1e-14
    np.testing.assert_allclose(O.renorm_update(W, np.zeros_like(W)), W, rtol=1e-15)


def test_gd_step_lowers_loss_before_renorm():
    W1, W2, W3, K, V, eta = _tiny(n=16, seed=11)
    eta = eta * 0.05
    L0 = O.chunk_loss(W1, W2, W3, K, V, eta)
    g = O.chunk_gradient(W1, W2, W3, K, V, eta)
    L1 = O.chunk_loss(W1 - g[0], W2 - g[1], W3 - g[2], K, V, eta)
    assert L1 < L0


# ------------------------------------------------------------------- orders
def test_causal_single_chunk_reads_initial_weights():
    W1, W2, W3, K, V, eta = _tiny(n=10, seed=12)
    Q = np.random.default_rng(13).normal(size=K.shape)
    o, Wf = O.sequence_causal((W1, W2, W3), Q, K, V, eta, chunk=10, opt="gd")
    np.testing.assert_array_equal(o, O.fast_weight_apply(W1, W2, W3, Q))
    Wu = O.chunk_update((W1, W2, W3), K, V, eta, "gd")
    for a, b in zip(Wf, Wu):
        np.testing.assert_array_equal(a, b)


def test_causal_chunks_read_only_earlier_chunks():
    W1, W2, W3, K, V, eta = _tiny(n=12, seed=14)
    Q = np.random.default_rng(15).normal(size=K.shape)
    o, _ = O.sequence_causal((W1, W2, W3), Q, K, V, eta, chunk=4, opt="muon")
    np.testing.assert_array_equal(o[:4], O.fast_weight_apply(W1, W2, W3, Q[:4]))
    W = O.chunk_update((W1, W2, W3), K[:4], V[:4], eta[:4], "muon")
    np.testing.assert_array_equal(o[4:8], O.fast_weight_apply(*W, Q[4:8]))
    # changing a later chunk's keys does not change earlier outputs
    K2 = K.copy()
    K2[8:] += 1.0
    o2, _ = O.sequence_causal((W1, W2, W3), Q, K2, V, eta, chunk=4, opt="muon")
    np.testing.assert_array_equal(o2[:8], o[:8])


def test_set_mode_is_update_then_apply_and_slices_sum():
    W1, W2, W3, K, V, eta = _tiny(n=20, seed=16)
    Q = np.random.default_rng(17).normal(size=(5, K.shape[1]))
    o, Wf = O.sequence_set((W1, W2, W3), Q, K, V, eta, opt="muon")
    Wu = O.chunk_update((W1, W2, W3), K, V, eta, "muon")
    np.testing.assert_allclose(o, O.fast_weight_apply(*Wu, Q), rtol=0, atol=0)
    o2, W2f = O.sequence_set((W1, W2, W3), Q, K, V, eta, opt="muon", token_slice=7)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------- momentum
def _chunks(seed, n_chunks=3, chunk=5, d=4, dh=8):
    W1, W2, W3, _, _, _ = _tiny(d=d, dh=dh, n=1, seed=seed)
    g = np.random.default_rng(seed + 100)
    K = g.normal(size=(n_chunks * chunk, d))
    V = g.normal(size=(n_chunks * chunk, d))
    eta = 0.02 + 0.01 * g.random(n_chunks * chunk)
    return (W1, W2, W3), K, V, eta


def test_momentum_with_zero_beta_is_gradient_descent():
    W, K, V, eta = _chunks(7)
    o_m, W_m = O.sequence_causal(W, K, K, V, eta, 5, "momentum", beta=0.0)
    o_g, W_g = O.sequence_causal(W, K, K, V, eta, 5, "gd")
    np.testing.assert_array_equal(o_m, o_g)
    for a, b in zip(W_m, W_g):
        np.testing.assert_array_equal(a, b)


def test_momentum_step_is_geometric_sum_of_past_chunk_gradients():
    # Unrolled: the step after chunk c is -sum_{j <= c} beta^(c-j) g_j, with
    # g_j the chunk gradient at the weights chunk j read. Rebuild the
    # trajectory from that closed sum and compare with the oracle's run.
    beta, chunk = 0.9, 5
    W, K, V, eta = _chunks(8, n_chunks=4, chunk=chunk)
    _, W_final = O.sequence_causal(W, K, K, V, eta, chunk, "momentum", beta=beta)
    Wc, grads = W, []
    for c in range(4):
        sl = slice(c * chunk, (c + 1) * chunk)
        grads.append(O.chunk_gradient(*Wc, K[sl], V[sl], eta[sl]))
        step = [-sum(beta ** (c - j) * grads[j][m] for j in range(c + 1)) for m in range(3)]
        Wc = tuple(O.renorm_update(Wc[m], step[m]) for m in range(3))
    for a, b in zip(W_final, Wc):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_momentum_first_chunk_equals_gradient_descent():
    # the velocity starts at zero: after one chunk momentum and GD agree for any beta
    W, K, V, eta = _chunks(9, n_chunks=1)
    _, W_m = O.sequence_causal(W, K, K, V, eta, 5, "momentum", beta=0.9)
    _, W_g = O.sequence_causal(W, K, K, V, eta, 5, "gd")
    for a, b in zip(W_m, W_g):
        np.testing.assert_array_equal(a, b)


# ------------------------------------------------- linear fast-weight memory
def test_linear_gradient_matches_central_differences():
    g = np.random.default_rng(31)
    d, n = 5, 9
    W = g.normal(size=(d, d)) / math.sqrt(d)
    K, V = g.normal(size=(n, d)), g.normal(size=(n, d))
    eta = 0.02 + 0.01 * g.random(n)
    G = O.linear_chunk_gradient(W, K, V, eta)
    h = 1e-6
    for i in range(d):
        for j in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[i, j] += h
            Wm[i, j] -= h
            fd = (O.linear_chunk_loss(Wp, K, V, eta) - O.linear_chunk_loss(Wm, K, V, eta)) / (2 * h)
            assert abs(G[i, j] - fd) < 1e-8 * max(1.0, abs(fd))


def test_linear_readout_special_cases():
    g = np.random.default_rng(32)
    X = g.normal(size=(6, 4))
    np.testing.assert_array_equal(O.linear_apply(np.eye(4), X), X)
    P = np.eye(4)[[2, 0, 3, 1]]          # row i of P picks coordinate perm[i]
    np.testing.assert_array_equal(O.linear_apply(P, X), X[:, [2, 0, 3, 1]])


def test_linear_single_token_step_is_rank_one():
    # one token: the GD step -dL/dW is eta v k^T, a rank-one matrix
    g = np.random.default_rng(33)
    d = 6
    W = g.normal(size=(d, d))
    k, v = g.normal(size=(1, d)), g.normal(size=(1, d))
    step = -O.linear_chunk_gradient(W, k, v, np.array([0.3]))
    assert np.linalg.matrix_rank(step) == 1
    np.testing.assert_allclose(step @ k[0], 0.3 * v[0] * (k[0] @ k[0]), rtol=1e-13)


def test_linear_causal_and_set_orders():
    g = np.random.default_rng(34)
    d, n = 4, 12
    W = (g.normal(size=(d, d)),)
    Q, K, V = g.normal(size=(n, d)), g.normal(size=(n, d)), g.normal(size=(n, d))
    eta = 0.05 * np.ones(n)
    # causal, one chunk: the readout sees the initial weights
    o, _ = O.sequence_causal(W, Q, K, V, eta, n, "gd")
    np.testing.assert_array_equal(o, O.linear_apply(W[0], Q))
    # set: one step on all tokens, then the read with the new weights
    o2, W2 = O.sequence_set(W, Q, K, V, eta, "gd")
    W_exp = O.renorm_update(W[0], -O.linear_chunk_gradient(W[0], K, V, eta))
    np.testing.assert_allclose(W2[0], W_exp, rtol=1e-14)
    np.testing.assert_allclose(o2, Q @ W_exp.T, rtol=1e-13)


# ------------------------------------------------------------- Muon step
def test_muon_step_lowers_the_chunk_loss_for_a_small_rate():
    # A Muon step moves every matrix against its gradient: <dL/dW, NS5(dL/dW)>
    # is the sum of the gradient's singular values times positive quintic
    # images of them, so for a small rate the chunk loss (pinned above by
    # finite differences) drops, and by the first-order amount <g, D>.
    W1, W2, W3, K, V, eta = _tiny(n=16, seed=21)
    W = (W1, W2, W3)
    L0 = O.chunk_loss(*W, K, V, eta)
    g = O.chunk_gradient(*W, K, V, eta)
    for lr in (1e-4, 1e-3):
        D = [O.optimizer_delta(gm, "muon", lr=lr) for gm in g]
        first_order = sum(float(np.sum(gm * Dm)) for gm, Dm in zip(g, D))
        assert first_order < 0.0
        L1 = O.chunk_loss(*(Wm + Dm for Wm, Dm in zip(W, D)), K, V, eta)
        assert L1 < L0
        assert abs((L1 - L0) - first_order) < 0.05 * abs(first_order)


@pytest.mark.parametrize("shape", [(6, 10), (10, 6)])
def test_muon_step_is_minus_lr_times_the_quintic_spectrum(shape):
    # For G = U diag(s) V^T the step is -lr U diag(phi(s / |s|)) V^T, phi the
    # scalar quintic map applied five times: the rate scales it, the sign is
    # negative, and the singular vectors are the gradient's. The bf16 rounding
    # points move the spectrum by a few percent on small matrices (the
    # closed-form test above allows 8e-2 for the same reason).
    g = np.random.default_rng(22)
    m, n = shape
    k = min(m, n)
    U, V = _orth(m, g), _orth(n, g)
    s = np.sort(g.uniform(0.5, 2.0, size=k))[::-1]
    G = U[:, :k] @ np.diag(s) @ V[:, :k].T
    phi = _scalar_ns(s / (np.linalg.norm(s) + O.NS_EPS))
    for lr in (0.02, 0.5):
        D = O.optimizer_delta(G, "muon", lr=lr)
        core = U[:, :k].T @ D @ V[:, :k]            # diag(-lr phi) up to rounding drift
        want = -lr * np.diag(phi)
        assert np.linalg.norm(core - want) / np.linalg.norm(want) < 8e-2
        # next to nothing outside the gradient's singular subspaces (only the
        # rounding of the bf16 operands leaks there)
        inside = U[:, :k] @ core @ V[:, :k].T
        assert np.linalg.norm(D - inside) / np.linalg.norm(D) < 2e-2


def test_gd_step_is_minus_the_gradient():
    g = np.random.default_rng(23).normal(size=(5, 7))
    np.testing.assert_array_equal(O.optimizer_delta(g, "gd"), -g)


def test_renorm_of_a_row_updated_to_zero_stores_the_zero_row():
    # a row whose updated norm is 0 cannot be rescaled to its old norm: it is
    # stored as updated (zero), not restored
    W = np.array([[3.0, 4.0], [1.0, -2.0]])
    D = np.array([[-3.0, -4.0], [0.5, 0.5]])
    out = O.renorm_update(W, D)
    assert np.all(out[0] == 0.0)
    np.testing.assert_allclose(np.linalg.norm(out[1]), np.linalg.norm(W[1]), rtol=1e-15)


# ------------------------------------------------------- whole-workload driver
def test_run_workload_gives_every_batch_entry_its_heads_initial_weights():
    # Two batch entries x two heads, built by hand: entry 1 repeats entry 0's
    # tokens, the heads have different initial weights. The fast weights are
    # per (b, h), initialised from head h for every b: both entries of a head
    # end identical, the heads differ, and the first causal chunk of (b, h)
    # reads head h's initial weights (brute-force readout loops above pin
    # fast_weight_apply).
    import lact_inputs as li
    g = np.random.default_rng(24)
    d, dh, n, ch = 4, 8, 6, 3
    w = li.Workload(0, "hand-built", 2, 2, d, dh, "f32", "causal", "gd", n, n, ch, 0)
    tok = lambda: np.repeat(g.normal(size=(1, 2, n, d)).astype(np.float32), 2, axis=0)
    q, k, v = tok(), tok(), tok()
    eta = np.repeat((0.05 + 0.01 * g.random((1, 2, n))).astype(np.float32), 2, axis=0)
    Wh = [(g.normal(size=s) * 0.5).astype(np.float32) for s in ((2, dh, d), (2, d, dh), (2, dh, d))]
    inp = li.Inputs(q, k, v, eta, *Wh)
    O_, W1, W2, W3 = O.run_workload(w, inp)
    for Wf in (O_, W1, W2, W3):
        np.testing.assert_array_equal(Wf[0], Wf[1])
        assert not np.allclose(Wf[0, 0], Wf[0, 1])
    for b in range(2):
        for h in range(2):
            first = O.fast_weight_apply(*(x[h].astype(np.float64) for x in Wh), q[b, h, :ch].astype(np.float64))
            np.testing.assert_allclose(O_[b, h, :ch], first, rtol=1e-13)
    # only the listed heads are computed
    O2, *_ = O.run_workload(w, inp, heads=[(1, 0)])
    np.testing.assert_array_equal(O2[1, 0], O_[1, 0])
    assert np.all(O2[0] == 0.0) and np.all(O2[1, 1] == 0.0)

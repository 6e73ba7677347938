"""Pins of the gated-DeltaNet replay oracle (oracle/gdn.py) against facts that
do not come from the oracle itself: closed forms of the gated delta rule,
central finite differences, an explicit-matrix brute force, and planted
mistakes that one of these must reject."""
import numpy as np
import pytest
import torch

from oracle.gdn import gdn_replay


def _case(H=2, dk=5, dv=4, R=7, seed=0, g0=None, b0=None, unit_k=True):
    rng = np.random.default_rng(seed)
    s0 = rng.standard_normal((H, dv, dk))
    q = rng.standard_normal((R, H, dk))
    k = rng.standard_normal((R, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((R, H, dv))
    g = np.log(rng.uniform(0.7, 1.0, (R, H))) if g0 is None else np.full((R, H), g0)
    b = rng.uniform(0.1, 0.9, (R, H)) if b0 is None else np.full((R, H), b0)
    d_o = rng.standard_normal((R, H, dv))
    return s0, q, k, v, g, b, d_o


def test_no_decay_no_write_keeps_the_captured_state():
    """g = 0, b = 0: S_t = S_0, so o_t = S_0 q_t, dq_t = S_0^T dO_t, dk = dv = 0,
    dg_t = sum_{s>=t} dO_s^T S_0 q_s, db_t = (v_t - S_0 k_t)^T G_t k_t with
    G_t = sum_{s>=t} dO_s q_s^T."""
    s0, q, k, v, g, b, d_o = _case(g0=0.0, b0=0.0)
    r = gdn_replay(s0, q, k, v, g, b, d_o)
    R, H = g.shape
    for h in range(H):
        S = s0[h]
        np.testing.assert_allclose(r["o"][:, h], q[:, h] @ S.T, atol=1e-12)
        np.testing.assert_allclose(r["dq"][:, h], d_o[:, h] @ S, atol=1e-12)
        for t in range(R):
            G = sum(np.outer(d_o[s, h], q[s, h]) for s in range(t, R))
            np.testing.assert_allclose(r["dg"][t, h], np.sum(G * S), atol=1e-10)
            w = v[t, h] - S @ k[t, h]
            np.testing.assert_allclose(r["dbeta"][t, h], w @ G @ k[t, h], atol=1e-10)
    assert np.abs(r["dk"]).max() < 1e-12 and np.abs(r["dv"]).max() < 1e-12
    np.testing.assert_allclose(r["s_final"], s0, atol=1e-12)


def test_full_write_stores_the_value_under_its_key():
    """b = 1 and |k_t| = 1: S_t k_t = a S_{t-1} (k_t - k_t) + v_t = v_t, whatever
    the decay; with q_t = k_t the output is v_t."""
    s0, q, k, v, g, b, d_o = _case(b0=1.0)
    r = gdn_replay(s0, k, k, v, g, b)
    np.testing.assert_allclose(r["o"], v, atol=1e-12)
    H = g.shape[1]
    for h in range(H):
        np.testing.assert_allclose(r["s_final"][h] @ k[-1, h], v[-1, h], atol=1e-12)


def _brute(s0, q, k, v, g, b):
    R, H, dk = q.shape
    o = np.zeros((R, H, v.shape[2]))
    fin = np.zeros_like(s0)
    for h in range(H):
        S = s0[h].copy()
        for t in range(R):
            kt = k[t, h][:, None]
            S = np.exp(g[t, h]) * S @ (np.eye(dk) - b[t, h] * kt @ kt.T) + b[t, h] * v[t, h][:, None] @ kt.T
            o[t, h] = S @ q[t, h]
        fin[h] = S
    return o, fin


def test_explicit_matrix_brute_force():
    s0, q, k, v, g, b, _ = _case(H=3, dk=6, dv=3, R=9, seed=3, unit_k=False)
    r = gdn_replay(s0, q, k, v, g, b)
    o, fin = _brute(s0, q, k, v, g, b)
    np.testing.assert_allclose(r["o"], o, atol=1e-12)
    np.testing.assert_allclose(r["s_final"], fin, atol=1e-12)


@pytest.mark.parametrize("name", ["q", "k", "v", "g", "beta"])
def test_finite_differences(name):
    s0, q, k, v, g, b, d_o = _case(H=2, dk=3, dv=4, R=5, seed=7, unit_k=False)
    args = {"q": q, "k": k, "v": v, "g": g, "beta": b}
    r = gdn_replay(s0, q, k, v, g, b, d_o)
    grad = r["d" + name]
    eps = 1e-6
    x = args[name]
    num = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        for sgn in (1, -1):
            xx = x.copy()
            xx[i] += sgn * eps
            a2 = dict(args, **{name: xx})
            o = gdn_replay(s0, a2["q"], a2["k"], a2["v"], a2["g"], a2["beta"])["o"]
            num[i] += sgn * np.sum(o * d_o) / (2 * eps)
    np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-7)


def test_planted_mistakes_are_caught():
    """A write scaled by the decay, or a missing decay, breaks one of the pins."""
    s0, q, k, v, g, b, _ = _case(b0=1.0, seed=11)

    def scaled_write(s0, q, k, v, g, b):  # a_t * b_t v_t k_t^T instead of b_t v_t k_t^T
        R, H, dk = q.shape
        o = np.zeros((R, H, v.shape[2]))
        for h in range(H):
            S = s0[h].copy()
            for t in range(R):
                a = np.exp(g[t, h])
                S = a * (S - b[t, h] * np.outer(S @ k[t, h], k[t, h]) + b[t, h] * np.outer(v[t, h], k[t, h]))
                o[t, h] = S @ q[t, h]
        return o

    assert np.abs(scaled_write(s0, k, k, v, g, b) - v).max() > 1e-3  # fails the full-write pin
    o_nodecay, _ = _brute(s0, q, k, v, np.zeros_like(g), b)
    assert np.abs(o_nodecay - gdn_replay(s0, q, k, v, g, b)["o"]).max() > 1e-3


def test_empty_response():
    s0, q, k, v, g, b, d_o = _case(R=0)
    r = gdn_replay(s0, q, k, v, g, b, d_o)
    assert r["o"].shape == (0, 2, 4)
    np.testing.assert_allclose(r["s_final"], s0)


def _chunkwise(s0, q, k, v, g, b, C):
    """The same rule in chunkwise form, derived independently of the oracle's
    loop.  Within a chunk, with gamma_t the running product of the decays and
    e_t = b_t (v_t - a_t S_{t-1} k_t):
        S_t = gamma_t S_0 + sum_{s<=t} (gamma_t / gamma_s) e_s k_s^T,
    so the e_t solve a unit lower-triangular system
        (I + A) E = diag(b) (V - diag(gamma) K S_0^T),
        A_ts = b_t (gamma_t / gamma_s) k_t . k_s   (s < t),
    and O = diag(gamma) Q S_0^T + (tril(Gamma) * Q K^T) E,
        S_C = gamma_C S_0 + E^T diag(gamma_C / gamma) K."""
    R, H, _ = q.shape
    o = np.zeros((R, H, v.shape[2]))
    fin = np.zeros_like(s0)
    for h in range(H):
        S = s0[h].copy()
        for c0 in range(0, R, C):
            sl = slice(c0, min(R, c0 + C))
            Q, K, V = q[sl, h], k[sl, h], v[sl, h]
            gam = np.exp(np.cumsum(g[sl, h]))
            bt = b[sl, h]
            ratio = gam[:, None] / gam[None, :]
            n = len(gam)
            A = np.tril(bt[:, None] * ratio * (K @ K.T), -1)
            E = np.linalg.solve(np.eye(n) + A, bt[:, None] * (V - gam[:, None] * (K @ S.T)))
            o[sl, h] = gam[:, None] * (Q @ S.T) + (np.tril(ratio) * (Q @ K.T)) @ E
            S = gam[-1] * S + E.T @ ((gam[-1] / gam)[:, None] * K)
        fin[h] = S
    return o, fin


@pytest.mark.parametrize("C", [1, 4, 16])
def test_chunkwise_form_equals_the_recurrence(C):
    s0, q, k, v, g, b, _ = _case(H=2, dk=6, dv=5, R=13, seed=17, unit_k=False)
    r = gdn_replay(s0, q, k, v, g, b)
    o, fin = _chunkwise(s0, q, k, v, g, b, C)
    np.testing.assert_allclose(r["o"], o, atol=1e-11)
    np.testing.assert_allclose(r["s_final"], fin, atol=1e-11)


def _chunk_grads(S, Q, K, V, g, b, dO, G_end):
    """Backward of one chunk of the chunkwise form, derived by hand: the
    gradients for Q, K, V, g, b and dL/dS at the chunk's start, given dO and
    dL/dS at its end.  All products are dense; the one solve is the
    transposed triangular system of the forward."""
    n = len(g)
    c = np.cumsum(g)
    gam = np.exp(c)
    Gam = np.exp(c[:, None] - c[None, :])
    L = np.tril(np.ones((n, n)))
    KK = K @ K.T
    A = np.tril(b[:, None] * Gam * KK, -1)
    X = V - gam[:, None] * (K @ S.T)
    E = np.linalg.solve(np.eye(n) + A, b[:, None] * X)
    P = L * Gam * (Q @ K.T)
    w = np.exp(c[-1] - c)
    # O = diag(gam) Q S^T + P E;  S_end = gam_n S + E^T diag(w) K
    dE = P.T @ dO + (w[:, None] * K) @ G_end.T
    dP = dO @ E.T
    dW = E @ G_end
    dS = dO.T @ (gam[:, None] * Q) + gam[-1] * G_end
    dgam = (dO * (Q @ S.T)).sum(1)
    LdP = L * Gam * dP
    dQ = gam[:, None] * (dO @ S) + LdP @ K
    dK = LdP.T @ Q
    dGam = L * dP * (Q @ K.T)
    dU = np.linalg.solve((np.eye(n) + A).T, dE)       # E = (I + A)^-1 U
    dA = -np.tril(dU @ E.T, -1)
    db = (dA * Gam * KK).sum(1) + (dU * X).sum(1)
    dGam += dA * b[:, None] * KK
    dKK = dA * b[:, None] * Gam
    dK += (dKK + dKK.T) @ K
    dX = b[:, None] * dU                               # U = diag(b) X
    dV = dX
    dgam -= (dX * (K @ S.T)).sum(1)
    dK += -gam[:, None] * (dX @ S) + w[:, None] * dW
    dS -= dX.T @ (gam[:, None] * K)
    # back to the log-decays through gam, Gam, w and gam_n, then g = diff(c)
    r = dGam * Gam
    rw = (dW * K).sum(1) * w
    dc = dgam * gam + r.sum(1) - r.sum(0) - rw
    dc[-1] += rw.sum() + (G_end * S).sum() * gam[-1]
    dg = np.cumsum(dc[::-1])[::-1]
    return dQ, dK, dV, dg, db, dS


@pytest.mark.parametrize("C", [1, 4, 8, 23])
def test_chunkwise_backward_equals_the_oracle_gradients(C):
    """The oracle's gradients (autograd of its step loop) against a chunkwise
    backward derived by hand: forward over the chunks keeping each chunk's
    starting state, then the chunks in reverse, carrying dL/dS."""
    s0, q, k, v, g, b, d_o = _case(H=2, dk=6, dv=5, R=23, seed=3, unit_k=False)
    want = gdn_replay(s0, q, k, v, g, b, d_o)
    R, H, _ = q.shape
    got = {x: np.zeros_like(want[x]) for x in ("dq", "dk", "dv", "dg", "dbeta")}
    for h in range(H):
        chunks = [(c0, min(R, c0 + C)) for c0 in range(0, R, C)]
        starts, S = [], s0[h].copy()
        for c0, c1 in chunks:
            starts.append(S)
            S = gdn_replay(S[None], q[c0:c1, h:h + 1], k[c0:c1, h:h + 1], v[c0:c1, h:h + 1],
                           g[c0:c1, h:h + 1], b[c0:c1, h:h + 1])["s_final"][0]
        G = np.zeros_like(S)
        for (c0, c1), S0 in reversed(list(zip(chunks, starts))):
            sl = slice(c0, c1)
            dQ, dK, dV, dg, db, G = _chunk_grads(S0, q[sl, h], k[sl, h], v[sl, h], g[sl, h],
                                                 b[sl, h], d_o[sl, h], G)
            got["dq"][sl, h], got["dk"][sl, h], got["dv"][sl, h] = dQ, dK, dV
            got["dg"][sl, h], got["dbeta"][sl, h] = dg, db
    for x in got:
        np.testing.assert_allclose(got[x], want[x], atol=1e-10, err_msg=x)


def test_state_gradient_is_linear_across_a_chunk():
    """dL/dS at a chunk's start depends on dL/dS at its end through one fixed
    matrix, G_start = G_end M + C with M = gamma_C I - W^T (I + A)^-1
    diag(gamma b) K: the chunks' backward can run in parallel, with only
    this product chained over them."""
    rng = np.random.default_rng(0)
    n, dk, dv = 7, 5, 4
    S, Q, K = rng.standard_normal((dv, dk)), rng.standard_normal((n, dk)), rng.standard_normal((n, dk))
    V, dO = rng.standard_normal((n, dv)), rng.standard_normal((n, dv))
    g, b = np.log(rng.uniform(0.7, 1, n)), rng.uniform(0.1, 0.9, n)
    G1 = rng.standard_normal((dv, dk))
    dS1 = _chunk_grads(S, Q, K, V, g, b, dO, G1)[5]
    dS0 = _chunk_grads(S, Q, K, V, g, b, dO, np.zeros((dv, dk)))[5]
    c = np.cumsum(g)
    gam = np.exp(c)
    A = np.tril(b[:, None] * np.exp(c[:, None] - c[None, :]) * (K @ K.T), -1)
    W = np.exp(c[-1] - c)[:, None] * K
    M = gam[-1] * np.eye(dk) - W.T @ np.linalg.solve(np.eye(n) + A, np.diag(gam * b) @ K)
    np.testing.assert_allclose(dS1 - dS0, G1 @ M, atol=1e-12)


def _cp_prep(K, Q, V, dO, g, b):
    """Chunk-local solves of the chunk-parallel form (no state, no dL/dS):
    E0 = T diag(b) V, ZK = T diag(b gamma) K, dU0 = T^T P^T dO, ZW = T^T W,
    with T = (I + A)^-1."""
    n = len(g)
    c = np.cumsum(g)
    gam = np.exp(c)
    Gam = np.exp(c[:, None] - c[None, :])
    IA = np.eye(n) + b[:, None] * np.tril(Gam * (K @ K.T), -1)
    Pt = np.tril(Gam * (Q @ K.T)).T
    W = np.exp(c[-1] - c)[:, None] * K
    return (np.linalg.solve(IA, b[:, None] * V), np.linalg.solve(IA, (b * gam)[:, None] * K),
            np.linalg.solve(IA.T, Pt @ dO), np.linalg.solve(IA.T, W))


def _chunk_parallel(s0, q, k, v, g, b, d_o, C, chains="explicit"):
    """The replay and its gradients in three stages: chunk-local solves (all
    chunks independent), then the two linear chains over the chunks (the state
    forward, E = E0 - ZK S^T, S <- gamma_C S + E^T W; dL/dS backward,
    dU = dU0 + ZW G^T, G <- gamma_C G + (gamma dO)^T Q - (gamma b dU)^T K),
    then every output chunk by chunk from its starting state, its final dL/dS,
    E and dU (independent again).  chains="affine" runs the same chains with
    E and dU expanded into per-chunk terms formed beforehand:
    S <- gamma_C S - S M + F, G <- gamma_C G - G M' + F', with M = ZK^T W,
    F = E0^T W, M' = ZW^T diag(gamma b) K, F' = (gamma dO)^T Q - (gamma b dU0)^T K;
    E and dU then come from S and G chunk by chunk."""
    R = len(g)
    chunks = [(a, min(R, a + C)) for a in range(0, R, C)]
    pre = [_cp_prep(k[a:e], q[a:e], v[a:e], d_o[a:e], g[a:e], b[a:e]) for a, e in chunks]
    S, S_start, E = s0.copy(), [], []
    G, G_end, dU = np.zeros_like(s0), [None] * len(chunks), [None] * len(chunks)
    if chains == "affine":
        terms = []
        for (a, e), (E0, ZK, dU0, ZW) in zip(chunks, pre):
            c = np.cumsum(g[a:e])
            gam, W = np.exp(c), np.exp(c[-1] - c)[:, None] * k[a:e]
            gb = (gam * b[a:e])[:, None]
            terms.append((np.exp(c[-1]), ZK.T @ W, E0.T @ W, ZW.T @ (gb * k[a:e]),
                          (gam[:, None] * d_o[a:e]).T @ q[a:e] - (gb * dU0).T @ k[a:e]))
        for (a, e), (E0, ZK, _, _), (gc, M, F, _, _) in zip(chunks, pre, terms):
            S_start.append(S)
            E.append(E0 - ZK @ S.T)
            S = gc * S - S @ M + F
        out = {"s_final": S}
        for ci in reversed(range(len(chunks))):
            gc, _, _, Mg, Fg = terms[ci]
            G_end[ci] = G
            dU[ci] = pre[ci][2] + pre[ci][3] @ G.T
            G = gc * G - G @ Mg + Fg
    else:
        for (a, e), (E0, ZK, _, _) in zip(chunks, pre):
            S_start.append(S)
            c = np.cumsum(g[a:e])
            E.append(E0 - ZK @ S.T)
            S = np.exp(c[-1]) * S + E[-1].T @ (np.exp(c[-1] - c)[:, None] * k[a:e])
        out = {"s_final": S}
        for ci in reversed(range(len(chunks))):
            a, e = chunks[ci]
            G_end[ci] = G
            c = np.cumsum(g[a:e])
            gam = np.exp(c)
            dU[ci] = pre[ci][2] + pre[ci][3] @ G.T
            G = np.exp(c[-1]) * G + (gam[:, None] * d_o[a:e]).T @ q[a:e] - \
                ((gam * b[a:e])[:, None] * dU[ci]).T @ k[a:e]
    res = {x: np.zeros_like(t) for x, t in (("o", v), ("dq", q), ("dk", k), ("dv", v),
                                             ("dg", g), ("dbeta", b))}
    for ci, (a, e) in enumerate(chunks):
        S0, Gc, Ec, dUc = S_start[ci], G_end[ci], E[ci], dU[ci]
        Q, K, V, dO, gg, bb = q[a:e], k[a:e], v[a:e], d_o[a:e], g[a:e], b[a:e]
        n = e - a
        c = np.cumsum(gg)
        gam, w = np.exp(c), np.exp(c[-1] - c)
        Gam = np.exp(c[:, None] - c[None, :])
        L = np.tril(np.ones((n, n)))
        P = L * Gam * (Q @ K.T)
        GK = np.tril(Gam * (K @ K.T), -1)
        dP, dW = dO @ Ec.T, Ec @ Gc
        LdP = L * Gam * dP
        dA = -np.tril(dUc @ Ec.T, -1)
        Msym = dA * bb[:, None] * Gam
        Msym = Msym + Msym.T
        res["o"][a:e] = gam[:, None] * (Q @ S0.T) + P @ Ec
        res["dq"][a:e] = gam[:, None] * (dO @ S0) + LdP @ K
        res["dk"][a:e] = LdP.T @ Q + Msym @ K - ((gam * bb)[:, None] * dUc) @ S0 + w[:, None] * dW
        res["dv"][a:e] = bb[:, None] * dUc
        res["dbeta"][a:e] = (dA * GK).sum(1) + (dUc * (V - gam[:, None] * (K @ S0.T))).sum(1)
        dgam = (dO * (Q @ S0.T)).sum(1) - (bb[:, None] * dUc * (K @ S0.T)).sum(1)
        r = dP * P + dA * bb[:, None] * GK
        rw = (dW * K).sum(1) * w
        dc = dgam * gam + r.sum(1) - r.sum(0) - rw
        dc[-1] += rw.sum() + (Gc * S0).sum() * gam[-1]
        res["dg"][a:e] = np.cumsum(dc[::-1])[::-1]
    out.update(res)
    return out


@pytest.mark.parametrize("chains", ["explicit", "affine"])
@pytest.mark.parametrize("C", [1, 4, 8, 23])
def test_chunk_parallel_form_equals_the_oracle(C, chains):
    s0, q, k, v, g, b, d_o = _case(H=1, dk=6, dv=5, R=23, seed=2, unit_k=False)
    want = gdn_replay(s0, q, k, v, g, b, d_o)
    got = _chunk_parallel(s0[0], q[:, 0], k[:, 0], v[:, 0], g[:, 0], b[:, 0], d_o[:, 0], C, chains)
    for x in ("o", "dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(got[x], want[x][:, 0], atol=1e-10, err_msg=x)
    np.testing.assert_allclose(got["s_final"], want["s_final"][0], atol=1e-10)

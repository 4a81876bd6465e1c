"""FP64 per-token oracle of the gated delta rule with a per-channel decay (KDA).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name a sibling "Cake packed KDA" training family beside the GDN one
("perf(cake_kda) ... #7097" page and its "#7117" table notes: a chunked
training backend for packed documents, single-device and context-parallel)
but print no formula.  The plainest reading, and the one taken here, is the
GDN recurrence of gdn_oracle.c with its scalar decay a_t = exp(g_t) replaced
by one decay per key channel, a_t = exp(g_t) with g_t in R^dk:

  q^, k^ = l2norm(q), l2norm(k)   (or q, k when the norm is off)
  S'_t = Diag(a_t) S_{t-1}                       (dk x dv, row i scaled by a_t[i])
  S_t  = S'_t + beta_t k^_t (v_t - S'_t^T k^_t)^T
  o_t  = scale S_t^T q^_t

per document (S = 0 at each start) and value head; value head h reads q/k head
h / G.  The backward is the reverse mode of those four lines, token by token
from the end; per token, with dS the adjoint of S_t:

  dS += scale q^ do^T;  dq^ = scale S_t do
  u = v - S'^T k^:  dbeta = k^^T dS u;  du = beta dS^T k^;  dv = du
  dk^ = beta dS u - S' du;  dS' = dS - k^ du^T
  dg = a . rowsum(dS' . S_{t-1});  dS_{t-1} = Diag(a) dS'

followed by the L2-norm backward of q and k.  Shapes follow ref.group: q, k
[L, dk]; v [G, L, dv]; g [G, L, dk]; beta [G, L]; dO [G, L, dv].  numpy
vector operations over the channels serve as steps; nothing is blocked or
reordered beyond the lines above.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def _l2(x, on, eps):
    if not on:
        return x.copy(), np.ones(x.shape[0])
    n = np.sqrt((x * x).sum(-1) + eps)
    return x / n[:, None], n


def _l2_back(x, n, dxh, on):
    """d|x|-normalise backward: dx = dxh / n - x (x . dxh) / n^3 per row."""
    if not on:
        return dxh
    return dxh / n[:, None] - x * ((x * dxh).sum(-1) / n ** 3)[:, None]


def group(q, k, v, g, beta, dO=None, *, l2norm=True, scale=128 ** -0.5, eps=EPS, s_in=None):
    """Forward (+ backward when dO is given) of one document, one q/k group.

    Returns o [G, L, dv] and, with dO: dq, dk [L, dk], dv [G, L, dv],
    dg [G, L, dk], dbeta [G, L]; s_out [G, dk, dv] (the state after the last
    token).  s_in [G, dk, dv] is the state entering the document (zero if None).
    """
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    L, dk = q.shape
    G, _, dv = v.shape
    qh, nq = _l2(q, l2norm, eps)
    kh, nk = _l2(k, l2norm, eps)
    a = np.exp(g)                                        # [G, L, dk]
    S = np.zeros((G, dk, dv)) if s_in is None else np.array(s_in, dtype=np.float64).reshape(G, dk, dv)
    states = np.zeros((L + 1, G, dk, dv))               # S_{t-1} entering token t, then S_L
    o = np.zeros((G, L, dv))
    for t in range(L):
        states[t] = S
        Sp = a[:, t, :, None] * S                        # S'_t = Diag(a_t) S_{t-1}
        u = v[:, t] - np.einsum("gij,i->gj", Sp, kh[t])  # v - S'^T k^
        S = Sp + beta[:, t, None, None] * kh[t][None, :, None] * u[:, None, :]
        o[:, t] = scale * np.einsum("gij,i->gj", S, qh[t])
    states[L] = S
    out = dict(o=o, s_out=S.copy())
    if dO is None:
        return out
    dO = np.asarray(dO, dtype=np.float64)
    dqh = np.zeros((L, dk))
    dkh = np.zeros((L, dk))
    dvv = np.zeros((G, L, dv))
    dg = np.zeros((G, L, dk))
    db = np.zeros((G, L))
    dS = np.zeros((G, dk, dv))
    for t in range(L - 1, -1, -1):
        S_prev, S_t = states[t], states[t + 1]
        Sp = a[:, t, :, None] * S_prev
        u = v[:, t] - np.einsum("gij,i->gj", Sp, kh[t])
        # o_t = scale S_t^T q^
        dS = dS + scale * qh[t][None, :, None] * dO[:, t][:, None, :]
        dqh[t] += scale * np.einsum("gij,gj->i", S_t, dO[:, t])
        # S_t = S' + beta k^ u^T
        db[:, t] = np.einsum("i,gij,gj->g", kh[t], dS, u)
        du = beta[:, t, None] * np.einsum("gij,i->gj", dS, kh[t])
        dvv[:, t] = du
        dkh[t] += np.einsum("g,gij,gj->i", beta[:, t], dS, u)
        # u = v - S'^T k^
        dkh[t] -= np.einsum("gij,gj->i", Sp, du)
        dSp = dS - kh[t][None, :, None] * du[:, None, :]
        # S' = Diag(a) S_{t-1}
        dg[:, t] = a[:, t] * (dSp * S_prev).sum(-1)
        dS = a[:, t, :, None] * dSp
    out.update(dq=_l2_back(q, nq, dqh, l2norm), dk=_l2_back(k, nk, dkh, l2norm), dv=dvv, dg=dg, dbeta=db,
               ds_in=dS)
    return out


def chunk_forward(q, k, v, g, beta, *, l2norm=True, scale=128 ** -0.5, chunk=64, eps=EPS):
    """The chunk form of the same forward (the algebra a chunked kernel follows).

    Unrolling the recurrence over a chunk from its entering state S, with the
    per-channel cumulative log decay G_r = sum_{i<=r} g_i (a dk vector),
    gamma_r = exp(G_r) and the relative decays exp(G_r - G_c) (c <= r, every
    entry <= 1):
      M_rc = k^_r . (exp(G_r - G_c) k^_c)   A = strict_tril(diag(beta) M)
      T = (I + A)^-1,  U = T diag(beta) V,  W = T diag(beta) (gamma . K^)
      X = U - W S                          (X_r = beta_r times the new value u_r)
      O = scale ((gamma . Q^) S + tril_incl(P) X),  P_rc = q^_r . (exp(G_r - G_c) k^_c)
      S_next = Diag(gamma_L) S + ((exp(G_L - G_c) k^_c) rows)^T X
    which is the GDN chunk form with each decay moved inside the channel sums.
    Returns o [G, L, dv] and the states entering each chunk [n_chunks, G, dk, dv].
    """
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    L, dk = q.shape
    Gh, _, dv = v.shape
    qh, _ = _l2(q, l2norm, eps)
    kh, _ = _l2(k, l2norm, eps)
    bounds = [(c0, min(c0 + chunk, L)) for c0 in range(0, L, chunk)]
    o = np.zeros((Gh, L, dv))
    S_tape = np.zeros((len(bounds), Gh, dk, dv))
    for h in range(Gh):
        S = np.zeros((dk, dv))
        for c, (s, e) in enumerate(bounds):
            S_tape[c, h] = S
            n = e - s
            Gc = np.cumsum(g[h, s:e], axis=0)                        # [n, dk]
            gam = np.exp(Gc)
            low = np.tril(np.ones((n, n), dtype=bool))                # c <= r
            D = np.where(low[:, :, None], Gc[:, None, :] - Gc[None, :, :], -np.inf)
            R = np.exp(D)                                             # [r, c, channel], 0 above the diagonal
            M = np.einsum("ri,rci,ci->rc", kh[s:e], R, kh[s:e])
            P = np.einsum("ri,rci,ci->rc", qh[s:e], R, kh[s:e])
            b = beta[h, s:e]
            A = np.tril(b[:, None] * M, -1)
            T = np.linalg.inv(np.eye(n) + A)
            U = T @ (b[:, None] * v[h, s:e])
            W = T @ (b[:, None] * gam * kh[s:e])
            X = U - W @ S
            o[h, s:e] = scale * ((gam * qh[s:e]) @ S + P @ X)
            Kd = np.exp(Gc[-1][None, :] - Gc) * kh[s:e]
            S = gam[-1][:, None] * S + Kd.T @ X
    return dict(o=o, S=S_tape)


def chunk_backward(q, k, v, g, beta, dO, *, l2norm=True, scale=128 ** -0.5, chunk=64, eps=EPS):
    """The reverse of chunk_forward, chunk by chunk from the end (the algebra a
    chunked gradient kernel follows).  Per chunk, with dS the adjoint of the
    state leaving it and the forward's intermediates recomputed:
      dX = scale P^T dO + Kd dS                     dP = scale dO X^T (c <= r)
      dS_in = scale (gamma . Q^)^T dO + Diag(gamma_L) dS - W^T dX
      dU = dX,  dW = -dX S^T,  dT = dU (beta V)^T + dW (beta gamma . K^)^T
      dA = -T^T dT T^T (strictly lower),  dM = diag(beta) dA
    then dM, dP, the gamma and Kd terms go back through the per-channel decay
    products to q^, k^ and the cumulative log decay, and dg is its reverse
    cumulative sum within the chunk.  Returns the dict of group()'s gradients.
    """
    q, k, v, g, beta, dO = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, dO))
    L, dk = q.shape
    Gh, _, dv = v.shape
    qh, nq = _l2(q, l2norm, eps)
    kh, nk = _l2(k, l2norm, eps)
    states = chunk_forward(q, k, v, g, beta, l2norm=l2norm, scale=scale, chunk=chunk, eps=eps)["S"]
    bounds = [(c0, min(c0 + chunk, L)) for c0 in range(0, L, chunk)]
    dqh = np.zeros((L, dk))
    dkh = np.zeros((L, dk))
    dvv = np.zeros((Gh, L, dv))
    dg = np.zeros((Gh, L, dk))
    db = np.zeros((Gh, L))
    ds_in = np.zeros((Gh, dk, dv))
    for h in range(Gh):
        dS = np.zeros((dk, dv))
        for c in range(len(bounds) - 1, -1, -1):
            s, e = bounds[c]
            n = e - s
            S = states[c, h]
            Q, K, V, b = qh[s:e], kh[s:e], v[h, s:e], beta[h, s:e]
            # the forward of this chunk
            Gc = np.cumsum(g[h, s:e], axis=0)
            gam = np.exp(Gc)
            low = np.tril(np.ones((n, n), dtype=bool))
            R = np.exp(np.where(low[:, :, None], Gc[:, None, :] - Gc[None, :, :], -np.inf))
            M = np.einsum("ri,rci,ci->rc", K, R, K)
            P = np.einsum("ri,rci,ci->rc", Q, R, K)
            A = np.tril(b[:, None] * M, -1)
            T = np.linalg.inv(np.eye(n) + A)
            Y = b[:, None] * gam * K                      # W = T Y
            W = T @ Y
            X = T @ (b[:, None] * V) - W @ S
            E = np.exp(Gc[-1][None, :] - Gc)              # Kd = E . K
            Kd = E * K
            # O = scale ((gamma . Q) S + P X);  S_next = Diag(gamma_L) S + Kd^T X
            dOc = dO[h, s:e]
            dX = scale * P.T @ dOc + Kd @ dS
            dP = np.where(low, scale * dOc @ X.T, 0.0)
            dQg = scale * dOc @ S.T                       # adjoint of gamma . Q
            dQ = gam * dQg
            dgam = Q * dQg
            dS_prev = scale * (gam * Q).T @ dOc + gam[-1][:, None] * dS - W.T @ dX
            dGL = gam[-1] * (dS * S).sum(-1)              # through Diag(gamma_L)
            dKd = X @ dS.T
            dK = E * dKd
            dE = K * dKd * E                              # d(G_L - G_c) per entry
            dGL += dE.sum(0)
            dGc = -dE
            # X = U - W S,  U = T (beta V),  W = T Y
            dU = dX
            dW = -dX @ S.T
            dT = dU @ (b[:, None] * V).T + dW @ Y.T
            TdU = T.T @ dU
            dvv[h, s:e] = b[:, None] * TdU
            dbc = (V * TdU).sum(-1)
            dY = T.T @ dW
            dK += b[:, None] * gam * dY
            dgam += b[:, None] * K * dY
            dbc += (gam * K * dY).sum(-1)
            # T = (I + A)^-1,  A = strict_tril(diag(beta) M)
            dA = np.tril(-T.T @ dT @ T.T, -1)
            dbc += (dA * M).sum(-1)
            dM = b[:, None] * dA
            # M_rc = K_r . (R_rc . K_c),  P_rc = Q_r . (R_rc . K_c)
            dK += np.einsum("rc,rci,ci->ri", dM, R, K) + np.einsum("rc,rci,ri->ci", dM, R, K)
            dQ += np.einsum("rc,rci,ci->ri", dP, R, K)
            dK += np.einsum("rc,rci,ri->ci", dP, R, Q)
            dRR = (dM[:, :, None] * K[:, None, :] * K[None, :, :] + dP[:, :, None] * Q[:, None, :] * K[None, :, :]) * R
            dGc += dRR.sum(1) - dRR.sum(0)                # R_rc = exp(G_r - G_c)
            dGc += dgam * gam                             # gamma = exp(G)
            dGc[-1] += dGL                                # G_L = G of the last row
            dg[h, s:e] = np.cumsum(dGc[::-1], axis=0)[::-1]
            db[h, s:e] = dbc
            dqh[s:e] += dQ
            dkh[s:e] += dK
            dS = dS_prev
        ds_in[h] = dS
    return dict(dq=_l2_back(q, nq, dqh, l2norm), dk=_l2_back(k, nk, dkh, l2norm), dv=dvv, dg=dg, dbeta=db,
                ds_in=ds_in)

"""The chunk-64 (WY / UT) form of the GDN recurrence in FP64 numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).

It restates, for one document and one value head, the chunked algorithm whose
programs the flashinfer Cake GDN pages name (the "GLM prep" gate prefix rows,
the intra program's Akk / Aqk rows, the WY program's w and u, the K1 state
walk writing an h tape every 64 tokens and the v_new rows, the output from
the state tapes, and the adjoint walk; "feat(cake_gdn_kcp) ... #8172" page,
the #8181 section and the commit notes on the context-parallel route's local
programs; "#8542" page, the saved-set table listing gamma, gcum, Akk, h,
v_new, w, u, Aqk).  The equations are the ones that follow from the per-token
recurrence of gdn_oracle.c by unrolling it over a chunk.

Per chunk of length L <= 64 with local positions r (numpy index 0..L-1):
  G_r = sum_{i<=r} g_i,  gamma_r = exp(G_r),  Gam_rj = exp(G_r - G_j) (r >= j)
  A   = strict_tril(diag(beta) (K K^T . Gam))      T = (I + A)^-1
  W   = T diag(beta gamma) K                       U = T diag(beta) V
  Vn  = U - W S                                   (S = state entering)
  O   = scale (diag(gamma) Q S + tril(Q K^T . Gam) Vn)
  S'  = gamma_L S + Kd^T Vn,  Kd_r = exp(G_L - G_r) k_r
The backward is the reverse of those equations, chunk by chunk from the end
(dS' = 0 after the last chunk).  Library matmuls and np.linalg.inv serve as
steps; nothing is blocked or reordered beyond the equations above.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6


def l2(x, on, eps=EPS):
    if not on:
        return x.copy(), np.ones(x.shape[0])
    n = np.sqrt((x * x).sum(-1) + eps)
    return x / n[:, None], n


def chunk_fwd(qh, kh, v, g, beta, S, scale):
    """One chunk of one v-head.  Returns (O, S_next, intermediates)."""
    L = len(g)
    G = np.cumsum(g)
    gam = np.exp(G)
    D = G[:, None] - G[None, :]
    low_incl = np.tril(np.ones((L, L), dtype=bool))
    Gam = np.where(low_incl, np.exp(np.where(low_incl, D, 0.0)), 0.0)
    KK = kh @ kh.T
    A = np.tril(beta[:, None] * KK * Gam, -1)
    T = np.linalg.inv(np.eye(L) + A)
    W = T @ ((beta * gam)[:, None] * kh)
    U = T @ (beta[:, None] * v)
    Vn = U - W @ S
    Aqk = (qh @ kh.T) * Gam
    O = scale * (gam[:, None] * (qh @ S) + Aqk @ Vn)
    dec = np.exp(G[-1] - G)
    Kd = dec[:, None] * kh
    S_next = gam[-1] * S + Kd.T @ Vn
    inter = dict(G=G, gam=gam, Gam=Gam, KK=KK, A=A, T=T, W=W, U=U, Vn=Vn, Aqk=Aqk,
                 dec=dec, Kd=Kd, S=S)
    return O, S_next, inter


def chunk_bwd(qh, kh, v, beta, dO, dSn, it, scale):
    """Reverse of chunk_fwd.  dSn = gradient of the state leaving the chunk.
    Returns (dS entering, dqh, dkh, dv, dbeta, dG)."""
    G, gam, Gam, A, T, W, Vn, Aqk, dec, Kd, S = (it[x] for x in (
        "G", "gam", "Gam", "A", "T", "W", "Vn", "Aqk", "dec", "Kd", "S"))
    KK = it["KK"]
    L = len(G)
    P = scale
    dG = np.zeros(L)
    # O = P diag(gam) Q S
    QS = qh @ S
    dqh = P * gam[:, None] * (dO @ S.T)
    dG += P * gam * (QS * dO).sum(1)
    dS = P * (gam[:, None] * qh).T @ dO
    # O += P Aqk Vn,  Aqk = (Q K^T) . Gam (lower incl. diagonal)
    dAqk = P * (dO @ Vn.T) * (Gam > 0)
    dVn = P * Aqk.T @ dO
    dqh += (dAqk * Gam) @ kh
    dkh = (dAqk * Gam).T @ qh
    dG += (dAqk * Aqk).sum(1) - (dAqk * Aqk).sum(0)
    # S' = gam_L S + Kd^T Vn
    dS += gam[-1] * dSn
    dG[-1] += gam[-1] * (S * dSn).sum()
    dKd = Vn @ dSn.T
    dVn += Kd @ dSn
    dkh += dec[:, None] * dKd
    z = dec * (kh * dKd).sum(1)
    dG[-1] += z.sum()
    dG -= z
    # Vn = U - W S
    dU = dVn
    dW = -dVn @ S.T
    dS -= W.T @ dVn
    # U = T diag(beta) V ;  W = T diag(beta gam) K
    X = T.T @ dU
    dv = beta[:, None] * X
    dbeta = (v * X).sum(1)
    Y = T.T @ dW
    dkh += (beta * gam)[:, None] * Y
    bk = (kh * Y).sum(1)
    dbeta += gam * bk
    dG += beta * gam * bk
    dT = dU @ (beta[:, None] * v).T + dW @ ((beta * gam)[:, None] * kh).T
    # T = (I + A)^-1  ->  dA = -T^T dT T^T on the strict lower triangle
    dA = np.tril(-T.T @ dT @ T.T, -1)
    # A = strict_tril(diag(beta) (K K^T . Gam))
    dbeta += (dA * Gam * KK).sum(1)
    B = dA * beta[:, None] * Gam
    dkh += B @ kh + B.T @ kh
    dG += (dA * A).sum(1) - (dA * A).sum(0)
    return dS, dqh, dkh, dv, dbeta, dG


def group(q, k, v, g, beta, dO=None, *, l2norm=True, scale=128 ** -0.5, chunk=64, eps=EPS):
    """Chunked forward (+ backward) of one document for one q/k head group.
    Shapes as oracle.ref.group: q, k [L, dk]; v, dO [G, L, dv]; g, beta [G, L].
    Returns o (and dq, dk, dv, dg, dbeta) plus per-chunk S and intermediates."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    L, dk = q.shape
    Gh, _, dv = v.shape
    qh, nq = l2(q, l2norm, eps)
    kh, nk = l2(k, l2norm, eps)
    bounds = [(c0, min(c0 + chunk, L)) for c0 in range(0, L, chunk)]
    o = np.zeros((Gh, L, dv))
    S_tape = np.zeros((len(bounds), Gh, dk, dv))
    inters = [[None] * len(bounds) for _ in range(Gh)]
    for h in range(Gh):
        S = np.zeros((dk, dv))
        for c, (s, e) in enumerate(bounds):
            S_tape[c, h] = S
            O, S, it = chunk_fwd(qh[s:e], kh[s:e], v[h, s:e], g[h, s:e], beta[h, s:e], S, scale)
            o[h, s:e] = O
            inters[h][c] = it
    out = dict(o=o, S=S_tape, inter=inters)
    if dO is None:
        return out
    dO = np.asarray(dO, dtype=np.float64)
    dqh = np.zeros((L, dk))
    dkh = np.zeros((L, dk))
    dvv = np.zeros((Gh, L, dv))
    dg = np.zeros((Gh, L))
    dbeta = np.zeros((Gh, L))
    dS_tape = np.zeros((len(bounds), Gh, dk, dv))
    for h in range(Gh):
        dSn = np.zeros((dk, dv))
        for c in range(len(bounds) - 1, -1, -1):
            s, e = bounds[c]
            dS_tape[c, h] = dSn
            dSn, dq_c, dk_c, dv_c, db_c, dG_c = chunk_bwd(
                qh[s:e], kh[s:e], v[h, s:e], beta[h, s:e], dO[h, s:e], dSn, inters[h][c], scale)
            dqh[s:e] += dq_c
            dkh[s:e] += dk_c
            dvv[h, s:e] = dv_c
            dbeta[h, s:e] = db_c
            dg[h, s:e] = np.cumsum(dG_c[::-1])[::-1]
    if l2norm:
        dq = dqh / nq[:, None] - q * ((q * dqh).sum(1) / nq ** 3)[:, None]
        dkk = dkh / nk[:, None] - k * ((k * dkh).sum(1) / nk ** 3)[:, None]
    else:
        dq, dkk = dqh, dkh
    out.update(dq=dq, dk=dkk, dv=dvv, dg=dg, dbeta=dbeta, dS=dS_tape)
    return out

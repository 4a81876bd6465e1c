"""Pins of the per-channel-decay (KDA) oracle, oracle/kda.py, on the CPU.

The pages print no KDA formula; the oracle's reading (the GDN recurrence with
one decay per key channel) is pinned by what the mathematics fixes:
  * a decay that is the same on every channel is the GDN recurrence, so the
    result must equal the independent C oracle of GDN (gdn_oracle.c), with
    the per-channel gate gradients summing to the GDN gate gradient;
  * a closed form: when only the first token writes (beta = 0 afterwards) the
    state is Diag(prod of the decays) beta k^_0 v_0^T, so each output is a
    per-channel weighted dot product written out here by plain loops;
  * central finite differences of <o, dO> with respect to every input,
    including the entering state.
"""
import numpy as np
import pytest

from oracle import kda, ref

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _inputs(rng, L, dk, dv, G, per_channel=True):
    q = rng.standard_normal((L, dk))
    k = rng.standard_normal((L, dk))
    v = rng.standard_normal((G, L, dv))
    if per_channel:
        g = -rng.uniform(0.02, 0.6, (G, L, dk))
    else:
        g = -rng.uniform(0.02, 0.6, (G, L))
    beta = rng.uniform(0.1, 0.9, (G, L))
    dO = rng.standard_normal((G, L, dv))
    return q, k, v, g, beta, dO


@pytest.mark.parametrize("l2norm", [True, False])
def test_uniform_decay_is_gdn(l2norm):
    rng = np.random.default_rng(11)
    L, dk, dv, G = 37, 8, 5, 3
    q, k, v, g, beta, dO = _inputs(rng, L, dk, dv, G, per_channel=False)
    if not l2norm:   # keep the unnormalised recurrence contractive
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    scale = dk ** -0.5
    r = ref.group(q, k, v, g, beta, dO, l2norm=l2norm, scale=scale)
    gk = np.repeat(g[:, :, None], dk, axis=2)
    o = kda.group(q, k, v, gk, beta, dO, l2norm=l2norm, scale=scale)
    for name in ("o", "dq", "dk", "dv", "dbeta"):
        np.testing.assert_allclose(o[name], r[name], rtol=1e-10, atol=1e-12, err_msg=name)
    np.testing.assert_allclose(o["dg"].sum(-1), r["dg"], rtol=1e-10, atol=1e-12)


def test_first_token_only_closed_form():
    rng = np.random.default_rng(12)
    L, dk, dv = 9, 6, 4
    q, k, v, g, beta, _ = _inputs(rng, L, dk, dv, 1)
    beta[0, 1:] = 0.0
    scale = 0.7
    o = kda.group(q, k, v, g, beta, l2norm=True, scale=scale)["o"][0]
    qn = [q[t] / np.sqrt(sum(x * x for x in q[t]) + kda.EPS) for t in range(L)]
    kn0 = k[0] / np.sqrt(sum(x * x for x in k[0]) + kda.EPS)
    for t in range(L):
        w = 0.0
        for i in range(dk):
            decay = 1.0
            for s in range(1, t + 1):
                decay *= np.exp(g[0, s, i])
            w += decay * kn0[i] * qn[t][i]
        np.testing.assert_allclose(o[t], scale * beta[0, 0] * w * v[0, 0], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("l2norm", [True, False])
def test_finite_differences(l2norm):
    rng = np.random.default_rng(13)
    L, dk, dv, G = 5, 4, 3, 2
    q, k, v, g, beta, dO = _inputs(rng, L, dk, dv, G)
    if not l2norm:
        q *= 0.4
        k *= 0.4
    s_in = 0.3 * rng.standard_normal((G, dk, dv))
    scale = 0.6
    args = dict(q=q, k=k, v=v, g=g, beta=beta, s_in=s_in)

    def f(a):
        return float((kda.group(a["q"], a["k"], a["v"], a["g"], a["beta"], l2norm=l2norm, scale=scale,
                                s_in=a["s_in"])["o"] * dO).sum())

    r = kda.group(q, k, v, g, beta, dO, l2norm=l2norm, scale=scale, s_in=s_in)
    grads = dict(q=r["dq"], k=r["dk"], v=r["dv"], g=r["dg"], beta=r["dbeta"], s_in=r["ds_in"])
    h = 1e-6
    for name, x in args.items():
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = {n: a.copy() for n, a in args.items()}
            xm = {n: a.copy() for n, a in args.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            num[idx] = (f(xp) - f(xm)) / (2 * h)
        np.testing.assert_allclose(grads[name], num, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("l2norm", [True, False])
def test_chunk_form_matches_the_recurrence(l2norm):
    """The chunk form (several chunks and a ragged tail) equals the per-token
    recurrence: outputs and the state entering each chunk."""
    rng = np.random.default_rng(14)
    L, dk, dv, G, C = 45, 6, 5, 2, 16
    q, k, v, g, beta, _ = _inputs(rng, L, dk, dv, G)
    if not l2norm:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    r = kda.group(q, k, v, g, beta, l2norm=l2norm, scale=0.5)
    c = kda.chunk_forward(q, k, v, g, beta, l2norm=l2norm, scale=0.5, chunk=C)
    np.testing.assert_allclose(c["o"], r["o"], rtol=1e-10, atol=1e-12)
    for i, t0 in enumerate(range(0, L, C)):
        ent = kda.group(q[:t0], k[:t0], v[:, :t0], g[:, :t0], beta[:, :t0], l2norm=l2norm, scale=0.5)["s_out"] \
            if t0 > 0 else np.zeros((G, dk, dv))
        np.testing.assert_allclose(c["S"][i], ent, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("l2norm", [True, False])
def test_chunk_backward_matches_the_recurrence(l2norm):
    """The chunk-form backward equals the per-token reverse mode on every
    gradient, over several chunks and a ragged tail."""
    rng = np.random.default_rng(15)
    L, dk, dv, G, C = 45, 6, 5, 2, 16
    q, k, v, g, beta, dO = _inputs(rng, L, dk, dv, G)
    if not l2norm:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    r = kda.group(q, k, v, g, beta, dO, l2norm=l2norm, scale=0.5)
    c = kda.chunk_backward(q, k, v, g, beta, dO, l2norm=l2norm, scale=0.5, chunk=C)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "ds_in"):
        np.testing.assert_allclose(c[name], r[name], rtol=1e-9, atol=1e-11, err_msg=name)

"""Pins of the FP64 oracle against things fixed independently of it.

Each test checks the oracle against the definition of the gated delta rule
(state S_t = a_t S_{t-1} + beta_t k_t (v_t - a_t S_{t-1}^T k_t)^T, output
o_t = scale S_t^T q_t, reset at every document start) through a property that
does not reuse the oracle's own code: a hand-worked example, central finite
differences, linearity/adjoint identities, closed forms of the special cases
(beta = 0, orthonormal keys, g = 0), document independence, and the
equivalence of its per-token and chunked forms.
"""
import os

import numpy as np
import pytest

from oracle import chunked, ref, tables

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_case(rng, doc_lens, H, HV, dk, dv, glo=0.5, ghi=3.0):
    T = sum(doc_lens)
    x = rng.uniform(glo, ghi, (T, HV))
    return dict(
        q=rng.standard_normal((T, H, dk)), k=rng.standard_normal((T, H, dk)),
        v=rng.standard_normal((T, HV, dv)), g=-np.log1p(np.exp(-x)),
        beta=1.0 / (1.0 + np.exp(-rng.standard_normal((T, HV)))),
        dO=rng.standard_normal((T, HV, dv)),
        cu_seqlens=np.concatenate([[0], np.cumsum(doc_lens)]).astype(np.int32))


def full(inp, H, HV, l2norm, scale, with_grad=True, threads=1):
    T, _, dk = inp["q"].shape
    dv = inp["v"].shape[2]
    res = ref.run(inp, H, HV, l2norm=l2norm, scale=scale, with_grad=with_grad, threads=threads)
    return ref.assemble(res, T, H, HV, dk, dv, inp["cu_seqlens"], with_grad=with_grad)


def test_hand_worked_example():
    vals = {}
    with open(os.path.join(HERE, "golden", "hand_worked_d2.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, t, *xs = line.split()
            vals.setdefault(name, {})[int(t)] = [float(x) for x in xs]
    get = lambda n: np.array([vals[n][0], vals[n][1]])
    q, k, v, dO = get("q"), get("k"), get("v")[None], get("dO")[None]
    g = np.log(get("a"))[:, 0][None]
    beta = get("beta")[:, 0][None]
    for impl in (ref.group, chunked.group):
        r = impl(q, k, v, g, beta, dO, l2norm=False, scale=1.0)
        np.testing.assert_allclose(r["o"][0], get("o"), atol=1e-14)
        np.testing.assert_allclose(r["dq"], get("dq"), atol=1e-14)
        np.testing.assert_allclose(r["dk"], get("dk"), atol=1e-14)
        np.testing.assert_allclose(r["dv"][0], get("dv"), atol=1e-14)
        np.testing.assert_allclose(r["dg"][0], get("dg")[:, 0], atol=1e-14)
        np.testing.assert_allclose(r["dbeta"][0], get("dbeta")[:, 0], atol=1e-14)


@pytest.mark.parametrize("l2norm", [True, False])
def test_finite_differences(l2norm):
    """Central differences of loss = <dO, o> against every gradient, on 7
    tokens over 2 documents, d = 4, H = 1, HV = 2."""
    rng = np.random.default_rng(11)
    H, HV, dk, dv = 1, 2, 4, 4
    inp = rand_case(rng, [3, 4], H, HV, dk, dv)
    scale = 0.7
    grads = full(inp, H, HV, l2norm, scale)

    def loss(x):
        return float((full(x, H, HV, l2norm, scale, with_grad=False)["o"] * inp["dO"]).sum())

    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta")):
        num = np.zeros_like(inp[name])
        for idx in np.ndindex(inp[name].shape):
            xp = dict(inp); xp[name] = inp[name].copy(); xp[name][idx] += h
            xm = dict(inp); xm[name] = inp[name].copy(); xm[name][idx] -= h
            num[idx] = (loss(xp) - loss(xm)) / (2 * h)
        err = np.abs(num - grads[gname]).max() / np.abs(num).max()
        assert err < 1e-6, (name, err)


def test_adjoint_dv():
    """o is linear in v, so <dO, o(v)> equals <v, dv>."""
    rng = np.random.default_rng(5)
    H, HV = 2, 4
    inp = rand_case(rng, [70, 5, 130], H, HV, 8, 6)
    r = full(inp, H, HV, True, 0.3)
    lhs = float((inp["dO"] * r["o"]).sum())
    rhs = float((inp["v"] * r["dv"]).sum())
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), 1.0)


@pytest.mark.parametrize("L,chunk", [(1, 64), (63, 64), (64, 64), (65, 64), (200, 64), (77, 16)])
@pytest.mark.parametrize("l2norm", [True, False])
def test_chunked_equals_per_token(L, chunk, l2norm):
    rng = np.random.default_rng(L + 7 * chunk)
    G, dk, dv = 2, 16, 8
    q, k = rng.standard_normal((L, dk)), rng.standard_normal((L, dk))
    if not l2norm:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v, dO = rng.standard_normal((G, L, dv)), rng.standard_normal((G, L, dv))
    g = -np.log1p(np.exp(-rng.uniform(1, 4, (G, L))))
    beta = rng.uniform(0, 1, (G, L))
    a = ref.group(q, k, v, g, beta, dO, l2norm=l2norm, scale=0.4, chunk_states=True, chunk=chunk)
    b = chunked.group(q, k, v, g, beta, dO, l2norm=l2norm, scale=0.4, chunk=chunk)
    for n in ("o", "dq", "dk", "dv", "dg", "dbeta", "S"):
        assert np.abs(a[n] - b[n]).max() <= 1e-12 * max(np.abs(b[n]).max(), 1.0), n


def test_beta_zero_closed_form():
    """beta = 0 keeps S = 0: o and every gradient but dbeta vanish exactly, and
    dbeta_t = scale sum_{s>=t} exp(G_s - G_t) (q^_s . k^_t)(dO_s . v_t), the
    first-order (decayed linear attention) term."""
    rng = np.random.default_rng(3)
    L, G, dk, dv, scale = 40, 2, 8, 5, 0.6
    q, k = rng.standard_normal((L, dk)), rng.standard_normal((L, dk))
    v, dO = rng.standard_normal((G, L, dv)), rng.standard_normal((G, L, dv))
    g = -rng.uniform(0.01, 0.3, (G, L))
    r = ref.group(q, k, v, g, np.zeros((G, L)), dO, l2norm=True, scale=scale)
    for n in ("o", "dq", "dk", "dv", "dg"):
        assert np.all(r[n] == 0.0), n
    qh = q / np.sqrt((q * q).sum(1) + ref.EPS)[:, None]
    kh = k / np.sqrt((k * k).sum(1) + ref.EPS)[:, None]
    for h in range(G):
        Gc = np.cumsum(g[h])
        expect = np.zeros(L)
        for t in range(L):
            for s in range(t, L):
                expect[t] += scale * np.exp(Gc[s] - Gc[t]) * (qh[s] @ kh[t]) * (dO[h, s] @ v[h, t])
        np.testing.assert_allclose(r["dbeta"][h], expect, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("gate", ["decayed", "zero"])
def test_orthonormal_keys(gate):
    """With mutually orthogonal keys the delta correction vanishes and o is
    decayed (g = 0: plain causal) linear attention with weights beta:
    o_t = scale sum_{s<=t} exp(G_t - G_s) (q^_t . k^_s) beta_s v_s."""
    rng = np.random.default_rng(4)
    L, G, dk, dv, scale = 24, 3, 32, 7, 0.9
    k = np.zeros((L, dk))
    k[np.arange(L), rng.permutation(dk)[:L]] = rng.uniform(0.5, 2.0, L)
    q = rng.standard_normal((L, dk))
    v = rng.standard_normal((G, L, dv))
    g = -rng.uniform(0.01, 0.5, (G, L)) if gate == "decayed" else np.zeros((G, L))
    beta = rng.uniform(0, 1, (G, L))
    for l2norm in (True, False):
        r = ref.group(q, k, v, g, beta, None, l2norm=l2norm, scale=scale)
        nq = np.sqrt((q * q).sum(1) + ref.EPS) if l2norm else np.ones(L)
        nk = np.sqrt((k * k).sum(1) + ref.EPS) if l2norm else np.ones(L)
        qh, kh = q / nq[:, None], k / nk[:, None]
        for h in range(G):
            Gc = np.cumsum(g[h])
            W = np.tril(np.exp(Gc[:, None] - Gc[None, :])) * (qh @ kh.T)
            expect = scale * W @ (beta[h][:, None] * v[h])
            np.testing.assert_allclose(r["o"][h], expect, rtol=1e-12, atol=1e-12)


def test_document_reset():
    """A packed run equals the documents run one by one, and a document's
    results do not depend on another document's inputs."""
    rng = np.random.default_rng(9)
    H, HV, dk, dv = 2, 4, 8, 8
    lens = [50, 1, 80]
    inp = rand_case(rng, lens, H, HV, dk, dv)
    packed = full(inp, H, HV, True, 0.5)
    cu = inp["cu_seqlens"]
    for d in range(len(lens)):
        s, e = cu[d], cu[d + 1]
        one = {n: inp[n][s:e] for n in ("q", "k", "v", "g", "beta", "dO")}
        one["cu_seqlens"] = np.array([0, e - s], dtype=np.int32)
        r = full(one, H, HV, True, 0.5)
        for n in ("o", "dq", "dk", "dv", "dg", "dbeta"):
            assert np.array_equal(r[n], packed[n][s:e]), (d, n)
    pert = {n: (x.copy() if isinstance(x, np.ndarray) else x) for n, x in inp.items()}
    for n in ("q", "k", "v", "g", "beta", "dO"):
        pert[n][: cu[1]] = rng.standard_normal(pert[n][: cu[1]].shape) * 0.1 + \
            (pert[n][: cu[1]] if n in ("g", "beta") else 0)
    r = full(pert, H, HV, True, 0.5)
    for n in ("o", "dq", "dk", "dv", "dg", "dbeta"):
        assert np.array_equal(r[n][cu[1]:], packed[n][cu[1]:]), n


def test_scale_and_columns():
    """o is proportional to scale, and the value columns evolve independently
    (running on v[..., cols] gives o[..., cols])."""
    rng = np.random.default_rng(2)
    H, HV = 1, 2
    inp = rand_case(rng, [90], H, HV, 8, 12)
    a = full(inp, H, HV, True, 0.25, with_grad=False)["o"]
    b = full(inp, H, HV, True, 0.75, with_grad=False)["o"]
    np.testing.assert_allclose(b, 3 * a, rtol=1e-13, atol=1e-15)
    cols = [1, 5, 6, 11]
    sub = dict(inp)
    sub["v"] = inp["v"][:, :, cols].copy()
    c = full(sub, H, HV, True, 0.25, with_grad=False)["o"]
    np.testing.assert_array_equal(c, a[:, :, cols])


def test_group_mapping():
    """v-head h reads q/k head h // (HV/H): zero keys on q/k head 0 leave
    v-heads 0 and 1 (of HV = 4, H = 2) with u = beta v but no output from
    other heads' keys, i.e. o = 0 for them, while v-heads 2, 3 are non-zero."""
    rng = np.random.default_rng(1)
    H, HV = 2, 4
    inp = rand_case(rng, [33], H, HV, 8, 8)
    inp["q"][:, 0] = 0.0
    o = full(inp, H, HV, False, 1.0, with_grad=False)["o"]
    assert np.all(o[:, 0:2] == 0.0)
    assert np.all(np.abs(o[:, 2:4]).max(axis=(0, 2)) > 0)


def test_window_truncation():
    """A sampled output window computed from a warmed-up sub-range matches
    the whole-document result to the damping bound that window() reports."""
    rng = np.random.default_rng(8)
    H, HV, dk, dv = 1, 2, 16, 16
    L = 3000
    inp = rand_case(rng, [L], H, HV, dk, dv, glo=2.0, ghi=6.0)
    whole = full(inp, H, HV, True, 0.5)
    t0, t1 = 1400, 1500
    a, b, left, right = ref.window(inp["g"].T, t0, t1, warm=256)
    assert a % 64 == 0 and left < 1e-12 and right < 1e-12
    res = ref.run(inp, H, HV, l2norm=True, scale=0.5, units=[ref.Unit(0, 0, t0, t1, a, b)])
    win = ref.assemble(res, L, H, HV, dk, dv, inp["cu_seqlens"])
    for n in ("o", "dq", "dk", "dv", "dg", "dbeta"):
        ref_ = whole[n][t0:t1]
        assert np.abs(win[n][t0:t1] - ref_).max() <= 1e-9 * np.abs(ref_).max(), n


def test_chunk_tables_enumeration():
    t = tables.chunk_tables([0, 0, 64, 65, 200, 200], chunk=64)
    assert t["chunk_offsets"].tolist() == [0, 0, 1, 2, 5, 5]
    assert t["chunk_doc"].tolist() == [1, 2, 3, 3, 3]
    assert t["chunk_tok0"].tolist() == [0, 64, 65, 129, 193]
    assert t["chunk_len"].tolist() == [64, 1, 64, 64, 7]


# ---------------------------------------------------------------------------
# per-document boundary states (S_in / S_out and their gradients)
# ---------------------------------------------------------------------------
def full_states(inp, H, HV, l2norm, scale, with_grad=True):
    T, _, dk = inp["q"].shape
    dv = inp["v"].shape[2]
    res = ref.run(inp, H, HV, l2norm=l2norm, scale=scale, with_grad=with_grad, threads=1, states=True)
    return ref.assemble(res, T, H, HV, dk, dv, inp["cu_seqlens"], with_grad=with_grad, states=True)


@pytest.mark.parametrize("l2norm", [True, False])
@pytest.mark.parametrize("m", [1, 33, 64, 69])
def test_boundary_states_split(l2norm, m):
    """A document cut at token m and run as two segments, the second starting
    from the first one's S_out (forward) and the first ending on the second
    one's dS_in (backward), gives the whole document's outputs, gradients and
    final state bit for bit: the boundary states carry exactly what the zero-
    start whole-document oracle (pinned above) passes from token m-1 to m."""
    rng = np.random.default_rng(40 + m)
    G, dk, dv, L = 2, 8, 6, 70
    q, k = rng.standard_normal((L, dk)), rng.standard_normal((L, dk))
    v, dO = rng.standard_normal((G, L, dv)), rng.standard_normal((G, L, dv))
    g, b = -rng.uniform(0.01, 0.3, (G, L)), rng.uniform(0.0, 1.0, (G, L))
    kw = dict(l2norm=l2norm, scale=0.4, states=True)
    whole = ref.group(q, k, v, g, b, dO, **kw)
    second = ref.group(q[m:], k[m:], v[:, m:], g[:, m:], b[:, m:], dO[:, m:],
                       s_in=ref.group(q[:m], k[:m], v[:, :m], g[:, :m], b[:, :m], **kw)["s_out"], **kw)
    first = ref.group(q[:m], k[:m], v[:, :m], g[:, :m], b[:, :m], dO[:, :m], ds_out=second["ds_in"], **kw)
    assert np.array_equal(np.concatenate([first["o"], second["o"]], 1), whole["o"])
    assert np.array_equal(second["s_out"], whole["s_out"])
    for n in ("dq", "dk"):
        assert np.array_equal(np.concatenate([first[n], second[n]], 0), whole[n]), n
    for n in ("dv", "dg", "dbeta"):
        assert np.array_equal(np.concatenate([first[n], second[n]], 1), whole[n]), n
    assert np.array_equal(first["ds_in"], whole["ds_in"])


@pytest.mark.parametrize("l2norm", [True, False])
def test_boundary_states_finite_differences(l2norm):
    """Central differences of loss = <dO, o> + <dS_out, S_out> with a nonzero
    S_in, on 7 tokens over 2 documents: the gradient with respect to S_in is
    ds_in, and the token gradients include the S_out term."""
    rng = np.random.default_rng(17)
    H, HV, dk, dv = 1, 2, 4, 3
    inp = rand_case(rng, [3, 4], H, HV, dk, dv)
    inp["s_in"] = 0.5 * rng.standard_normal((2, HV, dk, dv))
    inp["ds_out"] = rng.standard_normal((2, HV, dk, dv))
    scale = 0.7
    grads = full_states(inp, H, HV, l2norm, scale)

    def loss(x):
        r = full_states(x, H, HV, l2norm, scale, with_grad=False)
        return float((r["o"] * inp["dO"]).sum() + (r["s_out"] * inp["ds_out"]).sum())

    h = 1e-6
    for name, gname in (("s_in", "ds_in"), ("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"),
                        ("beta", "dbeta")):
        num = np.zeros_like(inp[name])
        for idx in np.ndindex(inp[name].shape):
            xp = dict(inp); xp[name] = inp[name].copy(); xp[name][idx] += h
            xm = dict(inp); xm[name] = inp[name].copy(); xm[name][idx] -= h
            num[idx] = (loss(xp) - loss(xm)) / (2 * h)
        err = np.abs(num - grads[gname]).max() / np.abs(num).max()
        assert err < 1e-6, (name, err)


def test_boundary_states_empty_document():
    """An empty document passes S_in through to S_out and dS_out back to dS_in."""
    rng = np.random.default_rng(3)
    G, dk, dv = 2, 4, 3
    s_in, ds_out = rng.standard_normal((G, dk, dv)), rng.standard_normal((G, dk, dv))
    z = np.zeros((0, dk))
    r = ref.group(z, z, np.zeros((G, 0, dv)), np.zeros((G, 0)), np.zeros((G, 0)), np.zeros((G, 0, dv)),
                  s_in=s_in, ds_out=ds_out, states=True)
    assert np.array_equal(r["s_out"], s_in) and np.array_equal(r["ds_in"], ds_out)

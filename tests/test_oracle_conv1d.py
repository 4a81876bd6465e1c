"""Pins of the FP64 conv1d + SiLU oracle against things fixed independently of
it: the impulse response (the kernel's tap order and the bias), SiLU itself
through scipy's logistic function, central finite differences of every
gradient, document restarts and causality."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import conv1d


def case(rng, doc_lens, C, W):
    T = sum(doc_lens)
    return (rng.standard_normal((T, C)), rng.standard_normal((C, W)), rng.standard_normal(C),
            np.concatenate([[0], np.cumsum(doc_lens)]).astype(np.int64))


def test_impulse_response():
    """A unit impulse at token t0 gives z[t0 + j] = b + w[:, W-1-j] for j < W
    (and z = b elsewhere): tap i multiplies x[t - (W-1) + i]."""
    rng = np.random.default_rng(1)
    C, W, T, t0 = 5, 4, 12, 3
    w, b = rng.standard_normal((C, W)), rng.standard_normal(C)
    x = np.zeros((T, C))
    x[t0] = 1.0
    y = conv1d.forward(x, w, b, np.array([0, T]))
    z = np.tile(b, (T, 1))
    for j in range(W):
        z[t0 + j] = b + w[:, W - 1 - j]
    assert np.allclose(y, z * expit(z), rtol=1e-15, atol=1e-15)


def test_width_one_is_pointwise_silu():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((9, 4))
    y = conv1d.forward(x, np.ones((4, 1)), None, np.array([0, 4, 9]))
    assert np.allclose(y, x * expit(x), rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("W", [1, 2, 4])
def test_finite_differences(W):
    rng = np.random.default_rng(10 + W)
    x, w, b, cu = case(rng, [2, 5, 1], 3, W)
    dy = rng.standard_normal(x.shape)
    dx, dw, db = conv1d.backward(x, w, b, cu, dy)

    def loss(xx, ww, bb):
        return float((conv1d.forward(xx, ww, bb, cu) * dy).sum())

    h = 1e-6
    for arr, grad, which in ((x, dx, 0), (w, dw, 1), (b, db, 2)):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args_p, args_m = [x.copy(), w.copy(), b.copy()], [x.copy(), w.copy(), b.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - grad).max() / np.abs(num).max()
        assert err < 1e-7, (which, err)


def test_document_restart_and_causality():
    rng = np.random.default_rng(4)
    x, w, b, cu = case(rng, [6, 3, 7], 4, 4)
    y = conv1d.forward(x, w, b, cu)
    # packed == documents one by one
    for d in range(3):
        s, e = cu[d], cu[d + 1]
        assert np.array_equal(y[s:e], conv1d.forward(x[s:e], w, b, np.array([0, e - s])))
    # a change at token t touches no earlier output and nothing in other documents
    x2 = x.copy()
    x2[7] += 1.0
    y2 = conv1d.forward(x2, w, b, cu)
    changed = np.nonzero(np.abs(y2 - y).max(axis=1))[0]
    assert changed.min() == 7 and changed.max() <= 8   # inside the second document [6, 9)

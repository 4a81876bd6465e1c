"""FP64 oracle of the short causal convolution + SiLU front of the GDN layer.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages time every call of their packed GDN layer together with a short
causal convolution, followed by SiLU, over the 10,240 packed q/k/v channels
at (H, HV) = (16, 48), restarting at every document ("#8542" page: the B23
shape description, the family's conv1d + SiLU training backend, and the
save-set table, which keeps at most three history rows: a kernel four taps
wide).  The pages print no formula; the plainest reading, written out here
for one depthwise (per-channel) kernel of width W and packed documents:

  z[t, c] = b[c] + sum_{i=0}^{W-1} w[c, i] * x[t - (W-1) + i, c]
            (x[s, c] = 0 for s before the document start of t)
  y[t, c] = silu(z[t, c]) = z sigma(z)

and its backward, with dz = dy * sigma(z) (1 + z (1 - sigma(z))):

  dx[s, c] = sum_i w[c, i] * dz[s + (W-1) - i, c]   (terms inside s's document)
  dw[c, i] = sum_t dz[t, c] * x[t - (W-1) + i, c]    db[c] = sum_t dz[t, c]

Shapes: x, y, dy, dx [T, C]; w, dw [C, W]; b, db [C]; cu_seqlens [N + 1].
Each document is handled by whole-array shifts of its rows (numpy); nothing
is blocked or reordered beyond the sums above.
"""
from __future__ import annotations

import numpy as np


def _z(x, w, b, cu):
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = x.shape
    W = w.shape[1]
    z = np.zeros((T, C))
    for d in range(len(cu) - 1):
        s, e = int(cu[d]), int(cu[d + 1])
        for i in range(W):
            sh = W - 1 - i                       # x[t - sh] feeds z[t] through w[:, i]
            if e - s > sh:
                z[s + sh:e] += w[:, i] * x[s:e - sh]
    if b is not None:
        z += np.asarray(b, dtype=np.float64)
    return z


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def forward(x, w, b, cu):
    """y = silu(causal depthwise conv(x) + b), per document."""
    z = _z(x, w, b, cu)
    return z * _sigmoid(z)


def backward(x, w, b, cu, dy):
    """(dx, dw, db) of sum(y * dy)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    z = _z(x, w, b, cu)
    sg = _sigmoid(z)
    dz = np.asarray(dy, dtype=np.float64) * sg * (1.0 + z * (1.0 - sg))
    T, C = x.shape
    W = w.shape[1]
    dx = np.zeros((T, C))
    dw = np.zeros((C, W))
    for d in range(len(cu) - 1):
        s, e = int(cu[d]), int(cu[d + 1])
        for i in range(W):
            sh = W - 1 - i
            if e - s > sh:
                dx[s:e - sh] += w[:, i] * dz[s + sh:e]
                dw[:, i] += (dz[s + sh:e] * x[s:e - sh]).sum(axis=0)
    db = dz.sum(axis=0)
    return dx, dw, db

"""ctypes binding and driver of the FP64 per-token oracle (gdn_oracle.c).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The unit of work is one (document, q/k head group): the G = HV/H consecutive
value heads that share q/k head j are v-heads j*G .. j*G+G-1 (the usual
grouped-head convention; the pages' "(H, HV) = query/key heads and value
heads" on the "feat(cake_gdn_kcp) ... #8172" page fixes only the counts).
Groups are independent, so they run on a thread pool; ctypes drops the GIL
during the C call.

Sampling on large workloads: an output window [t0, t1) of a long document is
computed from a sub-range [a, b) of the document that extends the window by a
warm-up W on the left (forward) and on the right (backward), starting from a
zero state.  Because ||I - beta k^ k^T|| <= 1 for ||k^|| <= 1 and
0 <= beta <= 1, the state that the truncation drops is damped by at least
prod_{a <= s < t0} exp(g_s) (and the dropped future adjoint likewise by the
product over [t1, b)); `window()` returns those products so a test can check
that they are far below the tolerance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdn_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libgdn_oracle.so")
EPS = 1e-6
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, IEEE double, no fast-math)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", SRC, "-o", tmp, "-lm"])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        L.gdn_oracle_group.restype = ctypes.c_int
        L.gdn_oracle_group.argtypes = [ctypes.c_int] * 4 + [dp] * 6 + [
            ctypes.c_int, ctypes.c_double, ctypes.c_double] + [dp] * 7 + [ctypes.c_int]
        L.gdn_oracle_group_states.restype = ctypes.c_int
        L.gdn_oracle_group_states.argtypes = L.gdn_oracle_group.argtypes + [dp] * 4
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def group(q, k, v, g, beta, dO=None, *, l2norm=True, scale=128 ** -0.5, eps=EPS,
          chunk_states=False, chunk=64, s_in=None, ds_out=None, states=False):
    """Forward (+ backward if dO is given) of one document segment, one group.

    q, k [L, dk]; v [G, L, dv]; g, beta [G, L]; dO [G, L, dv]; all float64.
    s_in, ds_out [G, dk, dv] (optional): the state entering the segment and the
    gradient with respect to the state leaving it.
    Returns a dict with o [G,L,dv] and, with dO: dq, dk [L,dk], dv [G,L,dv],
    dg, dbeta [G,L]; with chunk_states: S [nchunks, G, dk, dv] entering each
    chunk; with states: s_out [G,dk,dv] and, with dO, ds_in [G,dk,dv]."""
    q, k, v, g, beta = (np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    L, dk = q.shape
    G, _, dv = v.shape
    out = dict(o=np.zeros((G, L, dv)))
    if dO is not None:
        dO = np.ascontiguousarray(dO, dtype=np.float64)
        out.update(dq=np.zeros((L, dk)), dk=np.zeros((L, dk)), dv=np.zeros((G, L, dv)),
                   dg=np.zeros((G, L)), dbeta=np.zeros((G, L)))
    if chunk_states:
        out["S"] = np.zeros(((L + chunk - 1) // chunk, G, dk, dv))
    if states:
        out["s_out"] = np.zeros((G, dk, dv))
        if dO is not None:
            out["ds_in"] = np.zeros((G, dk, dv))
    s_in = None if s_in is None else np.ascontiguousarray(s_in, dtype=np.float64).reshape(G, dk, dv)
    ds_out = None if ds_out is None else np.ascontiguousarray(ds_out, dtype=np.float64).reshape(G, dk, dv)
    rc = lib().gdn_oracle_group_states(L, dk, dv, G, _p(q), _p(k), _p(v), _p(g), _p(beta), _p(dO),
                                       int(bool(l2norm)), float(eps), float(scale), _p(out["o"]),
                                       _p(out.get("dq")), _p(out.get("dk")), _p(out.get("dv")),
                                       _p(out.get("dg")), _p(out.get("dbeta")), _p(out.get("S")),
                                       int(chunk), _p(s_in), _p(out.get("s_out")), _p(ds_out),
                                       _p(out.get("ds_in")))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_group_states failed ({rc})")
    return out


def _f64(x):
    """torch tensor or numpy array -> float64 numpy (exact widening)."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


@dataclass
class Unit:
    """One oracle job: document `doc`, q/k head `j`, token window [t0, t1)
    (document-relative) computed from the sub-range [a, b)."""
    doc: int
    j: int
    t0: int
    t1: int
    a: int
    b: int


def window(g_doc: np.ndarray, t0: int, t1: int, warm: int, chunk: int = 64, tol: float = 1e-12):
    """Choose the sub-range [a, b) for the output window [t0, t1) of a document
    whose per-token gates (all v-heads of the group) are g_doc [Gh, Ld].  The
    left edge is chunk-aligned so chunk states line up.  The warm-ups grow from
    `warm` until the damping products fall below `tol` (or hit the document
    edges).  Returns (a, b, left_damping, right_damping)."""
    Ld = g_doc.shape[1]
    gmax = g_doc.max(axis=0)  # the least damping across the group's heads
    w = warm
    while True:
        a = max(0, ((t0 - w) // chunk) * chunk)
        b = min(Ld, t1 + w)
        left = float(np.exp(gmax[a:t0].sum())) if a > 0 else 0.0
        right = float(np.exp(gmax[t1:b].sum())) if b < Ld else 0.0
        if (left <= tol and right <= tol) or (a == 0 and b == Ld):
            return a, b, left, right
        w *= 2


def run(inputs: dict, H: int, HV: int, *, l2norm: bool, scale: float, units=None,
        with_grad: bool = True, chunk_states: bool = False, threads: int | None = None,
        states: bool = False):
    """Run the oracle over `units` (default: every document x group, whole
    documents).  `inputs` holds q, k, v, g, beta, dO (torch or numpy, token
    major) and cu_seqlens, and optionally the per-document boundary states
    s_in, ds_out [N, HV, dk, dv] (whole-document units only).  With `states`
    each result also holds s_out and (with gradients) ds_in of its group.
    Returns a list of (Unit, result dict)."""
    cu = np.asarray(inputs["cu_seqlens"], dtype=np.int64)
    G = HV // H
    if units is None:
        units = []
        for d in range(len(cu) - 1):
            Ld = int(cu[d + 1] - cu[d])
            for j in range(H):
                units.append(Unit(d, j, 0, Ld, 0, Ld))

    def job(u: Unit):
        s = int(cu[u.doc]) + u.a
        e = int(cu[u.doc]) + u.b
        hs = slice(u.j * G, (u.j + 1) * G)
        q = _f64(inputs["q"][s:e, u.j])
        k = _f64(inputs["k"][s:e, u.j])
        v = _f64(inputs["v"][s:e, hs]).transpose(1, 0, 2).copy()
        g = _f64(inputs["g"][s:e, hs]).T.copy()
        beta = _f64(inputs["beta"][s:e, hs]).T.copy()
        dO = _f64(inputs["dO"][s:e, hs]).transpose(1, 0, 2).copy() if with_grad else None
        bnd = {}
        for name in ("s_in", "ds_out"):
            if inputs.get(name) is not None:
                assert u.a == 0 and u.b == int(cu[u.doc + 1] - cu[u.doc]), "boundary states need whole documents"
                bnd[name] = _f64(inputs[name][u.doc, hs])
        return u, group(q, k, v, g, beta, dO, l2norm=l2norm, scale=scale,
                        chunk_states=chunk_states, states=states, **bnd)

    nthr = threads or os.cpu_count() or 1
    if nthr == 1 or len(units) == 1:
        return [job(u) for u in units]
    with ThreadPoolExecutor(max_workers=nthr) as ex:
        return list(ex.map(job, units))


def assemble(results, T: int, H: int, HV: int, dk: int, dv: int, cu, with_grad=True, states=False):
    """Scatter whole-document unit results into token-major FP64 arrays
    o [T,HV,dv], dq/dk [T,H,dk], dv [T,HV,dv], dg/dbeta [T,HV], and with
    `states` the per-document s_out (and ds_in) [N,HV,dk,dv]."""
    cu = np.asarray(cu, dtype=np.int64)
    G = HV // H
    out = dict(o=np.zeros((T, HV, dv)))
    if with_grad:
        out.update(dq=np.zeros((T, H, dk)), dk=np.zeros((T, H, dk)), dv=np.zeros((T, HV, dv)),
                   dg=np.zeros((T, HV)), dbeta=np.zeros((T, HV)))
    if states:
        out["s_out"] = np.zeros((len(cu) - 1, HV, dk, dv))
        if with_grad:
            out["ds_in"] = np.zeros((len(cu) - 1, HV, dk, dv))
    for u, r in results:
        if states:
            out["s_out"][u.doc, u.j * G:(u.j + 1) * G] = r["s_out"]
            if with_grad:
                out["ds_in"][u.doc, u.j * G:(u.j + 1) * G] = r["ds_in"]
        s = int(cu[u.doc]) + u.a
        w0, w1 = s + (u.t0 - u.a), s + (u.t1 - u.a)
        r0, r1 = u.t0 - u.a, u.t1 - u.a
        hs = slice(u.j * G, (u.j + 1) * G)
        out["o"][w0:w1, hs] = r["o"][:, r0:r1].transpose(1, 0, 2)
        if with_grad:
            out["dq"][w0:w1, u.j] = r["dq"][r0:r1]
            out["dk"][w0:w1, u.j] = r["dk"][r0:r1]
            out["dv"][w0:w1, hs] = r["dv"][:, r0:r1].transpose(1, 0, 2)
            out["dg"][w0:w1, hs] = r["dg"][:, r0:r1].T
            out["dbeta"][w0:w1, hs] = r["dbeta"][:, r0:r1].T
    return out

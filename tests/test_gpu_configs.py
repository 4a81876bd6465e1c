"""Parity of the full-size workloads (8192 to 524,288 tokens, H = 16, HV = 48)
against the FP64 oracle, in the launch configuration bench.py times.

The oracle runs on sampled (document, q/k-head group) units, all value heads
of the group at once so dq / dk are complete sums: whole documents where they
are short, otherwise output windows computed from a warmed-up sub-range whose
damping product is checked to be below 1e-12 (oracle.ref.window).  Samples
always include the first and last document; on the split workload they
include windows across segment boundaries."""
import numpy as np
import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from oracle import ref
from tests.gdn_testutil import compare

pytestmark = pytest.mark.gpu
GRADS = ("o", "dq", "dk", "dv", "dg", "dbeta")


def run_gpu(w, x):
    import linear_attention_gdn_gb300 as gdn
    cu_dev = torch.from_numpy(w.cu_seqlens).cuda()
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments)
    buf = gdn.Buffers(prob, w.cu_seqlens)
    out = dict(o=torch.empty((w.T, w.HV, 128), dtype=torch.bfloat16, device="cuda"),
               dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]), dv=torch.empty_like(x["v"]),
               dg=torch.empty_like(x["g"]), dbeta=torch.empty_like(x["beta"]))
    gdn.gdn_fwd(prob, x["q"], x["k"], x["v"], x["g"], x["beta"], cu_dev, w.cu_seqlens, out["o"], buf.saved,
                buf.workspace)
    gdn.gdn_bwd(prob, x["q"], x["k"], x["v"], x["g"], x["beta"], cu_dev, w.cu_seqlens, x["dO"], buf.saved,
                out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"], buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 0
    seg = gdn.gdn_plan_segment_chunks(prob, w.cu_seqlens)
    del buf
    return out, seg


def sample_units(w, x, seg_chunks, n_groups, rng, whole_max=16384, win=512):
    cu = w.cu_seqlens
    G = w.HV // w.H
    docs = sorted({0, w.N - 1} | set(rng.choice(w.N, size=min(w.N, 4), replace=False).tolist()))
    docs = [d for d in docs if cu[d + 1] > cu[d]]
    units = []
    for i in range(n_groups):
        d = docs[i % len(docs)]
        j = int(rng.integers(w.H))
        Ld = int(cu[d + 1] - cu[d])
        if Ld <= whole_max:
            units.append(ref.Unit(d, j, 0, Ld, 0, Ld))
            continue
        starts = [0, Ld - win, int(rng.integers(win, Ld - 2 * win))]
        if seg_chunks * 64 < Ld:   # across a segment boundary of the split
            b = seg_chunks * 64 * int(rng.integers(1, max(2, Ld // (seg_chunks * 64))))
            starts.append(max(0, min(Ld - win, b - win // 2)))
        t0 = starts[i % len(starts)]
        gdoc = x["g"][cu[d]:cu[d + 1], j * G:(j + 1) * G].double().cpu().numpy().T
        a, b_, left, right = ref.window(gdoc, t0, t0 + win, warm=1024)
        assert left <= 1e-12 and right <= 1e-12
        units.append(ref.Unit(d, j, t0, t0 + win, a, b_))
    return units


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_full_size_parity(idx):
    w = inputs.workload(idx)
    x = inputs.generate(w, "cuda")
    got, seg = run_gpu(w, x)
    rng = np.random.default_rng(100 + idx)
    if idx == 1:
        units = None   # the whole workload
    else:
        units = sample_units(w, x, seg, 12, rng)
    res = ref.run(x, w.H, w.HV, l2norm=w.l2norm, scale=w.scale, units=units)
    cu = w.cu_seqlens
    G = w.HV // w.H
    # every sampled (document, q/k-head group) unit is compared on its own, so that one bad unit
    # cannot hide under the others
    for u, r in res:
        s0 = int(cu[u.doc]) + u.t0
        s1 = int(cu[u.doc]) + u.t1
        r0, r1 = u.t0 - u.a, u.t1 - u.a
        hs = slice(u.j * G, (u.j + 1) * G)
        tag = f"workload{idx}/doc{u.doc}/group{u.j}/tokens{u.t0}-{u.t1}"
        for name in GRADS:
            if name in ("dq", "dk"):
                gv = got[name][s0:s1, u.j].double().cpu().numpy()
                rv = r[name][r0:r1]
            elif name in ("dg", "dbeta"):
                gv = got[name][s0:s1, hs].double().cpu().numpy()
                rv = r[name][:, r0:r1].T
            else:
                gv = got[name][s0:s1, hs].double().cpu().numpy()
                rv = r[name][:, r0:r1].transpose(1, 0, 2)
            compare(f"{tag}/{name}", gv, rv)

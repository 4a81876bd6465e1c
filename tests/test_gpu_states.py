"""GPU parity of the per-document boundary states (gdn_fwd_states /
gdn_bwd_states: S_in, S_out and their gradients) against the FP64 oracle,
through the C ABI."""
import numpy as np
import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from oracle import ref
from tests.gdn_testutil import compare, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta")

CASES = [
    ("tiny", inputs.workload(0)),
    # ragged documents and an empty one (its states pass straight through)
    ("ragged_empty", inputs.custom([1, 63, 0, 65, 130], 2, 6, seed=21)),
    # a long document cut into four segments: S_in enters through the first segment's
    # zero-start walk, dS_out through the last segment's reverse walk and the merges
    ("split4", inputs.custom([1000, 70], 1, 2, seed=22, segments=4)),
]


def boundary(w, seed, scale=0.2):
    gen = torch.Generator().manual_seed(seed)
    s_in = scale * torch.randn((w.N, w.HV, 128, 128), generator=gen, dtype=torch.float32)
    ds_out = scale * torch.randn((w.N, w.HV, 128, 128), generator=gen, dtype=torch.float32)
    return s_in, ds_out


@pytest.mark.parametrize("form", [0, 1], ids=["full_form", "replay_form"])
@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_boundary_states_parity(name, w, form):
    """Both saved forms: the replay form's backward rebuilds the UT blocks and V_new from a saved set
    that already holds S_in's effect, and its walks take dS_out in the same way."""
    import linear_attention_gdn_gb300 as gdn
    x = inputs.generate(w, "cpu")
    d = to_dev(x)
    s_in, ds_out = boundary(w, 100 + len(name))
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments, saved_form=form)
    buf = gdn.Buffers(prob, w.cu_seqlens, fill=255)
    nan = float("nan")
    o = torch.full((w.T, w.HV, 128), nan, dtype=torch.bfloat16, device="cuda")
    s_out = torch.full((w.N, w.HV, 128, 128), nan, dtype=torch.float32, device="cuda")
    ds_in = torch.full((w.N, w.HV, 128, 128), nan, dtype=torch.float32, device="cuda")
    gr = dict(dq=torch.full((w.T, w.H, 128), nan, dtype=torch.bfloat16, device="cuda"),
              dk=torch.full((w.T, w.H, 128), nan, dtype=torch.bfloat16, device="cuda"),
              dv=torch.full((w.T, w.HV, 128), nan, dtype=torch.bfloat16, device="cuda"),
              dg=torch.full((w.T, w.HV), nan, dtype=torch.float32, device="cuda"),
              dbeta=torch.full((w.T, w.HV), nan, dtype=torch.float32, device="cuda"))
    gdn.gdn_fwd_states(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens,
                       s_in.cuda(), o, s_out, buf.saved, buf.workspace)
    gdn.gdn_bwd_states(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"],
                       ds_out.cuda(), buf.saved, gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], ds_in,
                       buf.workspace)
    st = gdn.gdn_device_status(buf.workspace)
    assert st == 0, gdn.gdn_status_string(st)
    xs = dict(x)
    xs["s_in"], xs["ds_out"] = s_in.double().numpy(), ds_out.double().numpy()
    res = ref.run(xs, w.H, w.HV, l2norm=w.l2norm, scale=w.scale, states=True)
    r = ref.assemble(res, w.T, w.H, w.HV, 128, 128, w.cu_seqlens, states=True)
    compare(f"{name}/o", o.double().cpu().numpy(), r["o"])
    for n in GRADS:
        compare(f"{name}/{n}", gr[n].double().cpu().numpy(), r[n])
    compare(f"{name}/s_out", s_out.double().cpu().numpy(), r["s_out"])
    compare(f"{name}/ds_in", ds_in.double().cpu().numpy(), r["ds_in"])


def test_document_cut_across_calls():
    """A document run as two calls joined at a chunk boundary by S_out -> S_in
    (forward) and dS_in -> dS_out (backward) gives the one-call outputs and
    gradients bit for bit: the FP32 boundary state is exactly what the one-call
    walk carries across that chunk boundary in its registers."""
    import linear_attention_gdn_gb300 as gdn
    w = inputs.custom([640], 1, 3, seed=23)
    x = inputs.generate(w, "cpu")
    d = to_dev(x)
    whole_prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm)
    whole = gdn.Buffers(whole_prob, w.cu_seqlens, fill=255)
    o_w = torch.empty((w.T, w.HV, 128), dtype=torch.bfloat16, device="cuda")
    g_w = [torch.empty_like(d[n]) for n in ("q", "k", "v", "g", "beta")]
    gdn.gdn_fwd(whole_prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o_w, whole.saved,
                whole.workspace)
    gdn.gdn_bwd(whole_prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"],
                whole.saved, *g_w, whole.workspace)
    m = 256   # the cut, at a chunk boundary
    parts = []
    for lo, hi in ((0, m), (m, w.T)):
        cu = np.array([0, hi - lo], dtype=np.int32)
        prob = gdn.problem(hi - lo, 1, w.H, w.HV, w.scale, w.l2norm)
        sl = {n: d[n][lo:hi].contiguous() for n in ("q", "k", "v", "g", "beta", "dO")}
        parts.append((prob, cu, sl, gdn.Buffers(prob, cu, fill=255)))
    s_mid = torch.empty((1, w.HV, 128, 128), dtype=torch.float32, device="cuda")
    ds_mid = torch.empty_like(s_mid)
    outs, grads = [], []
    for i, (prob, cu, sl, buf) in enumerate(parts):
        o = torch.empty((cu[1], w.HV, 128), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_fwd_states(prob, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], torch.from_numpy(cu).cuda(), cu,
                           s_mid if i == 1 else None, o, s_mid if i == 0 else None, buf.saved, buf.workspace)
        outs.append(o)
    for i in (1, 0):
        prob, cu, sl, buf = parts[i]
        gg = [torch.empty_like(sl[n]) for n in ("q", "k", "v", "g", "beta")]
        gdn.gdn_bwd_states(prob, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], torch.from_numpy(cu).cuda(), cu,
                           sl["dO"], ds_mid if i == 0 else None, buf.saved, *gg, ds_mid if i == 1 else None,
                           buf.workspace)
        grads.insert(0, gg)
    torch.cuda.synchronize()
    for buf in (whole, parts[0][3], parts[1][3]):
        st = gdn.gdn_device_status(buf.workspace)
        assert st == 0, gdn.gdn_status_string(st)
    assert torch.equal(torch.cat(outs), o_w)
    for j, n in enumerate(("dq", "dk", "dv", "dg", "dbeta")):
        assert torch.equal(torch.cat([grads[0][j], grads[1][j]]), g_w[j]), n

"""GPU parity of the backward (and the checkpointed step) against the FP64
oracle, through the C ABI; bitwise reproducibility; saved-set refusal."""
import numpy as np
import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from oracle import ref
from tests.gdn_testutil import compare, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta")


def alloc_grads(w):
    nan = float("nan")
    return dict(dq=torch.full((w.T, w.H, 128), nan, dtype=torch.bfloat16, device="cuda"),
                dk=torch.full((w.T, w.H, 128), nan, dtype=torch.bfloat16, device="cuda"),
                dv=torch.full((w.T, w.HV, 128), nan, dtype=torch.bfloat16, device="cuda"),
                dg=torch.full((w.T, w.HV), nan, dtype=torch.float32, device="cuda"),
                dbeta=torch.full((w.T, w.HV), nan, dtype=torch.float32, device="cuda"))


def run_fwd_bwd(w, d, nan_fill=True):
    import linear_attention_gdn_gb300 as gdn
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments)
    buf = gdn.Buffers(prob, w.cu_seqlens, fill=255 if nan_fill else None)
    o = torch.full((w.T, w.HV, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    gr = alloc_grads(w)
    gdn.gdn_fwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o, buf.saved,
                buf.workspace)
    gdn.gdn_bwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"], buf.saved,
                gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], buf.workspace)
    st = gdn.gdn_device_status(buf.workspace)
    assert st == 0, gdn.gdn_status_string(st)
    return prob, buf, o, gr


CASES = [
    ("tiny", inputs.workload(0)),
    ("ragged_g3", inputs.custom([1, 63, 64, 65, 0, 130, 200], 2, 6, seed=5)),
    ("nol2_g1", inputs.custom([100, 28], 1, 1, l2norm=False, prenorm_qk=True, seed=6)),
    ("split4", inputs.custom([1000, 70], 1, 2, seed=7, segments=4)),
    # nine value heads per q/k head; gates steep enough (about -1 per token) that a chunk's
    # cumulative gate spans more than 2^100, past the factored per-token exponentials
    ("g9_steep", inputs.custom([150, 64, 1, 97], 1, 9, g_lo=-1.5, g_hi=-0.5, seed=11)),
    # four value heads per q/k head and more (chunk, q/k head) items than SMs, ragged and empty documents
    ("items_g4", inputs.custom([700, 0, 1300, 64, 33, 2100], 3, 12, seed=12)),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_backward_parity(name, w):
    x = inputs.generate(w, "cpu")
    d = to_dev(x)
    prob, buf, o, gr = run_fwd_bwd(w, d)
    res = ref.run(x, w.H, w.HV, l2norm=w.l2norm, scale=w.scale)
    r = ref.assemble(res, w.T, w.H, w.HV, 128, 128, w.cu_seqlens)
    compare(f"{name}/o", o.double().cpu().numpy(), r["o"])
    for n in GRADS:
        compare(f"{name}/{n}", gr[n].double().cpu().numpy(), r[n])


def test_bitwise_reproducible_and_ckpt_equivalent():
    import linear_attention_gdn_gb300 as gdn
    w = inputs.custom([300, 77, 640], 2, 6, seed=9, segments=0)
    d = to_dev(inputs.generate(w, "cpu"))
    _, _, o1, g1 = run_fwd_bwd(w, d)
    _, _, o2, g2 = run_fwd_bwd(w, d, nan_fill=False)
    assert torch.equal(o1, o2)
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n
    # the checkpointed step (fwd without states, fwd with states, bwd) gives
    # the same bits as fwd + bwd
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm)
    buf = gdn.Buffers(prob, w.cu_seqlens, fill=255)
    o3 = torch.full_like(o1, float("nan"))
    g3 = alloc_grads(w)
    gdn.gdn_ckpt_fwd_bwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"], o3,
                         g3["dq"], g3["dk"], g3["dv"], g3["dg"], g3["dbeta"], buf.saved, buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 0
    assert torch.equal(o1, o3)
    for n in GRADS:
        assert torch.equal(g1[n], g3[n]), n


def test_saved_mismatch_refused():
    """A saved set from another problem (different scale) is refused on the
    device: status GDN_ERR_SAVED_MISMATCH and the gradients stay unwritten."""
    import linear_attention_gdn_gb300 as gdn
    w = inputs.workload(0)
    d = to_dev(inputs.generate(w, "cpu"))
    prob, buf, o, gr = run_fwd_bwd(w, d)
    other = gdn.problem(w.T, w.N, w.H, w.HV, 0.5 * w.scale, w.l2norm)
    g2 = alloc_grads(w)
    gdn.gdn_bwd(other, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"], buf.saved,
                g2["dq"], g2["dk"], g2["dv"], g2["dg"], g2["dbeta"], buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 4
    for n in GRADS:
        assert torch.isnan(g2[n].float()).all(), n


@pytest.mark.parametrize("dev_cu", [
    [0, 192, 320],    # the two documents' lengths swapped: same total, same chunk count
    [0, 128, 300],    # the last document cut short: the device copy ends before T
    [0, 200, 160],    # decreasing
])
def test_disagreeing_device_cu_seqlens_refused(dev_cu):
    """The host copy of cu_seqlens plans the call and the device copy drives the
    kernels.  A device copy that differs from the host copy is caught by the
    table kernel (GDN_ERR_INVALID_ARG) before any kernel indexes with it; every
    output stays unwritten."""
    import linear_attention_gdn_gb300 as gdn
    w = inputs.workload(0)   # host cu_seqlens [0, 128, 320]
    d = to_dev(inputs.generate(w, "cpu"))
    bad = torch.tensor(dev_cu, dtype=torch.int32, device="cuda")
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm)
    buf = gdn.Buffers(prob, w.cu_seqlens, fill=255)
    o = torch.full((w.T, w.HV, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_fwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], bad, w.cu_seqlens, o, buf.saved, buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 1
    assert torch.isnan(o.float()).all()
    gr = alloc_grads(w)
    gdn.gdn_bwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], bad, w.cu_seqlens, d["dO"], buf.saved,
                gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 1
    for n in GRADS:
        assert torch.isnan(gr[n].float()).all(), n

"""The device-side timeout path, driven on purpose without faulting the GPU.

Every wait inside the kernels is bounded (about one second); when one runs
out, the kernel records GDN_ERR_TIMEOUT in the call's error word, finishes
without leaving copies or MMAs in flight, and every later kernel of the call
skips its work.  The library has a test-only hook for this: with
GDN_TEST_WITHHOLD_LOAD set, one CTA of the replay form's V_new kernel never
requests its first tiles, so its wait for them is the one that runs out.  The
test checks the status, that no gradient was written, and that the context is
still usable: the same call without the hook gives the full form's results."""
import os

import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from tests.gdn_testutil import to_dev
from tests.test_gpu_bwd import GRADS, alloc_grads

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    import linear_attention_gdn_gb300 as gdn
    w = inputs.custom([130, 64], 2, 4, seed=21)
    d = to_dev(inputs.generate(w, "cpu"))
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, saved_form=gdn.SAVED_REPLAY)
    buf = gdn.Buffers(prob, w.cu_seqlens, fill=255)
    o = torch.empty((w.T, w.HV, 128), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_fwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o, buf.saved,
                buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 0
    gr = alloc_grads(w)
    os.environ["GDN_TEST_WITHHOLD_LOAD"] = "1"
    try:
        gdn.gdn_bwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"],
                    buf.saved, gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], buf.workspace)
        assert gdn.gdn_device_status(buf.workspace) == 6   # GDN_ERR_TIMEOUT
    finally:
        del os.environ["GDN_TEST_WITHHOLD_LOAD"]
    for n in GRADS:
        assert torch.isnan(gr[n].float()).all(), n
    # the context is still usable: the same backward, now complete, equals the full form's
    gdn.gdn_bwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"], buf.saved,
                gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 0
    pf = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm)
    bf = gdn.Buffers(pf, w.cu_seqlens)
    gf = alloc_grads(w)
    gdn.gdn_fwd(pf, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o, bf.saved, bf.workspace)
    gdn.gdn_bwd(pf, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"], bf.saved,
                gf["dq"], gf["dk"], gf["dv"], gf["dg"], gf["dbeta"], bf.workspace)
    assert gdn.gdn_device_status(bf.workspace) == 0
    for n in GRADS:
        assert torch.equal(gr[n], gf[n]), n

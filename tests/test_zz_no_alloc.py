"""gdn_fwd_noalloc: the forward for callers that cannot allocate device memory
(hosts that pass only inputs and outputs, or paths where cudaMalloc's device
synchronisation is not allowed).  It runs with the library's fixed 64 MiB
device array as its workspace; its output must match gdn_fwd's on the same
inputs, call after call, since every call reuses the same array."""
import numpy as np
import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from tests.gdn_testutil import compare, to_dev

pytestmark = pytest.mark.gpu


def fwd_with_workspace(gdn, w, d):
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm)
    buf = gdn.Buffers(prob, w.cu_seqlens)
    o = torch.full((w.T, w.HV, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_fwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o, None, buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 0
    return o


def fwd_no_alloc(gdn, w, d):
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm)
    o = torch.full((w.T, w.HV, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_fwd_noalloc(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o)
    torch.cuda.synchronize()
    return o


def test_no_alloc_forward_matches_gdn_fwd_twice():
    import linear_attention_gdn_gb300 as gdn
    # two different problems back to back: the second call finds the first
    # call's contents in the shared array.  Both entry points run the same
    # kernels on the same inputs, so the outputs must agree bit for bit (the
    # tolerance comparison is only there to say by how much, should they not).
    cases = [inputs.custom([1, 63, 64, 65, 0, 130, 200], 2, 6, seed=5), inputs.workload(0)]
    for w in cases:
        d = to_dev(inputs.generate(w, "cpu", with_grad=False))
        want = fwd_with_workspace(gdn, w, d)
        got = fwd_no_alloc(gdn, w, d)
        if not torch.equal(got, want):
            compare(f"noalloc/{w.name}", got.double().cpu().numpy(), want.double().cpu().numpy())
            raise AssertionError(f"noalloc/{w.name}: not bitwise equal to gdn_fwd")


def test_no_alloc_refuses_problems_beyond_the_fixed_scratch():
    import linear_attention_gdn_gb300 as gdn
    w = inputs.custom([64 * 200], 16, 48, seed=1)     # 200 chunks x 48 heads: far above 64 MiB
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm)
    q = torch.zeros((w.T, w.H, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((w.T, w.HV, 128), dtype=torch.bfloat16, device="cuda")
    gb = torch.zeros((w.T, w.HV), dtype=torch.float32, device="cuda")
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_fwd_noalloc(prob, q, q, v, gb, gb, cu, w.cu_seqlens, v)
    assert e.value.status == 3   # GDN_ERR_WORKSPACE_TOO_SMALL

"""GPU parity of the causal conv1d + SiLU front (gdn_conv1d_fwd / _bwd)
against the FP64 oracle, through the C ABI; bitwise reproducibility."""
import numpy as np
import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from oracle import conv1d
from tests.gdn_testutil import compare

pytestmark = pytest.mark.gpu

CASES = [
    # ragged, single-token and empty documents; one partial channel block
    ("ragged", [1, 2, 3, 70, 0, 129], 64, 4, True),
    ("c520_w3", [300, 17], 520, 3, True),
    ("w1_nobias", [5, 40], 256, 1, False),
    ("w2", [33, 0, 64], 128, 2, True),
    # several token ranges per channel block, their cuts falling inside documents
    ("ranges", [2500, 700, 1, 2900], 1024, 4, True),
]


def run(case, d):
    import linear_attention_gdn_gb300 as gdn
    T, C = d["x"].shape
    W = d["w"].shape[1]
    cu = d["cu_seqlens"]
    prob = gdn.conv_problem(T, len(cu) - 1, C, W)
    cu_dev = torch.from_numpy(cu).cuda()
    x, w, dy = d["x"].cuda(), d["w"].cuda(), d["dy"].cuda()
    b = d["b"].cuda() if d["b"] is not None else None
    y = torch.full((T, C), float("nan"), dtype=torch.bfloat16, device="cuda")
    dx = torch.full_like(y, float("nan"))
    dw = torch.full((C, W), float("nan"), dtype=torch.float32, device="cuda")
    db = torch.full((C,), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.full((max(gdn.gdn_conv1d_workspace_bytes(prob, cu), 16),), 255, dtype=torch.uint8, device="cuda")
    gdn.gdn_conv1d_fwd(prob, x, w, b, cu_dev, cu, y)
    gdn.gdn_conv1d_bwd(prob, x, w, b, cu_dev, cu, dy, dx, dw, db, ws)
    assert gdn.gdn_device_status(ws) == 0   # the backward's status word (it syncs the stream)
    return y, dx, dw, db


@pytest.mark.parametrize("name,docs,C,W,bias", CASES, ids=[c[0] for c in CASES])
def test_conv1d_parity(name, docs, C, W, bias):
    d = inputs.conv_inputs(docs, C, W, seed=len(name) + C, with_bias=bias)
    y, dx, dw, db = run(name, d)
    x64 = d["x"].double().numpy()
    w64 = d["w"].double().numpy()
    b64 = d["b"].double().numpy() if d["b"] is not None else None
    ry = conv1d.forward(x64, w64, b64, d["cu_seqlens"])
    rdx, rdw, rdb = conv1d.backward(x64, w64, b64, d["cu_seqlens"], d["dy"].double().numpy())
    compare(f"{name}/y", y.double().cpu().numpy(), ry)
    compare(f"{name}/dx", dx.double().cpu().numpy(), rdx)
    compare(f"{name}/dw", dw.double().cpu().numpy(), rdw)
    compare(f"{name}/db", db.double().cpu().numpy(), rdb)


def test_conv1d_b23_sampled_channels():
    """The pages' B23 shape (4 documents 12288/8192/7168/5120, 10,240 packed
    q/k/v channels): every output of 96 channels spread over all channel
    blocks against the oracle (channels are independent), and run-to-run
    bitwise equality of everything."""
    docs, C = [12288, 8192, 7168, 5120], 10240
    d = inputs.conv_inputs(docs, C, 4, seed=23)
    y, dx, dw, db = run("b23", d)
    y2, dx2, dw2, db2 = run("b23", d)
    assert torch.equal(y, y2) and torch.equal(dx, dx2) and torch.equal(dw, dw2) and torch.equal(db, db2)
    ch = np.unique(np.concatenate([np.arange(0, C, 113), [C - 1]]))[:96]
    x64 = d["x"][:, ch].double().numpy()
    w64 = d["w"][ch].double().numpy()
    b64 = d["b"][ch].double().numpy()
    cu = d["cu_seqlens"]
    ry = conv1d.forward(x64, w64, b64, cu)
    rdx, rdw, rdb = conv1d.backward(x64, w64, b64, cu, d["dy"][:, ch].double().numpy())
    compare("b23/y", y[:, ch].double().cpu().numpy(), ry)
    compare("b23/dx", dx[:, ch].double().cpu().numpy(), rdx)
    compare("b23/dw", dw[ch].double().cpu().numpy(), rdw)
    compare("b23/db", db[ch].double().cpu().numpy(), rdb)

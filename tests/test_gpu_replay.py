"""The replay saved form on the GPU, through the C ABI.

The replay form keeps only the state tape (and the segment transfers) from
the forward; the backward runs the UT / WY preparation again and recomputes
V_new = U - W S from the saved states.  It computes exactly what the full
form computes, so every output and gradient must agree bit for bit with the
full form's; the recomputed intermediates (T, V_new) and the adjoint walk's
tapes (dS', dV_new) are also compared, stage by stage, with the chunked FP64
oracle's intermediates."""
import numpy as np
import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from oracle import chunked, tables
from tests.gdn_testutil import compare, to_dev
from tests.test_gpu_bwd import GRADS, alloc_grads
from tests.test_gpu_fwd import CASES

pytestmark = pytest.mark.gpu


def run(w, d, form, ckpt=False):
    import linear_attention_gdn_gb300 as gdn
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments, saved_form=form)
    buf = gdn.Buffers(prob, w.cu_seqlens, fill=255)
    o = torch.full((w.T, w.HV, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    gr = alloc_grads(w)
    if ckpt:
        gdn.gdn_ckpt_fwd_bwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"],
                             o, gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], buf.saved, buf.workspace)
    else:
        gdn.gdn_fwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o, buf.saved,
                    buf.workspace)
        gdn.gdn_bwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"],
                    buf.saved, gr["dq"], gr["dk"], gr["dv"], gr["dg"], gr["dbeta"], buf.workspace)
    st = gdn.gdn_device_status(buf.workspace)
    assert st == 0, gdn.gdn_status_string(st)
    torch.cuda.synchronize()
    return prob, buf, o, gr


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
def test_replay_form_equals_full_form(name, w):
    import linear_attention_gdn_gb300 as gdn
    d = to_dev(inputs.generate(w, "cpu"))
    _, bf, o_f, g_f = run(w, d, gdn.SAVED_FULL)
    _, br, o_r, g_r = run(w, d, gdn.SAVED_REPLAY)
    assert br.saved_bytes < bf.saved_bytes
    assert torch.equal(o_f, o_r), f"{name}/o"
    for n in GRADS:
        assert torch.equal(g_f[n], g_r[n]), f"{name}/{n}"


def test_replay_ckpt_equals_replay_fwd_bwd():
    import linear_attention_gdn_gb300 as gdn
    w = inputs.custom([300, 77, 640], 2, 6, seed=9)
    d = to_dev(inputs.generate(w, "cpu"))
    _, _, o1, g1 = run(w, d, gdn.SAVED_REPLAY)
    _, _, o2, g2 = run(w, d, gdn.SAVED_REPLAY, ckpt=True)
    assert torch.equal(o1, o2)
    for n in GRADS:
        assert torch.equal(g1[n], g2[n]), n


def test_saved_form_mismatch_refused():
    """A full-form saved set handed to a replay-form backward (and the reverse) is refused on the device."""
    import linear_attention_gdn_gb300 as gdn
    w = inputs.workload(0)
    d = to_dev(inputs.generate(w, "cpu"))
    for made, used in ((gdn.SAVED_FULL, gdn.SAVED_REPLAY), (gdn.SAVED_REPLAY, gdn.SAVED_FULL)):
        prob, buf, _, _ = run(w, d, made)
        other = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, saved_form=used)
        ws = torch.empty((gdn.gdn_saved_bytes(other, w.cu_seqlens)[1],), dtype=torch.uint8, device="cuda")
        g2 = alloc_grads(w)
        gdn.gdn_bwd(other, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, d["dO"],
                    buf.saved, g2["dq"], g2["dk"], g2["dv"], g2["dg"], g2["dbeta"], ws)
        assert gdn.gdn_device_status(ws) == 4
        for n in GRADS:
            assert torch.isnan(g2[n].float()).all(), n


def _sw(R, C):
    """element index of (row i, col j) in a BF16 swizzled tile of R rows and C columns"""
    i = np.arange(R)[:, None]
    j = np.arange(C)[None, :]
    off = (j >> 6) * (R * 128) + i * 128 + ((((j & 63) >> 3) ^ (i & 7)) << 4) + (j & 7) * 2
    return off // 2


def _tiles(ws, off, n_blocks, block_bytes, start, R, C):
    """[n_blocks, R, C] float64 from BF16 tiles at byte `start` of each block of the region at `off`."""
    raw = ws[off: off + n_blocks * block_bytes].view(n_blocks, block_bytes)[:, start: start + R * C * 2]
    x = raw.contiguous().view(torch.bfloat16).double().cpu().numpy().reshape(n_blocks, R * C)
    return x[:, _sw(R, C)]


@pytest.mark.parametrize("name,w", [CASES[0], CASES[1]], ids=[CASES[0][0], CASES[1][0]])
def test_stage_parity_replay_intermediates(name, w):
    """T (the UT inverse) and the matrices that define W = T' K and U = T'' V, the gated Aqk and the
    per-token scalars of the UT blocks, V_new (recomputed from the saved states), the adjoint walk's dS'
    (gradient of the state leaving each chunk) and dV_new, against the chunked FP64 oracle's
    intermediates."""
    import linear_attention_gdn_gb300 as gdn
    x = inputs.generate(w, "cpu")
    d = to_dev(x)
    prob, buf, _, _ = run(w, d, gdn.SAVED_REPLAY)
    o_cb, o_vn, o_ds, o_dv = gdn.gdn_backward_tape_offsets(prob, w.cu_seqlens)
    NC, HV, H, G = w.num_chunks, w.HV, w.H, w.HV // w.H
    nb = NC * HV
    ws = buf.workspace
    T_gpu = _tiles(ws, o_cb, nb, 33792, 24576, 64, 64).reshape(NC, HV, 64, 64)
    Tp_gpu = _tiles(ws, o_cb, nb, 33792, 0, 64, 64).reshape(NC, HV, 64, 64)        # T' = T diag(beta gamma rk)
    Tpp_gpu = _tiles(ws, o_cb, nb, 33792, 8192, 64, 64).reshape(NC, HV, 64, 64)    # T'' = T diag(beta)
    Aqk_gpu = _tiles(ws, o_cb, nb, 33792, 16384, 64, 64).reshape(NC, HV, 64, 64)
    scal = ws[o_cb: o_cb + nb * 33792].view(nb, 33792)[:, 32768: 32768 + 129 * 4].contiguous()
    scal = scal.view(torch.float32).double().cpu().numpy().reshape(NC, HV, 129)   # sc[64], kd[64], e^{G_L}
    vn_gpu = _tiles(ws, o_vn, nb, 16384, 0, 128, 64).reshape(NC, HV, 128, 64)        # [dv][token]
    ds_gpu = _tiles(ws, o_ds, nb, 32768, 0, 128, 128).reshape(NC, HV, 128, 128)      # dS'^T [dv][dk]
    dvn_gpu = _tiles(ws, o_dv, nb, 16384, 0, 128, 64).reshape(NC, HV, 128, 64)       # [dv][token]
    t = tables.chunk_tables(w.cu_seqlens)
    f64 = lambda a: a.double().numpy()
    keys = ("T", "Tp", "Tpp", "Aqk", "sc", "kd", "gL", "Vn", "dS", "dVn")
    got = {k: [] for k in keys}
    ref = {k: [] for k in keys}
    cu = w.cu_seqlens
    for doc in range(w.N):
        s0, s1 = int(cu[doc]), int(cu[doc + 1])
        if s1 == s0:
            continue
        for j in range(H):
            hs = slice(j * G, (j + 1) * G)
            out = chunked.group(f64(x["q"][s0:s1, j]), f64(x["k"][s0:s1, j]),
                                f64(x["v"][s0:s1, hs]).transpose(1, 0, 2), f64(x["g"][s0:s1, hs]).T,
                                f64(x["beta"][s0:s1, hs]).T, f64(x["dO"][s0:s1, hs]).transpose(1, 0, 2),
                                l2norm=w.l2norm, scale=w.scale)
            qd, kd_ = f64(x["q"][s0:s1, j]), f64(x["k"][s0:s1, j])
            rq = 1 / np.sqrt((qd * qd).sum(1) + 1e-6) if w.l2norm else np.ones(s1 - s0)
            rk = 1 / np.sqrt((kd_ * kd_).sum(1) + 1e-6) if w.l2norm else np.ones(s1 - s0)
            for h in range(G):
                hv = j * G + h
                for c, it in enumerate(out["inter"][h]):
                    gc = int(t["chunk_offsets"][doc]) + c
                    L = len(it["G"])
                    b_c = f64(x["beta"][s0 + 64 * c: s0 + 64 * c + L, hv])
                    rk_c, rq_c = rk[64 * c: 64 * c + L], rq[64 * c: 64 * c + L]
                    got["T"].append(T_gpu[gc, hv, :L, :L])
                    ref["T"].append(it["T"])
                    # W = T' K (raw k rows) and U = T'' V: the matrices that define them
                    got["Tp"].append(Tp_gpu[gc, hv, :L, :L])
                    ref["Tp"].append(it["T"] * (b_c * it["gam"] * rk_c)[None, :])
                    got["Tpp"].append(Tpp_gpu[gc, hv, :L, :L])
                    ref["Tpp"].append(it["T"] * b_c[None, :])
                    got["Aqk"].append(Aqk_gpu[gc, hv, :L, :L])
                    ref["Aqk"].append(np.tril(it["Aqk"]))
                    got["sc"].append(scal[gc, hv, :L])
                    ref["sc"].append(w.scale * it["gam"] * rq_c)
                    got["kd"].append(scal[gc, hv, 64: 64 + L])
                    ref["kd"].append(it["dec"] * rk_c)
                    got["gL"].append(scal[gc, hv, 128: 129])
                    ref["gL"].append(it["gam"][-1:])
                    got["Vn"].append(vn_gpu[gc, hv, :, :L].T)
                    ref["Vn"].append(it["Vn"])
                    got["dS"].append(ds_gpu[gc, hv].T)
                    ref["dS"].append(out["dS"][c, h])
                    dO_c = f64(x["dO"][s0 + 64 * c: s0 + 64 * c + L, hv])
                    got["dVn"].append(dvn_gpu[gc, hv, :, :L].T)
                    ref["dVn"].append(w.scale * it["Aqk"].T @ dO_c + it["Kd"] @ out["dS"][c, h])
    for k in got:
        compare(f"{name}/{k}", np.concatenate([a.ravel() for a in got[k]]),
                np.concatenate([a.ravel() for a in ref[k]]))


@pytest.mark.parametrize("idx", [3, 4])
def test_replay_form_equals_full_form_full_size(idx):
    """The full-size workloads: the 166-document pack with L2 off, and the 524,288-token document whose
    walks are split into segments (its backward merges read the saved segment transfers in both
    forms).  Every output and gradient agrees bit for bit between the saved forms."""
    import linear_attention_gdn_gb300 as gdn
    w = inputs.workload(idx)
    x = inputs.generate(w, "cuda")
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    res = {}
    for form in (gdn.SAVED_FULL, gdn.SAVED_REPLAY):
        prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments, saved_form=form)
        buf = gdn.Buffers(prob, w.cu_seqlens)
        out = dict(o=torch.empty((w.T, w.HV, 128), dtype=torch.bfloat16, device="cuda"),
                   dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]), dv=torch.empty_like(x["v"]),
                   dg=torch.empty_like(x["g"]), dbeta=torch.empty_like(x["beta"]))
        gdn.gdn_fwd(prob, x["q"], x["k"], x["v"], x["g"], x["beta"], cu, w.cu_seqlens, out["o"], buf.saved,
                    buf.workspace)
        gdn.gdn_bwd(prob, x["q"], x["k"], x["v"], x["g"], x["beta"], cu, w.cu_seqlens, x["dO"], buf.saved,
                    out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"], buf.workspace)
        assert gdn.gdn_device_status(buf.workspace) == 0
        res[form] = out
        del buf
        torch.cuda.empty_cache()
    for n in ("o",) + GRADS:
        assert torch.equal(res[gdn.SAVED_FULL][n], res[gdn.SAVED_REPLAY][n]), f"workload{idx}/{n}"

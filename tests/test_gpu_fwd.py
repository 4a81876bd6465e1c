"""GPU parity of the forward path against the FP64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from linear_attention_gdn_gb300 import inputs
from oracle import ref, tables
from tests.gdn_testutil import compare, decode_tape, to_dev

pytestmark = pytest.mark.gpu


def run_fwd(w, d, save=True, nan_fill=True):
    import linear_attention_gdn_gb300 as gdn
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments)
    buf = gdn.Buffers(prob, w.cu_seqlens, fill=255 if nan_fill else None)
    o = torch.full((w.T, w.HV, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_fwd(prob, d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_dev"], w.cu_seqlens, o,
                buf.saved if save else None, buf.workspace)
    assert gdn.gdn_device_status(buf.workspace) == 0
    torch.cuda.synchronize()
    return prob, buf, o


def oracle_full(w, d, chunk_states=False):
    res = ref.run(d, w.H, w.HV, l2norm=w.l2norm, scale=w.scale, with_grad=False, chunk_states=chunk_states)
    return res, ref.assemble(res, w.T, w.H, w.HV, 128, 128, w.cu_seqlens, with_grad=False)


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
def test_forward_parity(name, w):
    d = to_dev(inputs.generate(w, "cpu", with_grad=False))
    prob, buf, o = run_fwd(w, d)
    res, r = oracle_full(w, {**d, "q": d["q"].cpu(), "k": d["k"].cpu(), "v": d["v"].cpu(),
                             "g": d["g"].cpu(), "beta": d["beta"].cpu()}, chunk_states=True)
    compare(f"{name}/o", o.double().cpu().numpy(), r["o"])
    # stage parity: the saved state entering every chunk
    t = tables.chunk_tables(w.cu_seqlens)
    tape = decode_tape(buf.saved, w.num_chunks, w.HV)
    G = w.HV // w.H
    ref_tape = np.zeros_like(tape)
    for u, rr in res:
        c0 = t["chunk_offsets"][u.doc]
        n = rr["S"].shape[0]
        ref_tape[c0:c0 + n, u.j * G:(u.j + 1) * G] = rr["S"]
    compare(f"{name}/tape", tape, ref_tape)


def test_chunk_tables_bitexact():
    import linear_attention_gdn_gb300 as gdn
    for lens in ([128, 192], [1, 0, 64, 65, 0, 0, 300, 7], [64 * 5000], [3] * 2000):
        w = inputs.custom(lens, 1, 1, seed=1)
        d = to_dev(inputs.generate(w, "cuda", with_grad=False))
        prob, buf, o = run_fwd(w, d, save=False)
        offs, nc = gdn.gdn_chunk_table_offsets(prob, w.cu_seqlens)
        t = tables.chunk_tables(w.cu_seqlens)
        assert nc == len(t["chunk_doc"])
        ws = buf.workspace
        get = lambda off, n: ws[off: off + 4 * n].view(torch.int32).cpu().numpy()
        assert np.array_equal(get(offs[0], w.N + 1), t["chunk_offsets"])
        assert np.array_equal(get(offs[1], nc), t["chunk_doc"])
        assert np.array_equal(get(offs[2], nc), t["chunk_tok0"])
        assert np.array_equal(get(offs[3], nc), t["chunk_len"])

"""Host-side logic of the C ABI, without a GPU: the library loads and exports
every symbol include/gdn.h declares, byte queries follow the documented
layout, and invalid problems / arguments are refused before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import linear_attention_gdn_gb300 as gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "gdn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:gdn_status|const char \*|int32_t)\s*\**\s*(gdn_\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol():
    gdn.load()
    syms = declared_symbols()
    assert len(syms) >= 8, syms
    for s in syms:
        assert hasattr(gdn.lib, s), s
        assert s in gdn.EXPORTS


def test_status_strings():
    for code in range(9):
        assert gdn.gdn_status_string(code)
    assert "KDA" in gdn.gdn_status_string(8)
    assert gdn.gdn_status_string(99) == "unknown status"


def test_saved_and_workspace_bytes():
    p = gdn.problem(320, 2, 2, 4)
    saved, ws = gdn.gdn_saved_bytes(p, [0, 128, 320])
    # header + 5 chunks x 4 v-heads x (32 KiB BF16 state + 33 KiB UT block + 16 KiB V_new^T), no split
    assert saved == 4096 + 5 * 4 * 32768 + 5 * 4 * 33792 + 5 * 4 * 16384
    assert ws > 5 * 4 * 33792
    p = gdn.problem(64 * 40, 1, 1, 2, segments=4)
    saved, _ = gdn.gdn_saved_bytes(p, [0, 64 * 40])
    assert gdn.gdn_plan_segment_chunks(p, [0, 64 * 40]) == 10
    # 4 segments -> 3 transfer operators per v-head in FP32, then the UT blocks and V_new^T tiles
    assert saved == 4096 + 40 * 2 * 32768 + 3 * 2 * 128 * 128 * 4 + 40 * 2 * 33792 + 40 * 2 * 16384


def test_replay_form_saved_bytes():
    # the replay form keeps the header and the BF16 state tape (plus M_seg when a document is split)
    p = gdn.problem(320, 2, 2, 4, saved_form=gdn.SAVED_REPLAY)
    saved, ws = gdn.gdn_saved_bytes(p, [0, 128, 320])
    assert saved == 4096 + 5 * 4 * 32768
    full_saved, full_ws = gdn.gdn_saved_bytes(gdn.problem(320, 2, 2, 4), [0, 128, 320])
    assert full_saved - saved == 5 * 4 * (33792 + 16384)
    assert ws - full_ws == 5 * 4 * 16384   # the recomputed V_new^T tiles
    p = gdn.problem(64 * 40, 1, 1, 2, segments=4, saved_form=gdn.SAVED_REPLAY)
    saved, _ = gdn.gdn_saved_bytes(p, [0, 64 * 40])
    assert saved == 4096 + 40 * 2 * 32768 + 3 * 2 * 128 * 128 * 4
    # at the 4-document bench workload: 24 KiB of states per token, under 30 KB
    w = [0, 98304, 163840, 221184, 262144]
    saved, _ = gdn.gdn_saved_bytes(gdn.problem(262144, 4, 16, 48, saved_form=gdn.SAVED_REPLAY), w)
    assert saved / 262144 < 30e3
    offs = gdn.gdn_backward_tape_offsets(gdn.problem(320, 2, 2, 4, saved_form=gdn.SAVED_REPLAY), [0, 128, 320])
    assert all(o > 0 and o % 1024 == 0 for o in offs)
    offs = gdn.gdn_backward_tape_offsets(gdn.problem(320, 2, 2, 4), [0, 128, 320])
    assert offs[0] == 0 and offs[1] == 0 and offs[2] > 0 and offs[3] > 0


def test_bad_saved_form_refused():
    p = gdn.problem(320, 2, 2, 4, saved_form=2)
    with pytest.raises(gdn.GDNError) as e:
        gdn.gdn_saved_bytes(p, [0, 128, 320])
    assert e.value.status == 1


@pytest.mark.parametrize("cu,T,N,H,HV,dk,code", [
    ([0, 10, 5], 5, 2, 1, 1, 128, 1),      # decreasing cu_seqlens
    ([1, 10], 9, 1, 1, 1, 128, 1),         # cu[0] != 0
    ([0, 10], 11, 1, 1, 1, 128, 1),        # cu[N] != T
    ([0, 10], 10, 1, 2, 3, 128, 2),        # HV not a multiple of H
    ([0, 10], 10, 1, 1, 1, 64, 2),         # dk != 128
])
def test_invalid_problems_refused(cu, T, N, H, HV, dk, code):
    p = gdn.problem(T, N, H, HV, dk=dk)
    cu_a = np.array(cu, dtype=np.int32)
    s, w = ctypes.c_size_t(), ctypes.c_size_t()
    st = gdn.lib.gdn_saved_bytes(ctypes.byref(p), cu_a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                 ctypes.byref(s), ctypes.byref(w))
    assert st == code


def test_invalid_arguments_refused_before_launch():
    """Null, misaligned or undersized buffers return INVALID_ARG /
    WORKSPACE_TOO_SMALL from host checks (fake device addresses are never
    dereferenced)."""
    p = gdn.problem(320, 2, 2, 4)
    cu = np.array([0, 128, 320], dtype=np.int32)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    saved, ws = gdn.gdn_saved_bytes(p, cu)
    A = 1 << 20   # a fake, aligned address
    args = lambda q=A, o=A, sv=A, wsp=A, wsb=ws: (ctypes.byref(p), ctypes.c_void_p(q), ctypes.c_void_p(A),
                                                  ctypes.c_void_p(A), ctypes.c_void_p(A), ctypes.c_void_p(A),
                                                  ctypes.cast(ctypes.c_void_p(A), ctypes.POINTER(ctypes.c_int32)),
                                                  cup, ctypes.c_void_p(o) if o else None,
                                                  ctypes.c_void_p(sv) if sv else None,
                                                  ctypes.c_void_p(wsp) if wsp else None, wsb, None)
    assert gdn.lib.gdn_fwd(*args(q=A + 2)) == 1          # misaligned q
    assert gdn.lib.gdn_fwd(*args(o=0, sv=0)) == 1         # nothing to write
    assert gdn.lib.gdn_fwd(*args(wsp=0)) == 1             # no workspace
    assert gdn.lib.gdn_fwd(*args(wsb=100)) == 3           # workspace too small
    bw = lambda sv, wsb: gdn.lib.gdn_bwd(ctypes.byref(p), *[ctypes.c_void_p(A)] * 5,
                                          ctypes.cast(ctypes.c_void_p(A), ctypes.POINTER(ctypes.c_int32)), cup,
                                          ctypes.c_void_p(A), ctypes.c_void_p(sv) if sv else None,
                                          *[ctypes.c_void_p(A)] * 5, ctypes.c_void_p(A), wsb, None)
    assert bw(0, ws) == 1                                 # backward needs the saved set
    assert bw(A, 10) == 3


def test_conv1d_problem_checks_and_workspace():
    """The conv1d front refuses C not a multiple of 8 and W outside 1..4, and
    its backward workspace is the 16-byte status word plus one FP32 partial of
    dw and db per 1,024-token range (host checks only)."""
    cu = np.array([0, 1000, 2500], dtype=np.int32)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    n = ctypes.c_size_t(0)
    for C, W, code in ((12, 4, 1), (16, 5, 2), (16, 0, 1), (16, 4, 0)):
        p = gdn.conv_problem(2500, 2, C, W)
        assert gdn.lib.gdn_conv1d_workspace_bytes(ctypes.byref(p), cup, ctypes.byref(n)) == code
    assert n.value == 16 + 3 * (4 + 1) * 16 * 4


def test_kda_saved_and_workspace_bytes():
    """The per-channel-decay entry points: the full form's saved set = header + (BF16 state + BF16
    V_new^T + the 82,944-byte block of decay products and UT tiles) per chunk and value head; the
    replay form leaves the blocks out (the backward forms them again).  The workspace holds the
    per-chunk blocks and the backward's tapes in either form."""
    p = gdn.problem(320, 2, 2, 4)
    saved, ws = gdn.gdn_kda_saved_bytes(p, [0, 128, 320])
    assert saved == 4096 + 5 * 4 * (32768 + 16384 + 82944)
    assert ws >= 5 * 4 * (82944 + 32768 + 16384)
    p2 = gdn.problem(320, 2, 2, 4, saved_form=gdn.SAVED_REPLAY)
    saved2, ws2 = gdn.gdn_kda_saved_bytes(p2, [0, 128, 320])
    assert saved2 == 4096 + 5 * 4 * (32768 + 16384)
    assert ws2 == ws


def test_kda_invalid_arguments_refused_before_launch():
    p = gdn.problem(128, 1, 1, 2)
    cu = np.array([0, 128], dtype=np.int32)
    cup = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    fake = ctypes.c_void_p(1 << 20)   # 16-byte aligned, never dereferenced: every check fails first
    # o is required
    st = gdn.lib.gdn_kda_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, fake, cup, None, None, fake, 1 << 30,
                             None)
    assert st == 1
    # misaligned input
    bad = ctypes.c_void_p((1 << 20) + 4)
    st = gdn.lib.gdn_kda_fwd(ctypes.byref(p), bad, fake, fake, fake, fake, fake, cup, fake, None, fake, 1 << 30,
                             None)
    assert st == 1
    # workspace too small
    st = gdn.lib.gdn_kda_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, fake, cup, fake, None, fake, 16, None)
    assert st == 3
    # backward without a saved set
    st = gdn.lib.gdn_kda_bwd(ctypes.byref(p), fake, fake, fake, fake, fake, fake, cup, fake, None, fake, fake,
                             fake, fake, fake, fake, 1 << 30, None)
    assert st == 1
    # unsupported head size
    p3 = gdn.problem(128, 1, 1, 2, dk=64)
    s = ctypes.c_size_t(0)
    assert gdn.lib.gdn_kda_saved_bytes(ctypes.byref(p3), cup, ctypes.byref(s), ctypes.byref(s)) == 2

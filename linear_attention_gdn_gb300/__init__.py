"""Python binding of libgdn, the sm_103a chunked Gated DeltaNet training path.

The functions below carry the C ABI's names (include/gdn.h) and only marshal
arguments: torch tensors become device pointers, host arrays become host
pointers, a non-OK status raises GDNError.  Every step of the path runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and importing
this package fails if the compiled library is missing (build it with
``python -m linear_attention_gdn_gb300.build`` or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

LIB_PATH = _build.LIB
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_WORKSPACE_TOO_SMALL",
          4: "GDN_ERR_SAVED_MISMATCH", 5: "GDN_ERR_CUDA", 6: "GDN_ERR_TIMEOUT", 7: "GDN_ERR_DEVICE",
          8: "GDN_ERR_GATE_RANGE"}
EXPORTS = ("gdn_saved_bytes", "gdn_fwd", "gdn_bwd", "gdn_ckpt_fwd_bwd", "gdn_status_string",
           "gdn_device_status", "gdn_plan_segment_chunks", "gdn_chunk_table_offsets", "gdn_profile_enable",
           "gdn_profile_read", "gdn_fwd_noalloc", "gdn_fwd_states", "gdn_bwd_states", "gdn_conv1d_workspace_bytes",
           "gdn_conv1d_fwd", "gdn_conv1d_bwd", "gdn_backward_tape_offsets", "gdn_kda_saved_bytes", "gdn_kda_fwd",
           "gdn_kda_bwd", "gdn_tensor_probe")
SAVED_FULL, SAVED_REPLAY = 0, 1   # gdn_problem.saved_form


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({gdn_status_string(status)})")


class gdn_kernel_stat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_longlong), ("timed_launches", ctypes.c_longlong),
                ("total_ms", ctypes.c_double)]


class gdn_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("N", ctypes.c_int32), ("H", ctypes.c_int32), ("HV", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("scale", ctypes.c_float),
                ("l2norm", ctypes.c_int32), ("segments", ctypes.c_int32), ("saved_form", ctypes.c_int32)]


class gdn_conv_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("N", ctypes.c_int32), ("C", ctypes.c_int32), ("W", ctypes.c_int32)]


def conv_problem(T, N, C, W=4) -> gdn_conv_problem:
    return gdn_conv_problem(int(T), int(N), int(C), int(W))


def problem(T, N, H, HV, scale=128 ** -0.5, l2norm=True, segments=0, dk=128, dv=128,
            saved_form=SAVED_FULL) -> gdn_problem:
    return gdn_problem(int(T), int(N), int(H), int(HV), int(dk), int(dv), float(scale), int(bool(l2norm)),
                       int(segments), int(saved_form))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libgdn.so not built ({LIB_PATH}); run linear_attention_gdn_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, sz, i32p = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_int32)
    pp = ctypes.POINTER(gdn_problem)
    L.gdn_saved_bytes.argtypes = [pp, i32p, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.gdn_fwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, sz, vp]
    L.gdn_bwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.gdn_ckpt_fwd_bwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.gdn_fwd_states.argtypes = [pp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, sz, vp]
    L.gdn_bwd_states.argtypes = [pp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.gdn_status_string.argtypes = [ctypes.c_int]
    L.gdn_status_string.restype = ctypes.c_char_p
    L.gdn_device_status.argtypes = [vp, vp]
    L.gdn_plan_segment_chunks.argtypes = [pp, i32p]
    L.gdn_plan_segment_chunks.restype = ctypes.c_int32
    L.gdn_chunk_table_offsets.argtypes = [pp, i32p, ctypes.POINTER(sz), i32p]
    L.gdn_backward_tape_offsets.argtypes = [pp, i32p, ctypes.POINTER(sz)]
    L.gdn_kda_saved_bytes.argtypes = [pp, i32p, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.gdn_kda_fwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, sz, vp]
    L.gdn_kda_bwd.argtypes = [pp, vp, vp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.gdn_fwd_noalloc.argtypes = [pp, vp, vp, vp, vp, vp, i32p, i32p, vp, vp]
    L.gdn_fwd_noalloc.restype = ctypes.c_int
    cp = ctypes.POINTER(gdn_conv_problem)
    L.gdn_conv1d_workspace_bytes.argtypes = [cp, i32p, ctypes.POINTER(sz)]
    L.gdn_conv1d_fwd.argtypes = [cp, vp, vp, vp, vp, i32p, vp, vp]
    L.gdn_conv1d_bwd.argtypes = [cp, vp, vp, vp, vp, i32p, vp, vp, vp, vp, vp, sz, vp]
    for name in ("gdn_conv1d_workspace_bytes", "gdn_conv1d_fwd", "gdn_conv1d_bwd", "gdn_fwd_states",
                 "gdn_bwd_states"):
        getattr(L, name).restype = ctypes.c_int
    L.gdn_tensor_probe.argtypes = [ctypes.c_int32, vp, ctypes.POINTER(ctypes.c_double), vp]
    L.gdn_tensor_probe.restype = ctypes.c_int
    L.gdn_profile_enable.argtypes = [ctypes.c_int]
    L.gdn_profile_enable.restype = None
    L.gdn_profile_read.argtypes = [ctypes.POINTER(gdn_kernel_stat), ctypes.c_int]
    L.gdn_profile_read.restype = ctypes.c_int
    for name in ("gdn_saved_bytes", "gdn_fwd", "gdn_bwd", "gdn_ckpt_fwd_bwd", "gdn_device_status",
                 "gdn_chunk_table_offsets", "gdn_backward_tape_offsets"):
        getattr(L, name).restype = ctypes.c_int
    return L


class _Lazy:
    """The library handle, loaded on first use (importing the package must not
    require the library, so that the build step can import it)."""
    _h = None

    def __getattr__(self, name):
        if _Lazy._h is None:
            _Lazy._h = _load()
        return getattr(_Lazy._h, name)


lib = _Lazy()


def load():
    """Load libgdn.so now and check that it exports every ABI symbol."""
    for name in EXPORTS:
        getattr(lib, name)
    return lib


def _ptr(x):
    """Device/host address of a tensor or array; None -> NULL."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return ctypes.c_void_p(x.data_ptr())
    if isinstance(x, np.ndarray):
        return ctypes.c_void_p(x.ctypes.data)
    return ctypes.c_void_p(int(x))


def _cu_host(cu):
    a = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st, where):
    if st != 0:
        raise GDNError(st, where)


def gdn_status_string(status: int) -> str:
    return lib.gdn_status_string(int(status)).decode()


def gdn_saved_bytes(prob: gdn_problem, cu_seqlens_host):
    cu, cup = _cu_host(cu_seqlens_host)
    s, w = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib.gdn_saved_bytes(ctypes.byref(prob), cup, ctypes.byref(s), ctypes.byref(w)), "gdn_saved_bytes")
    return s.value, w.value


def gdn_plan_segment_chunks(prob: gdn_problem, cu_seqlens_host) -> int:
    cu, cup = _cu_host(cu_seqlens_host)
    return int(lib.gdn_plan_segment_chunks(ctypes.byref(prob), cup))


def gdn_chunk_table_offsets(prob: gdn_problem, cu_seqlens_host):
    cu, cup = _cu_host(cu_seqlens_host)
    offs = (ctypes.c_size_t * 4)()
    nc = ctypes.c_int32(0)
    _check(lib.gdn_chunk_table_offsets(ctypes.byref(prob), cup, offs, ctypes.byref(nc)), "gdn_chunk_table_offsets")
    return list(offs), nc.value


def gdn_backward_tape_offsets(prob: gdn_problem, cu_seqlens_host):
    """Workspace byte offsets of the UT blocks, V_new^T, dS' and dV_new^T tapes a gdn_bwd call leaves
    (the first two only in the replay saved form); see include/gdn.h."""
    cu, cup = _cu_host(cu_seqlens_host)
    offs = (ctypes.c_size_t * 4)()
    _check(lib.gdn_backward_tape_offsets(ctypes.byref(prob), cup, offs), "gdn_backward_tape_offsets")
    return list(offs)


def gdn_fwd(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, o, saved, workspace, ws_bytes=None,
            stream=None):
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_fwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                       ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(o),
                       _ptr(saved), _ptr(workspace), ws_bytes, _stream(stream)), "gdn_fwd")


def gdn_kda_saved_bytes(prob: gdn_problem, cu_seqlens_host):
    """(saved bytes, workspace bytes) of the per-channel-decay (KDA) entry points."""
    cu, cup = _cu_host(cu_seqlens_host)
    s, w = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib.gdn_kda_saved_bytes(ctypes.byref(prob), cup, ctypes.byref(s), ctypes.byref(w)),
           "gdn_kda_saved_bytes")
    return s.value, w.value


def gdn_kda_fwd(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, o, saved, workspace, ws_bytes=None,
                stream=None):
    """KDA forward: g is FP32 [T, HV, 128] (a log decay per key channel); see include/gdn.h."""
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_kda_fwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(o),
                           _ptr(saved), _ptr(workspace), ws_bytes, _stream(stream)), "gdn_kda_fwd")


def gdn_kda_bwd(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, dO, saved, dq, dk, dv, dg, dbeta,
                workspace, ws_bytes=None, stream=None):
    """KDA backward: dg is FP32 [T, HV, 128]; see include/gdn.h."""
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_kda_bwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(dO),
                           _ptr(saved), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(workspace),
                           ws_bytes, _stream(stream)), "gdn_kda_bwd")


def gdn_fwd_states(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, s_in, o, s_out, saved, workspace,
                   ws_bytes=None, stream=None):
    """gdn_fwd with per-document boundary states: s_in, s_out FP32 [N, HV, 128, 128] (either may be None);
    see include/gdn.h."""
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_fwd_states(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(s_in),
                              _ptr(o), _ptr(s_out), _ptr(saved), _ptr(workspace), ws_bytes, _stream(stream)),
           "gdn_fwd_states")


def gdn_fwd_noalloc(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, o, stream=None):
    """gdn_fwd without a caller workspace or saved set (the library's fixed
    64 MiB device array serves as the workspace); see include/gdn.h."""
    cu, cup = _cu_host(cu_seqlens_host)
    _check(lib.gdn_fwd_noalloc(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(o),
                               _stream(stream)), "gdn_fwd_noalloc")


def gdn_bwd(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, dO, saved, dq, dk, dv, dg, dbeta,
            workspace, ws_bytes=None, stream=None):
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_bwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                       ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(dO),
                       _ptr(saved), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(workspace),
                       ws_bytes, _stream(stream)), "gdn_bwd")


def gdn_bwd_states(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, dO, ds_out, saved, dq, dk, dv, dg,
                   dbeta, ds_in, workspace, ws_bytes=None, stream=None):
    """gdn_bwd with per-document boundary states: ds_out, ds_in FP32 [N, HV, 128, 128] (either may be None);
    see include/gdn.h."""
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_bwd_states(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                              ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(dO),
                              _ptr(ds_out), _ptr(saved), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                              _ptr(ds_in), _ptr(workspace), ws_bytes, _stream(stream)), "gdn_bwd_states")


def gdn_ckpt_fwd_bwd(prob, q, k, v, g, beta, cu_seqlens_dev, cu_seqlens_host, dO, o, dq, dk, dv, dg, dbeta,
                     saved_scratch, workspace, ws_bytes=None, stream=None):
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_ckpt_fwd_bwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(dO),
                                _ptr(o), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(saved_scratch),
                                _ptr(workspace), ws_bytes, _stream(stream)), "gdn_ckpt_fwd_bwd")


def gdn_profile_enable(on: int) -> None:
    lib.gdn_profile_enable(int(on))


def gdn_profile_read(out, max_entries: int) -> int:
    return int(lib.gdn_profile_read(out, int(max_entries)))


def gdn_profile_read_all() -> dict:
    """{kernel name: {launches, timed_launches, total_ms}} since the last read."""
    arr = (gdn_kernel_stat * 32)()
    n = gdn_profile_read(arr, 32)
    return {arr[i].name.decode(): {"launches": arr[i].launches, "timed_launches": arr[i].timed_launches,
                                   "total_ms": arr[i].total_ms} for i in range(min(n, 32))}


def gdn_device_status(workspace, stream=None) -> int:
    return int(lib.gdn_device_status(_ptr(workspace), _stream(stream)))


def gdn_tensor_probe(iters, dev_err, stream=None) -> float:
    """Launch the tensor-pipe probe (include/gdn.h) on `stream`; dev_err is a zeroed device int32
    tensor.  Returns the FLOP count of the launch (the caller times it)."""
    flops = ctypes.c_double(0.0)
    _check(lib.gdn_tensor_probe(int(iters), _ptr(dev_err), ctypes.byref(flops), _stream(stream)),
           "gdn_tensor_probe")
    return flops.value


# ---------------------------------------------------------------------------
# allocation helpers (torch owns the memory; the library allocates nothing)
# ---------------------------------------------------------------------------
def gdn_conv1d_workspace_bytes(prob, cu_seqlens_host) -> int:
    cu, cup = _cu_host(cu_seqlens_host)
    n = ctypes.c_size_t(0)
    _check(lib.gdn_conv1d_workspace_bytes(ctypes.byref(prob), cup, ctypes.byref(n)), "gdn_conv1d_workspace_bytes")
    return int(n.value)


def gdn_conv1d_fwd(prob, x, w, b, cu_seqlens_dev, cu_seqlens_host, y, stream=None):
    """The short causal conv1d + SiLU front (see include/gdn.h): x, y [T, C] BF16; w [C, W], b [C] FP32."""
    cu, cup = _cu_host(cu_seqlens_host)
    _check(lib.gdn_conv1d_fwd(ctypes.byref(prob), _ptr(x), _ptr(w), _ptr(b),
                              ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(y),
                              _stream(stream)), "gdn_conv1d_fwd")


def gdn_conv1d_bwd(prob, x, w, b, cu_seqlens_dev, cu_seqlens_host, dy, dx, dw, db, workspace, ws_bytes=None,
                   stream=None):
    cu, cup = _cu_host(cu_seqlens_host)
    ws_bytes = workspace.numel() * workspace.element_size() if ws_bytes is None else ws_bytes
    _check(lib.gdn_conv1d_bwd(ctypes.byref(prob), _ptr(x), _ptr(w), _ptr(b),
                              ctypes.cast(_ptr(cu_seqlens_dev), ctypes.POINTER(ctypes.c_int32)), cup, _ptr(dy),
                              _ptr(dx), _ptr(dw), _ptr(db), _ptr(workspace), ws_bytes, _stream(stream)),
           "gdn_conv1d_bwd")


class Buffers:
    """Caller-side saved set and workspace for one problem, allocated with torch."""

    def __init__(self, prob: gdn_problem, cu_seqlens_host, device="cuda", fill=None, kda=False):
        import torch
        sizes = gdn_kda_saved_bytes if kda else gdn_saved_bytes
        self.saved_bytes, self.ws_bytes = sizes(prob, cu_seqlens_host)
        mk = (lambda n: torch.full((max(n, 1024),), fill, dtype=torch.uint8, device=device)) if fill is not None \
            else (lambda n: torch.empty((max(n, 1024),), dtype=torch.uint8, device=device))
        self.saved = mk(self.saved_bytes)
        self.workspace = mk(self.ws_bytes)

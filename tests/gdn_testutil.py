"""Shared helpers of the GPU parity tests: the accuracy budget, the saved-tape
decoder, and drivers that run the library and the oracle on one workload."""
import numpy as np
import torch

from oracle import ref, tables

# accuracy budget of the pages' FP64 comparisons ("feat(cake_gdn_kcp) ... #8172"
# page, #8181 section): rel-RMS <= 1e-2, max-abs <= 2e-2 * max|ref|, finite
REL_RMS = 1e-2
MAX_ABS = 2e-2


def compare(name, x, r, rel_rms=REL_RMS, max_abs=MAX_ABS):
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert x.shape == r.shape, (name, x.shape, r.shape)
    assert np.isfinite(x).all(), f"{name}: non-finite values"
    nr = np.linalg.norm(r)
    if nr == 0:
        assert np.abs(x).max() == 0, name
        return 0.0, 0.0
    rr = np.linalg.norm(x - r) / nr
    ma = np.abs(x - r).max() / np.abs(r).max()
    assert rr <= rel_rms and ma <= max_abs, f"{name}: rel-RMS {rr:.3e}, max-abs/max|ref| {ma:.3e}"
    return rr, ma


def _sw_index():
    """element index of (row i, col j) in a BF16 SwTile(128 x 128)"""
    i = np.arange(128)[:, None]
    j = np.arange(128)[None, :]
    off = (j >> 6) * (128 * 128) + i * 128 + ((((j & 63) >> 3) ^ (i & 7)) << 4) + (j & 7) * 2
    return off // 2


SW = _sw_index()


def decode_tape(saved: torch.Tensor, NC: int, HV: int):
    """BF16 states entering each chunk, as S [NC, HV, dk, dv] float64."""
    raw = saved[4096: 4096 + NC * HV * 32768].view(torch.bfloat16).view(NC, HV, 16384)
    st = raw.double().cpu().numpy()[:, :, SW]          # [NC, HV, dv(i), dk(j)] = S^T
    return st.transpose(0, 1, 3, 2)


def to_dev(inp, device="cuda"):
    out = {}
    for n, x in inp.items():
        out[n] = x.to(device) if hasattr(x, "to") else x
    out["cu_dev"] = torch.from_numpy(np.asarray(inp["cu_seqlens"], dtype=np.int32)).to(device)
    return out

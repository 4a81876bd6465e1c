"""Seeded synthetic workloads for the chunked Gated DeltaNet training path.

This module only draws inputs; it holds none of the method's arithmetic.  Both
the CUDA path's tests/bench and the CPU oracle take their inputs from here, so
that both sides see exactly the same BF16 / FP32 values.

The workloads mirror the shapes the flashinfer Cake GDN pages time and test:
packed variable-length documents, head dim 128, (H, HV) = (16, 48) query/key
and value heads, BF16 q/k/v and output gradient, FP32 gate g and beta
("feat(cake_gdn_kcp) ... #8172" page, #8181 section, which fixes the head
dimension at 128, q/k/v and the output gradient in BF16 and g, beta in FP32;
the "shape A" pack of 4 documents 98304/65536/57344/40960 is from the "#8542"
page, Conventions).

Value distributions (all seeded):
  q, k, v, dO ~ N(0, 1), rounded to BF16
  g = logsigmoid(U(lo, hi))   (FP32; per token and v-head)
  beta = sigmoid(N(0, 1))     (FP32; per token and v-head)
One generator draws in the fixed order q, k, v, g, beta, dO.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

CHUNK = 64
HEAD_DIM = 128


@dataclass
class Workload:
    name: str
    doc_lens: list
    H: int
    HV: int
    l2norm: bool
    g_lo: float
    g_hi: float
    seed: int
    prenorm_qk: bool = False     # q, k normalised in FP32 on the host, then BF16
    segments: int = 0            # 0 = planner's choice, >0 = forced P
    scale: float = HEAD_DIM ** -0.5
    dk: int = HEAD_DIM
    dv: int = HEAD_DIM
    ops: tuple = ("fwd", "fwd+bwd")

    @property
    def T(self) -> int:
        return int(sum(self.doc_lens))

    @property
    def N(self) -> int:
        return len(self.doc_lens)

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.doc_lens)]).astype(np.int32)

    @property
    def num_chunks(self) -> int:
        return int(sum((n + CHUNK - 1) // CHUNK for n in self.doc_lens))


def loguniform_doc_lens(total: int, lo: int, hi: int, seed: int) -> list:
    """Document lengths floor(exp(U(ln lo, ln hi))) drawn until they cover
    `total` tokens; the last one is truncated so the sum is exactly `total`."""
    rng = np.random.default_rng(seed)
    lens, acc = [], 0
    while acc < total:
        n = int(math.floor(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
        n = max(1, min(n, total - acc))
        lens.append(n)
        acc += n
    return lens


def workload(idx: int) -> Workload:
    """The five workloads: 0 = tiny (2 docs, H=2/HV=4), 1 = one 8192-token doc,
    2 = four docs, 262144 tokens, 3 = log-uniform short docs, 262144 tokens,
    L2 norm off (q, k pre-normalised), 4 = one 524288-token doc with a stronger
    gate (U(3, 8)) and the intra-GPU segment split."""
    if idx == 0:
        return Workload("tiny_2doc_h2_hv4", [128, 192], 2, 4, True, 2.0, 6.0, 0)
    if idx == 1:
        return Workload("doc8k_h16_hv48", [8192], 16, 48, True, 2.0, 6.0, 1)
    if idx == 2:
        return Workload("pack4_262k_h16_hv48", [98304, 65536, 57344, 40960], 16, 48,
                        True, 2.0, 6.0, 2, ops=("fwd", "fwd+bwd", "ckpt"))
    if idx == 3:
        return Workload("loguniform_262k_h16_hv48", loguniform_doc_lens(262144, 64, 8192, 3),
                        16, 48, False, 2.0, 6.0, 3, prenorm_qk=True, ops=("fwd+bwd",))
    if idx == 4:
        return Workload("doc524k_h16_hv48", [524288], 16, 48, True, 3.0, 8.0, 4,
                        ops=("fwd+bwd",))
    raise ValueError(f"no workload {idx}")


def custom(doc_lens, H, HV, l2norm=True, g_lo=2.0, g_hi=6.0, seed=0, prenorm_qk=False,
           segments=0, name="custom") -> Workload:
    return Workload(name, list(doc_lens), H, HV, l2norm, g_lo, g_hi, seed,
                    prenorm_qk=prenorm_qk, segments=segments)


def generate(w: Workload, device="cpu", with_grad=True) -> dict:
    """Draw the inputs of workload `w` on `device` with one seeded generator.

    Returns q, k [T,H,dk] BF16; v [T,HV,dv] BF16; g, beta [T,HV] FP32;
    dO [T,HV,dv] BF16 (if with_grad); cu_seqlens (host int32 numpy)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    T, H, HV = w.T, w.H, w.HV

    def normal(shape):
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)

    q = normal((T, H, w.dk))
    k = normal((T, H, w.dk))
    if w.prenorm_qk:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    q = q.to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    v = normal((T, HV, w.dv)).to(torch.bfloat16)
    x = torch.rand((T, HV), generator=gen, device=dev, dtype=torch.float32)
    g = torch.nn.functional.logsigmoid(w.g_lo + (w.g_hi - w.g_lo) * x)
    beta = torch.sigmoid(normal((T, HV)))
    out = dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=w.cu_seqlens)
    if with_grad:
        out["dO"] = normal((T, HV, w.dv)).to(torch.bfloat16)
    return out


def generate_kda(w: Workload, device="cpu", with_grad=True) -> dict:
    """Inputs of the per-channel-decay (KDA) form for workload `w`: as generate(),
    except g [T,HV,dk] FP32, one log decay per key channel,
    g = logsigmoid(U(g_lo, g_hi)) drawn per (token, v-head, channel)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    T, H, HV = w.T, w.H, w.HV

    def normal(shape):
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)

    q = normal((T, H, w.dk))
    k = normal((T, H, w.dk))
    if w.prenorm_qk:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    q = q.to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    v = normal((T, HV, w.dv)).to(torch.bfloat16)
    x = torch.rand((T, HV, w.dk), generator=gen, device=dev, dtype=torch.float32)
    g = torch.nn.functional.logsigmoid(w.g_lo + (w.g_hi - w.g_lo) * x)
    beta = torch.sigmoid(normal((T, HV)))
    out = dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=w.cu_seqlens)
    if with_grad:
        out["dO"] = normal((T, HV, w.dv)).to(torch.bfloat16)
    return out


def conv_inputs(doc_lens, C: int, W: int = 4, seed: int = 0, with_bias: bool = True) -> dict:
    """Seeded inputs of the causal conv1d + SiLU front: x, dy [T, C] ~ N(0, 1) in
    BF16; taps w [C, W] ~ N(0, 0.5^2) and bias b [C] ~ N(0, 0.1^2) in FP32 (the
    pages give no initialisation; these keep z = conv + b of order one).  One
    generator draws x, w, b, dy in that order."""
    gen = torch.Generator().manual_seed(seed)
    T = int(sum(doc_lens))
    x = torch.randn((T, C), generator=gen).to(torch.bfloat16)
    w = 0.5 * torch.randn((C, W), generator=gen)
    b = 0.1 * torch.randn((C,), generator=gen)
    dy = torch.randn((T, C), generator=gen).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(doc_lens)]).astype(np.int32)
    return dict(x=x, w=w, b=b if with_bias else None, dy=dy, cu_seqlens=cu)

"""Benchmark of the GB300 chunked Gated DeltaNet training step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 2] [--op fwd+bwd|fwd|ckpt] [--kda]

A step is one pass of the whole hot path over one batch: gdn_fwd (writing the
saved states) + gdn_bwd on the packed 4-document workload of 262,144 tokens
with H = 16 q/k heads, HV = 48 value heads, head dim 128 (the pages' "shape
A").  Inputs are seeded synthetic tensors already resident in HBM; they are
far larger than L2 (no flush needed).  Prints one JSON line.

Multi-GPU: the path has no exchange step, so N GPUs run N independent
replicas (one process per GPU under torchrun); value = all tokens processed /
the slowest rank's time.

--impl reference times the FP64 CPU oracle (the only other implementation
there is) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN fwd+bwd Mtokens/s on 1 GB300 (H16/HV48, d=128); % BF16 tensor-core peak"
UNIT = "Mtokens/s"
D = 128
C = 64


# ---------------------------------------------------------------------------
# algorithmic work: the method's own FLOPs and HBM bytes (the dense tile
# products of the chunked algorithm, KK^T and QK^T once per q/k head, the O(C^3)
# inverse not counted; bytes = the method's inputs read once, its outputs
# written once and the BF16 state saved every 64 tokens written once and read
# once).  Per full chunk and value head this is the method's count:
#   fwd  F_f = HV (6 d^2 + 6 C d) + H (4 C d) FLOP / token,
#        57,728 B / token at (16, 48): q, k, v, g, beta in; o, states out
#   bwd  F_b = HV (14 d^2 + 24 C d) + H (4 C d) FLOP / token,
#        78,592 B / token: q, k, v, g, beta, dO, states in; dq, dk, dv, dg, dbeta out
# Partial chunks use their real length L in place of C.  Each kernel is
# credited with the method tensors it reads or writes (so a tensor two kernels
# read counts for both) and with its share of the products; the intermediate
# tapes this design keeps in HBM (dS', V_new^T, dV_new^T, T blocks) are never
# credited: they are reported apart, as design bytes.
# ---------------------------------------------------------------------------
def chunk_lens(w):
    out = []
    for n in w.doc_lens:
        out += [C] * (n // C) + ([n % C] if n % C else [])
    return out


# per kernel: coefficients (a, b, c) of HV (a L d^2 + b L^2 d) + H (c L^2 d) per chunk of L tokens
KERNEL_FLOP_TERMS = {
    "prep_kernel": (0, 0, 4),        # KK^T, QK^T
    "fwd_scan_kernel": (6, 6, 0),    # W S, S Q, Kd^T V_new; W, U, Aqk V_new
    "fwd_walk_kernel": (6, 6, 4),    # the same with the UT stage (KK^T, QK^T) inside the walk
    "bwd_scan_kernel": (6, 4, 0),    # dS' K^T, dV_new W, dO' Q; W, dO^T Aqk
    "bwd_walk_kernel": (6, 4, 4),    # the same with the UT stage inside the walk
    "grad_kernel": (8, 20, 4),       # the rest of F_b
    "vnew_kernel": (2, 4, 0),        # replay form: W, U and W S again
}


def kernel_flops(name, w):
    """Method FLOPs of one launch of `name` on workload w (real chunk lengths)."""
    a, b, c = KERNEL_FLOP_TERMS.get(name, (0, 0, 0))
    return sum(w.HV * (a * L * D * D + b * L * L * D) + w.H * c * L * L * D for L in chunk_lens(w))


def method_tensors(w):
    """Bytes of each tensor the method reads or writes once (states: one BF16 128 x 128 per chunk and value
    head)."""
    T, H, HV, NC = w.T, w.H, w.HV, w.num_chunks
    qk, vh, gb = T * H * D * 2 * 2, T * HV * D * 2, T * HV * 4 * 2
    return {"qk": qk, "k": qk // 2, "v": vh, "gb": gb, "o": vh, "dO": vh, "states": NC * HV * D * D * 2,
            "dqdk": qk, "dv": vh, "dgdb": gb}


KERNEL_METHOD_TENSORS = {
    "prep_kernel": ("qk", "gb"),
    "fwd_scan_kernel": ("qk", "v", "o", "states"),
    "fwd_walk_kernel": ("qk", "v", "gb", "o", "states"),
    "bwd_scan_kernel": ("qk", "dO"),
    "bwd_walk_kernel": ("qk", "v", "gb", "dO", "states"),
    "grad_kernel": ("qk", "v", "gb", "dO", "states", "dqdk", "dv", "dgdb"),
    "vnew_kernel": ("k", "v", "states"),
}


def kernel_bytes(name, w):
    """Method bytes of one launch of `name` (the method's tensors it reads or writes)."""
    m = method_tensors(w)
    return sum(m[t] for t in KERNEL_METHOD_TENSORS.get(name, ()))


def step_bytes(w, op):
    m = method_tensors(w)
    fwd = m["qk"] + m["v"] + m["gb"] + m["o"] + m["states"]
    fwd_nosave = fwd - m["states"]
    bwd = m["qk"] + m["v"] + m["gb"] + m["dO"] + m["states"] + m["dqdk"] + m["dv"] + m["dgdb"]
    return {"fwd": fwd, "fwd+bwd": fwd + bwd, "ckpt": fwd_nosave + fwd + bwd}[op]


def step_flops(w, op):
    Ls = chunk_lens(w)
    f_fwd = sum(w.HV * (6 * L * D * D + 6 * L * L * D) + w.H * 4 * L * L * D for L in Ls)
    f_bwd = sum(w.HV * (14 * L * D * D + 24 * L * L * D) + w.H * 4 * L * L * D for L in Ls)
    return {"fwd": f_fwd, "fwd+bwd": f_fwd + f_bwd, "ckpt": 2 * f_fwd + f_bwd}[op]


# The per-channel-decay (KDA) form on the same shapes: the decay products M = K^ (exp(G_r - G_c) . K^)^T
# and P are per value head (the decay differs per head), and g, dg are [T, HV, 128] FP32:
#   fwd  F_f = HV (6 d^2 + 10 C d) FLOP / token
#   bwd  F_b = HV (14 d^2 + 28 C d) FLOP / token (the GDN count with its KK^T, QK^T term per value head)
# bytes: the GDN method tensors with g (and dg) 128 FP32 values per token and value head.
def kda_step_flops(w):
    Ls = chunk_lens(w)
    return sum(w.HV * ((6 + 14) * L * D * D + (10 + 28) * L * L * D) for L in Ls)


def kda_step_bytes(w):
    m = method_tensors(w)
    g_extra = w.T * w.HV * (D - 1) * 4   # g (or dg) per channel instead of per token
    fwd = m["qk"] + m["v"] + m["gb"] + g_extra + m["o"] + m["states"]
    bwd = m["qk"] + m["v"] + m["gb"] + g_extra + m["dO"] + m["states"] + m["dqdk"] + m["dv"] + m["dgdb"] + g_extra
    return fwd + bwd


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        m = json.load(open(p))
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained", m["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def source_hash():
    """Hash of the GDN kernels' sources (the conv1d front, profiled apart, and
    the tensor-core probe, which is not on the path, are left out) with comments
    and whitespace removed, so that a change to a comment keeps the committed
    ncu figures valid."""
    h = hashlib.sha256()
    cs = os.path.join(ROOT, "linear_attention_gdn_gb300", "csrc")
    for f in sorted(os.listdir(cs)):
        if f in ("gdn_conv1d.cu", "gdn_probe.cu"):
            continue
        t = open(os.path.join(cs, f), encoding="utf-8").read()
        t = re.sub(r"/\*.*?\*/", " ", t, flags=re.S)
        t = re.sub(r"//[^\n]*", " ", t)
        h.update(f.encode() + b"\0" + " ".join(t.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the current sources (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    m = json.load(open(p))
    if m.get("source_hash") != source_hash():
        return None
    k = m.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch_full")


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi"] + (["-i", str(self.gpu)] if self.gpu else []) +
                                         [f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a while to start: wait for its first sample (up to 5 s) and keep
            # only the samples taken from here on, i.e. during the timed region
            t0 = time.time()
            while not self.lines and self.proc.poll() is None and time.time() - t0 < 5:
                time.sleep(0.01)
            self.lines.clear()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
# ---------------------------------------------------------------------------
# replica timing (N independent replicas, one process per GPU): shared by the
# GPU run and the multi-process CPU tests
# ---------------------------------------------------------------------------
def make_allmax(world, device):
    """max over ranks of a float (identity for one process)."""
    def allmax(v):
        if world <= 1:
            return v
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(v)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return t.item()
    return allmax


def timed_replicas(step, K, W, barrier, allmax, clock):
    """W untimed steps, then K timed steps bracketed by `barrier` (all ranks,
    device synchronised); returns the slowest rank's ms per step.  `clock()`
    returns (start, stop_ms): start() marks the beginning, stop_ms() the
    elapsed milliseconds (CUDA events on the launching stream on a GPU)."""
    for _ in range(W):
        step()
    barrier()
    start, stop_ms = clock()
    start()
    for _ in range(K):
        step()
    ms = stop_ms()
    barrier()
    return allmax(ms / K)


def replica_rate(world, tokens_per_replica, ms_per_step):
    """whole-job Mtokens/s: the units all ranks processed over the slowest rank's time."""
    return world * tokens_per_replica / ms_per_step / 1e3


def parse_cpulist(text):
    """CPU ids of a sysfs cpulist ("0-3,8,10-11")."""
    cpus = set()
    for part in text.strip().split(","):
        if part:
            a, _, b = part.partition("-")
            cpus |= set(range(int(a), int(b or a) + 1))
    return cpus


def bind_gpu_local_cpus(dev):
    """Run this process on the host cores next to the GPU (sysfs local_cpulist of its PCI
    function), so that the pinned host buffers of the end-to-end pass are allocated on the
    memory node the GPU's link reaches directly.  A process-local setting (the caller puts the
    previous set back with os.sched_setaffinity); returns what was done, or why not."""
    import torch
    pr = torch.cuda.get_device_properties(dev)
    ids = [getattr(pr, k, None) for k in ("pci_domain_id", "pci_bus_id", "pci_device_id")]
    if any(v is None for v in ids):
        return {"cpus": "unchanged", "why": "no PCI id from the runtime"}
    path = "/sys/bus/pci/devices/%04x:%02x:%02x.0" % tuple(ids)
    try:
        local = parse_cpulist(open(path + "/local_cpulist").read())
        node = open(path + "/numa_node").read().strip()
    except OSError:
        return {"cpus": "unchanged", "why": "no sysfs entry " + path}
    mine = os.sched_getaffinity(0)
    use = local & mine
    if not use:
        return {"cpus": "unchanged", "why": "no GPU-local core in this process's set", "numa_node": node}
    if use != mine:
        os.sched_setaffinity(0, use)
    return {"cpus": len(use), "of": len(mine), "numa_node": node}


def run_ours(args, rank, world, local_rank):
    import torch

    import linear_attention_gdn_gb300 as gdn
    from linear_attention_gdn_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = inputs.workload(args.workload)
    x = inputs.generate(w, dev)
    cu_dev = torch.from_numpy(w.cu_seqlens).to(dev)
    form = gdn.SAVED_REPLAY if args.form == "replay" else gdn.SAVED_FULL
    prob = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments, saved_form=form)
    buf = gdn.Buffers(prob, w.cu_seqlens, device=dev)
    stream = torch.cuda.current_stream(dev)
    o = torch.empty((w.T, w.HV, D), dtype=torch.bfloat16, device=dev)
    dq, dk = torch.empty_like(x["q"]), torch.empty_like(x["k"])
    dv = torch.empty_like(x["v"])
    dg, db = torch.empty_like(x["g"]), torch.empty_like(x["beta"])

    def step(op, xx=x):
        if op in ("fwd", "fwd+bwd"):
            gdn.gdn_fwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens, o,
                        buf.saved, buf.workspace, stream=stream)
        if op == "fwd+bwd":
            gdn.gdn_bwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens, xx["dO"],
                        buf.saved, dq, dk, dv, dg, db, buf.workspace, stream=stream)
        if op == "ckpt":
            gdn.gdn_ckpt_fwd_bwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens,
                                 xx["dO"], o, dq, dk, dv, dg, db, buf.saved, buf.workspace, stream=stream)
        if op == "fwd+bwd replay form":   # the replay saved form: states only, the backward recomputes
            gdn.gdn_fwd(prob_r, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens, o,
                        buf_r.saved, buf_r.workspace, stream=stream)
            gdn.gdn_bwd(prob_r, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens, xx["dO"],
                        buf_r.saved, dq, dk, dv, dg, db, buf_r.workspace, stream=stream)
        if op == "fwd+bwd with states":   # per-document S_in in, S_out out; dS_out in, dS_in out
            gdn.gdn_fwd_states(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens,
                               bnd["s_in"], o, bnd["s_out"], buf.saved, buf.workspace, stream=stream)
            gdn.gdn_bwd_states(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens,
                               xx["dO"], bnd["ds_out"], buf.saved, dq, dk, dv, dg, db, bnd["ds_in"],
                               buf.workspace, stream=stream)

    bnd = {}
    prob_r = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments, saved_form=gdn.SAVED_REPLAY)
    buf_r = gdn.Buffers(prob_r, w.cu_seqlens, device=dev) if not args.quick else None

    def time_workload(idx, K, W):
        """fwd + bwd of workload `idx` on its own inputs and buffers (freed afterwards)."""
        ww = inputs.workload(idx)
        xx = inputs.generate(ww, dev)
        cu_w = torch.from_numpy(ww.cu_seqlens).to(dev)
        pw = gdn.problem(ww.T, ww.N, ww.H, ww.HV, ww.scale, ww.l2norm, ww.segments)
        bw = gdn.Buffers(pw, ww.cu_seqlens, device=dev)
        ow = torch.empty((ww.T, ww.HV, D), dtype=torch.bfloat16, device=dev)
        gr = (torch.empty_like(xx["q"]), torch.empty_like(xx["k"]), torch.empty_like(xx["v"]),
              torch.empty_like(xx["g"]), torch.empty_like(xx["beta"]))

        def st():
            gdn.gdn_fwd(pw, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_w, ww.cu_seqlens, ow, bw.saved,
                        bw.workspace, stream=stream)
            gdn.gdn_bwd(pw, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_w, ww.cu_seqlens, xx["dO"],
                        bw.saved, *gr, bw.workspace, stream=stream)
        t_w = timed_replicas(st, K, W, barrier, allmax, event_clock)
        stw = gdn.gdn_device_status(bw.workspace, stream)
        assert stw == 0, gdn.gdn_status_string(stw)
        seg = gdn.gdn_plan_segment_chunks(pw, ww.cu_seqlens)
        max_chunks = max((n + C - 1) // C for n in ww.doc_lens)
        pk_ = peaks()
        fl = step_flops(ww, "fwd+bwd")
        res = {"ms": round(t_w, 4), "Mtokens_per_s": round(replica_rate(world, ww.T, t_w), 3),
               "TFLOP_per_s": round(world * fl / t_w / 1e9, 1),
               "tensor_frac": round(world * fl / t_w / 1e9 / pk_["bf16_tflops_sustained"], 4),
               "tokens": ww.T, "docs": ww.N, "l2norm": ww.l2norm,
               "segments_of_longest_doc": -(-max_chunks // seg) if seg else None, "segment_chunks": seg}
        del xx, bw, ow, gr
        torch.cuda.empty_cache()
        return res

    def time_kda(K, W):
        """fwd + bwd of the per-channel-decay (KDA) form on the bench workload's shapes (own inputs with
        g [T, HV, 128], own buffers, freed afterwards); per-kernel times from the launch events."""
        xx = inputs.generate_kda(w, dev)
        pk_ = gdn.problem(w.T, w.N, w.H, w.HV, w.scale, w.l2norm, w.segments)
        bk = gdn.Buffers(pk_, w.cu_seqlens, device=dev, kda=True)
        ok_ = torch.empty((w.T, w.HV, D), dtype=torch.bfloat16, device=dev)
        gr = (torch.empty_like(xx["q"]), torch.empty_like(xx["k"]), torch.empty_like(xx["v"]),
              torch.empty_like(xx["g"]), torch.empty_like(xx["beta"]))

        def st():
            gdn.gdn_kda_fwd(pk_, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens, ok_,
                            bk.saved, bk.workspace, stream=stream)
            gdn.gdn_kda_bwd(pk_, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu_dev, w.cu_seqlens, xx["dO"],
                            bk.saved, *gr, bk.workspace, stream=stream)
        t_k = timed_replicas(st, K, W, barrier, allmax, event_clock)
        stk = gdn.gdn_device_status(bk.workspace, stream)
        assert stk == 0, gdn.gdn_status_string(stk)
        gdn.gdn_profile_read_all()
        gdn.gdn_profile_enable(1)
        timed_replicas(st, K, 1, barrier, allmax, event_clock)
        gdn.gdn_profile_enable(0)
        ks = gdn.gdn_profile_read_all()
        pk2 = peaks()
        fl, by = kda_step_flops(w), kda_step_bytes(w)
        res = {"ms": round(t_k, 4), "Mtokens_per_s": round(replica_rate(world, w.T, t_k), 3),
               "TFLOP_per_s": round(world * fl / t_k / 1e9, 1),
               "tensor_frac": round(world * fl / t_k / 1e9 / pk2["bf16_tflops_sustained"], 4),
               "method_GB_per_s": round(by / (t_k * 1e-3) / 1e9, 1),
               "hbm_frac": round(by / (t_k * 1e-3) / 1e9 / pk2["hbm_gbs"], 4),
               "saved_bytes_per_token": round(bk.saved_bytes / w.T, 1),
               "counting": "F = HV (20 d^2 + 38 C d) FLOP / token; bytes: the method tensors with g, dg "
                           "[T, HV, 128] FP32",
               "kernels_ms_per_step": {k: round(v["total_ms"] / (K + 1), 4) for k, v in ks.items()
                                       if v["timed_launches"]}}
        del xx, bk, ok_, gr
        torch.cuda.empty_cache()
        return res

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    allmax = make_allmax(world, dev)

    def event_clock():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def stop_ms():
            e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1)
        return (lambda: e0.record(stream)), stop_ms

    def timed(op, K, W):
        return timed_replicas(lambda: step(op), K, W, barrier, allmax, event_clock)

    if args.kda:   # the per-channel-decay form alone
        res = time_kda(args.steps, args.warmup)
        return {"metric": "KDA fwd+bwd Mtokens/s on 1 GB300 (H16/HV48, d=128)", "value": res["Mtokens_per_s"],
                "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": res["ms"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic", "config": {"workload": w.name, "op": "kda fwd+bwd"},
                "kda": res}
    op = args.op
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    gdn.gdn_profile_read_all()                      # reset the launch counters
    with ClockSampler(uuid) as clk:
        ms = timed(op, args.steps, args.warmup)
    launches = gdn.gdn_profile_read_all()
    st = gdn.gdn_device_status(buf.workspace, stream)
    assert st == 0, gdn.gdn_status_string(st)
    n_launch = sum(v["launches"] for v in launches.values())
    n_launch = int(round(n_launch * args.steps / (args.steps + args.warmup)))

    # per-kernel device times over a second timed pass with launch events (its warm-up step included:
    # every step of the pass is recorded)
    gdn.gdn_profile_enable(1)
    timed(op, args.steps, 1)
    gdn.gdn_profile_enable(0)
    kstats = gdn.gdn_profile_read_all()
    prof_steps = args.steps + 1

    # (the end-to-end pass runs right after the main timing, before the extra timings below)
    # end to end through the C ABI with pinned host buffers: every step copies
    # its inputs in and all of its outputs back
    e2e = None
    if not args.no_e2e:
        # End to end through the C ABI: every step copies its inputs in from pinned host memory and
        # its results back out.  As in a training loop, the copies of neighbouring steps overlap the
        # compute: step i + 1's inputs go in on one copy stream (into the other of two device input
        # sets) and step i - 1's results come out on another while step i runs; events order every
        # buffer reuse.
        names_in = ("q", "k", "v", "g", "beta", "dO")
        cpus_before = os.sched_getaffinity(0)
        host_binding = bind_gpu_local_cpus(dev)   # before the pinned buffers are allocated
        h_in = {n: x[n].to("cpu").pin_memory() for n in names_in}
        h_cu = torch.from_numpy(w.cu_seqlens).pin_memory()
        d_in = [{n: torch.empty_like(x[n]) for n in names_in} for _ in range(2)]
        d_cu = [torch.empty_like(cu_dev) for _ in range(2)]
        outs = [tuple(torch.empty_like(t) for t in ((o, dq, dk, dv, dg, db) if op != "fwd" else (o,)))
                for _ in range(2)]
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs[0]]
        bi = sum(t.numel() * t.element_size() for t in h_in.values()) + w.cu_seqlens.nbytes
        bo = sum(t.numel() * t.element_size() for t in h_out)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set b landed (fwd+bwd: all but dO)
        ev_in2 = [torch.cuda.Event() for _ in range(2)]    # fwd+bwd: dO of set b landed
        ev_fwd = [torch.cuda.Event() for _ in range(2)]    # fwd+bwd: the forward of set b finished
        ev_used = [torch.cuda.Event() for _ in range(2)]   # the step on set b finished
        ev_out = [torch.cuda.Event() for _ in range(2)]    # results of set b copied out

        def step_on(b):
            xx, cu, (oo, *gr) = d_in[b], d_cu[b], outs[b]
            if op in ("fwd", "fwd+bwd"):
                gdn.gdn_fwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu, w.cu_seqlens, oo,
                            buf.saved, buf.workspace, stream=stream)
            if op == "fwd+bwd":
                gdn.gdn_bwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu, w.cu_seqlens, xx["dO"],
                            buf.saved, *gr, buf.workspace, stream=stream)
            if op == "ckpt":
                gdn.gdn_ckpt_fwd_bwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu, w.cu_seqlens,
                                     xx["dO"], oo, *gr, buf.saved, buf.workspace, stream=stream)

        # fwd+bwd: the forward starts once its own inputs are in (dO follows on the same copy stream)
        # and o goes out as soon as the forward is done, so the first and last steps of the pass
        # overlap their copies with compute too
        split = op == "fwd+bwd"

        def run_e2e(K, e_start=None, e_end=None):
            if e_start is not None:
                e_start.record(s_in)
            for i in range(K):
                b = i % 2
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_used[b])
                    d_cu[b].copy_(h_cu, non_blocking=True)
                    for n in names_in:
                        if not (split and n == "dO"):
                            d_in[b][n].copy_(h_in[n], non_blocking=True)
                    ev_in[b].record(s_in)
                    if split:
                        d_in[b]["dO"].copy_(h_in["dO"], non_blocking=True)
                        ev_in2[b].record(s_in)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])
                if split:
                    xx, cu, (oo, *gr) = d_in[b], d_cu[b], outs[b]
                    gdn.gdn_fwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu, w.cu_seqlens, oo,
                                buf.saved, buf.workspace, stream=stream)
                    ev_fwd[b].record(stream)
                    stream.wait_event(ev_in2[b])
                    gdn.gdn_bwd(prob, xx["q"], xx["k"], xx["v"], xx["g"], xx["beta"], cu, w.cu_seqlens, xx["dO"],
                                buf.saved, *gr, buf.workspace, stream=stream)
                else:
                    step_on(b)
                ev_used[b].record(stream)
                with torch.cuda.stream(s_out):
                    if split:
                        s_out.wait_event(ev_fwd[b])
                        h_out[0].copy_(outs[b][0], non_blocking=True)   # o
                    s_out.wait_event(ev_used[b])
                    for hb, dbuf in list(zip(h_out, outs[b]))[1 if split else 0:]:
                        hb.copy_(dbuf, non_blocking=True)
                    ev_out[b].record(s_out)
            if e_end is not None:
                e_end.record(s_out)

        run_e2e(2)
        barrier()
        ke = max(3, args.steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(uuid) as clk_e2e:
            t0 = time.perf_counter()
            run_e2e(ke, e0, e1)
            barrier()
        ms_e2e = allmax(max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3) / ke)
        os.sched_setaffinity(0, cpus_before)
        st = gdn.gdn_device_status(buf.workspace, stream)
        assert st == 0, gdn.gdn_status_string(st)
        e2e = {"value": round(replica_rate(world, w.T, ms_e2e), 3), "unit": UNIT, "h2d_bytes_per_step": int(bi),
               "d2h_bytes_per_step": int(bo), "ms_per_step": round(ms_e2e, 3),
               "overlap": "step i+1's host-to-device and step i-1's device-to-host copies run on two copy streams "
                          "while step i computes; the forward starts once its own inputs are in and o goes out "
                          "once the forward is done", "host_cpus": host_binding, "clocks": clk_e2e.summary()}

    extra = {}
    if not args.quick:
        bnd.update({n: 0.1 * torch.randn((w.N, w.HV, D, D), device=dev) for n in ("s_in", "ds_out")})
        bnd.update({n: torch.empty((w.N, w.HV, D, D), device=dev) for n in ("s_out", "ds_in")})
        for other in ("fwd", "ckpt", "fwd+bwd with states", "fwd+bwd replay form"):
            if other != op:
                if other == "fwd+bwd replay form":
                    gdn.gdn_profile_read_all()
                    gdn.gdn_profile_enable(1)
                t_o = timed(other, max(3, args.steps // 2), 2)
                fl = step_flops(w, "fwd+bwd" if other.startswith("fwd+bwd") else other)
                extra[other] = {"ms": round(t_o, 4), "Mtokens_per_s": round(replica_rate(world, w.T, t_o), 3),
                                "TFLOP_per_s": round(world * fl / t_o / 1e9, 1)}
                if other == "fwd+bwd replay form":
                    gdn.gdn_profile_enable(0)
                    ks = gdn.gdn_profile_read_all()
                    n_st = max(3, args.steps // 2) + 2
                    extra[other].update({
                        "saved_bytes_per_token": round(buf_r.saved_bytes / w.T, 1),
                        "full_form_saved_bytes_per_token": round(buf.saved_bytes / w.T, 1),
                        "kernels_ms_per_step": {k: round(v["total_ms"] / n_st, 4) for k, v in ks.items()
                                                if v["timed_launches"]}})
        # the short causal conv1d + SiLU front over the workload's packed q/k/v channels (4 taps),
        # timed alone: fwd reads x and writes y, bwd reads x and dy and writes dx (BF16 [T, C])
        C_qkv = (2 * w.H + w.HV) * D
        cp = gdn.conv_problem(w.T, w.N, C_qkv, 4)
        cx = torch.randn((w.T, C_qkv), device=dev).to(torch.bfloat16)
        cdy = torch.randn_like(cx)
        cw, cb = 0.5 * torch.randn((C_qkv, 4), device=dev), 0.1 * torch.randn((C_qkv,), device=dev)
        cy, cdx = torch.empty_like(cx), torch.empty_like(cx)
        cdw, cdb = torch.empty_like(cw), torch.empty_like(cb)
        cws = torch.empty((max(gdn.gdn_conv1d_workspace_bytes(cp, w.cu_seqlens), 16),), dtype=torch.uint8,
                          device=dev)
        row_bytes = w.T * C_qkv * 2
        for name, fn, nbytes in (
                ("conv1d_silu fwd", lambda: gdn.gdn_conv1d_fwd(cp, cx, cw, cb, cu_dev, w.cu_seqlens, cy,
                                                               stream=stream), 2 * row_bytes),
                ("conv1d_silu bwd", lambda: gdn.gdn_conv1d_bwd(cp, cx, cw, cb, cu_dev, w.cu_seqlens, cdy, cdx,
                                                               cdw, cdb, cws, stream=stream), 3 * row_bytes)):
            t_c = timed_replicas(fn, max(3, args.steps // 2), 2, barrier, allmax, event_clock)
            extra[name] = {"ms": round(t_c, 4), "channels": C_qkv, "taps": 4,
                           "GB_per_s": round(nbytes / (t_c * 1e-3) / 1e9, 1),
                           "Mtokens_per_s": round(replica_rate(world, w.T, t_c), 3)}
        del cx, cdy, cy, cdx
        # fwd+bwd of the other full-size workloads (8,192-token document; ~156 log-uniform
        # documents of 262,144 tokens with L2 off; one 524,288-token document split into segments)
        for widx in (1, 3, 4):
            if widx != args.workload:
                extra[f"workload{widx} fwd+bwd"] = time_workload(widx, max(3, args.steps // 2), 2)
        # the per-channel-decay form on the same workload
        extra["kda fwd+bwd"] = time_kda(max(3, args.steps // 2), 2)

    if rank != 0:
        return None
    pk = peaks()
    probe = tensor_probe(gdn, torch, dev, stream)
    kt = {k: v for k, v in kstats.items() if v["timed_launches"] > 0}
    top = max(kt, key=lambda k: kt[k]["total_ms"])
    per_launch_ms = kt[top]["total_ms"] / kt[top]["timed_launches"]
    roof = roofline(top, w, per_launch_ms, pk)
    k_tflops = kernel_flops(top, w) / (per_launch_ms * 1e-3) / 1e12
    roof.update({"tensor_frac_of_probe": round(k_tflops / probe["tflops"], 4),
                 "tensor_frac_of_nominal": round(k_tflops / NOMINAL_BF16_TFLOPS, 4)})
    tot = sum(u["total_ms"] for u in kt.values())
    kernels = {}
    for k, v in kt.items():
        f, b = kernel_flops(k, w), kernel_bytes(k, w)
        kernels[k] = {"launches_per_step": round(v["launches"] / prof_steps, 2),
                      "ms_per_step": round(v["total_ms"] / prof_steps, 4), "share": round(v["total_ms"] / tot, 4),
                      "TFLOP_per_s": round(f * v["timed_launches"] / v["total_ms"] / 1e9, 1) if f else None,
                      "method_GB_per_s": round(b * v["timed_launches"] / v["total_ms"] / 1e6, 1) if b else None}
    tflops = world * step_flops(w, op) / ms / 1e9
    step_gbs = world * step_bytes(w, op) / ms / 1e6
    in_gb = sum(x[n].numel() * x[n].element_size() for n in ("q", "k", "v", "g", "beta", "dO")) / 1e9
    return {
        "metric": METRIC, "value": round(replica_rate(world, w.T, ms), 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.T, "docs": w.doc_lens, "H": w.H, "HV": w.HV, "dk": D,
                   "dv": D, "chunk": C, "l2norm": w.l2norm, "op": op, "saved_form": args.form,
                   "l2_flush": f"none needed: {in_gb:.1f} GB of inputs per step exceed the 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "tflops": round(tflops, 1), "tensor_frac_of_step": round(tflops / pk["bf16_tflops_sustained"], 4),
        "tensor_frac_of_step_probe": round(tflops / probe["tflops"], 4),
        "tensor_frac_of_step_nominal": round(tflops / NOMINAL_BF16_TFLOPS, 4), "tensor_probe": probe,
        "step_method_GB_per_s": round(step_gbs, 1), "hbm_frac_of_step": round(step_gbs / pk["hbm_gbs"], 4),
        "roofline": roof, "kernels": kernels, "gpu_launches": n_launch, "clocks": clk.summary(),
        "e2e": e2e, "ops": extra,
    }


NOMINAL_BF16_TFLOPS = 2250.0   # the vendor's dense BF16 tensor-core figure for one GB300


def tensor_probe(gdn, torch, dev, stream, reps=3, iters=200000):
    """The library's tensor-pipe probe (one CTA per SM issuing M = 128, N = 256, K = 16 BF16 tcgen05
    products on operands resident in shared memory): best of `reps` launches, in TFLOP/s, with the SM
    clocks sampled while it runs."""
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    gdn.gdn_tensor_probe(200, err, stream)   # warm-up (module load, clocks)
    best = 0.0
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fl = gdn.gdn_tensor_probe(iters, err, stream)
            e1.record(stream)
            e1.synchronize()
            best = max(best, fl / e0.elapsed_time(e1) / 1e9)
    assert int(err.item()) == 0, "tensor probe: a bounded wait ran out"
    return {"tflops": round(best, 1), "nominal_tflops": NOMINAL_BF16_TFLOPS,
            "what": "tcgen05 BF16 M128 N256 K16 products back to back, operands resident in shared memory, "
                    "one CTA per SM, FP32 accumulation in TMEM",
            "iters": iters, "reps": reps, "clocks": clk.summary()}


def roofline(kernel, w, launch_ms, pk):
    """The roofline object of one kernel: method FLOPs and bytes of one launch (the method's per-token
    counts over the workload's real chunks) over its measured launch time, against the binding roof (the
    larger of the two time floors at those counts)."""
    fl, by = kernel_flops(kernel, w), kernel_bytes(kernel, w)
    t_tensor = fl / (pk["bf16_tflops_sustained"] * 1e12)
    t_hbm = by / (pk["hbm_gbs"] * 1e9)
    if fl > 0 and t_tensor >= t_hbm:
        achieved = fl / (launch_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops_sustained"], 4)}
        note = f"{pk['src']} sustained BF16 (the kernel is timed inside a multi-ms step)"
    else:
        achieved = by / (launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4)}
        note = f"{pk['src']} HBM copy bandwidth"
    traffic = ncu_traffic(kernel)
    roof.update({"traffic": traffic, "kernel": kernel, "peak_note": note, "launch_ms": round(launch_ms, 4),
                 "method_flops_per_launch": fl, "method_bytes_per_launch": by,
                 "tensor_frac": round(fl / (launch_ms * 1e-3) / 1e12 / pk["bf16_tflops_sustained"], 4),
                 "hbm_frac": round(by / (launch_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                 "traffic_over_method_bytes": round(traffic / by, 3) if traffic and by else None,
                 "counting": "method FLOPs / bytes per the method's per-token counts (real chunk lengths); "
                             "the design's own intermediate tapes are not credited (traffic shows them)"})
    return roof


# ---------------------------------------------------------------------------
# the FP64 CPU oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------
def oracle_sample(w, tokens_per_unit, units, threads):
    """Run `units` q/k-head-group jobs of the oracle, fwd+bwd, each over a
    `tokens_per_unit`-token document (an exact sub-problem with the workload's
    head counts and distributions), in parallel.  Returns (seconds, rate in
    Mtokens/s of the full HV-head problem)."""
    from linear_attention_gdn_gb300 import inputs
    from oracle import ref

    small = inputs.custom([tokens_per_unit], w.H, w.HV, w.l2norm, w.g_lo, w.g_hi, seed=w.seed)
    x = inputs.generate(small, "cpu")
    G = w.HV // w.H
    us = [ref.Unit(0, u % w.H, 0, tokens_per_unit, 0, tokens_per_unit) for u in range(units)]
    t0 = time.perf_counter()
    ref.run(x, w.H, w.HV, l2norm=w.l2norm, scale=w.scale, units=us, threads=threads)
    dt = time.perf_counter() - t0
    return dt, units * tokens_per_unit * G / w.HV / dt / 1e6


def cpu_count():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    from linear_attention_gdn_gb300 import inputs
    w = inputs.workload(args.workload)
    threads = cpu_count()
    tpu = 1024
    res = []
    for i in range(args.warmup + args.steps):
        dt, rate = oracle_sample(w, tpu, threads, threads)
        if i >= args.warmup:
            res.append((dt, rate))
    dt = statistics.median(t[0] for t in res)
    rate = statistics.median(t[1] for t in res)
    sample = (f"{threads} q/k-head groups x {tpu}-token document (3 value heads each), fwd+bwd, per step; "
              f"rate scaled to all {w.HV} value heads")
    return {"impl": "reference", "metric": METRIC, "value": round(rate, 6), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "op": "fwd+bwd", "sample": sample},
            "cpu_baseline": {"value": round(rate, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(rate, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--op", default="fwd+bwd", choices=("fwd", "fwd+bwd", "ckpt"))
    ap.add_argument("--kda", action="store_true",
                    help="time only the per-channel-decay (KDA) fwd+bwd on the workload (for profiling)")
    ap.add_argument("--form", default="full", choices=("full", "replay"),
                    help="saved form of the timed step (the other one is timed in ops)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the extra fwd / ckpt timings")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args), allow_nan=False), flush=True)
        return
    args.warmup = max(args.warmup, 3)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu and not args.kda:
            from linear_attention_gdn_gb300 import inputs
            w = inputs.workload(args.workload)
            threads = cpu_count()
            units = 6 * threads   # about 10-15 s of oracle work on the host cores
            dt, rate = oracle_sample(w, 8192, units, threads)
            out["cpu_baseline"] = {"value": round(rate, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                                   "sample": f"{units} q/k-head groups x 8192-token document, fwd+bwd, "
                                             f"{dt:.1f} s; rate scaled to all {w.HV} value heads"}
        print(json.dumps(out, allow_nan=False), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

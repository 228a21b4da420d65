#!/usr/bin/env python
"""Benchmark of the tiled exact-attention library on one or more GB300s.

Workload: causal attention, B=1, H=16, N=16384, D=128, bf16 inputs drawn
i.i.d. N(0,1) (synthetic, seeded).  One step is one pass of the hot path
over that batch: the forward (O, LSE) and, when the library has it, the
recompute backward (dQ, dK, dV) -- every launch through the C ABI.

Metric: attention TFLOPS = 4*B*H*N^2*D / t, halved for causal; the
backward counts 2.5x the forward.  Printed as ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 launch with torch.distributed.run: every rank runs the same
per-GPU workload on its own GPU (weak scaling, no collective on the data
path); the step time is the max over ranks.  ``--impl reference`` times
the fp64 CPU oracle on the host cores on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOPS (4·B·H·N²·D, causal/2) and % of GB300 dense BF16 peak"
WORKLOAD = dict(name="causal_fwd_bwd_B1_H16_N16384_D128", B=1, Hq=16, Hkv=16, N=16384, D=128,
                causal=True)
L2_BYTES = 129 << 20         # GB300 L2
L2_FLUSH_BYTES = 256 << 20   # > L2


def attn_flops(B, H, N, D, causal, window=None):
    """Forward FLOPs by the pages' count 4*B*H*N^2*D (blog.ans20xx.com day26,
    'CUDA event 计时模板'), halved for the causal mask.  A causal sliding
    window of W < N keys counts N*W - W^2/2 (query, key) pairs per head, the
    same continuous count that gives N^2/2 at W = N."""
    if causal and window and window < N:
        return 4.0 * B * H * D * (N * window - window * window / 2)
    f = 4.0 * B * H * N * N * D
    return f / 2 if causal else f


def bwd_flops(B, H, N, D, causal, window=None):
    return 2.5 * attn_flops(B, H, N, D, causal, window)


def tile_pairs(B, H, N, causal, window=None):
    """(128-row query tile, 128-key tile) pairs the kernels process."""
    n_qt = (N + 127) // 128
    if not causal:
        return B * H * n_qt * n_qt
    if not window or window >= N:
        return B * H * n_qt * (n_qt + 1) // 2
    return B * H * sum(qt - max(0, qt * 128 - window + 1) // 128 + 1 for qt in range(n_qt))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def source_digest(files):
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# The plain forward kernel (two query tiles per block) and the residual
# forward (bias / emitted logits) live in separate files.
FWD_SOURCES = ["tiled_attention_02_gb300/csrc/attn_fwd_pp.cu",
               "tiled_attention_02_gb300/csrc/sm103_ptx.cuh"]
RES_FWD_SOURCES = ["tiled_attention_02_gb300/csrc/attn_fwd.cu",
                   "tiled_attention_02_gb300/csrc/sm103_ptx.cuh"]
BWD_SOURCES = ["tiled_attention_02_gb300/csrc/attn_bwd.cu",
               "tiled_attention_02_gb300/csrc/sm103_ptx.cuh"]
DEC_SOURCES = ["tiled_attention_02_gb300/csrc/attn_decode.cu",
               "tiled_attention_02_gb300/csrc/sm103_ptx.cuh"]


def profiled(kernel_tag, digest, units):
    """What the committed ncu summary ``profiles/<kernel_tag>.md`` says about
    this kernel, if it was captured on the same kernel source (digest):
    DRAM bytes per launch (``traffic``), scaled to `units` (query-tile x
    kv-tile pairs) when the capture ran a smaller case, and the tensor
    pipe's active cycles in percent of peak (``tensor_pipe_active_pct``, as
    captured).  Empty when absent or stale."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return {}
    text = open(path).read()
    m_d = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m_d or m_d.group(1) != digest:
        return {}
    out = {"profile": f"profiles/{kernel_tag}.md"}
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_u = re.search(r"units_per_launch:\s*([0-9.eE+]+)", text)
    if m_b and m_u:
        cap_units = float(m_u.group(1))
        out["traffic"] = float(m_b.group(1)) * units / cap_units
        out["traffic_basis"] = ("measured at this size" if cap_units == units else
                                f"scaled by units from a capture of {cap_units:.0f} units")
    m_t = re.search(r"tensor_pipe_active_pct:\s*([0-9.eE+]+)", text)
    if m_t:
        out["tensor_pipe_active_pct"] = float(m_t.group(1))
    return out


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id is not None:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ------------------------------------------------------------ distributed

def dist_setup(want_cuda: bool):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if want_cuda else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------- CPU (oracle)

def oracle_sample(R: int, rng_seed: int = 0):
    """A bounded, self-contained sample of the workload for the fp64 oracle:
    the last R query rows and the last R key rows of one head.  Under the
    causal mask those key rows are attended only by those query rows, so the
    sample needs nothing outside itself: forward rows (O, LSE), Delta, dQ of
    the R query rows, dK and dV of the R key rows.  Work is counted with the
    benchmark's own convention: 4*D*|J_i| per forward row, 2.5x for the
    backward."""
    import numpy as np
    import torch
    W = WORKLOAD
    N, D = W["N"], W["D"]
    g = torch.Generator().manual_seed(rng_seed)
    shape = (1, 1, N, D)
    q, k, v, do = (torch.randn(*shape, generator=g).to(torch.bfloat16).float().numpy()
                   .astype(np.float64) for _ in range(4))
    rows = np.arange(N - R, N, dtype=np.int64)
    fl = sum(4.0 * D * (int(i) + 1) for i in rows)
    return dict(q=q, k=k, v=v, do=do, rows=rows, flops=fl * 3.5,
                desc=f"last {R} query rows and last {R} key rows of one head (N={N}, D={D}, "
                     f"causal): forward rows, Delta, dQ, dK, dV in fp64")


def run_oracle_sample(orc, s):
    W = WORKLOAD
    scale = 1.0 / math.sqrt(W["D"])
    orc.forward(s["q"], s["k"], s["v"], scale=scale, causal=True, rows=s["rows"])
    orc.backward_sampled(s["q"], s["k"], s["v"], s["do"], scale=scale, causal=True,
                         q_rows=s["rows"], k_rows=s["rows"])


def cpu_baseline(min_seconds=10.0, max_seconds=30.0, R=256):
    import oracle as orc
    orc.build()
    s = oracle_sample(R)
    n, flops, t0 = 0, 0.0, time.perf_counter()
    while True:
        run_oracle_sample(orc, s)
        n += 1
        flops += s["flops"]
        el = time.perf_counter() - t0
        if el >= min_seconds or el * (n + 1) / n > max_seconds:
            break
    return {"value": flops / el / 1e12, "unit": "TFLOPS", "cores": orc.get_threads(),
            "kind": "oracle", "sample": f"{s['desc']}; {n} repetitions, {el:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_setup(want_cuda=False)
    if rank != 0:
        return 0
    import oracle as orc
    orc.build()
    s = oracle_sample(args.ref_rows)
    for _ in range(args.warmup):
        run_oracle_sample(orc, s)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run_oracle_sample(orc, s)
        times.append(time.perf_counter() - t0)
    per = sum(times) / len(times)
    value = s["flops"] / per / 1e12
    cores = orc.get_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(WORKLOAD, world, wants_flush("auto", workload_bytes(WORKLOAD)),
                                  workload_bytes(WORKLOAD)),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": s["desc"]},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def line_config(W, world, do_flush, bytes_per_step):
    """The JSON line's `config`, the same for both arms."""
    kind = W.get("kind", "fwd_bwd")
    return dict(config_block(world, W),
                step={"fwd_bwd": "forward + backward", "fwd": "forward",
                      "decode": "one decode step (stream-K over one block per SM, then merge)",
                      "chain_train": "four chained layers forward, then backward "
                                     "through the block (fp32 residual and gradient)",
                      "chain": "four chained forward layers, fp32 residual in place"}[kind],
                l2=l2_note(do_flush, bytes_per_step))


def workload_bytes(W):
    """Algorithmic bytes of one step of W (as the GPU arm counts them)."""
    B, Hq, Hkv, N, D = W["B"], W["Hq"], W["Hkv"], W["N"], W["D"]
    io = 2 * (B * Hq * N * D) * 2 + 2 * (B * Hkv * N * D) * 2 + B * Hq * N * 4
    bw = 4 * (B * Hq * N * D) * 2 + 4 * (B * Hkv * N * D) * 2 + B * Hq * N * 4
    return io + (bw if W.get("kind", "fwd_bwd") == "fwd_bwd" else 0)


def config_block(world, W=None):
    W = W or WORKLOAD
    cfg = {"workload": W["name"], "B": W["B"], "H": W["Hq"], "Hkv": W["Hkv"], "N": W["N"],
           "D": W["D"], "causal": W["causal"], "scale": 1 / math.sqrt(W["D"]),
           "parallelism": f"replicas x{world} (independent problems, no collective)"}
    if W.get("kind") in ("chain", "chain_train"):
        cfg["layers"] = W["layers"]
    if W.get("window"):
        cfg["window"] = W["window"]
    return cfg


# Optional workloads for manual measurement (the default line is WORKLOAD).
EXTRA_WORKLOADS = {
    "noncausal_fwd": dict(name="noncausal_fwd_B8_H32_N2048_D128", kind="fwd", B=8, Hq=32,
                          Hkv=32, N=2048, D=128, causal=False),
    "causal_fwd_d64": dict(name="causal_fwd_B2_H16_N4096_D64", kind="fwd", B=2, Hq=16, Hkv=16,
                           N=4096, D=64, causal=True),
    "residual_chain": dict(name="residual_chain_4layers_B1_H20_KV4_N4096_D128", kind="chain",
                           layers=4, B=1, Hq=20, Hkv=4, N=4096, D=128, causal=True),
    "tiny": dict(name="tiny_fwd_B1_H1_N128_D64", kind="fwd", B=1, Hq=1, Hkv=1, N=128, D=64,
                 causal=False),
    # Head dims 80 and 96 on the default step's shape (FLOPs at the true D).
    "causal_fwd_bwd_d80": dict(name="causal_fwd_bwd_B1_H16_N16384_D80", B=1, Hq=16, Hkv=16,
                               N=16384, D=80, causal=True),
    "causal_fwd_bwd_d96": dict(name="causal_fwd_bwd_B1_H16_N16384_D96", B=1, Hq=16, Hkv=16,
                               N=16384, D=96, causal=True),
    # Training step of the block residual chain: 4 layers forward, 4 backward.
    "residual_chain_train": dict(name="residual_chain_train_4layers_B1_H20_KV4_N4096_D128",
                                 kind="chain_train", layers=4, B=1, Hq=20, Hkv=4, N=4096, D=128,
                                 causal=True),
    # Decode step (flash decode): one new query row per head over a 16384-row
    # cache, grouped heads 32 : 8 (every K/V byte serves 4 query rows).
    "decode": dict(name="decode_B16_H32_KV8_N16384_D128", kind="decode", B=16, Hq=32, Hkv=8,
                   N=16384, D=128, causal=True),
    "profile_chain_train_small": dict(name="residual_chain_train_4layers_B1_H10_KV2_N2048_D128",
                                      kind="chain_train", layers=4, B=1, Hq=10, Hkv=2, N=2048,
                                      D=128, causal=True),
    "profile_decode_small": dict(name="decode_B4_H32_KV8_N16384_D128", kind="decode", B=4,
                                 Hq=32, Hkv=8, N=16384, D=128, causal=True),
    # One plain layer of the residual chain's shape (no bias, no emitted logits),
    # forward + backward: what the residual adds is measured against it.
    "gqa_fwd_bwd": dict(name="causal_fwd_bwd_B1_H20_KV4_N4096_D128", B=1, Hq=20, Hkv=4, N=4096,
                        D=128, causal=True),
    # Causal sliding window of 4096 keys on the default step's shape.
    "swa_fwd_bwd": dict(name="swa4096_fwd_bwd_B1_H16_N16384_D128", B=1, Hq=16, Hkv=16, N=16384,
                        D=128, causal=True, window=4096),
    # Smaller cases of the default step and of the residual chain for
    # multi-pass ncu captures: inputs still larger than L2, well under 1 GB.
    "profile_small": dict(name="causal_fwd_bwd_B1_H16_N8192_D128", B=1, Hq=16, Hkv=16, N=8192,
                          D=128, causal=True),
    "profile_chain_small": dict(name="residual_chain_4layers_B1_H8_KV2_N4096_D128", kind="chain",
                                layers=4, B=1, Hq=8, Hkv=2, N=4096, D=128, causal=True),
}


def chain_layer_bytes(W, layer):
    """Algorithmic HBM bytes of one chained layer: Q, K, V read, O and LSE
    written, plus the kept (j <= i under the causal mask) fp32 logits read
    from the previous layer (layers 1..L-1) and written for the next (layers
    0..L-2)."""
    B, Hq, Hkv, N, D, L = W["B"], W["Hq"], W["Hkv"], W["N"], W["D"], W["layers"]
    kept = N * (N + 1) // 2 if W["causal"] else N * N
    base = 2 * (B * Hq * N * D) * 2 + 2 * (B * Hkv * N * D) * 2 + B * Hq * N * 4
    return base + (layer > 0) * B * Hq * kept * 4 + (layer < L - 1) * B * Hq * kept * 4


# ---------------------------------------------------------------- GPU arm

def build_workload(W, ta, dev, rank, sh):
    """One independent set of device buffers for workload W and the phases
    that run on them: (phases, host inputs, device inputs, results), where a
    phase is (label, fn, flops, algorithmic bytes) and a step runs every
    phase in order."""
    import torch
    from tiled_attention_02_gb300.inputs import make_chain, make_qkv
    kind = W.get("kind", "fwd_bwd")
    B, Hq, Hkv, N, D, causal = W["B"], W["Hq"], W["Hkv"], W["N"], W["D"], W["causal"]
    scale = 1.0 / math.sqrt(D)
    phases = []
    host_inputs, dev_inputs, results = [], [], []
    if kind == "decode":
        from tiled_attention_02_gb300.inputs import make_decode
        x = make_decode(B, Hq, Hkv, N, D, seed=rank)
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        ws = torch.empty(max(ta.attn_decode_workspace_size(B, Hq, Hkv, N, D), 256),
                         dtype=torch.uint8, device=dev)

        def dec():
            s = ta.raw_attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, Hq, Hkv, N, D, scale, ws.data_ptr(),
                                   ws.numel(), sh)
            assert s == 0, s
        # algorithmic bytes: the K/V cache once, the query rows, O and LSE
        dec_bytes = 2 * (B * Hkv * N * D) * 2 + 2 * (B * Hq * D) * 2 + B * Hq * 4
        phases.append(("decode", dec, 4.0 * B * Hq * N * D, dec_bytes))
        # The K/V cache is state that stays on the device across decode
        # steps; a step's input is its query rows.
        host_inputs += [x["q"]]
        dev_inputs += [q]
        results = [o]
    elif kind == "chain_train":
        # 4-layer block, forward then backward: every layer keeps its emitted
        # logits (the next layer's bias, needed again by the backward), and
        # one fp32 buffer carries the logit gradient down the block in place.
        L = W["layers"]
        layers = make_chain(B, Hq, Hkv, N, D, layers=L, seed=rank, with_do=True)
        dl = [{n: x[n].to(dev) for n in ("q", "k", "v", "do")} for x in layers]
        outs = [(torch.empty_like(x["q"]),
                 torch.empty((B, Hq, N), dtype=torch.float32, device=dev)) for x in dl]
        S = [torch.empty((B, Hq, N, N), dtype=torch.float32, device=dev) for _ in range(L - 1)]
        gbuf = torch.empty((B, Hq, N, N), dtype=torch.float32, device=dev)
        grads = [(torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]))
                 for x in dl]
        ws = torch.empty(max(ta.attn_bwd_workspace_size(B, Hq, Hkv, N, D), 256),
                         dtype=torch.uint8, device=dev)
        kept = B * Hq * (N * (N + 1) // 2 if causal else N * N) * 4
        for i in range(L):
            def layer_f(i=i):
                x, (o, lse) = dl[i], outs[i]
                st = ta.raw_attn_fwd(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                     S[i - 1].data_ptr() if i > 0 else None, o.data_ptr(),
                                     lse.data_ptr(), B, Hq, Hkv, N, D, scale, causal,
                                     S[i].data_ptr() if i < L - 1 else None, sh)
                assert st == 0, st
            phases.append((f"fwd{i}", layer_f, attn_flops(B, Hq, N, D, causal),
                           chain_layer_bytes(W, i)))
        io_b = 5 * (B * Hq * N * D) * 2 + 2 * 2 * (B * Hkv * N * D) * 2 + B * Hq * N * 4
        for i in reversed(range(L)):
            def layer_b(i=i):
                x, (o, lse) = dl[i], outs[i]
                dq, dk, dv = grads[i]
                st = ta.raw_attn_bwd_residual(
                    x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
                    lse.data_ptr(), x["do"].data_ptr(), S[i - 1].data_ptr() if i > 0 else None,
                    gbuf.data_ptr() if i < L - 1 else None, dq.data_ptr(), dk.data_ptr(),
                    dv.data_ptr(), gbuf.data_ptr() if i > 0 else None, B, Hq, Hkv, N, D, scale,
                    causal, ws.data_ptr(), ws.numel(), sh)
                assert st == 0, st
            by = io_b + kept * ((i > 0) + (i < L - 1) + (i > 0))
            phases.append((f"bwd{i}", layer_b, bwd_flops(B, Hq, N, D, causal), by))
        for i, x in enumerate(layers):
            for n in ("q", "k", "v", "do"):
                host_inputs.append(x[n])
                dev_inputs.append(dl[i][n])
        results = [grads[0][0]]
    elif kind == "chain":
        layers = make_chain(B, Hq, Hkv, N, D, layers=W["layers"], seed=rank)
        dl = [{n: x[n].to(dev) for n in ("q", "k", "v")} for x in layers]
        outs = [(torch.empty_like(x["q"]),
                 torch.empty((B, Hq, N), dtype=torch.float32, device=dev)) for x in dl]
        buf = torch.empty((B, Hq, N, N), dtype=torch.float32, device=dev)
        L = W["layers"]
        for i in range(L):
            def layer(i=i):
                x, (o, lse) = dl[i], outs[i]
                s = ta.raw_attn_fwd(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                    buf.data_ptr() if i > 0 else None, o.data_ptr(),
                                    lse.data_ptr(), B, Hq, Hkv, N, D, scale, causal,
                                    buf.data_ptr() if i < L - 1 else None, sh)
                assert s == 0, s
            phases.append((f"layer{i}", layer, attn_flops(B, Hq, N, D, causal),
                           chain_layer_bytes(W, i)))
        for i, x in enumerate(layers):
            for n in ("q", "k", "v"):
                host_inputs.append(x[n])
                dev_inputs.append(dl[i][n])
        results = [outs[-1][0]]
    else:
        x = make_qkv(B, Hq, Hkv, N, D, seed=rank, with_do=(kind == "fwd_bwd"))
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)

        window = W.get("window")

        def fwd():
            if window:
                s = ta.raw_attn_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), None,
                                           o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, N, D, scale,
                                           window, None, sh)
            else:
                s = ta.raw_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), None,
                                    o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, N, D, scale,
                                    causal, None, sh)
            assert s == 0, s
        io_bytes = 2 * (B * Hq * N * D) * 2 + 2 * (B * Hkv * N * D) * 2 + B * Hq * N * 4
        phases.append(("fwd", fwd, attn_flops(B, Hq, N, D, causal, window), io_bytes))
        host_inputs += [x["q"], x["k"], x["v"]]
        dev_inputs += [q, k, v]
        results = [o]
        if kind == "fwd_bwd":
            do = x["do"].to(dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty(max(ta.attn_bwd_workspace_size(B, Hq, Hkv, N, D), 256),
                             dtype=torch.uint8, device=dev)

            def bwd():
                if window:
                    s = ta.raw_attn_bwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               o.data_ptr(), lse.data_ptr(), do.data_ptr(),
                                               dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B,
                                               Hq, Hkv, N, D, scale, window, ws.data_ptr(),
                                               ws.numel(), sh)
                else:
                    s = ta.raw_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                        lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                        dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, D, scale,
                                        causal, ws.data_ptr(), ws.numel(), sh)
                assert s == 0, s
            bwd_bytes = 4 * (B * Hq * N * D) * 2 + 4 * (B * Hkv * N * D) * 2 + B * Hq * N * 4
            phases.append(("bwd", bwd, bwd_flops(B, Hq, N, D, causal, window), bwd_bytes))
            host_inputs.append(x["do"])
            dev_inputs.append(do)
            results = [dq, dk, dv]
    return phases, host_inputs, dev_inputs, results


LAUNCHES = {"fwd": 1, "bwd": 3, "decode": 2, **{f"bwd{i}": 3 for i in range(8)}}


def pct_stats(xs):
    """median / p90 / min of a list of times, as the pages' CUDA-event bench
    template reports them (p90 by nearest rank)."""
    ys = sorted(xs)
    return {"median": statistics.median(ys), "p90": ys[max(0, math.ceil(0.9 * len(ys)) - 1)],
            "min": ys[0]}


def wants_flush(l2_mode, bytes_per_step):
    """Between timed steps either flush L2 (write a buffer larger than it) or
    rely on a step's own traffic being more than twice the L2, which leaves
    nothing of the previous step resident."""
    return l2_mode == "flush" or (l2_mode == "auto" and bytes_per_step <= 2 * L2_BYTES)


def l2_note(do_flush, bytes_per_step):
    return (f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MB write)" if do_flush else
            f"no flush: inputs larger than L2 (a step moves {bytes_per_step / 2**20:.0f} MB, "
            f"over twice the {L2_BYTES >> 20} MB L2)")


def time_steps(phases, stream, n, do_flush, flush):
    """n steps, each phase bracketed by CUDA events on the launching stream;
    returns per-step lists of per-phase milliseconds."""
    import torch
    nph = len(phases)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(n)]
    for i in range(n):
        if do_flush:
            flush.fill_(float(i))   # untimed: evicts the previous step's data from L2
        ev[i][0].record(stream)
        for j, (_, fn, _, _) in enumerate(phases):
            fn()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    return [[e[j].elapsed_time(e[j + 1]) for j in range(nph)] for e in ev]


def kernel_entries(W, phases, ph_ms, pk):
    """Roofline entry per phase: achieved rate from the CUDA-event time
    (`ph_ms`: milliseconds per launch of each phase) against the measured
    peak, with DRAM traffic and tensor-pipe activity from the committed ncu
    summary of the same kernel source."""
    kind = W.get("kind", "fwd_bwd")
    B, Hq, Hkv, N, D, causal = W["B"], W["Hq"], W["Hkv"], W["N"], W["D"], W["causal"]
    units = tile_pairs(B, Hq, N, causal, W.get("window"))   # 128x128 tile pairs
    tag = (f"{'causal' if causal else 'noncausal'}_B{B}_H{Hq}_N{N}_D{D}"
           + (f"_W{W['window']}" if W.get("window") else ""))
    kernels = {}
    for (lbl, _, fl, by), avg in zip(phases, ph_ms):
        if kind == "decode":
            dg = source_digest(DEC_SOURCES)
            ach = by / (avg * 1e-3) / 1e9
            kernels[lbl] = dict({"kernel": f"decode_split_kernel<{D}> + decode_merge_kernel",
                                 "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                                 "unit": "GB/s", "frac": ach / pk["hbm_gbs"]},
                                **profiled(f"decode_split_kernel_{W['name']}", dg, B * Hkv * N),
                                bytes_per_launch=by, flops_per_launch=fl,
                                tflops=fl / (avg * 1e-3) / 1e12, avg_launch_ms=avg,
                                launches_timed=2, source_digest=dg)
            continue
        if kind in ("chain", "chain_train"):
            is_b = lbl.startswith("bwd")
            dg = source_digest(BWD_SOURCES if is_b else RES_FWD_SOURCES)
            ach = by / (avg * 1e-3) / 1e9
            if is_b:
                prof = profiled(f"bwd_main_kernel_residual_chain_train_B{B}_H{Hq}_N{N}_D{D}", dg,
                                units) if lbl in ("bwd1", "bwd2") else {}
            else:
                mid = lbl in ("fwd1", "fwd2", "layer1", "layer2")
                prof = profiled(f"fwd_kernel_chain_{tag}", dg, units) if mid else {}
            kernels[lbl] = dict({"kernel": (f"bwd_main_kernel<{D},causal,residual> (+pre, dQ "
                                            f"convert)" if is_b else
                                            f"fwd_kernel<{D},causal,bias/emit>"),
                                 "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                                 "unit": "GB/s", "frac": ach / pk["hbm_gbs"]},
                                **prof, bytes_per_launch=by, flops_per_launch=fl,
                                tflops=fl / (avg * 1e-3) / 1e12, avg_launch_ms=avg,
                                launches_timed=3 if is_b else 1, source_digest=dg)
            continue
        is_bwd = lbl == "bwd"
        dg = source_digest(BWD_SOURCES if is_bwd else FWD_SOURCES)
        ach = fl / (avg * 1e-3) / 1e12
        kname = "bwd_main_kernel" if is_bwd else "fwd_pp_kernel"
        kernels[lbl] = dict({"kernel": f"{kname}<{D},{'causal' if causal else 'noncausal'}>",
                             "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                             "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"]},
                            **profiled(f"{kname}_{tag}", dg, units),
                            flops_per_launch=fl, units_per_launch=units, avg_launch_ms=avg,
                            launches_timed=3 if is_bwd else 1, source_digest=dg)
        if is_bwd:
            kernels[lbl]["timing_note"] = ("CUDA events around attn_bwd: preprocess + main + "
                                           "dQ convert; the main kernel dominates (ncu launch "
                                           "list)")
    return kernels


# The other configurations, timed after the default line in the same run
# with the pages' CUDA-event template: 20 warm-up and 100 timed iterations,
# median / p90 / min (blog.ans20xx.com day26, "CUDA event 计时模板").
CONFIG_SET = (("C1", "tiny"), ("C2", "noncausal_fwd"), ("C3", "causal_fwd_d64"),
              ("C4", "residual_chain"), ("C4_train", "residual_chain_train"))
# The pages' own figure for C3's shape: flash-attn v2 forward on an H100-SXM,
# 11.9 ms median, counted 4*B*H*S^2*D without the causal halving
# (blog.ans20xx.com day26, "报告格式").
PAGES_C3_FA2_H100 = {"ms": 11.9, "tflops_unhalved": 11.57, "hardware": "H100-SXM-80GB"}


def time_config(W, ta, dev, sh, stream, flush, l2_mode, pk, n_warm=20, n_iter=100):
    phases, _, _, _ = build_workload(W, ta, dev, 0, sh)
    kind = W.get("kind", "fwd_bwd")
    bytes_step = sum(ph[3] for ph in phases)
    flops_step = sum(ph[2] for ph in phases)
    do_flush = wants_flush(l2_mode, bytes_step)
    for _ in range(n_warm):
        for _, fn, _, _ in phases:
            fn()
    import torch
    torch.cuda.synchronize()
    assert ta.attn_last_device_status() == 0
    per = time_steps(phases, stream, n_iter, do_flush, flush)
    assert ta.attn_last_device_status() == 0
    step_ms = [sum(p) for p in per]
    st = pct_stats(step_ms)
    ph_med = [statistics.median(p[j] for p in per) for j in range(len(phases))]
    out = {"workload": W["name"], "ms": st, "iters": n_iter, "warmup": n_warm,
           "l2": l2_note(do_flush, bytes_step),
           "gpu_launches_per_iter": sum(LAUNCHES.get(lbl, 1) for lbl, *_ in phases)}
    kernels = kernel_entries(W, phases, ph_med, pk)
    if W["name"].startswith("tiny"):
        out["us"] = {k: 1e3 * v for k, v in st.items()}
        out["bound"] = "launch latency (4.19 MFLOP; a rate is not meaningful)"
        return out
    out["tflops"] = flops_step / (st["median"] * 1e-3) / 1e12
    if kind in ("chain", "chain_train"):
        out["gbs"] = bytes_step / (st["median"] * 1e-3) / 1e9
        out["bound"] = "hbm"
        out["frac"] = out["gbs"] / pk["hbm_gbs"]
        out["peak"] = pk["hbm_gbs"]
        out["phases"] = {lbl: {"ms_median": kernels[lbl]["avg_launch_ms"],
                               "gbs": kernels[lbl]["achieved"], "frac": kernels[lbl]["frac"],
                               **{k: kernels[lbl][k] for k in ("traffic",
                                                               "tensor_pipe_active_pct")
                                  if kernels[lbl].get(k) is not None}}
                         for lbl in kernels}
    else:
        k0 = kernels["fwd"]
        out.update({"bound": "tensor", "frac": k0["frac"], "peak": pk["bf16_tflops"],
                    "kernel": k0["kernel"]})
        for key in ("traffic", "tensor_pipe_active_pct", "profile"):
            if k0.get(key) is not None:
                out[key] = k0[key]
        if W["causal"]:
            out["tflops_unhalved"] = 2 * out["tflops"]
        if W["name"] == EXTRA_WORKLOADS["causal_fwd_d64"]["name"]:
            out["pages_context"] = dict(PAGES_C3_FA2_H100,
                                        note="another machine: context, not a target")
    return out


def run_ours(args):
    import torch
    world, rank, local = dist_setup(want_cuda=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import tiled_attention_02_gb300 as ta
    ta.build()
    W = WORKLOAD if args.workload == "step" else EXTRA_WORKLOADS[args.workload]
    kind = W.get("kind", "fwd_bwd")
    B, Hq, N, D, causal = W["B"], W["Hq"], W["N"], W["D"], W["causal"]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    pk = peaks()

    phases, host_inputs, dev_inputs, results = build_workload(W, ta, dev, rank, sh)
    launches_per_step = sum(LAUNCHES.get(lbl, 1) for lbl, *_ in phases)

    def step():
        for _, fn, _, _ in phases:
            fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert ta.attn_last_device_status() == 0

    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_id.startswith("GPU-"):
            gpu_id = "GPU-" + gpu_id
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    bytes_step = sum(ph[3] for ph in phases)
    flops_step = sum(ph[2] for ph in phases)
    do_flush = wants_flush(args.l2, bytes_step)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)   # let the sampler start before the load
    # ---- the K timed steps (the line's value)
    per = time_steps(phases, stream, args.steps, do_flush, flush)
    barrier(world)
    status = ta.attn_last_device_status()
    assert status == 0, ta.attn_status_string(status)
    step_ms = [sum(p) for p in per]
    nph = len(phases)
    ph_avg = [max_over_ranks(sum(p[j] for p in per) / len(per), world, dev) for j in range(nph)]
    ms_step = max_over_ranks(sum(step_ms) / args.steps, world, dev)
    value = world * flops_step / (ms_step * 1e-3) / 1e12
    # ---- the same step back to back for at least a second, under the same
    # clock sampling (a steadier figure and enough clock samples)
    sustained = None
    if not args.no_sustained:
        n_sus = max(args.steps, int(math.ceil(args.sustained_s / max(ms_step * 1e-3, 1e-6))))
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if do_flush:
            per_s = time_steps(phases, stream, n_sus, do_flush, flush)
            sus_ms = sum(sum(p) for p in per_s) / n_sus
        else:
            s0.record(stream)
            for _ in range(n_sus):
                step()
            s1.record(stream)
            torch.cuda.synchronize(dev)
            sus_ms = s0.elapsed_time(s1) / n_sus
        sus_ms = max_over_ranks(sus_ms, world, dev)
        sustained = {"steps": n_sus, "seconds": n_sus * sus_ms * 1e-3, "ms_per_step": sus_ms,
                     "value": world * flops_step / (sus_ms * 1e-3) / 1e12}
        assert ta.attn_last_device_status() == 0
    # ---- the other configurations (rank 0's GPU, default line only)
    configs = None
    if args.workload == "step" and not args.no_configs and rank == 0:
        configs = {}
        for cid, wname in CONFIG_SET:
            configs[cid] = time_config(EXTRA_WORKLOADS[wname], ta, dev, sh, stream, flush,
                                       args.l2, pk)
            torch.cuda.empty_cache()
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()

    # ------------------------------------------------------------ e2e
    # Every step copies its inputs from pinned host memory to the device and
    # its results back, all inside the timed region.  Steps are pipelined the
    # way a host program would run them: two sets of device buffers, the
    # upload of step i+1 and the download of step i-1 on two copy streams
    # while step i computes.  The serial form (copy in, compute, copy out, on
    # one stream) is timed too and reported beside it.
    e2e = None
    if not args.no_e2e:
        pinned = [t.pin_memory() for t in host_inputs]
        outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in results]
        h2d = sum(t.numel() * t.element_size() for t in pinned)
        d2h = sum(t.numel() * t.element_size() for t in outs_h)
        phases_b, _, dev_inputs_b, results_b = build_workload(W, ta, dev, rank, sh)
        sets = [(phases, dev_inputs, results), (phases_b, dev_inputs_b, results_b)]
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        n_e2e = max(4, min(args.steps, 50))

        def serial_step():
            for d, h in zip(dev_inputs, pinned):
                d.copy_(h, non_blocking=True)
            step()
            for h, d in zip(outs_h, results):
                h.copy_(d, non_blocking=True)

        def pipelined(n):
            computed = [None, None]   # event: the set's last compute is done
            downloaded = [None, None]  # event: the set's results have been copied out
            start = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            up.wait_event(start)
            last = None
            for i in range(n):
                ph, di, re = sets[i % 2]
                with torch.cuda.stream(up):
                    if computed[i % 2] is not None:
                        up.wait_event(computed[i % 2])   # step i-2 has read these inputs
                    for d, h in zip(di, pinned):
                        d.copy_(h, non_blocking=True)
                    loaded = torch.cuda.Event()
                    loaded.record(up)
                stream.wait_event(loaded)
                if downloaded[i % 2] is not None:
                    stream.wait_event(downloaded[i % 2])   # step i-2's results are out
                for _, fn, _, _ in ph:
                    fn()
                done = torch.cuda.Event()
                done.record(stream)
                computed[i % 2] = done
                with torch.cuda.stream(down):
                    down.wait_event(done)
                    for h, d in zip(outs_h, re):
                        h.copy_(d, non_blocking=True)
                    last = torch.cuda.Event()
                    last.record(down)
                downloaded[i % 2] = last
            stream.wait_event(last)
            end = torch.cuda.Event(enable_timing=True)
            end.record(stream)
            return start, end

        for _ in range(2):
            serial_step()
        pipelined(2)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            serial_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        serial_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        barrier(world)
        p0, p1 = pipelined(n_e2e)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(p0.elapsed_time(p1) / n_e2e, world, dev)
        assert ta.attn_last_device_status() == 0
        e2e = {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": n_e2e,
               "overlap": "two device buffer sets; step i+1's upload and step i-1's download "
                          "run on two copy streams while step i computes",
               "serial_ms_per_step": serial_ms,
               "serial_value": world * flops_step / (serial_ms * 1e-3) / 1e12}

    # ------------------------------------------------------- roofline
    # The dominant kernel by device time decides the roofline entry; every
    # phase is reported under "kernels".
    kernels = kernel_entries(W, phases, ph_avg, pk)
    for j, (lbl, *_rest) in enumerate(phases):
        kernels[lbl]["ms"] = pct_stats([p[j] for p in per])
    dom = max(kernels, key=lambda kk: kernels[kk]["avg_launch_ms"])
    roof = dict(kernels[dom])
    roof["peak_source"] = (f"{pk['source']} HBM copy" if roof["bound"] == "hbm"
                           else f"{pk['source']} bf16 burst")
    if configs is not None and kind == "fwd_bwd":
        configs["C5"] = {"workload": W["name"], "ms": pct_stats(step_ms), "iters": args.steps,
                         "tflops": value / world, "frac": value / world / pk["bf16_tflops"],
                         "peak": pk["bf16_tflops"], "bound": "tensor",
                         "phases": {lbl: {kk: kernels[lbl][kk] for kk in
                                          ("kernel", "ms", "achieved", "frac", "traffic",
                                           "tensor_pipe_active_pct") if kk in kernels[lbl]}
                                    for lbl in kernels},
                         "note": "the line's own K timed steps"}

    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: q,k,v(,dO) ~ N(0,1) bf16, seeded",
            "config": line_config(W, world, do_flush, bytes_step),
            "ms": pct_stats(step_ms),
            "pct_of_bf16_peak": 100.0 * value / world / pk["bf16_tflops"],
            "hbm_gbs_step": world * bytes_step / (ms_step * 1e-3) / 1e9,
            "roofline": roof, "kernels": kernels, "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps, "e2e": e2e}
    if sustained is not None:
        line["sustained"] = sustained
    if configs is not None:
        line["configs"] = configs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_min_s, args.cpu_max_s)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="step", choices=["step", *EXTRA_WORKLOADS],
                    help="step (default): the causal fwd+bwd line; others for manual runs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations (C1-C4) after the default line")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the back-to-back run of the step after the K timed steps")
    ap.add_argument("--sustained-s", type=float, default=1.0,
                    help="length of the back-to-back run (seconds)")
    ap.add_argument("--l2", choices=["auto", "flush", "none"], default="auto",
                    help="between timed steps: flush L2, or not (auto: flush unless a step's "
                         "algorithmic bytes exceed twice the L2 size)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-min-s", type=float, default=10.0)
    ap.add_argument("--cpu-max-s", type=float, default=30.0)
    ap.add_argument("--ref-rows", type=int, default=64,
                    help="query/key rows per oracle sample step (reference arm)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

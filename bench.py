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
L2_FLUSH_BYTES = 256 << 20   # > 129 MB L2


def attn_flops(B, H, N, D, causal):
    """Forward FLOPs by the pages' count 4*B*H*N^2*D (blog.ans20xx.com day26,
    'CUDA event 计时模板'), halved for the causal mask."""
    f = 4.0 * B * H * N * N * D
    return f / 2 if causal else f


def bwd_flops(B, H, N, D, causal):
    return 2.5 * attn_flops(B, H, N, D, causal)


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


FWD_SOURCES = ["tiled_attention_02_gb300/csrc/attn_fwd.cu",
               "tiled_attention_02_gb300/csrc/sm103_ptx.cuh"]


def profiled_traffic(kernel_tag, digest, units):
    """DRAM bytes per launch from the committed ncu summary for this kernel,
    scaled to `units` (query-tile x kv-tile pairs) when it was captured on a
    smaller case; None if absent or if the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_d = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_u = re.search(r"units_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_d and m_b and m_u) or m_d.group(1) != digest:
        return None
    return float(m_b.group(1)) * units / float(m_u.group(1))


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
            "config": config_block(world),
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": s["desc"]},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_block(world):
    W = WORKLOAD
    return {"workload": W["name"], "B": W["B"], "H": W["Hq"], "Hkv": W["Hkv"], "N": W["N"],
            "D": W["D"], "causal": W["causal"], "scale": 1 / math.sqrt(W["D"]),
            "parallelism": f"replicas x{world} (independent problems, no collective)",
            "l2": "flushed between timed steps (256 MB write)"}


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch
    world, rank, local = dist_setup(want_cuda=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import tiled_attention_02_gb300 as ta
    from tiled_attention_02_gb300.inputs import make_qkv
    ta.build()
    W = WORKLOAD
    B, Hq, Hkv, N, D, causal = W["B"], W["Hq"], W["Hkv"], W["N"], W["D"], W["causal"]
    scale = 1.0 / math.sqrt(D)
    x = make_qkv(B, Hq, Hkv, N, D, seed=rank, with_do=True)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(ta.attn_bwd_workspace_size(B, Hq, Hkv, N, D), 256), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    # Does this build have the backward?
    st = ta.raw_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                         lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                         dv.data_ptr(), 1, 1, 1, 128, D, scale, 1, ws.data_ptr(),
                         ws.numel(), sh)
    have_bwd = (st == ta.ATTN_OK)
    torch.cuda.synchronize(dev)

    def fwd():
        s = ta.raw_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, o.data_ptr(),
                            lse.data_ptr(), B, Hq, Hkv, N, D, scale, causal, None, sh)
        assert s == 0, s

    def bwd():
        s = ta.raw_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                            dv.data_ptr(), B, Hq, Hkv, N, D, scale, causal, ws.data_ptr(),
                            ws.numel(), sh)
        assert s == 0, s

    launches_per_step = 1 + (3 if have_bwd else 0)
    for _ in range(args.warmup):
        fwd()
        if have_bwd:
            bwd()
    torch.cuda.synchronize(dev)
    assert ta.attn_last_device_status() == 0

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_id.startswith("GPU-"):
            gpu_id = "GPU-" + gpu_id
    except Exception:
        gpu_id = str(local)
    sampler = ClockSampler(gpu_id)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)   # let the sampler start before the load
    for i in range(args.steps):
        flush.fill_(float(i))       # untimed: evicts the previous step's data from L2
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        if have_bwd:
            bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    status = ta.attn_last_device_status()
    assert status == 0, ta.attn_status_string(status)

    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev] if have_bwd else [0.0] * args.steps
    step_ms = [a + b for a, b in zip(fwd_ms, bwd_ms)]
    ms_step = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    fwd_avg = max_over_ranks(sum(fwd_ms) / len(fwd_ms), world, dev)
    bwd_avg = max_over_ranks(sum(bwd_ms) / len(bwd_ms), world, dev) if have_bwd else 0.0
    f_fwd = attn_flops(B, Hq, N, D, causal)
    f_bwd = bwd_flops(B, Hq, N, D, causal) if have_bwd else 0.0
    flops_step = f_fwd + f_bwd
    value = world * flops_step / (ms_step * 1e-3) / 1e12

    # ------------------------------------------------------------ e2e
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (x[n].pin_memory() for n in ("q", "k", "v", "do"))
        outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory()
                for t in ((dq, dk, dv) if have_bwd else (o,))]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv) + ((hdo,) if have_bwd else ()))
        d2h = sum(t.numel() * t.element_size() for t in outs)

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            if have_bwd:
                do.copy_(hdo, non_blocking=True)
            fwd()
            if have_bwd:
                bwd()
                outs[0].copy_(dq, non_blocking=True)
                outs[1].copy_(dk, non_blocking=True)
                outs[2].copy_(dv, non_blocking=True)
            else:
                outs[0].copy_(o, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(3, min(args.steps, 20))
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        e2e = {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    # ------------------------------------------------------- roofline
    pk = peaks()
    n_qt = (N + 127) // 128
    units = B * Hq * (n_qt * (n_qt + 1) // 2 if causal else n_qt * n_qt)   # 128x128 tile pairs
    digest = source_digest(FWD_SOURCES)
    achieved = f_fwd / (fwd_avg * 1e-3) / 1e12
    roof = {"kernel": "fwd_kernel<128,causal>", "bound": "tensor", "achieved": achieved,
            "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
            "peak_source": f"{pk['source']} bf16 burst",
            "traffic": profiled_traffic("fwd_kernel_causal_B1_H16_N16384_D128", digest, units),
            "flops_per_launch": f_fwd, "units_per_launch": units,
            "avg_launch_ms": fwd_avg, "source_digest": digest}

    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: q,k,v,dO ~ N(0,1) bf16, seeded",
            "config": dict(config_block(world),
                           step="forward + backward" if have_bwd else
                           "forward only (backward not in this build)"),
            "fwd_tflops": f_fwd / (fwd_avg * 1e-3) / 1e12,
            "bwd_tflops": (f_bwd / (bwd_avg * 1e-3) / 1e12) if have_bwd else None,
            "pct_of_bf16_peak": 100.0 * value / world / pk["bf16_tflops"],
            "roofline": roof, "clocks": clocks, "gpu_launches": launches_per_step * args.steps,
            "e2e": e2e}
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
    ap.add_argument("--no-e2e", action="store_true")
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

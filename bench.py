"""Throughput of the scaled FP8 casts on GB300 (GB/s moved, read + write).

Default workload, one step = the whole hot path over one batch:
  * the per-step cast of every weight, activation and activation gradient of
    a 24-layer decoder (hidden 2048, FFN 8192, batch 4 x seq 4096): 384 bf16
    tensors, 14,092,861,440 elements, weights and activations to E4M3,
    gradients to E5M2, per-tensor max-window scaling (window 16), in one
    grouped launch (fp8q_cast_multi);
  * the MX E4M3 cast (OCP rule) of the bf16 [16384, 8192] tanh activations.
Algorithmic bytes: 3 B per element for the per-tensor cast (2 read + 1
written), 3.03125 B per element for MX (+1 E8M0 byte per 32).

Run: python bench.py [--steps K] [--warmup W] [--impl ours|reference]
     [--workload decoder|single|mx] [--n N]  (torchrun for --gpus N > 1:
     replicas, one full workload per GPU).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 scaled-cast GB/s (read+write) and fraction of GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decoder", choices=["decoder", "single", "mx"])
    p.add_argument("--n", type=int, default=1 << 26, help="elements for --workload single")
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# workload construction (device-resident inputs and outputs)
# ---------------------------------------------------------------------------

class Workload:
    def __init__(self, kind: str, n: int, device):
        import torch

        from tensor_scaling_cast_gb300 import fp8q as F
        from tensor_scaling_cast_gb300 import synthetic as S
        self.kind, self.F, self.torch = kind, F, torch
        self.xs, self.fmts, self.handles = [], [], []
        self.mx_x = None
        if kind == "decoder":
            self.specs = S.decoder_tensor_specs()
            for sp in self.specs:
                self.xs.append(S.decoder_tensor(sp, 0, device))
                self.fmts.append(sp[2])
            self.mx_x = S.mx_tanh(device)
            self.name = ("decoder_1b1 per-step cast (384 bf16 tensors, 14,092,861,440 elements; "
                         "E4M3 weights/activations, E5M2 gradients; max-window 16) + MX E4M3 OCP "
                         "cast of bf16 [16384, 8192] tanh(N(0,2))")
        elif kind == "single":
            g = torch.Generator(device=device)
            g.manual_seed(1)
            self.xs.append(torch.randn(n, generator=g, device=device).to(torch.bfloat16))
            self.fmts.append(F.E4M3)
            self.name = f"single bf16 tensor of {n} elements, E4M3, max-window 16"
        else:
            self.mx_x = S.mx_tanh(device)
            self.name = "MX E4M3 OCP cast of bf16 [16384, 8192] tanh(N(0,2))"
        self.handles = [F.fp8q_create(f, 16, 0, 0) for f in self.fmts]
        self.qs = [torch.empty(x.numel(), dtype=torch.uint8, device=device) for x in self.xs]
        m = max(1, len(self.xs))
        self.sinv = torch.empty(m, dtype=torch.float32, device=device)
        self.amax = torch.empty(m, dtype=torch.float32, device=device)
        self.clipped = torch.empty(m, dtype=torch.int64, device=device)
        if self.mx_x is not None:
            r, c = self.mx_x.shape
            self.mx_q = torch.empty(r, c, dtype=torch.uint8, device=device)
            self.mx_e8 = torch.empty(r, c // 32, dtype=torch.uint8, device=device)
            self.mx_clip = torch.empty(1, dtype=torch.int64, device=device)
        self.cast_elems = sum(x.numel() for x in self.xs)
        self.mx_elems = 0 if self.mx_x is None else self.mx_x.numel()
        self.cast_bytes = 3 * self.cast_elems
        self.mx_bytes = 0 if self.mx_x is None else self.mx_elems * 2 + self.mx_elems + self.mx_elems // 32
        self.step_bytes = self.cast_bytes + self.mx_bytes

    def step(self, ev=None):
        F = self.F
        if ev is not None:
            ev[0].record()
        if self.xs:
            F.fp8q_cast_multi(self.handles, self.xs, self.qs, self.sinv, self.amax, self.clipped)
        if ev is not None:
            ev[1].record()
        if self.mx_x is not None:
            F.mx_cast(self.mx_x, F.E4M3, 0, self.mx_q, self.mx_e8, self.mx_clip)
        if ev is not None:
            ev[2].record()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc = index, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def cpu_oracle_sample(seconds: float, inputs=None):
    """Cast decoder_1b1 tensors (step 0 = current scaling, then a delayed
    step) through the oracle until about `seconds` of work; returns
    (GB/s, cores, description)."""
    import numpy as np
    import torch

    from oracle import coracle, policy
    from tensor_scaling_cast_gb300 import synthetic as S
    coracle.build()
    cores = os.cpu_count() or 1
    specs = S.decoder_tensor_specs()
    done_bytes, done_elems, elapsed, names = 0, 0, 0.0, []
    i = 0
    while elapsed < seconds and i < len(specs):
        sp = specs[i]
        x = inputs[i] if inputs is not None else S.decoder_tensor(sp, 0, "cpu")
        xb = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)
        st = policy.ScalingState(sp[2], 16)
        st.step(xb, cores)                       # fill the window (not timed)
        t0 = time.perf_counter()
        st.step(xb, cores)                       # one delayed-scaling cast
        elapsed += time.perf_counter() - t0
        done_bytes += 3 * xb.size
        done_elems += xb.size
        names.append(sp[0])
        i += 1
    desc = (f"oracle.c max-window cast of {len(names)} decoder_1b1 tensors ({names[0]}..{names[-1]}), "
            f"{done_elems} elements, {elapsed:.1f} s on {cores} threads")
    return done_bytes / elapsed / 1e9, cores, desc


def run_reference(args, rank: int):
    if rank != 0:
        return
    gbs, cores, desc = cpu_oracle_sample(max(3.0, args.cpu_seconds))
    line = {"metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "decoder_1b1 per-step cast (sample, see cpu_baseline)",
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank: int, world: int):
    import torch
    import torch.distributed as dist

    from tensor_scaling_cast_gb300 import build
    from tensor_scaling_cast_gb300 import fp8q as F

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    F.load()
    W = Workload(args.workload, args.n, dev)
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):
        W.step()
    torch.cuda.synchronize()

    # device-resident timed region
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    l0 = F.launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for k in range(K):
        W.step(evs[k])
    t_end.record()
    torch.cuda.synchronize()
    launches = F.launch_count() - l0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_step = ms / K
    cast_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) if W.xs else 0.0
    mx_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) if W.mx_x is not None else 0.0
    value = world * W.step_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = peaks()

    # dominant kernel roofline
    if W.xs:
        dom, dom_ms, dom_bytes = "cast_group_kernel", cast_ms, W.cast_bytes
    else:
        dom, dom_ms, dom_bytes = "mx_kernel", mx_ms, W.mx_bytes
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    parts = {}
    if W.xs:
        parts["grouped_cast"] = {"ms": round(cast_ms, 4), "bytes": W.cast_bytes,
                                 "GB/s": round(W.cast_bytes / (cast_ms * 1e-3) / 1e9, 1),
                                 "frac": round(W.cast_bytes / (cast_ms * 1e-3) / 1e9 / peak, 4)}
    if W.mx_x is not None:
        parts["mx_cast"] = {"ms": round(mx_ms, 4), "bytes": W.mx_bytes,
                            "GB/s": round(W.mx_bytes / (mx_ms * 1e-3) / 1e9, 1),
                            "frac": round(W.mx_bytes / (mx_ms * 1e-3) / 1e9 / peak, 4)}

    # end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(W, args.e2e_steps, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and args.workload == "decoder":
        gbs, cores, desc = cpu_oracle_sample(args.cpu_seconds, inputs=W.xs)
        cpu = {"value": round(gbs, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": W.name, "elements_per_step": W.cast_elems + W.mx_elems,
                       "bytes_per_step": W.step_bytes, "io": "bf16 in, FP8 (+E8M0) out",
                       "l2": f"inputs larger than L2 ({W.step_bytes / 1e9:.1f} GB moved per step)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback",
                         "bytes_per_launch": dom_bytes, "traffic": None},
            "parts": parts,
            "gpu_launches": launches,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def run_e2e(W, steps: int, world: int, dev):
    """Same step through the public API with host buffers: pinned H2D of the
    step's inputs, the casts, D2H of every output (q, E8M0, scalars)."""
    import torch
    import torch.distributed as dist
    F = W.F
    h_x = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in W.xs]
    for hx, x in zip(h_x, W.xs):
        hx.copy_(x)
    h_q = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for q in W.qs]
    n = max(1, len(W.xs))
    h_small = torch.empty(3 * n, dtype=torch.float32, pin_memory=True)
    h_clip = torch.empty(n, dtype=torch.int64, pin_memory=True)
    if W.mx_x is not None:
        h_mx = torch.empty(W.mx_x.shape, dtype=W.mx_x.dtype, pin_memory=True)
        h_mx.copy_(W.mx_x)
        h_mq = torch.empty(W.mx_q.shape, dtype=torch.uint8, pin_memory=True)
        h_me = torch.empty(W.mx_e8.shape, dtype=torch.uint8, pin_memory=True)
        h_mc = torch.empty(1, dtype=torch.int64, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in W.xs) + (0 if W.mx_x is None else W.mx_x.numel() * 2)
    d2h = sum(q.numel() for q in W.qs) + (3 * 4 * n if W.xs else 0) + (8 * n if W.xs else 0)
    if W.mx_x is not None:
        d2h += W.mx_q.numel() + W.mx_e8.numel() + 8

    def one():
        for hx, x in zip(h_x, W.xs):
            x.copy_(hx, non_blocking=True)
        if W.mx_x is not None:
            W.mx_x.copy_(h_mx, non_blocking=True)
        W.step()
        for hq, q in zip(h_q, W.qs):
            hq.copy_(q, non_blocking=True)
        if W.xs:
            h_small[0:n].copy_(W.sinv, non_blocking=True)
            h_small[n:2 * n].copy_(W.amax, non_blocking=True)
            h_clip.copy_(W.clipped, non_blocking=True)
        if W.mx_x is not None:
            h_mq.copy_(W.mx_q, non_blocking=True)
            h_me.copy_(W.mx_e8, non_blocking=True)
            h_mc.copy_(W.mx_clip, non_blocking=True)

    one()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return {"value": round(world * W.step_bytes / (ms / steps * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 3), "steps": steps}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    run_ours(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

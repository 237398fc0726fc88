"""Throughput of the scaled FP8 casts on GB300 (GB/s moved, read + write).

Default workload (``--workload decoder``), one step = the whole hot path over
one batch:
  * the per-step cast of every weight, activation and activation gradient of
    a 24-layer decoder (hidden 2048, FFN 8192, batch 4 x seq 4096): 384 bf16
    tensors, 14,092,861,440 elements, weights and activations to E4M3,
    gradients to E5M2, per-tensor max-window scaling (window 16), in one
    grouped launch (fp8q_cast_multi);
  * the MX E4M3 cast (OCP rule) of the bf16 [16384, 8192] tanh activations.
Algorithmic bytes: 3 B per element for a bf16 per-tensor cast (2 read + 1
written), 5 B for fp32, 3.03125 B per element for bf16 MX (+1 E8M0 byte per
32).  The other workloads (current, spike, grad, mx, single) measure the
remaining configurations and small profiling cases with the same JSON line.

Run: python bench.py [--steps K] [--warmup W] [--impl ours|reference]
     [--workload decoder|current|spike|grad|mx|transpose|single] [--n N]
     [--sigma-is-variance]
(torchrun for --gpus N > 1: replicas, one full workload per GPU).

Besides the timed figures, each line carries `results` (what the
configurations ask to report, computed with the library outside the timed
region) and `inputs_sha256` (the SHA-256 of every input tensor's bytes), so
the reported fractions can be tied to the exact inputs that produced them.
Lines also carry `parts_after_clean_l2` (except the CUDA-graph workloads):
each part timed alone after a read of 1 GiB that leaves no dirty line in
L2, i.e. without the write-back of the previous part's (or step's) output
that a part absorbs inside the timed steps (`parts`).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8 scaled-cast GB/s (read+write) and fraction of GB300 HBM peak"
# The arithmetic of the path: bf16 (or fp32) elements in, 8-bit float codes
# out, the scale applied and the element converted in fp32.
DTYPE = "bf16 in -> fp8 e4m3/e5m2 out (fp32 scale arithmetic)"
DECODER_NAME = ("decoder_1b1 per-step cast (384 bf16 tensors, 14,092,861,440 elements; "
                "E4M3 weights/activations, E5M2 gradients; max-window 16) + MX E4M3 OCP "
                "cast of bf16 [16384, 8192] tanh(N(0,2))")


def decoder_config(world: int) -> dict:
    """The `config` of the default (decoder_1b1) bench line; the reference
    arm reports the same one."""
    from tensor_scaling_cast_gb300 import synthetic as S
    cast = sum(r * c * 3 for _, (r, c), *_ in S.decoder_tensor_specs())
    mx = 16384 * 8192 * 3 + 16384 * 8192 // 32
    step = cast + mx
    return {"workload": DECODER_NAME, "bytes_per_step": step, "io": "bf16/fp32 in, FP8 (+E8M0) out",
            "l2": f"inputs larger than L2 ({step / 1e9:.2f} GB moved per step)",
            "parallelism": "replicas" if world > 1 else "single GPU"}
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decoder",
                   choices=["decoder", "current", "spike", "grad", "mx", "transpose", "single"])
    p.add_argument("--n", type=int, default=1 << 26, help="elements for --workload single")
    p.add_argument("--single-dtype", default="bf16", choices=["bf16", "fp32"],
                   help="input type for --workload single")
    p.add_argument("--group-policies", action="store_true",
                   help="--workload spike: cast the step's tensor under both policies in one grouped launch")
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-one-core", action="store_true",
                   help="skip the single-thread oracle baseline (run by default beside the all-core one)")
    p.add_argument("--sigma-is-variance", action="store_true",
                   help="read the MX activations' N(0,2) as variance 2 (sigma = sqrt 2) for the timed "
                        "input; results report both readings either way")
    return p.parse_args()


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over all ranks (the slowest rank's time); identity for
    one process.  device: where the collective's tensor lives (cuda for
    NCCL, cpu for gloo)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = ["tensor_scaling_cast_gb300/csrc/cast_kernels.cuh", "tensor_scaling_cast_gb300/csrc/state.cuh",
                  "tensor_scaling_cast_gb300/csrc/fp8q_device.cuh", "tensor_scaling_cast_gb300/csrc/fp8q_internal.cuh"]
TRAFFIC_FILE = "profiles/traffic_cast_group_kernel_decoder_1b1.md"


def captured_traffic():
    """DRAM bytes of one full-size grouped launch from the committed ncu
    capture, or None when the kernel sources changed since it was taken."""
    import hashlib
    try:
        h = hashlib.sha256()
        for f in KERNEL_SOURCES:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        fields = {}
        with open(os.path.join(ROOT, TRAFFIC_FILE)) as fh:
            for line in fh:
                if ":" in line and not line.startswith(("#", "|", " ")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("source_sha256") == h.hexdigest():
            return int(fields["traffic_bytes_per_launch"])
    except Exception:
        pass
    return None


def cast_bytes(x) -> int:
    return x.numel() * (x.element_size() + 1)


def mx_bytes(x) -> int:
    return x.numel() * (x.element_size() + 1) + x.numel() // 32


# ---------------------------------------------------------------------------
# workloads: parts launched in order each step, device-resident buffers
# ---------------------------------------------------------------------------

class Part:
    """One launch (or grouped launch) of a step."""

    def __init__(self, name, kernel, nbytes, run, inputs, outputs):
        self.name, self.kernel, self.bytes = name, kernel, nbytes
        self.run = run              # run(k): enqueue on the current stream
        self.inputs = inputs        # inputs(k) -> device tensors read at step k
        self.outputs = outputs      # outputs(k) -> device tensors written at step k


class Workload:
    def __init__(self, kind: str, n: int, device, host_io: bool = False, single_dtype: str = "bf16",
                 group_policies: bool = False, mx_sigma: float = 2.0):
        """host_io: inputs and outputs live in pinned host memory and the
        kernels read / write them directly over NVLink-C2C (zero-copy).
        group_policies (spike): both handles cast the step's tensor in one
        fp8q_cast_multi launch instead of one launch each."""
        import torch

        from tensor_scaling_cast_gb300 import fp8q as F
        from tensor_scaling_cast_gb300 import synthetic as S
        self.kind, self.device, self.host_io = kind, device, host_io
        self.handles = []

        def io_in(t):                   # an input tensor in the chosen memory
            if not host_io:
                return t
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            return h

        def io_out(shape, dtype):       # an output tensor in the chosen memory
            if host_io:
                return torch.empty(shape, dtype=dtype, pin_memory=True)
            return torch.empty(shape, dtype=dtype, device=dev)
        self.parts: list[Part] = []
        self.oracle_jobs = []       # (callable(nthreads) -> bytes) for the CPU baseline
        self.named_inputs = []      # (name, tensor) of every input, for the digests
        dev = device

        def grouped(name, xs, fmts, window, margin=0):
            hs = [F.fp8q_create(f, window, margin, 0) for f in fmts]
            self.handles += hs
            xs = [io_in(x) for x in xs]
            qs = [io_out((x.numel(),), torch.uint8) for x in xs]
            m = len(xs)
            outs = [torch.empty(m, dtype=torch.float32, device=dev),
                    torch.empty(m, dtype=torch.float32, device=dev),
                    torch.empty(m, dtype=torch.int64, device=dev)]
            run = lambda k: F.fp8q_cast_multi(hs, xs, qs, *outs)
            self.parts.append(Part(name, "cast_group_kernel", sum(cast_bytes(x) for x in xs), run,
                                   lambda k: xs, lambda k: qs + outs))
            for x, f in zip(xs, fmts):
                self.oracle_jobs.append(("cast", x, f, window, margin))

        def mx(name, x, headroom, rule=0, axis=0):
            r, c = x.shape
            q = io_out((r, c), torch.uint8)
            e8 = io_out((r, c // 32) if axis == 0 else (r // 32, c), torch.uint8)
            cl = torch.empty(1, dtype=torch.int64, device=dev)
            run = lambda k: F.mx_cast_ex(x, F.E4M3, rule, headroom, axis, q, e8, cl)
            self.parts.append(Part(name, "mx_kernel" if axis == 0 else "mx_colwise_kernel",
                                   mx_bytes(x), run, lambda k: [x], lambda k: [q, e8, cl]))
            self.oracle_jobs.append(("mx", x, 0, headroom, 0))

        if kind == "decoder":
            specs = S.decoder_tensor_specs()
            xs = [io_in(S.decoder_tensor(sp, 0, dev)) for sp in specs]
            grouped("grouped_cast", xs, [sp[2] for sp in specs], 16)
            xm = io_in(S.mx_tanh(dev, sigma=mx_sigma))
            mx("mx_cast", xm, 0)
            self.named_inputs = [(sp[0], x) for sp, x in zip(specs, xs)] + [("mx_tanh", xm)]
            self.name = DECODER_NAME if mx_sigma == 2.0 else DECODER_NAME.replace(
                "tanh(N(0,2))", f"tanh(N(0,2)) read as variance 2 (sigma {mx_sigma:.6g})")
        elif kind == "grad":
            xs = [io_in(x) for x in S.grad_group_step(1, dev)]
            grouped("grouped_cast", xs, [1] * len(xs), 16)
            self.named_inputs = [(f"grad{i}", x) for i, x in enumerate(xs)]
            self.name = (f"grad_group: 64 bf16 tensors ({sum(x.numel() for x in xs)} elements), "
                         "E5M2, max-window 16, one grouped launch")
        elif kind == "mx":
            x = io_in(S.mx_tanh(dev, sigma=mx_sigma))
            self.named_inputs = [("mx_tanh", x)]
            mx("mx_cast_ocp", x, 0)
            mx("mx_cast_headroom1", x, 1)
            mx("mx_cast_ceil", x, 0, rule=1)
            mx("mx_cast_nearest", x, 0, rule=2)
            mx("mx_cast_colwise_ocp", x, 0, axis=1)
            mx("mx_cast_colwise_ceil", x, 0, rule=1, axis=1)
            r, c = x.shape
            dq = [io_out((r, c), torch.uint8), io_out((r, c // 32), torch.uint8),
                  io_out((c, r), torch.uint8), io_out((c, r // 32), torch.uint8)]
            dcl = [torch.empty(1, dtype=torch.int64, device=dev) for _ in range(2)]
            for nm, rule in (("mx_cast_dual_ocp", 0), ("mx_cast_dual_ceil", 1)):
                self.parts.append(Part(nm, "mx_dual_kernel",
                                       x.numel() * (x.element_size() + 2) + 2 * (x.numel() // 32),
                                       lambda k, rule=rule: F.mx_cast_dual(x, F.E4M3, rule, 0, *dq, *dcl),
                                       lambda k: [x], lambda k: dq + dcl))
            self.name = ("MX E4M3 of bf16 [16384, 8192] tanh(N(0,2)): row-wise OCP, +1 headroom, "
                         "ceil and nearest scale rules; column-wise OCP and ceil; dual (row-wise + "
                         "transposed column-wise) OCP and ceil")
            if mx_sigma != 2.0:
                self.name = self.name.replace("tanh(N(0,2))", f"tanh(N(0,2)) read as variance 2 (sigma {mx_sigma:.6g})")
        elif kind == "transpose":
            x = io_in(S.mx_tanh(dev))
            self.named_inputs = [("mx_tanh", x)]
            r, c = x.shape
            g = F.fp8q_create(F.E4M3, 16, 0, 0)
            self.handles.append(g)
            q, qt = io_out((r, c), torch.uint8), io_out((c, r), torch.uint8)
            outs = torch.empty(3, dtype=torch.float32, device=dev)
            self.parts.append(Part("cast_transpose", "cast_transpose_kernel",
                                   x.numel() * (x.element_size() + 2),
                                   lambda k: F.fp8q_cast_transpose(g, x, q, qt, outs[0:1], outs[1:2]),
                                   lambda k: [x], lambda k: [q, qt]))
            self.oracle_jobs.append(("cast", x, 0, 16, 0))
            self.name = ("cast_transpose: bf16 [16384, 8192] -> E4M3 q [16384, 8192] and q^T "
                         "[8192, 16384], max-window 16, one launch")
        elif kind == "spike":
            seq = [S.spike_step(s, dev) for s in range(S.SPIKE_STEPS)]
            self.named_inputs = [(f"spike_step{s}", x) for s, x in enumerate(seq)]
            qs = []
            for name, w, m in (("most_recent_w1", 1, 0), ("max_window_w16_m1", 16, 1)):
                g = F.ScaledCast(F.E4M3, w, m)
                self.handles.append(g)
                q = torch.empty(seq[0].numel(), dtype=torch.uint8, device=dev)
                qs.append(q)
                if not group_policies:
                    run = (lambda g, q: lambda k: g(seq[k % len(seq)], q))(g, q)
                    self.parts.append(Part(name, "cast_group_kernel", cast_bytes(seq[0]), run,
                                           lambda k: [seq[k % len(seq)]], (lambda q: lambda k: [q])(q)))
                self.oracle_jobs.append(("cast", seq[0], 0, w, m))
            if group_policies:
                hs = [g.handle for g in self.handles]
                outs = [torch.empty(2, dtype=torch.float32, device=dev), torch.empty(2, dtype=torch.float32, device=dev),
                        torch.empty(2, dtype=torch.int64, device=dev)]
                run = lambda k: F.fp8q_cast_multi(hs, [seq[k % len(seq)]] * 2, qs, *outs)
                self.parts.append(Part("both_policies_grouped", "cast_group_kernel", 2 * cast_bytes(seq[0]), run,
                                       lambda k: [seq[k % len(seq)]], lambda k: qs + outs))
            self.name = ("spike_seq: bf16 [4096, 4096] E4M3, inputs rotating over the 16 steps "
                         "(512 MiB), most-recent and max-window-16 (margin 1) per step"
                         + (", both policies in one grouped launch" if group_policies else ""))
        elif kind == "current":
            x = S.current_4096(dev)
            self.named_inputs = [("current_4096", x)]
            g = F.ScaledCast(F.E4M3, 0, 0)
            self.handles.append(g)
            q = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
            self.parts.append(Part("current_scaling", "cast_group_kernel", 2 * 4 * x.numel() + x.numel(),
                                   lambda k: g(x, q), lambda k: [x], lambda k: [q]))
            self.oracle_jobs.append(("cast", x, 0, 0, 0))
            self.name = "current_4096: fp32 [4096] N(0,1), E4M3, current scaling (latency)"
        else:
            g = torch.Generator(device=dev)
            g.manual_seed(1)
            x = torch.randn(n, generator=g, device=dev)
            if single_dtype == "bf16":
                x = x.to(torch.bfloat16)
            grouped("cast", [x], [F.E4M3], 16)
            self.named_inputs = [("single", x)]
            self.name = f"single {single_dtype} tensor of {n} elements, E4M3, max-window 16"
        self.step_bytes = sum(p.bytes for p in self.parts)
        # small launches cannot be fed from Python fast enough: those
        # workloads are timed by replaying a CUDA graph of `graph_steps` steps
        self.graph_steps = {"current": 100, "spike": 16}.get(kind, 0)

    def step(self, k, ev=None):
        for i, p in enumerate(self.parts):
            if ev is not None:
                ev[i].record()
            p.run(k)
        if ev is not None:
            ev[len(self.parts)].record()


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

    def stop(self, t0: float, t1: float):
        """Samples taken between host times t0 and t1 (the timed region)."""
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
                "reasons": sorted(reasons), "samples": len(sm),
                "window_s": round(t1 - t0, 3)}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def _bits(x):
    import numpy as np
    import torch
    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.view(torch.int32).numpy().view(np.uint32)


def oracle_time(jobs, seconds: float, nthreads: int):
    """Run the oracle over the workload's tensors (a delayed-scaling cast per
    per-tensor job after one window-filling cast; an MX cast per MX job),
    round-robin, until about `seconds` of timed work.  Returns
    (GB/s, description)."""
    from oracle import coracle, policy
    coracle.build()
    done, elapsed, count, i, names = 0, 0.0, 0, 0, set()
    host = {}
    while elapsed < seconds and i < 64 * len(jobs):
        kind, x, fmt, a, b = jobs[i % len(jobs)]
        key = id(x)
        if key not in host:
            host[key] = _bits(x)
        xb = host[key]
        if kind == "cast":
            st = policy.ScalingState(fmt, a, b)
            if a > 0:
                st.step(xb.reshape(-1)[: 1 << 20], nthreads)   # fill the window (not timed)
            t0 = time.perf_counter()
            st.step(xb.reshape(-1), nthreads)
            elapsed += time.perf_counter() - t0
            done += xb.size * (xb.itemsize + 1)
        else:
            t0 = time.perf_counter()
            coracle.mx_cast(xb, 0, a, nthreads)
            elapsed += time.perf_counter() - t0
            done += xb.size * (xb.itemsize + 1) + xb.size // 32
        names.add(kind)
        count += 1
        i += 1
    desc = (f"oracle.c: {count} casts ({'/'.join(sorted(names))}) of this workload's tensors, "
            f"{done / 1e9:.2f} GB moved, {elapsed:.1f} s on {nthreads} thread(s)")
    return done / elapsed / 1e9, desc


def run_reference(args, rank: int):
    """The reference arm: the CPU oracle as it stands, on the host cores, no
    GPU.  Each of the W + K steps casts a bounded slice of the decoder_1b1
    workload (round-robin over one layer's 16 tensors, delayed scaling with
    a filled window), sized so the whole run takes about a minute."""
    if rank != 0:
        return
    import numpy as np

    from oracle import coracle, policy
    from tensor_scaling_cast_gb300 import synthetic as S
    coracle.build()
    cores = os.cpu_count() or 1
    specs = S.decoder_tensor_specs()[:16]
    xs, states = {}, {}

    def tensor(i):                              # generated and window-filled on first use
        if i not in xs:
            xs[i] = _bits(S.decoder_tensor(specs[i], 0, "cpu")).reshape(-1)
            st = policy.ScalingState(specs[i][2], 16)
            st.step(xs[i][: 1 << 20], cores)
            states[i] = st
        return xs[i], states[i]

    x0, _ = tensor(0)
    t0 = time.perf_counter()
    policy.ScalingState(0, 16).step(x0[: 1 << 22], cores)
    rate = (1 << 22) / max(1e-6, time.perf_counter() - t0)          # elements / s
    budget = max(2.0, 4 * args.cpu_seconds)
    per_step = int(min(1 << 26, max(1 << 16, rate * budget / (args.steps + args.warmup))))
    done, elapsed = 0, 0.0
    for k in range(args.warmup + args.steps):
        i = k % len(specs)
        x, st = tensor(i)
        off = ((k // len(specs)) * per_step) % max(1, x.size - per_step)
        sl = np.ascontiguousarray(x[off: off + per_step])
        t0 = time.perf_counter()
        st.step(sl, cores)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            elapsed += dt
            done += sl.size * 3
    gbs = done / elapsed / 1e9
    desc = (f"oracle.c delayed-scaling cast, {args.steps} timed steps of up to {per_step} elements "
            f"(slices of decoder_1b1 layer-0 tensors, round-robin), {elapsed:.1f} s on {cores} threads")
    line = {"metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * elapsed / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic", "impl": "reference",
            "config": decoder_config(args.gpus),
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
    sigma = math.sqrt(2.0) if args.sigma_is_variance else 2.0
    W = Workload(args.workload, args.n, dev, single_dtype=args.single_dtype, group_policies=args.group_policies,
                 mx_sigma=sigma)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.5)                            # sampler up before the GPU work starts
    warm = max(3, args.warmup)
    for k in range(warm):
        W.step(k)
    torch.cuda.synchronize()

    K = args.steps
    P = len(W.parts)
    graph = None
    if W.graph_steps:
        G = W.graph_steps
        K = max(G, (K // G) * G)
        l_cap = F.launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for k in range(G):
                W.step(warm + k)
        launches_per_graph = F.launch_count() - l_cap
        graph.replay()
        torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(P + 1)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    l0 = F.launch_count()
    host_t0 = time.time()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    if graph is not None:
        for _ in range(K // W.graph_steps):
            graph.replay()
    else:
        for k in range(K):
            W.step(warm + k, evs[k])
    t_end.record()
    torch.cuda.synchronize()
    host_t1 = time.time()
    launches = F.launch_count() - l0
    if graph is not None:
        launches = launches_per_graph * (K // W.graph_steps)
    clk = clocks.stop(host_t0, host_t1)
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    ms_step = ms / K
    value = world * W.step_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = peaks()

    parts = {}
    for i, p in enumerate(W.parts):
        if graph is None:
            ts = sorted(e[i].elapsed_time(e[i + 1]) for e in evs)
            pm = statistics.mean(ts)
            pct = {"p10": round(ts[len(ts) // 10], 5), "p50": round(ts[len(ts) // 2], 5),
                   "p90": round(ts[(9 * len(ts)) // 10], 5)}
        else:                       # graph replay: the step time split by bytes
            pm = ms_step * p.bytes / W.step_bytes
            pct = {"timing": f"CUDA-graph replay of {W.graph_steps} steps; step time split by bytes"}
        gbs = p.bytes / (pm * 1e-3) / 1e9
        parts[p.name] = {"kernel": p.kernel, "ms": round(pm, 5), "bytes": p.bytes,
                         "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), **pct}
    dom = max(W.parts, key=lambda p: parts[p.name]["ms"])
    dpart = parts[dom.name]

    copy_ref = copy_reference(dev, W.step_bytes)
    clean = parts_after_clean_l2(W, dev, min(K, 10), warm + K, peak) if not W.graph_steps else None
    results = workload_results(args.workload, dev) if rank == 0 else None
    digests = input_digests(W) if rank == 0 else None
    e2e = None
    if not args.no_e2e:
        need = pinned_bytes(W)
        ok, why = host_memory_allows(need)
        zero_copy_ok = args.workload in ("decoder", "grad", "mx", "single", "transpose")
        if not ok:
            e2e = {"value": None, "skipped": why}
        elif world > 1 and zero_copy_ok:
            # one pinned copy of the workload per rank: the zero-copy path only
            e2e = run_e2e_zero_copy(args, world, dev, sigma)
        else:
            staged = run_e2e(W, args.e2e_steps, world, dev, warm + K)
            if hasattr(torch._C, "_host_emptyCache"):
                torch._C._host_emptyCache()          # give the staging mirrors back
            e2e = staged
            if zero_copy_ok:
                zc = run_e2e_zero_copy(args, world, dev, sigma)
                # the headline is the faster of the two paths, reported with
                # its own timing, bytes and phases; the other sits beside it
                best, other, other_name = ((zc, staged, "staged_copy") if zc["value"] > staged["value"]
                                           else (staged, zc, "zero_copy"))
                e2e = dict(best)
                e2e[other_name] = other

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cores = os.cpu_count() or 1
        gbs, desc = oracle_time(W.oracle_jobs, args.cpu_seconds, cores)
        cpu = {"value": round(gbs, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": desc}
        if not args.no_cpu_one_core:
            g1, d1 = oracle_time(W.oracle_jobs, args.cpu_seconds, 1)
            cpu["one_core"] = {"value": round(g1, 4), "unit": "GB/s", "cores": 1, "sample": d1}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": warm, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic",
            "config": {"workload": W.name, "bytes_per_step": W.step_bytes,
                       "io": "bf16/fp32 in, FP8 (+E8M0) out",
                       "l2": f"inputs larger than L2 ({W.step_bytes / 1e9:.2f} GB moved per step)"
                       if args.workload in ("decoder", "grad", "mx", "spike", "single", "transpose")
                       else "tiny: L2-resident, latency only",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "frac_of_same_box_copy": round(dpart["GB/s"] / copy_ref["GB/s"], 4),
            "roofline": {"bound": "hbm", "kernel": dom.kernel, "achieved": dpart["GB/s"],
                         "peak": peak, "unit": "GB/s", "frac": dpart["frac"],
                         "peak_source": "measured: MEASURED_PEAKS.json hbm_gbs (copy)"
                         if peak_kind == "measured" else "fallback",
                         "bytes_per_launch": dom.bytes,
                         "traffic": captured_traffic() if (args.workload == "decoder"
                                                           and dom.kernel == "cast_group_kernel") else None},
            "parts": parts,
            "copy_reference": copy_ref,
            "gpu_launches": launches,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        if clean is not None:
            line["parts_after_clean_l2"] = clean
        if args.workload == "current":
            line["latency_us_per_cast"] = round(ms_step * 1e3, 2)
        if results is not None:
            line["results"] = results
        if digests is not None:
            line["inputs_sha256"] = digests
        print(json.dumps(line), flush=True)


def parts_after_clean_l2(W, dev, steps: int, k0: int, peak: float) -> dict:
    """Each part timed on its own right after a read of 1 GiB, which leaves
    no dirty line in the 129 MB L2: the part's own throughput, without the
    write-back of the previous part's output that it absorbs inside a step
    (CUDA events around the part only; outside the timed region of `value`)."""
    import torch
    flush = torch.ones(1 << 29, dtype=torch.float16, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in W.parts]
    tot = [0.0] * len(W.parts)
    for k in range(steps):
        for i, p in enumerate(W.parts):
            torch.sum(flush, dim=0, dtype=torch.float32, out=sink)
            evs[i][0].record()
            p.run(k0 + k)
            evs[i][1].record()
        torch.cuda.synchronize()
        for i in range(len(W.parts)):
            tot[i] += evs[i][0].elapsed_time(evs[i][1])
    del flush
    out = {}
    for i, p in enumerate(W.parts):
        ms = tot[i] / steps
        gbs = p.bytes / (ms * 1e-3) / 1e9
        out[p.name] = {"ms": round(ms, 5), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
    return out


def input_digests(W) -> dict:
    """SHA-256 of every input tensor's bytes, by tensor name (hashed on the
    host cores in parallel; hashlib releases the GIL on large buffers)."""
    import concurrent.futures as cf
    import hashlib

    def one(item):
        name, t = item
        a = _bits(t).reshape(-1)
        h = hashlib.sha256()
        step = 1 << 26
        for i in range(0, a.size, step):
            h.update(memoryview(a[i:i + step]).cast("B"))
        return name, h.hexdigest()
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        return dict(ex.map(one, W.named_inputs))


def mx_results(dev, rules=(("ocp", 0, 0, 0), ("headroom1", 0, 1, 0), ("ceil", 1, 0, 0),
                           ("nearest", 2, 0, 0), ("colwise_ocp", 0, 0, 1))):
    """Clipped fraction (and for row-wise blocks MSE and bias) of the MX
    E4M3 cast of tanh(N(0, s)) under both readings of the configuration's
    N(0,2): s = 2 the standard deviation (adopted), s = sqrt 2 (variance 2)."""
    import torch

    from tensor_scaling_cast_gb300 import fp8q as F
    from tensor_scaling_cast_gb300 import synthetic as S
    res = {}
    for key, sigma in (("sigma_2", 2.0), ("sigma_sqrt2_variance_reading", math.sqrt(2.0))):
        x = S.mx_tanh(dev, sigma=sigma)
        r, c = x.shape
        out = {}
        for name, rule, h, axis in rules:
            q = torch.empty(r, c, dtype=torch.uint8, device=dev)
            e8 = torch.empty((r, c // 32) if axis == 0 else (r // 32, c), dtype=torch.uint8, device=dev)
            cl = torch.empty(1, dtype=torch.int64, device=dev)
            F.mx_cast_ex(x, F.E4M3, rule, h, axis, q, e8, cl)
            entry = {"clipped_fraction": int(cl.item()) / x.numel()}
            if axis == 0:
                st = torch.empty(3, dtype=torch.float64, device=dev)
                F.mx_error_stats(x, q, e8, F.E4M3, st)
                mse, bias, _ = st.cpu().tolist()
                entry.update(mse=mse, bias=bias)
            out[name] = entry
            del q, e8
        res[key] = out
        del x
    return res


def workload_results(kind: str, dev):
    """The quantities each configuration asks to report, computed with the
    library on fresh handles outside the timed region."""
    import torch

    from tensor_scaling_cast_gb300 import fp8q as F
    from tensor_scaling_cast_gb300 import synthetic as S

    def f32(t):
        return float(t.item())

    if kind == "current":
        x = S.current_4096(dev)
        g = F.ScaledCast(F.E4M3, 0, 0)
        q, sinv, amax, clipped = g(x)
        g.close()
        return {"amax": f32(amax), "scale": 1.0 / f32(sinv), "scale_inv": f32(sinv),
                "clipped": int(clipped.item()), "fp8_bytes_head": q[:8].cpu().tolist()}
    if kind == "spike":
        seq = [S.spike_step(t, dev) for t in range(S.SPIKE_STEPS)]
        n = seq[0].numel()
        out = {}
        for name, kw in (("most_recent_w1", dict(window=1)),
                         ("max_window_w16_m1", dict(window=16, margin=1)),
                         ("smoothed_a0.1", dict(window=0, estimator=1, alpha=0.1)),
                         ("smoothed_a0.5", dict(window=0, estimator=1, alpha=0.5)),
                         ("max_window_w16_interval4", dict(window=16, interval=4))):
            g = F.ScaledCast(F.E4M3, **kw)
            fr = []
            for x in seq:
                _, _, _, c = g(x)
                fr.append(int(c.item()) / n)
            g.close()
            out[name] = [round(v, 7) for v in fr]
        return {"clipped_fraction_per_step": out, "spike_step": S.SPIKE_STEP}
    if kind == "transpose":
        return None
    if kind == "mx":
        return {"mx_e4m3": mx_results(dev)}
    if kind in ("grad", "decoder"):
        if kind == "grad":
            xs = S.grad_group_step(1, dev)
            fmts = [F.E5M2] * len(xs)
        else:
            specs = S.decoder_tensor_specs()[:16]            # layer 0
            xs = [S.decoder_tensor(sp, 0, dev) for sp in specs]
            fmts = [sp[2] for sp in specs]
        hs = [F.fp8q_create(f, 16) for f in fmts]
        m = len(xs)
        res = []
        for step in range(2):
            qs = [torch.empty(x.numel(), dtype=torch.uint8, device=dev) for x in xs]
            cl, nf, uf = (torch.empty(m, dtype=torch.int64, device=dev) for _ in range(3))
            F.fp8q_cast_multi_ex(hs, xs, qs, None, None, cl, nf, uf)
            ntot = sum(x.numel() for x in xs)
            res.append({"clipped_fraction": int(cl.sum()) / ntot, "underflow_fraction": int(uf.sum()) / ntot,
                        "nonfinite": int(nf.sum())})
            del qs
        for h in hs:
            F.fp8q_destroy(h)
        scope = "64 gradient tensors" if kind == "grad" else "layer 0 (16 tensors)"
        out = {"scope": scope, "step0_current_scaling": res[0], "step1_max_window": res[1]}
        if kind == "decoder":
            out["mx_e4m3"] = mx_results(dev, (("ocp", 0, 0, 0), ("headroom1", 0, 1, 0)))
        return out
    return None


def copy_reference(dev, step_bytes: int):
    """Device-to-device copy on this GPU, timed the same way: the
    achievable-copy figure for this box (read + write bytes / time), and
    the dominant kernel's rate as a fraction of it."""
    import torch
    n = min(1 << 30, max(1 << 26, step_bytes // 4)) // 2      # bf16 elements per buffer
    a = torch.empty(n, dtype=torch.bfloat16, device=dev).fill_(1.0)
    b = torch.empty_like(a)
    for _ in range(3):
        b.copy_(a)
    torch.cuda.synchronize()
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        b.copy_(a)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    gbs = 2 * a.numel() * 2 / (ms * 1e-3) / 1e9
    del a, b
    torch.cuda.empty_cache()
    return {"GB/s": round(gbs, 1), "bytes": 4 * n, "how": "torch copy_ of a bf16 buffer, mean of 20"}


def pinned_bytes(W) -> int:
    """Host bytes one pinned copy of a step's inputs and outputs takes."""
    seen, total = set(), 0
    for p in W.parts:
        for t in list(p.inputs(0)) + list(p.outputs(0)):
            if id(t) not in seen:
                seen.add(id(t))
                total += t.numel() * t.element_size()
    return total


def host_memory_allows(need: int):
    """True when this rank's share of the available host memory (shared by
    the ranks on this node) holds `need` bytes with a 25% margin."""
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        return True, ""
    local = max(1, int(os.environ.get("LOCAL_WORLD_SIZE", "1")))
    share = avail // local
    if need * 1.25 <= share:
        return True, ""
    return False, (f"e2e needs {need / 1e9:.1f} GB of pinned host memory per rank; "
                   f"{share / 1e9:.1f} GB available per rank")


def run_e2e_zero_copy(args, world: int, dev, sigma: float = 2.0):
    """The same step with inputs and outputs in pinned host memory passed
    straight to the C ABI: the kernels read the inputs and write the
    results over NVLink-C2C, so each step moves the same host bytes.  Its
    own bytes and timing: h2d = the host-resident inputs the kernels read,
    d2h = the host-resident outputs they write (the per-tensor amax, scale
    and count arrays stay on the device)."""
    import torch
    W = Workload(args.workload, args.n, dev, host_io=True, single_dtype=args.single_dtype,
                 group_policies=args.group_policies, mx_sigma=sigma)
    seen = set()

    def host_bytes(ts):
        total = 0
        for t in ts:
            if t.device.type == "cpu" and id(t) not in seen:
                seen.add(id(t))
                total += t.numel() * t.element_size()
        return total
    h2d = host_bytes(t for p in W.parts for t in p.inputs(0))
    d2h = host_bytes(t for p in W.parts for t in p.outputs(0))
    for k in range(3):
        W.step(k)
    torch.cuda.synchronize()
    steps = max(2, args.e2e_steps)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for k in range(steps):
        W.step(3 + k)
    b.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    for p in W.handles:
        if hasattr(p, "close"):
            p.close()
    per = ms / steps
    return {"value": round(world * W.step_bytes / (per * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(per, 3), "steps": steps,
            "phases_ms": {"casts_over_host_link": round(per, 3)},
            "host_link_GBps": round((h2d + d2h) / (per * 1e-3) / 1e9, 1),
            "path": "pinned host buffers passed to the fp8q C ABI; kernels read and write them over NVLink-C2C (zero-copy)"}


def run_e2e(W, steps: int, world: int, dev, k0: int):
    """Same step through the public API with host buffers: pinned H2D of the
    step's inputs, the casts, D2H of every output, all inside the timed
    region."""
    import torch
    import torch.distributed as dist
    mirror = {}

    def host_of(t):
        if id(t) not in mirror:
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            mirror[id(t)] = h
        return mirror[id(t)]

    def io(k):
        ins, outs = [], []
        for p in W.parts:
            ins += [t for t in p.inputs(k) if id(t) not in {id(u) for u in ins}]
            outs += p.outputs(k)
        return ins, outs

    ins0, outs0 = io(k0)
    h2d = sum(t.numel() * t.element_size() for t in ins0)
    d2h = sum(t.numel() * t.element_size() for t in outs0)

    def one(k, ev=None):
        ins, outs = io(k)
        if ev is not None:
            ev[0].record()
        for t in ins:
            t.copy_(host_of(t), non_blocking=True)
        if ev is not None:
            ev[1].record()
        W.step(k)
        if ev is not None:
            ev[2].record()
        for t in outs:
            host_of(t).copy_(t, non_blocking=True)
        if ev is not None:
            ev[3].record()

    for k in range(k0, k0 + 2):
        one(k)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for k in range(steps):
        one(k0 + 2 + k, evs[k])
    b.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    phase = [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i in range(3)]
    return {"value": round(world * W.step_bytes / (ms / steps * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 3), "steps": steps,
            "phases_ms": {"h2d": round(phase[0], 3), "casts": round(phase[1], 3),
                          "d2h": round(phase[2], 3)},
            "h2d_GBps": round(h2d / (phase[0] * 1e-3) / 1e9, 1) if phase[0] > 0 else None,
            "d2h_GBps": round(d2h / (phase[2] * 1e-3) / 1e9, 1) if phase[2] > 0 else None,
            "path": "pinned host -> cudaMemcpyAsync -> fp8q C ABI -> cudaMemcpyAsync -> pinned host"}


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

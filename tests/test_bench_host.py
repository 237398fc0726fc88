"""Host-side logic of bench.py that needs no GPU: the reference arm (the CPU
oracle), its behaviour on non-zero ranks, and the max-over-ranks timing
reduction under a world_size-2 gloo process group."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "1", "--cpu-seconds", "0.3"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == os.cpu_count()
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"]
    import bench
    assert d["dtype"] == bench.DTYPE
    assert d["config"] == bench.decoder_config(1)      # the same config as our arm's line


def test_decoder_config_bytes_match_the_workload_definition():
    """384 tensors of 3 bytes per element (2 in, 1 out) plus the MX cast of
    bf16 [16384, 8192] at 3 + 1/32 bytes per element."""
    import bench
    from tensor_scaling_cast_gb300 import synthetic as S
    specs = S.decoder_tensor_specs()
    assert len(specs) == 384
    n = sum(r * c for _, (r, c), *_ in specs)
    assert n == 14_092_861_440
    assert bench.decoder_config(1)["bytes_per_step"] == 3 * n + 3 * 16384 * 8192 + 16384 * 8192 // 32
    assert bench.decoder_config(2)["parallelism"] == "replicas"


def test_reference_arm_other_ranks_do_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                          "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0 and out.stdout.strip() == ""


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
    q.put((rank, got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_input_digests_are_sha256_of_each_tensors_bytes():
    """inputs_sha256 of a bench line: the SHA-256 of each input tensor's raw
    bytes, keyed by the tensor's name (bf16 and fp32, one tensor larger
    than the 2^26-element hashing stride)."""
    import hashlib
    import types

    import bench
    g = torch.Generator().manual_seed(3)
    a = torch.randn(1000, generator=g).to(torch.bfloat16)
    b = torch.randn((1 << 26) + 7, generator=g)
    d = bench.input_digests(types.SimpleNamespace(named_inputs=[("a", a), ("b", b)]))
    assert d == {"a": hashlib.sha256(a.view(torch.int16).numpy().tobytes()).hexdigest(),
                 "b": hashlib.sha256(b.numpy().tobytes()).hexdigest()}


def test_lines_name_the_arithmetic_not_just_a_float_type():
    import bench
    assert "bf16" in bench.DTYPE and "fp8" in bench.DTYPE and "fp32" in bench.DTYPE

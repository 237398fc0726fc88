"""Casts and loss-scale updates captured into CUDA graphs (stream capture),
through the C ABI, against the CPU oracle.

A captured call records nothing on the device while the stream captures;
every replay of the graph must then advance the handles' device state as
the same eager call would: every output byte, amax, scale_inv, clipped
count and the final window of every handle equal the oracle's over the
whole sequence.  A handle's first cast under a window takes the
current-scaling path chosen on the host, so it is refused while capturing.
"""
import os
import warnings

import numpy as np
import pytest
import torch

from oracle import policy
from tensor_scaling_cast_gb300 import fp8q as F

pytestmark = pytest.mark.gpu

NT = os.cpu_count() or 1
EINVAL = -1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    from tensor_scaling_cast_gb300 import build
    build.build()
    F.load()
    torch.cuda.set_device(0)


def host_bits(x: torch.Tensor) -> np.ndarray:
    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return x.view(torch.int32).numpy().view(np.uint32).reshape(-1)


def f32bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32).reshape(-1)


def step_inputs(t: int, shapes, dtypes):
    """Seeded inputs of step t, one per tensor, with a x64 spike on every
    97th element at step 3 (so that windows, hysteresis-free rises and
    clipping all occur)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(7000 + t)
    out = []
    for i, (shape, dt) in enumerate(zip(shapes, dtypes)):
        x = torch.randn(shape, generator=g, device="cuda") * (2.0 ** (i - 1))
        if t == 3:
            x.view(-1)[::97] *= 64.0
        out.append(x.to(dt))
    return out


def test_graph_replays_advance_state_like_eager_calls():
    """A grouped cast captured once after the handles' first (eager) cast,
    then replayed for steps 1-6 on new inputs copied into the captured
    buffers: windows 4, 2, 16 and 0 (current scaling each call), margin 1,
    both formats, bf16 and fp32."""
    fmts = [0, 1, 0, 1]
    windows = [4, 2, 16, 0]
    shapes = [(256, 320), (1000,), (64, 64), (3000,)]
    dtypes = [torch.bfloat16, torch.float32, torch.bfloat16, torch.bfloat16]
    hs = [F.fp8q_create(f, w, 1, 0) for f, w in zip(fmts, windows)]
    orc = [policy.ScalingState(f, w, 1, 0) for f, w in zip(fmts, windows)]
    bufs = [torch.empty(sh, dtype=dt, device="cuda") for sh, dt in zip(shapes, dtypes)]
    qs = [torch.empty(b.numel(), dtype=torch.uint8, device="cuda") for b in bufs]
    n = len(hs)
    sinv = torch.empty(n, dtype=torch.float32, device="cuda")
    amax = torch.empty(n, dtype=torch.float32, device="cuda")
    clipped = torch.empty(n, dtype=torch.int64, device="cuda")

    def load_step(t):
        for b, x in zip(bufs, step_inputs(t, shapes, dtypes)):
            b.copy_(x)

    def check(t):
        sb, ab, cb = f32bits(sinv), f32bits(amax), clipped.cpu().numpy()
        for i, b in enumerate(bufs):
            q_o, a_o, s_o, c_o, _ = orc[i].step(host_bits(b), NT)
            assert np.array_equal(qs[i].cpu().numpy(), q_o.reshape(-1)), (t, i)
            assert ab[i] == a_o and sb[i] == s_o and int(cb[i]) == c_o, (t, i)

    load_step(0)
    F.fp8q_cast_multi(hs, bufs, qs, sinv, amax, clipped)
    torch.cuda.synchronize()
    check(0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        F.fp8q_cast_multi(hs, bufs, qs, sinv, amax, clipped)
    # capturing ran nothing: the state is still the one after step 0
    assert [F.fp8q_scale_state(h)[1] for h in hs] == [1] * n
    for t in range(1, 7):
        load_step(t)
        graph.replay()
        torch.cuda.synchronize()
        check(t)
    # host reads of the state work after the replays
    for h, o in zip(hs, orc):
        assert F.fp8q_scale_state(h) == (o.prev_e, o.steps)
        hist = F.fp8q_amax_history(h, max(1, o.window))
        assert [int(np.float32(v).view(np.uint32)) for v in hist] == o.hist
        F.fp8q_destroy(h)


def test_graph_capture_refuses_a_first_windowed_cast():
    """The first cast of a window-4 handle under capture returns
    FP8Q_EINVAL and enqueues nothing; the same cast made eagerly afterwards
    is still the handle's first (current scaling)."""
    h = F.fp8q_create(0, 4, 0, 0)
    x = torch.randn(4096, device="cuda").to(torch.bfloat16)
    q = torch.empty(4096, dtype=torch.uint8, device="cuda")
    lib = F.load()
    graph = torch.cuda.CUDAGraph()
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")        # torch may note that the captured graph is empty
        with torch.cuda.graph(graph):
            st = lib.fp8q_cast(h, x.data_ptr(), F.BF16, x.numel(), q.data_ptr(), None, None, None,
                               torch.cuda.current_stream().cuda_stream)
    assert st == EINVAL
    assert F.fp8q_scale_state(h)[1] == 0
    sinv = torch.empty(1, dtype=torch.float32, device="cuda")
    F.fp8q_cast(h, x, q, sinv)
    torch.cuda.synchronize()
    o = policy.ScalingState(0, 4, 0, 0)
    q_o, _, s_o, _, _ = o.step(host_bits(x), NT)
    assert np.array_equal(q.cpu().numpy(), q_o.reshape(-1))
    assert f32bits(sinv)[0] == s_o
    assert F.fp8q_scale_state(h) == (o.prev_e, 1)
    F.fp8q_destroy(h)


def test_graph_replays_of_the_loss_scaler():
    """One loss-scale update captured once and replayed 12 times on
    non-finite counts rewritten before each replay: the scale, the skip
    flag and the clean-step count follow the oracle's state machine."""
    rng = np.random.default_rng(91)
    ls = F.fp8q_loss_scaler_create(1024.0, 3, 1.0, 2.0 ** 24)
    o = policy.LossScaler(1024.0, 3, 1.0, 2.0 ** 24)
    counts = torch.zeros(5, dtype=torch.int64, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    skip = torch.empty(1, dtype=torch.int32, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        F.fp8q_loss_scaler_update(ls, counts, scale, skip)
    for t in range(12):
        host = (rng.random(5) < 0.1).astype(np.int64) * rng.integers(1, 9, 5)
        counts.copy_(torch.from_numpy(host))
        graph.replay()
        torch.cuda.synchronize()
        want_skip = o.update(host.tolist())
        assert (float(scale.item()), bool(skip.item())) == (float(o.scale), want_skip), t
    assert F.fp8q_loss_scaler_read(ls) == (float(o.scale), o.good)
    F.fp8q_loss_scaler_destroy(ls)

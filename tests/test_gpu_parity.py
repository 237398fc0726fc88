"""Parity of the sm_103a kernels (through the C ABI) with the CPU oracle.

Bar: bit-exact for FP8 bytes, E8M0 bytes, amax, scale_inv and clipped counts;
error statistics (MSE and bias) within 1e-6 relative of the oracle's fp64
values.  Inputs come from the seeded generators; the oracle receives the
same bytes copied to the host.  Every output buffer handed to the library
carries guard bands (tests/canary.py) that must be intact after the call.
"""
import os

import numpy as np
import pytest
import torch

from canary import Guards
from oracle import coracle, policy
from tensor_scaling_cast_gb300 import fp8q as F
from tensor_scaling_cast_gb300 import synthetic

pytestmark = pytest.mark.gpu

G = Guards()

NT = os.cpu_count() or 1
EMAX = {0: 8, 1: 15}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the gpu tests")
    from tensor_scaling_cast_gb300 import build
    build.build()
    F.load()
    torch.cuda.set_device(0)


@pytest.fixture(autouse=True)
def _guards():
    G.release()
    yield
    G.check_and_release("at the end of the test")


def rel_close(got: float, want: float, tol: float = 1e-6) -> bool:
    """|got - want| <= tol * |want|; an exact zero must be matched exactly."""
    return abs(got - want) <= tol * abs(want)


def cast_guarded(g, x):
    """fp8q_cast through handle g into guarded outputs; returns (q, scale_inv,
    amax, clipped) once the guard bands are checked."""
    q = G.empty(x.shape, torch.uint8)
    sinv = G.empty(1, torch.float32)
    amax = G.empty(1, torch.float32)
    clipped = G.empty(1, torch.int64)
    F.fp8q_cast(g.handle, x, q, sinv, amax, clipped)
    G.check("after fp8q_cast")
    return q, sinv, amax, clipped


def host_bits(x: torch.Tensor) -> np.ndarray:
    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return x.view(torch.int32).numpy().view(np.uint32).reshape(-1)


def f32bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32).reshape(-1)


def from_bits(bits: np.ndarray, dtype) -> torch.Tensor:
    if dtype == torch.bfloat16:
        return torch.from_numpy(bits.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(bits.astype(np.uint32).view(np.int32).copy()).view(torch.float32)


def set_exponent(h: int, fmt: int, e: int):
    """Plant a one-entry window whose maximum makes the rule choose e."""
    F.fp8q_set_history(h, [float(2.0 ** (EMAX[fmt] - e))], None)


# ---------------------------------------------------------------------------
# the conversion itself, through the full kernel path
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [0, 1])
def test_every_bf16_pattern_every_scale(fmt):
    """All 65,536 bf16 bit patterns (zeros, subnormals, Inf, NaN included),
    four copies so the launch spans several chunks, at exponents covering the
    reachable range: bytes, amax, scale_inv and clipped count exact."""
    bits = np.tile(np.arange(65536, dtype=np.uint32).astype(np.uint16), 4)
    x = from_bits(bits, torch.bfloat16).cuda()
    h = F.fp8q_create(fmt, 1, 0, 0)
    q = G.empty(x.numel(), torch.uint8)
    out = G.empty(2, torch.float32)
    clipped = G.empty(1, torch.int64)
    lo = EMAX[fmt] - 127
    for e in sorted(set(list(range(lo, 127, 7)) + [lo, lo + 1, -1, 0, 1, 125, 126])):
        set_exponent(h, fmt, e)
        F.fp8q_cast(h, x, q, out[0:1], out[1:2], clipped)
        G.check(f"e={e}")
        q_o, a_o, c_o = coracle.cast(bits, fmt, e, NT)
        got = q.cpu().numpy()
        bad = np.nonzero(got != q_o)[0]
        assert bad.size == 0, (e, [(hex(int(bits[i])), hex(int(got[i])), hex(int(q_o[i]))) for i in bad[:8]])
        assert f32bits(out)[0] == np.float32(2.0 ** -e).view(np.uint32)
        assert f32bits(out)[1] == a_o
        assert int(clipped.item()) == c_o
    F.fp8q_destroy(h)


@pytest.mark.parametrize("fmt", [0, 1])
def test_random_fp32_patterns(fmt):
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=(1 << 20) + 5, dtype=np.uint64).astype(np.uint32)
    x = from_bits(bits, torch.float32).cuda()
    h = F.fp8q_create(fmt, 1, 0, 0)
    q = G.empty(x.numel(), torch.uint8)
    clipped = G.empty(1, torch.int64)
    for e in (EMAX[fmt] - 127, -60, -3, 0, 17, 90, 126):
        set_exponent(h, fmt, e)
        F.fp8q_cast(h, x, q, None, None, clipped)
        G.check(f"e={e}")
        q_o, _, c_o = coracle.cast(bits, fmt, e, NT)
        assert np.array_equal(q.cpu().numpy(), q_o), e
        assert int(clipped.item()) == c_o
    F.fp8q_destroy(h)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def run_steps(g, orc_state, xs):
    """Cast a sequence through one handle (a ScaledCast) and the oracle;
    compare all."""
    records = []
    for t, x in enumerate(xs):
        q, sinv, amax, clipped = cast_guarded(g, x)
        q_o, a_o, s_o, c_o, e_o = orc_state.step(host_bits(x), NT)
        assert np.array_equal(q.cpu().numpy().reshape(-1), q_o.reshape(-1)), f"bytes differ at step {t}"
        assert f32bits(amax)[0] == a_o, t
        assert f32bits(sinv)[0] == s_o, t
        assert int(clipped.item()) == c_o, t
        records.append((e_o, c_o))
        G.release()
    return records


def test_current_scaling_4096_fp32():
    x = synthetic.current_4096("cuda")
    g = F.ScaledCast(F.E4M3, window=0, margin=0)
    o = policy.ScalingState(0, window=0, margin=0)
    recs = run_steps(g, o, [x, x * 3.0, x * 1e-3])
    assert all(c == 0 for _, c in recs)             # current scaling never clips
    g.close()


@pytest.mark.parametrize("window,margin", [(1, 0), (16, 1)])
def test_spike_sequence(window, margin):
    """16 steps of bf16 4096x4096 with a x8 spike on 0.1% of step 9."""
    g = F.ScaledCast(F.E4M3, window=window, margin=margin)
    o = policy.ScalingState(0, window=window, margin=margin)
    xs = (synthetic.spike_step(s, "cuda") for s in range(synthetic.SPIKE_STEPS))
    recs = run_steps(g, o, xs)
    clipped = [c for _, c in recs]
    if window == 1:
        assert clipped[synthetic.SPIKE_STEP] > 0
    hist = g.history()
    assert [np.float32(v).view(np.uint32) for v in hist] == o.hist
    assert g.state() == (o.prev_e, 16)
    g.close()


def run_group_steps(fmts, windows, xs_steps, margin=0, hyst=0, names=None):
    """One fp8q_cast_multi per step over all tensors, every output byte,
    amax, scale_inv and clipped count of every step compared with the
    oracle, then the final window and exponent of every handle."""
    hs = [F.fp8q_create(f, w, margin, hyst) for f, w in zip(fmts, windows)]
    orc = [policy.ScalingState(f, w, margin, hyst) for f, w in zip(fmts, windows)]
    n = len(hs)
    names = names or list(range(n))
    for t, xs in enumerate(xs_steps):
        qs = [G.empty(x.numel(), torch.uint8) for x in xs]
        sinv = G.empty(n, torch.float32)
        amax = G.empty(n, torch.float32)
        clipped = G.empty(n, torch.int64)
        F.fp8q_cast_multi(hs, xs, qs, sinv, amax, clipped)
        G.check(f"step {t}")
        sb, ab, cb = f32bits(sinv), f32bits(amax), clipped.cpu().numpy()
        for i, x in enumerate(xs):
            q_o, a_o, s_o, c_o, e_o = orc[i].step(host_bits(x), NT)
            assert np.array_equal(qs[i].cpu().numpy(), q_o.reshape(-1)), (t, names[i])
            assert ab[i] == a_o and sb[i] == s_o and int(cb[i]) == c_o, (t, names[i])
        G.release()
        del qs, xs
        torch.cuda.empty_cache()
    for h, o, nm in zip(hs, orc, names):
        assert F.fp8q_scale_state(h) == (o.prev_e, o.steps), nm
        hist = F.fp8q_amax_history(h, max(1, o.window))
        assert [int(np.float32(v).view(np.uint32)) for v in hist] == o.hist, nm
        F.fp8q_destroy(h)


def test_two_streams_with_distinct_handles():
    """Two groups of handles cast on two streams with no ordering between
    them, four steps each (the launches may overlap on the GPU): every byte,
    amax, scale_inv and clipped count of both groups equal the oracle's."""
    specs = synthetic.decoder_tensor_specs(layers=1, hidden=256, ffn=1024, tokens=512)
    groups = [specs[0::2], specs[1::2]]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    hs = [[F.fp8q_create(sp[2], 4, 0, 0) for sp in grp] for grp in groups]
    orc = [[policy.ScalingState(sp[2], 4, 0, 0) for sp in grp] for grp in groups]
    for t in range(4):
        xs = [[synthetic.decoder_tensor(sp, t, "cuda") for sp in grp] for grp in groups]
        torch.cuda.synchronize()
        outs = []
        for gi, st in enumerate(streams):
            n = len(groups[gi])
            qs = [G.empty(x.numel(), torch.uint8) for x in xs[gi]]
            o = (G.empty(n, torch.float32), G.empty(n, torch.float32), G.empty(n, torch.int64))
            torch.cuda.synchronize()             # the guard fills are done before either stream starts
            outs.append((qs, o))
        for gi, st in enumerate(streams):
            qs, o = outs[gi]
            F.fp8q_cast_multi(hs[gi], xs[gi], qs, *o, stream=st)
        torch.cuda.synchronize()
        G.check(f"step {t}")
        for gi in range(2):
            qs, (sinv, amax, clipped) = outs[gi]
            sb, ab, cb = f32bits(sinv), f32bits(amax), clipped.cpu().numpy()
            for i, x in enumerate(xs[gi]):
                q_o, a_o, s_o, c_o, _ = orc[gi][i].step(host_bits(x), NT)
                assert np.array_equal(qs[i].cpu().numpy(), q_o.reshape(-1)), (t, gi, i)
                assert ab[i] == a_o and sb[i] == s_o and int(cb[i]) == c_o, (t, gi, i)
        G.release()
    for gi in range(2):
        for h, o in zip(hs[gi], orc[gi]):
            assert F.fp8q_scale_state(h) == (o.prev_e, o.steps)
            F.fp8q_destroy(h)


def test_grad_group_reduced_sizes():
    """64 gradient-like bf16 tensors (sides 64..512) -> E5M2, window 16, one
    grouped launch per step, 4 steps (step 0 is current scaling)."""
    steps = [synthetic.grad_group_step(s, "cuda", sides=(64, 128, 256, 512)) for s in range(4)]
    run_group_steps([1] * 64, [16] * 64, steps)


def test_grad_group_full_size_sixteen_steps():
    """The full 64-tensor group (sides 1024..8192, ~9.4e8 elements per
    step) over its whole 16-step sequence, one grouped launch per step:
    step 0 is current scaling, steps 1-15 fill the window-16 ring with 1-15
    entries; every byte, amax, scale_inv and clipped count of every step
    and the final ring of every handle compared."""
    hs_steps = (synthetic.grad_group_step(s, "cuda") for s in range(16))
    run_group_steps([1] * 64, [16] * 64, hs_steps)


def test_decoder_reduced_sizes():
    """Every weight / activation / gradient of a 2-layer decoder at reduced
    widths, E4M3 + E5M2 mixed in one launch, window 16, 8 steps."""
    sizes = dict(layers=2, hidden=256, ffn=1024, tokens=512)
    specs = synthetic.decoder_tensor_specs(**sizes)
    steps = ([synthetic.decoder_tensor(sp, s, "cuda") for sp in specs] for s in range(8))
    run_group_steps([sp[2] for sp in specs], [16] * len(specs), steps)


def test_decoder_full_size_eight_steps():
    """The benchmark's workload at full size and in its launch
    configuration: all 384 tensors of the 24-layer decoder (14,092,861,440
    elements per step) in one fp8q_cast_multi call per step, all 8 steps:
    step 0 (empty history: current scaling with the pre-pass), steps 1-7
    (max-window over 1-7 ring entries); every byte, amax, scale_inv and
    clipped count of every tensor and step, then every handle's ring and
    exponent, compared with the oracle."""
    specs = synthetic.decoder_tensor_specs()
    steps = ([synthetic.decoder_tensor(sp, step, "cuda") for sp in specs] for step in range(8))
    run_group_steps([sp[2] for sp in specs], [16] * len(specs), steps, names=[sp[0] for sp in specs])


@pytest.mark.parametrize("headroom", [0, 1])
def test_mx_tanh_full_size(headroom):
    """bf16 [16384, 8192] tanh(N(0,2)) -> MX E4M3: every element byte, every
    E8M0 byte, the clipped count; then the error statistics."""
    x = synthetic.mx_tanh("cuda")
    rows, cols = x.shape
    q = G.empty((rows, cols), torch.uint8)
    e8 = G.empty((rows, cols // 32), torch.uint8)
    cl = G.empty(1, torch.int64)
    F.mx_cast(x, F.E4M3, headroom, q, e8, cl)
    G.check()
    xb = host_bits(x).reshape(rows, cols)
    q_o, e8_o, c_o = coracle.mx_cast(xb, 0, headroom, NT)
    assert np.array_equal(e8.cpu().numpy(), e8_o)
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert int(cl.item()) == c_o
    if headroom == 1:
        assert c_o == 0
    out = G.empty(3, torch.float64)
    F.mx_error_stats(x, q, e8, F.E4M3, out)
    G.check("after mx_error_stats")
    mse, bias, n = out.cpu().tolist()
    mse_o, bias_o, n_o = coracle.mx_stats(xb, q_o, e8_o, 0, NT)
    assert int(n) == n_o
    assert rel_close(mse, mse_o), (mse, mse_o)
    assert rel_close(bias, bias_o), (bias, bias_o)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_edge_values(fmt, dtype):
    """Zero blocks, NaN / Inf blocks, subnormal and huge blocks, ragged row
    counts, fp32 and bf16, both formats, headroom 0..2."""
    rng = np.random.default_rng(41)
    rows, cols = 37, 96
    v = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-40, 40, size=(rows, 1)))
    v[0, :32] = 0.0
    v[0, 5] = -0.0
    v[1, 7] = np.nan
    v[2, 40] = -np.inf
    v[3, :] *= 1e-38
    v[4, 64:] = 3e38
    x = torch.from_numpy(v.astype(np.float32)).to(dtype).cuda()
    xb = host_bits(x).reshape(rows, cols)
    for h in (0, 1, 2):
        q = G.empty((rows, cols), torch.uint8)
        e8 = G.empty((rows, cols // 32), torch.uint8)
        cl = G.empty(1, torch.int64)
        F.mx_cast(x, fmt, h, q, e8, cl)
        G.check(f"headroom {h}")
        q_o, e8_o, c_o = coracle.mx_cast(xb, fmt, h)
        assert np.array_equal(e8.cpu().numpy(), e8_o), h
        assert np.array_equal(q.cpu().numpy(), q_o), h
        assert int(cl.item()) == c_o


def _mx_ex_gpu(x, fmt, rule, headroom, axis):
    rows, cols = x.shape
    q = G.empty((rows, cols), torch.uint8)
    e8 = G.empty((rows, cols // 32) if axis == 0 else (rows // 32, cols), torch.uint8)
    cl = G.empty(1, torch.int64)
    F.mx_cast_ex(x, fmt, rule, headroom, axis, q, e8, cl)
    G.check(f"mx_cast_ex fmt={fmt} rule={rule} h={headroom} axis={axis}")
    out = q.cpu().numpy(), e8.cpu().numpy(), int(cl.item())
    G.release()
    return out


@pytest.mark.parametrize("rule,axis", [(1, 0), (2, 0), (0, 1), (1, 1), (2, 1)])
def test_mx_rules_and_axes_full_size(rule, axis):
    """bf16 [16384, 8192] tanh(N(0,2)) -> MX E4M3 under the round-up (ceil)
    and nearest scale rules, row-wise and column-wise 32-blocks."""
    x = synthetic.mx_tanh("cuda")
    xb = host_bits(x).reshape(x.shape)
    q, e8, cl = _mx_ex_gpu(x, 0, rule, 0, axis)
    q_o, e8_o, c_o = coracle.mx_cast_ex(xb, 0, rule, 0, axis, NT)
    assert np.array_equal(e8, e8_o)
    assert np.array_equal(q, q_o)
    assert cl == c_o
    if rule == 1:
        assert c_o == 0                  # rounding the scale up never clips


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_ex_edge_values(dtype):
    """Every rule and direction, both formats, headroom 0..2, on a tensor with
    zero / NaN / Inf / subnormal / huge blocks and a ragged column tile."""
    rng = np.random.default_rng(43)
    rows, cols = 96, 320          # 320 = 256 + 64: a ragged column tile
    v = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-40, 40, size=(rows, 1)))
    v[:, 5] *= np.exp(rng.uniform(-30, 30))
    v[0:32, 0] = 0.0
    v[0, :32] = 0.0
    v[1, 7] = np.nan
    v[40, 40] = -np.inf
    v[3, :] *= 1e-38
    v[4, 64:] = 3e38
    x = torch.from_numpy(v.astype(np.float32)).to(dtype).cuda()
    xb = host_bits(x).reshape(rows, cols)
    for fmt in (0, 1):
        for rule in (0, 1, 2):
            for axis in (0, 1):
                for h in (0, 2):
                    q, e8, cl = _mx_ex_gpu(x, fmt, rule, h, axis)
                    q_o, e8_o, c_o = coracle.mx_cast_ex(xb, fmt, rule, h, axis)
                    assert np.array_equal(e8, e8_o), (fmt, rule, axis, h)
                    assert np.array_equal(q, q_o), (fmt, rule, axis, h)
                    assert cl == c_o, (fmt, rule, axis, h)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_colwise_ragged_and_offset(dtype):
    """Column-wise blocks with cols % 64 == 16 (a last sub-tile holding 16
    valid columns), a 16-column tensor, q 16-byte but not 32-byte aligned
    and E8M0 at an odd address."""
    rng = np.random.default_rng(44)
    for rows, cols in ((64, 336), (96, 16)):
        v = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-20, 20, size=(1, cols)))
        v[2, cols - 1] = np.nan
        v[33, 0] = np.inf
        x = torch.from_numpy(v.astype(np.float32)).to(dtype).cuda()
        xb = host_bits(x).reshape(rows, cols)
        q = G.empty((rows, cols), torch.uint8, offset=16)
        e8 = G.empty((rows // 32, cols), torch.uint8, offset=1)
        cl = G.empty(1, torch.int64)
        for fmt in (0, 1):
            for rule in (0, 1):
                F.mx_cast_ex(x, fmt, rule, 0, 1, q, e8, cl)
                G.check(f"{rows}x{cols} fmt={fmt} rule={rule}")
                q_o, e8_o, c_o = coracle.mx_cast_ex(xb, fmt, rule, 0, 1)
                assert np.array_equal(e8.cpu().numpy(), e8_o), (rows, cols, fmt, rule)
                assert np.array_equal(q.cpu().numpy(), q_o), (rows, cols, fmt, rule)
                assert int(cl.item()) == c_o, (rows, cols, fmt, rule)


def test_mx_ex_argument_checks():
    x = torch.zeros(48, 64, dtype=torch.bfloat16, device="cuda")
    q = G.empty((48, 64), torch.uint8)
    e8 = G.empty((2, 64), torch.uint8)
    with pytest.raises(F.Fp8qError):
        F.mx_cast_ex(x, 0, 0, 0, 1, q, e8)          # rows not a multiple of 32
    with pytest.raises(F.Fp8qError):
        F.mx_cast_ex(x[:32], 0, 3, 0, 0, q, e8)     # unknown rule


# ---------------------------------------------------------------------------
# edge cases of the per-tensor path
# ---------------------------------------------------------------------------

SIZES = [0, 1, 15, 16, 17, 31, 33, 4095, 4096, 4097, 8191, 8192, 8193, 16383, 16384, 16385, 65537,
         (1 << 20) + 3]


def _special_tensor(n, dtype, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(n) * np.exp(rng.uniform(-5, 5))
    if n > 20:
        v[3] = -0.0
        v[7] = 0.0
        v[11] = 1e-42
        v[13] = -1e-45
    return torch.from_numpy(v.astype(np.float32)).to(dtype).cuda()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("window", [0, 3])
def test_sizes_and_special_values(dtype, window):
    """Empty, tiny, ragged and chunk-boundary sizes; current scaling in one
    CTA and with the pre-pass; delayed steps; signed zeros, subnormals."""
    for fmt in (0, 1):
        for n in SIZES:
            g = F.ScaledCast(fmt, window=window, margin=1 if window else 0)
            o = policy.ScalingState(fmt, window=window, margin=1 if window else 0)
            xs = [_special_tensor(n, dtype, 100 + n + k) * (4.0 ** k) for k in range(3)]
            run_steps(g, o, xs)
            g.close()


def test_nonfinite_inputs():
    """NaN and Inf in the tensor: NaN -> sign|0x7F, Inf saturates and counts,
    amax becomes NaN, the next exponent is kept."""
    for dtype in (torch.bfloat16, torch.float32):
        for fmt in (0, 1):
            g = F.ScaledCast(fmt, window=2)
            o = policy.ScalingState(fmt, window=2)
            base = _special_tensor(50000, dtype, 7)
            a = base.clone()
            a[100] = float("inf")
            a[200] = float("-inf")
            b = base.clone()
            b[300] = float("nan")
            b[301] = -float("nan")
            run_steps(g, o, [base, a, b, base, base])
            g.close()


def test_hysteresis_sequence():
    rng = np.random.default_rng(9)
    xs = [torch.from_numpy((rng.standard_normal(30000) * s).astype(np.float32)).cuda()
          for s in (1, 0.5, 0.26, 0.1, 0.05, 1, 3, 0.2)]
    for h in (1, 2):
        g = F.ScaledCast(0, window=1, hysteresis=h)
        o = policy.ScalingState(0, window=1, hysteresis=h)
        run_steps(g, o, xs)
        g.close()


def test_group_over_512_tensors_mixed():
    """600 tensors of mixed size / dtype / format / window (two launches),
    several steps."""
    rng = np.random.default_rng(17)
    cnt = 600
    fmts = [int(f) for f in rng.integers(0, 2, cnt)]
    wins = [int(w) for w in rng.integers(0, 5, cnt)]
    sizes = [int(s) for s in rng.choice([1, 17, 1000, 8192, 16385, 40000], cnt)]
    dts = [torch.bfloat16 if rng.integers(0, 2) else torch.float32 for _ in range(cnt)]
    steps = [[_special_tensor(n, d, 1000 * s + i) for i, (n, d) in enumerate(zip(sizes, dts))]
             for s in range(3)]
    run_group_steps(fmts, wins, steps)


def test_resume_equals_continuous():
    """16 steps straight == 8 steps, save history + exponent, restore into a
    fresh handle, 8 more steps (byte for byte)."""
    xs = [synthetic.spike_step(s, "cuda", shape=(512, 1024)) for s in range(16)]
    a = F.ScaledCast(0, window=4, margin=1)
    full = [cast_guarded(a, x)[0].cpu() for x in xs]
    b = F.ScaledCast(0, window=4, margin=1)
    part = [cast_guarded(b, x)[0].cpu() for x in xs[:8]]
    saved, (prev_e, _) = b.history(), b.state()
    c = F.ScaledCast(0, window=4, margin=1)
    c.set_history(saved, prev_e)
    part += [cast_guarded(c, x)[0].cpu() for x in xs[8:]]
    assert all(torch.equal(u, v) for u, v in zip(full, part))
    for g in (a, b, c):
        g.close()


@pytest.mark.parametrize("estimator,alpha,interval,window", [
    (1, 0.5, 1, 0), (1, 0.1, 1, 4), (1, 1.0, 1, 0), (0, 1.0, 3, 1), (0, 1.0, 4, 16), (1, 0.25, 2, 2)])
def test_estimators_on_spike_sequence(estimator, alpha, interval, window):
    """Exponential smoothing and the recompute interval on the spike
    sequence (bf16 [2048, 2048], x8 spike at step 9), every step compared."""
    g = F.ScaledCast(F.E4M3, window, 0, 0, estimator=estimator, alpha=alpha, interval=interval)
    o = policy.ScalingState(0, window, 0, 0, estimator=estimator, alpha=alpha, interval=interval)
    xs = [synthetic.spike_step(s, "cuda", shape=(2048, 2048)) for s in range(16)]
    run_steps(g, o, xs)
    avg, steps = F.fp8q_get_estimator_state(g.handle)
    assert steps == 16
    if estimator == 1:
        assert np.float32(avg) == o.avg
    g.close()


def test_estimators_mixed_in_one_group():
    """One grouped launch holding max-window, smoothed and interval handles."""
    rng = np.random.default_rng(19)
    cfg = [(0, 16, 0, 1.0, 1), (1, 0, 1, 0.3, 1), (0, 1, 0, 1.0, 3), (1, 4, 1, 0.5, 2)] * 5
    hs = [F.fp8q_create_ex(f, w, 0, 0, est, a, k) for f, w, est, a, k in cfg]
    orc = [policy.ScalingState(f, w, 0, 0, estimator=est, alpha=a, interval=k) for f, w, est, a, k in cfg]
    for t in range(6):
        xs = [_special_tensor(int(n), torch.bfloat16, 100 * t + i) * float(np.exp(rng.uniform(-3, 3)))
              for i, n in enumerate(rng.choice([100, 8192, 20000, 70000], len(cfg)))]
        qs = [G.empty(x.numel(), torch.uint8) for x in xs]
        sinv = G.empty(len(cfg), torch.float32)
        amax = G.empty(len(cfg), torch.float32)
        clipped = G.empty(len(cfg), torch.int64)
        F.fp8q_cast_multi(hs, xs, qs, sinv, amax, clipped)
        G.check(f"step {t}")
        sb, ab, cb = f32bits(sinv), f32bits(amax), clipped.cpu().numpy()
        for i, x in enumerate(xs):
            q_o, a_o, s_o, c_o, _ = orc[i].step(host_bits(x), NT)
            assert np.array_equal(qs[i].cpu().numpy(), q_o.reshape(-1)), (t, i)
            assert (ab[i], sb[i], int(cb[i])) == (a_o, s_o, c_o), (t, i)
    for h in hs:
        F.fp8q_destroy(h)


@pytest.mark.parametrize("order", ["history_first", "estimator_first"])
def test_estimator_resume_equals_continuous(order):
    """Smoothed estimator with interval 3: 12 casts straight == 5 casts,
    save (history, exponent, average, steps), restore into a fresh handle
    in either order of the two restore calls, 7 casts -- byte for byte,
    and the restored handle ends in the continuous run's state."""
    xs = [synthetic.spike_step(s, "cuda", shape=(256, 1024)) for s in range(12)]
    kw = dict(estimator=1, alpha=0.3, interval=3)
    a = F.ScaledCast(0, 4, 0, 0, **kw)
    full = [cast_guarded(a, x)[0].cpu() for x in xs]
    b = F.ScaledCast(0, 4, 0, 0, **kw)
    part = [cast_guarded(b, x)[0].cpu() for x in xs[:5]]
    hist, (prev_e, _) = b.history(), b.state()
    avg, steps = F.fp8q_get_estimator_state(b.handle)
    c = F.ScaledCast(0, 4, 0, 0, **kw)
    if order == "history_first":
        c.set_history(hist, prev_e)
        F.fp8q_set_estimator_state(c.handle, avg, steps)
    else:
        F.fp8q_set_estimator_state(c.handle, avg, steps)
        c.set_history(hist, prev_e)
    assert F.fp8q_get_estimator_state(c.handle) == (avg, steps)
    assert c.state() == (prev_e, steps)
    part += [cast_guarded(c, x)[0].cpu() for x in xs[5:]]
    assert all(torch.equal(u, v) for u, v in zip(full, part))
    assert F.fp8q_get_estimator_state(c.handle) == F.fp8q_get_estimator_state(a.handle)
    assert c.history() == a.history() and c.state() == a.state()
    for g in (a, b, c):
        g.close()


def test_reset_clears_estimator_state():
    """fp8q_reset returns a handle to its state after fp8q_create: empty
    window, no previous exponent, no running average, zero casts."""
    g = F.ScaledCast(0, 4, 0, 0, estimator=1, alpha=0.5, interval=2)
    for s in range(3):
        cast_guarded(g, synthetic.spike_step(s, "cuda", shape=(64, 256)))
    assert F.fp8q_get_estimator_state(g.handle)[1] == 3
    g.reset()
    assert F.fp8q_get_estimator_state(g.handle) == (None, 0)
    assert g.state() == (None, 0) and g.history() == []
    g.close()


def _counted_group_step(hs, xs, underflow=True):
    n = len(hs)
    qs = [G.empty(x.numel(), torch.uint8) for x in xs]
    outs = [G.empty(n, torch.float32) for _ in range(2)]
    cl = G.empty(n, torch.int64)
    nf = G.full(n, -1, torch.int64)
    uf = G.full(n, -1, torch.int64) if underflow else None
    F.fp8q_cast_multi_ex(hs, xs, qs, outs[0], outs[1], cl, nf, uf)
    G.check("after fp8q_cast_multi_ex")
    return qs, outs, cl, nf, uf


def test_nonfinite_and_underflow_counts():
    """Per-tensor counts of NaN/Inf inputs and of finite nonzero inputs cast
    to zero, against the oracle, for both formats and dtypes, sizes across
    chunk boundaries; the bytes equal those of the launch without the
    underflow count."""
    rng = np.random.default_rng(61)
    specs = [(f, dt, n) for f in (0, 1) for dt in (torch.bfloat16, torch.float32)
             for n in (1, 100, 8193, 70001)]
    hs = [F.fp8q_create(f, 2) for f, _, _ in specs]
    hs2 = [F.fp8q_create(f, 2) for f, _, _ in specs]
    orc = [policy.ScalingState(f, 2) for f, _, _ in specs]
    for t in range(3):
        xs = []
        for i, (f, dt, n) in enumerate(specs):
            v = rng.standard_normal(n) * np.exp(rng.uniform(-30, 3, n))
            if n > 50:
                v[rng.integers(0, n, 5)] = np.nan
                v[rng.integers(0, n, 3)] = np.inf
                v[rng.integers(0, n, 7)] = 0.0
            xs.append(torch.from_numpy(v.astype(np.float32)).to(dt).cuda())
        qs, outs, cl, nf, uf = _counted_group_step(hs, xs, True)
        qs2, _, _, nf2, _ = _counted_group_step(hs2, xs, False)
        for i, x in enumerate(xs):
            q_o, a_o, s_o, c_o, _ = orc[i].step(host_bits(x), NT)
            assert np.array_equal(qs[i].cpu().numpy(), q_o), (t, i)
            assert torch.equal(qs[i], qs2[i])
            nf_o, uf_o = coracle.count_special(host_bits(x), q_o)
            assert (int(nf[i]), int(uf[i]), int(nf2[i])) == (nf_o, uf_o, nf_o), (t, i)
    for h in hs + hs2:
        F.fp8q_destroy(h)


def test_underflow_count_full_size_gradients():
    """Gradient-like tensors (magnitudes spread over 1e-8..1e2) underflow a
    lot under E5M2 with a max-window scale: counts exact at full size."""
    xs = synthetic.grad_group_step(2, "cuda")[:8]
    hs = [F.fp8q_create(1, 16) for _ in xs]
    orc = [policy.ScalingState(1, 16) for _ in xs]
    for t in range(2):
        qs, outs, cl, nf, uf = _counted_group_step(hs, xs, True)
        for i, x in enumerate(xs):
            q_o, *_ = orc[i].step(host_bits(x), NT)
            assert np.array_equal(qs[i].cpu().numpy(), q_o.reshape(-1))
            assert (int(nf[i]), int(uf[i])) == coracle.count_special(host_bits(x), q_o)
    assert int(uf.sum()) > 0
    for h in hs:
        F.fp8q_destroy(h)


def test_loss_scaler_against_oracle():
    """The device loss scaler follows the oracle's state machine on a random
    non-finite pattern, including the clamps."""
    rng = np.random.default_rng(62)
    for init, n, lo, hi in ((1024.0, 3, 1.0, 2.0 ** 24), (2.0 ** 23, 2, 1.0, 2.0 ** 24), (4.0, 1, 2.0, 64.0)):
        ls = F.fp8q_loss_scaler_create(init, n, lo, hi)
        o = policy.LossScaler(init, n, lo, hi)
        scale = G.empty(1, torch.float32)
        skip = G.empty(1, torch.int32)
        for t in range(40):
            counts = torch.from_numpy((rng.random(7) < 0.08).astype(np.int64) * rng.integers(1, 9, 7)).cuda()
            F.fp8q_loss_scaler_update(ls, counts, scale, skip)
            want_skip = o.update(counts.cpu().tolist())
            G.check(f"update {t}")
            assert (float(scale.item()), bool(skip.item())) == (float(o.scale), want_skip), t
        assert F.fp8q_loss_scaler_read(ls) == (float(o.scale), o.good)
        F.fp8q_loss_scaler_destroy(ls)


def test_loss_scaling_step_loop():
    """Casts of gradient tensors feed their non-finite counts to the scaler
    in one stream: an Inf in one tensor of a step halves the scale."""
    hs = [F.fp8q_create(1, 4) for _ in range(3)]
    ls = F.fp8q_loss_scaler_create(2.0 ** 16, 2)
    o = policy.LossScaler(2.0 ** 16, 2)
    scale = G.empty(1, torch.float32)
    skip = G.empty(1, torch.int32)
    for t in range(8):
        xs = [torch.randn(5000, device="cuda") * 1e-3 for _ in hs]
        if t in (2, 5):
            xs[1][17] = float("inf")
        qs, outs, cl, nf, uf = _counted_group_step(hs, xs, False)
        F.fp8q_loss_scaler_update(ls, nf, scale, skip)
        want = o.update(nf.cpu().tolist())
        G.check(f"update {t}")
        assert bool(skip.item()) == want == (t in (2, 5))
        assert float(scale.item()) == float(o.scale)
    F.fp8q_loss_scaler_destroy(ls)
    for h in hs:
        F.fp8q_destroy(h)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_per_tensor_error_stats(dtype):
    """MSE and bias of per-tensor casts (a clipping one: the window holds a
    smaller tensor's amax) within 1e-6 relative of the oracle, both formats,
    with non-finite inputs skipped; the count exact."""
    clean = synthetic.spike_step(9, "cuda", shape=(1024, 1024)).to(dtype)
    x = clean.clone()
    x.view(-1)[12345] = float("nan")
    x.view(-1)[54321] = float("-inf")
    for fmt in (0, 1):
        g = F.ScaledCast(fmt, window=1)
        cast_guarded(g, clean * 0.125)        # history from a smaller tensor: step 2 clips
        q, sinv, _, clipped = cast_guarded(g, x)
        assert int(clipped.item()) > 1
        out = G.empty(3, torch.float64)
        F.fp8q_error_stats(x, q, fmt, sinv, out)
        G.check("after fp8q_error_stats")
        mse, bias, n = out.cpu().tolist()
        e = -int(np.log2(sinv.item()))
        mse_o, bias_o, n_o = coracle.stats(host_bits(x), q.cpu().numpy().reshape(-1), fmt, e, NT)
        assert int(n) == n_o == x.numel() - 2
        assert rel_close(mse, mse_o), (mse, mse_o)
        assert rel_close(bias, bias_o), (bias, bias_o)
        g.close()


def test_argument_errors():
    h = F.fp8q_create(0, 4)
    x = torch.randn(1000, device="cuda")
    q = G.empty(1001, torch.uint8)
    with pytest.raises(F.Fp8qError) as ei:
        F.fp8q_cast(h, x[1:], q)                # misaligned input
    assert ei.value.status == -2
    with pytest.raises(F.Fp8qError) as ei:
        F.fp8q_cast_multi([h, h], [x, x], [q, q])   # same handle twice
    assert ei.value.status == -1
    with pytest.raises(F.Fp8qError):
        F.fp8q_set_history(h, [1.0] * 5)        # more than the window
    F.fp8q_destroy(h)

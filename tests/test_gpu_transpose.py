"""Parity of the fused cast + transpose kernels with the CPU oracle.

fp8q_cast_transpose: q must equal the oracle's per-tensor cast of x and qt
its transpose; amax, scale_inv, clipped and the history as for fp8q_cast.
mx_cast_dual: (q_row, e8m0_row) must equal the oracle's row-wise MX cast of
x and (q_colt, e8m0_colt) the row-wise MX cast of x^T.  All bit-exact.
Every output buffer carries guard bands (tests/canary.py) of at least one
32-row tile-store box on each side, checked after every call.
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

G = Guards(seed=0x7A9)

NT = os.cpu_count() or 1


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


def host_bits(x: torch.Tensor) -> np.ndarray:
    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.view(torch.int32).numpy().view(np.uint32)


def f32bits(t: torch.Tensor) -> int:
    return int(t.detach().cpu().view(torch.int32).numpy().view(np.uint32).reshape(-1)[0])


def _edge_tensor(rows, cols, dtype, seed):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-30, 30, size=(rows, 1)))
    v *= np.exp(rng.uniform(-10, 10, size=(1, cols)))
    v[0:32, 0] = 0.0
    v[0, :32] = 0.0
    v[1, 7] = np.nan
    v[40 % rows, 40 % cols] = -np.inf
    v[3, :] *= 1e-38
    v[4, cols // 2:] = 3e38
    return torch.from_numpy(v.astype(np.float32)).to(dtype).cuda()


def _dual_gpu(x, fmt, rule, headroom):
    rows, cols = x.shape
    qr = G.empty((rows, cols), torch.uint8)
    er = G.empty((rows, cols // 32), torch.uint8)
    qc = G.empty((cols, rows), torch.uint8)
    ec = G.empty((cols, rows // 32), torch.uint8)
    cr = G.empty(1, torch.int64)
    cc = G.empty(1, torch.int64)
    F.mx_cast_dual(x, fmt, rule, headroom, qr, er, qc, ec, cr, cc)
    G.check(f"mx_cast_dual {rows}x{cols} fmt={fmt} rule={rule} h={headroom}")
    assert F.fp8q_pipeline_status() == 0
    out = [t.cpu().numpy() for t in (qr, er, qc, ec)] + [int(cr.item()), int(cc.item())]
    G.release()
    return out


def _dual_oracle(xb, fmt, rule, headroom, nthreads=1):
    qr, er, cr = coracle.mx_cast_ex(xb, fmt, rule, headroom, 0, nthreads)
    qc, ec, cc = coracle.mx_cast_ex(np.ascontiguousarray(xb.T), fmt, rule, headroom, 0, nthreads)
    return qr, er, qc, ec, cr, cc


@pytest.mark.parametrize("rule", [0, 1, 2])
def test_mx_dual_full_size(rule):
    """bf16 [16384, 8192] tanh(N(0,2)) -> both MX E4M3 layouts in one pass."""
    x = synthetic.mx_tanh("cuda")
    got = _dual_gpu(x, 0, rule, 0)
    want = _dual_oracle(host_bits(x), 0, rule, 0, NT)
    names = ["q_row", "e8m0_row", "q_colt", "e8m0_colt"]
    for g, w, nm in zip(got[:4], want[:4], names):
        assert np.array_equal(g, w), nm
    assert got[4:] == list(want[4:])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_dual_edge_values(dtype):
    """Zero / NaN / Inf / subnormal / huge blocks, ragged column tiles,
    both formats, every rule, headroom 0 and 2.  Widths of 256 and 512
    columns give column-tile counts divisible by the warps of a CTA, so the
    row-block scale bytes go through the CTA's pooled table (with a ragged
    last row chunk at 96 and 160 rows); the other widths store them from
    each warp."""
    for rows, cols in ((96, 320), (32, 32), (64, 288), (160, 96), (96, 256), (160, 512)):
        x = _edge_tensor(rows, cols, dtype, rows * 7 + cols)
        xb = host_bits(x)
        for fmt in (0, 1):
            for rule in (0, 1, 2):
                for h in (0, 2):
                    got = _dual_gpu(x, fmt, rule, h)
                    want = _dual_oracle(xb, fmt, rule, h)
                    for g, w in zip(got[:4], want[:4]):
                        assert np.array_equal(g, w), (rows, cols, fmt, rule, h)
                    assert got[4:] == list(want[4:]), (rows, cols, fmt, rule, h)


@pytest.mark.parametrize("rule", [0, 1, 2])
def test_mx_e5m2_full_size_all_layouts(rule):
    """bf16 [16384, 8192] tanh(N(0,2)) scaled into the E5M2 range -> MX E5M2
    row-wise, column-wise and both at once (the dual), every rule: all bytes
    and counts equal the oracle's."""
    x = synthetic.mx_tanh("cuda") * 3.0e4
    xb = host_bits(x)
    rows, cols = x.shape
    want_r = coracle.mx_cast_ex(xb, 1, rule, 0, 0, NT)
    want_c = coracle.mx_cast_ex(xb, 1, rule, 0, 1, NT)
    for axis, want in ((0, want_r), (1, want_c)):
        q = G.empty((rows, cols), torch.uint8)
        e8 = G.empty((rows, cols // 32) if axis == 0 else (rows // 32, cols), torch.uint8)
        cl = G.empty(1, torch.int64)
        F.mx_cast_ex(x, 1, rule, 0, axis, q, e8, cl)
        G.check(f"axis {axis}")
        assert np.array_equal(q.cpu().numpy(), want[0]), axis
        assert np.array_equal(e8.cpu().numpy(), want[1]), axis
        assert int(cl.item()) == want[2], axis
        G.release()
        del q, e8
    got = _dual_gpu(x, 1, rule, 0)
    assert np.array_equal(got[0], want_r[0]) and np.array_equal(got[1], want_r[1])
    assert got[4] == want_r[2]
    # the transposed column-wise layout is the row-wise MX cast of x^T
    qc, ec, cc = coracle.mx_cast_ex(np.ascontiguousarray(xb.T), 1, rule, 0, 0, NT)
    assert np.array_equal(got[2], qc) and np.array_equal(got[3], ec)
    assert got[5] == cc == want_c[2]


def _clip_boundary_tensor(rows, cols, seed):
    """32 x 32 regions of one binade 2^k each (k from -120 to 120).  The
    region's diagonal holds +-1.9375 * 2^k, so every row block and every
    column block of the region has that maximum and, under the OCP rule,
    the shared exponent k - emax_elem.  The other entries sit on the clip
    thresholds of both formats (E4M3: 464 * 2^E = 1.8125 * 2^k, E5M2:
    61440 * 2^E = 1.875 * 2^k), one bf16 step above and below them, or
    well inside the range; all are exact bf16 values."""
    rng = np.random.default_rng(seed)
    step = 2.0 ** -7
    pool = np.array([1.8125, 1.8125 + step, 1.8125 - step, 1.875, 1.875 + step, 1.875 - step,
                     1.75, 1.0, 0.5, 0.0])
    v = rng.choice(pool, size=(rows, cols)) * rng.choice([-1.0, 1.0], size=(rows, cols))
    ks = rng.integers(-120, 121, size=(rows // 32, cols // 32))
    v *= np.exp2(np.repeat(np.repeat(ks, 32, axis=0), 32, axis=1))
    for i in range(rows // 32):
        for j in range(cols // 32):
            d = np.arange(32)
            v[32 * i + d, 32 * j + d] = 1.9375 * 2.0 ** int(ks[i, j]) * rng.choice([-1.0, 1.0], size=32)
    return v


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_clip_boundaries(dtype):
    """Elements exactly at, just above and just below the clip thresholds of
    both formats: the clipped counts and bytes of the MX dual, the
    column-wise and the row-wise MX casts equal the oracle's (every rule)."""
    rows, cols = 128, 320
    x = torch.from_numpy(_clip_boundary_tensor(rows, cols, 91).astype(np.float32)).to(dtype).cuda()
    xb = host_bits(x)
    for fmt in (0, 1):
        for rule in (0, 1, 2):
            got = _dual_gpu(x, fmt, rule, 0)
            want = _dual_oracle(xb, fmt, rule, 0)
            for g, w in zip(got[:4], want[:4]):
                assert np.array_equal(g, w), (fmt, rule)
            assert got[4:] == list(want[4:]), (fmt, rule)
            if rule == 0:
                assert got[4] > 0 and got[5] > 0          # the thresholds are crossed
            for axis in (0, 1):
                q = G.empty((rows, cols), torch.uint8)
                e8 = G.empty((rows, cols // 32) if axis == 0 else (rows // 32, cols), torch.uint8)
                cl = G.empty(1, torch.int64)
                F.mx_cast_ex(x, fmt, rule, 0, axis, q, e8, cl)
                G.check(f"fmt={fmt} rule={rule} axis={axis}")
                q_o, e8_o, c_o = coracle.mx_cast_ex(xb, fmt, rule, 0, axis, 1)
                assert np.array_equal(q.cpu().numpy(), q_o), (fmt, rule, axis)
                assert np.array_equal(e8.cpu().numpy(), e8_o), (fmt, rule, axis)
                assert int(cl.item()) == c_o, (fmt, rule, axis)


def _ct_steps(shape, dtype, fmt, window, steps, make, estimator=F.EST_MAX_WINDOW, alpha=1.0, interval=1):
    rows, cols = shape
    h = F.fp8q_create_ex(fmt, window, 1 if window else 0, 0, estimator, alpha, interval)
    o = policy.ScalingState(fmt, window, 1 if window else 0, 0, estimator, alpha, interval)
    for t in range(steps):
        x = make(t)
        q = G.empty((rows, cols), torch.uint8)
        qt = G.empty((cols, rows), torch.uint8)
        outs = G.empty(2, torch.float32)
        cl = G.empty(1, torch.int64)
        F.fp8q_cast_transpose(h, x, q, qt, outs[0:1], outs[1:2], cl)
        G.check(f"fp8q_cast_transpose {rows}x{cols} step {t}")
        q_o, a_o, s_o, c_o, _ = o.step(host_bits(x).reshape(-1), NT)
        q_o = q_o.reshape(rows, cols)
        assert np.array_equal(q.cpu().numpy(), q_o), t
        assert np.array_equal(qt.cpu().numpy(), q_o.T), t
        assert (f32bits(outs[0:1]), f32bits(outs[1:2]), int(cl.item())) == (s_o, a_o, c_o), t
        G.release()
    assert F.fp8q_pipeline_status() == 0
    hist = F.fp8q_amax_history(h, max(1, window))
    assert [np.float32(v).view(np.uint32) for v in hist] == o.hist
    F.fp8q_destroy(h)


@pytest.mark.parametrize("window", [0, 1, 16])
def test_cast_transpose_spike_sequence(window):
    """bf16 [4096, 4096] spike sequence (x8 at step 9): q and q^T each step,
    current scaling (pre-pass) on step 0 or every step."""
    _ct_steps((4096, 4096), torch.bfloat16, 0, window, 12,
              lambda t: synthetic.spike_step(t, "cuda"))


@pytest.mark.parametrize("estimator,alpha,interval", [(F.EST_SMOOTHED, 0.25, 1), (F.EST_MAX_WINDOW, 1.0, 3),
                                                     (F.EST_SMOOTHED, 0.5, 2)])
def test_cast_transpose_estimators(estimator, alpha, interval):
    """The transpose takes its exponent from the same device state as the
    grouped cast: exponential smoothing and a recompute interval over the
    spike sequence, q, q^T, scale, amax, clipped and history each step."""
    _ct_steps((1024, 2048), torch.bfloat16, 0, 8, 12,
              lambda t: synthetic.spike_step(t, "cuda", shape=(1024, 2048)),
              estimator, alpha, interval)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("fmt", [0, 1])
def test_cast_transpose_edge_values(dtype, fmt):
    for shape in ((96, 320), (32, 32), (64, 288)):
        _ct_steps(shape, dtype, fmt, 2, 3,
                  lambda t, shape=shape: _edge_tensor(shape[0], shape[1], dtype, 100 * t + shape[1]) * (4.0 ** t))


def _at(shape, offset):
    """A guarded device byte buffer starting `offset` bytes past a 256-byte
    boundary."""
    return G.empty(shape, torch.uint8, offset=offset)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_dual_offset_outputs(dtype):
    """Outputs 16-byte but not 32-byte aligned and E8M0 arrays at odd
    addresses: same bytes as the oracle."""
    rows, cols = 160, 288
    x = _edge_tensor(rows, cols, dtype, 77)
    xb = host_bits(x)
    qr = _at((rows, cols), 16)
    er = _at((rows, cols // 32), 1)
    qc = _at((cols, rows), 48)
    ec = _at((cols, rows // 32), 3)
    for fmt in (0, 1):
        F.mx_cast_dual(x, fmt, 0, 0, qr, er, qc, ec)
        G.check(f"fmt={fmt}")
        want = _dual_oracle(xb, fmt, 0, 0)
        for g, w in zip((qr, er, qc, ec), want[:4]):
            assert np.array_equal(g.cpu().numpy(), w), fmt


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_cast_transpose_offset_outputs(dtype):
    rows, cols = 96, 160
    x = _edge_tensor(rows, cols, dtype, 78)
    h = F.fp8q_create(0, 0)
    o = policy.ScalingState(0, 0)
    q = _at((rows, cols), 16)
    qt = _at((cols, rows), 48)
    F.fp8q_cast_transpose(h, x, q, qt)
    G.check()
    q_o = o.step(host_bits(x).reshape(-1), NT)[0].reshape(rows, cols)
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert np.array_equal(qt.cpu().numpy(), q_o.T)
    F.fp8q_destroy(h)


def test_cast_transpose_argument_checks():
    h = F.fp8q_create(0, 4)
    x = torch.zeros(48, 64, dtype=torch.bfloat16, device="cuda")
    q = G.empty((48, 64), torch.uint8)
    qt = G.empty((64, 48), torch.uint8)
    with pytest.raises(F.Fp8qError) as ei:
        F.fp8q_cast_transpose(h, x, q, qt)             # rows not a multiple of 32
    assert ei.value.status == -1
    F.fp8q_destroy(h)


def test_pipeline_wait_gives_up_and_is_reported():
    """Barrier waits that nothing completes (a bare one, and the per-warp tile
    pipeline's own wait) end at their deadline, are counted by
    fp8q_pipeline_status, and leave the device usable."""
    import time
    F.fp8q_pipeline_status()                          # clear
    t0 = time.time()
    F.fp8q_pipeline_selftest()
    torch.cuda.synchronize()
    assert 0.05 < time.time() - t0 < 30
    assert F.fp8q_pipeline_status() == 2              # the bare wait and the per-warp pipeline
    assert F.fp8q_pipeline_status() == 0              # read resets
    x = synthetic.mx_tanh("cuda", shape=(64, 256))
    got = _dual_gpu(x, 0, 0, 0)
    want = _dual_oracle(host_bits(x), 0, 0, 0)
    assert all(np.array_equal(g, w) for g, w in zip(got[:4], want[:4]))


def test_random_shapes_all_tiled_paths():
    """Randomly drawn shapes (ragged 64-column sub-tiles, partial row chunks,
    tails of 16 columns), both input types, both formats, every MX rule:
    column-wise MX, the MX dual and the per-tensor cast + transpose, byte for
    byte against the oracle."""
    rng = np.random.default_rng(2024)
    for trial in range(24):
        dtype = (torch.bfloat16, torch.float32)[trial % 2]
        fmt = (trial // 2) % 2
        rule = (trial // 4) % 3
        rows = 32 * int(rng.integers(1, 18))
        cols32 = 32 * int(rng.integers(1, 20))
        x = _edge_tensor(rows, cols32, dtype, 500 + trial) if trial % 3 == 0 else \
            torch.from_numpy((rng.standard_normal((rows, cols32)) *
                              np.exp(rng.uniform(-8, 8, size=(1, cols32)))).astype(np.float32)).to(dtype).cuda()
        xb = host_bits(x)
        # MX dual
        got = _dual_gpu(x, fmt, rule, trial % 3)
        want = _dual_oracle(xb, fmt, rule, trial % 3)
        for g, w in zip(got[:4], want[:4]):
            assert np.array_equal(g, w), (trial, rows, cols32)
        assert got[4:] == list(want[4:]), (trial, rows, cols32)
        # column-wise MX on a 16-column-aligned width
        cols16 = cols32 - 16 if cols32 > 32 and trial % 4 == 1 else cols32
        xc = x[:, :cols16].contiguous()
        xcb = host_bits(xc)
        q = G.empty((rows, cols16), torch.uint8)
        e8 = G.empty((rows // 32, cols16), torch.uint8)
        cl = G.empty(1, torch.int64)
        F.mx_cast_ex(xc, fmt, rule, 0, F.MX_COLWISE, q, e8, cl)
        G.check(f"trial {trial} column-wise")
        q_o, e8_o, c_o = coracle.mx_cast_ex(xcb, fmt, rule, 0, 1)
        assert np.array_equal(q.cpu().numpy(), q_o) and np.array_equal(e8.cpu().numpy(), e8_o), (trial, rows, cols16)
        assert int(cl.item()) == c_o, (trial, rows, cols16)
        # per-tensor cast + transpose, current scaling then a delayed step
        _ct_steps((rows, cols32), dtype, fmt, 2, 2, lambda t, x=x: x * (2.0 ** (3 * t)))
    assert F.fp8q_pipeline_status() == 0


@pytest.mark.parametrize("dtype,shape", [(torch.bfloat16, (16416, 4160)), (torch.float32, (8224, 1056))])
def test_large_ragged_shapes(dtype, shape):
    """Shapes that give every warp of a full grid several chunks, with a
    ragged last row chunk (rows / 32 odd) and, for fp32, a ragged last
    column chunk band: the MX dual, the column-wise MX cast and the
    per-tensor cast + transpose, byte for byte, twice in a row."""
    rows, cols = shape
    rng = np.random.default_rng(rows + cols)
    x = torch.from_numpy((rng.standard_normal(shape) * np.exp(rng.uniform(-6, 6, size=(rows, 1))))
                         .astype(np.float32)).to(dtype).cuda()
    xb = host_bits(x)
    for rule in (0, 1):
        want = _dual_oracle(xb, 0, rule, 0, NT)
        for _ in range(2):
            got = _dual_gpu(x, 0, rule, 0)
            for g, w, nm in zip(got[:4], want[:4], ["q_row", "e8m0_row", "q_colt", "e8m0_colt"]):
                assert np.array_equal(g, w), (shape, rule, nm)
            assert got[4:] == list(want[4:]), (shape, rule)
        q_o, e8_o, c_o = coracle.mx_cast_ex(xb, 0, rule, 0, 1, NT)
        for _ in range(2):
            q = G.empty((rows, cols), torch.uint8)
            e8 = G.empty((rows // 32, cols), torch.uint8)
            cl = G.empty(1, torch.int64)
            F.mx_cast_ex(x, 0, rule, 0, 1, q, e8, cl)
            G.check("column-wise")
            assert np.array_equal(q.cpu().numpy(), q_o) and np.array_equal(e8.cpu().numpy(), e8_o), (shape, rule)
            assert int(cl.item()) == c_o
            G.release()
    _ct_steps(shape, dtype, 0, 4, 3, lambda t: x * (2.0 ** t))
    assert F.fp8q_pipeline_status() == 0

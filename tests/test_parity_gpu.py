"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Integers (codes, block dots, tokens) must match exactly;
floats within the norm-relative tolerances of gpu_util."""
import numpy as np
import pytest

from oracle import oracle as orc
from q8_quantized_projection_gb300 import build, native, synth
from conftest import read_golden
from gpu_util import (QK, act_to_numpy, assert_codes_match, check_close, dev, host,
                      no_device_error, torch, upload_act, upload_weights)

pytestmark = pytest.mark.gpu

MODES = ["f32", "i8", "i8x2"]


@pytest.fixture(scope="module", autouse=True)
def lib():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    orc.build()
    native.load()
    yield
    no_device_error()


# ------------------------------------------------------------------- pack

@pytest.mark.parametrize("n,k", [(1, 32), (37, 96), (300, 4096), (5, 14336)])
def test_pack_bit_exact(n, k):
    rng = np.random.default_rng(10 + n + k)
    w = synth.f32_weights(rng, n, k)
    w[0, :QK] = 0.0
    if n > 3:
        w[1, QK:2 * QK] *= 1e-6
        w[2, :QK] *= 1e-3
        w[3, 0] = 65504.0 * 127 * 4      # overflowing scale
    q_o, s_o, ov_o = orc.q8_pack(w)
    t = torch()
    q = t.empty((n, k), dtype=t.int8, device="cuda")
    s = t.empty((n, k // QK), dtype=t.int16, device="cuda")
    ov = t.zeros(1, dtype=t.int32, device="cuda")
    native.q8_pack(dev(w), q, s, ov)
    assert np.array_equal(host(q), q_o)
    assert np.array_equal(host(s).view(np.uint16), s_o)
    assert int(host(ov)[0]) == ov_o


# ------------------------------------------------------------- producer

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("rows,k", [(1, 32), (3, 96), (1, 4096), (17, 4096), (2, 14336),
                                    (5, 4128), (256, 1024)])
@pytest.mark.parametrize("norm,with_gain", [(False, False), (True, False), (True, True)])
def test_act_quant_bit_exact(mode, rows, k, norm, with_gain):
    rng = np.random.default_rng(rows * 7 + k + (3 if norm else 0) + (5 if with_gain else 0))
    h = synth.activations(rng, rows, k)
    h[0, :QK] = 0.0
    g = synth.gain(rng, k) if with_gain else None
    x, r = orc.rmsnorm(h, g, 1e-5) if norm else (h, None)
    act_o = orc.quantize(mode, x)
    xq, xd = native.activation_buffers(mode, rows, k)
    native.act_quant(mode, dev(h), xq, xd, norm=norm, gain=dev(g) if g is not None else None,
                     eps=1e-5)
    assert_codes_match(act_to_numpy(mode, xq, xd), act_o, r, what=f"act_quant {mode} {rows}x{k}")


@pytest.mark.parametrize("mode", MODES)
def test_act_quant_rounding_order_golden(mode):
    """The hand-worked block of tests/golden/rmsnorm_order.txt: x = (h*rf)*g,
    where the other order of the two roundings moves a one-word code."""
    fx = {r[0]: r[1] for r in read_golden("rmsnorm_order.txt")}
    g0 = np.float32(float.fromhex(fx["g0"]))
    h = np.zeros((1, QK), np.float32)
    h[0, :2] = 3.0
    g = np.ones(QK, np.float32)
    g[0], g[1] = g0, g0 / np.float32(2)
    x, r = orc.rmsnorm(h, g, eps=0.0)
    assert float(x[0, 0]) == float.fromhex(fx["x0"])
    act_o = orc.quantize(mode, x)
    if mode == "i8":
        assert (int(act_o[0][0, 0]), int(act_o[0][0, 1])) == (int(fx["code0"]), int(fx["code1"]))
    xq, xd = native.activation_buffers(mode, 1, QK)
    native.act_quant(mode, dev(h), xq, xd, norm=True, gain=dev(g), eps=0.0)
    assert_codes_match(act_to_numpy(mode, xq, xd), act_o, None, what=f"golden order {mode}")


@pytest.mark.parametrize("mode", MODES)
def test_act_quant_near_tie_row(mode):
    """A row whose RMS scale lies 2^-44 from an f32 rounding boundary (K = 32,
    h = (1 - 2^-19, 1, ..., 1), eps = 0): the codes match the oracle's, or
    the mismatch is reported as a near tie (an expected failure)."""
    h = np.ones((2, QK), np.float32)
    h[0, 0] = np.float32(1 - 2.0 ** -19)
    h[1, 0] = np.float32(1.25)
    x, r = orc.rmsnorm(h, None, eps=0.0)
    assert orc.near_tie(r).tolist() == [True, False]
    act_o = orc.quantize(mode, x)
    xq, xd = native.activation_buffers(mode, 2, QK)
    native.act_quant(mode, dev(h), xq, xd, norm=True, eps=0.0)
    assert_codes_match(act_to_numpy(mode, xq, xd), act_o, r, what=f"near-tie row {mode}")


# ------------------------------------------------------------- block dots

@pytest.mark.parametrize("mode", ["i8", "i8x2"])
@pytest.mark.parametrize("n,k,rows", [(1, 32, 1), (37, 96, 3), (129, 4096, 2)])
def test_block_dots_bit_exact(mode, n, k, rows):
    rng = np.random.default_rng(n + k + rows)
    q, _ = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    act = orc.quantize(mode, x)
    isum_o = orc.block_dots(q, act[0], act[1] if mode == "i8x2" else None)
    t = torch()
    xq, _ = upload_act(mode, act, rows, k)
    isum = t.empty((rows, n, k // QK), dtype=t.int32, device="cuda")
    native.q8_debug_block_dots(mode, dev(q), xq, rows, isum, path=0)
    assert np.array_equal(host(isum), isum_o)


# ------------------------------------------------------------- projection

SHAPES = [(1, 32), (3, 64), (37, 96), (1000, 1024), (301, 4096), (77, 4128), (64, 14336),
          (5, 3104), (33, 11008), (19, 5120)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("rows", [1, 2, 3, 4, 5, 7, 8, 13, 16, 17])
def test_proj_parity(mode, n, k, rows):
    if rows > 3 and n * k > 1000 * 1024:
        rows = 3  # keep the oracle within seconds on the largest shapes
    rng = np.random.default_rng(1000 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    act = orc.quantize(mode, x)
    y_o, norm = orc.project(mode, q, s, act)
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    t = torch()
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    native.q8_proj(mode, qd, sd, xq, xd, rows, y)
    check_close(mode, host(y), y_o, norm, out_f64=False, what=f"{mode} {n}x{k} rows={rows}")
    if mode == "f32":
        y64 = t.empty((rows, n), dtype=t.float64, device="cuda")
        native.q8_proj(mode, qd, sd, xq, xd, rows, y64, out_f64=True)
        check_close(mode, host(y64), y_o, norm, out_f64=True, what=f"f64 {n}x{k} rows={rows}")
    y2 = t.empty((rows, n), dtype=t.float32, device="cuda")
    native.q8_proj_chunk(mode, qd, sd, xq, xd, rows, y2)
    check_close(mode, host(y2), y_o, norm, what=f"chunk {mode} {n}x{k} rows={rows}")


@pytest.mark.parametrize("n,k,rows", [(300, 4096, 2), (64, 14336, 2), (300, 4096, 8), (64, 14336, 13),
                                      (200, 2048, 40)])
def test_f32_batch_binade_spread(n, k, rows):
    """f32 activations whose 32-value blocks lie up to 2^130 apart within a
    row (and one all-zero row): at 2 rows the row-per-lane kernel (a row pair
    at K = 4096; one row a launch, planes built stage by stage, at K =
    14336), each block scaled to its row's largest binade; from 8 rows the
    tensor cores, each column's sum kept relative to the largest block binade
    seen so far and rescaled when a larger one comes (blocks far below are
    negligible): within 1e-9 of the norm, f32 and f64 outputs."""
    rng = np.random.default_rng(77 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k).astype(np.float64)
    scale = 2.0 ** rng.integers(-100, 30, size=(rows, k // 32))
    x = (x.reshape(rows, k // 32, 32) * scale[:, :, None]).reshape(rows, k).astype(np.float32)
    x[rows // 2] = 0.0
    act = orc.quantize("f32", x)
    y_o, norm = orc.project("f32", q, s, act)
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act("f32", act, rows, k)
    t = torch()
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    native.q8_proj("f32", qd, sd, xq, xd, rows, y)
    check_close("f32", host(y), y_o, norm, what=f"f32 spread {n}x{k} rows={rows}")
    y64 = t.empty((rows, n), dtype=t.float64, device="cuda")
    native.q8_proj("f32", qd, sd, xq, xd, rows, y64, out_f64=True)
    check_close("f32", host(y64), y_o, norm, out_f64=True, what=f"f64 spread {n}x{k} rows={rows}")
    assert np.all(host(y64)[rows // 2] == 0.0)
    no_device_error()


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k", [(300, 4096), (64, 14336), (129, 4128)])
@pytest.mark.parametrize("rows", [32, 64])
def test_proj_parity_large_batches(mode, n, k, rows):
    """q8_proj itself (not only q8_proj_chunk) at the largest batches of the
    batched-decode workload, K = 4096 and 14336 (tensor cores for the int8
    modes), and K = 4128 (not a multiple of 256: the CUDA-core kernels)."""
    rng = np.random.default_rng(2000 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    act = orc.quantize(mode, x)
    y_o, norm = orc.project(mode, q, s, act)
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    t = torch()
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    native.q8_proj(mode, qd, sd, xq, xd, rows, y)
    check_close(mode, host(y), y_o, norm, what=f"{mode} {n}x{k} rows={rows}")


@pytest.mark.parametrize("mode,rows", [("i8", 3), ("i8", 4), ("i8", 5), ("i8", 8),
                                       ("i8x2", 2), ("i8x2", 3), ("i8x2", 4)])
@pytest.mark.parametrize("n,k", [(6100, 2048), (5000, 5120), (9731, 1024), (4900, 14336)])
def test_batched_row_groups(mode, rows, n, k):
    """Batched int8 projections where each CTA owns several 32-row groups
    (N well above 32 x the SM count), ragged in N, with 1, 2, 5 and 14 stages
    of 1024 values per group; two calls give identical bits."""
    rng = np.random.default_rng(3000 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    act = orc.quantize(mode, x)
    y_o, norm = orc.project(mode, q, s, act)
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    t = torch()
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    native.q8_proj(mode, qd, sd, xq, xd, rows, y)
    check_close(mode, host(y), y_o, norm, what=f"{mode} {n}x{k} rows={rows}")
    y2 = t.full((rows, n), float("nan"), dtype=t.float32, device="cuda")
    native.q8_proj(mode, qd, sd, xq, xd, rows, y2)
    assert t.equal(y, y2)


@pytest.mark.parametrize("mode", MODES)
def test_largest_resident_row(mode):
    """K = 16384, the longest row a fused launch (and a one-row f32 launch)
    keeps in shared memory: q8_proj and q8_proj_fused at one row against the
    oracle, and the fused result bitwise equal to act_quant + q8_proj."""
    n, k = 300, 16384
    rng = np.random.default_rng(4242)
    q, s = synth.q8_weights(rng, n, k)
    h = synth.activations(rng, 1, k)
    g = synth.gain(rng, k)
    x, _ = orc.rmsnorm(h, g, 1e-5)
    y_o, norm = orc.project(mode, q, s, orc.quantize(mode, x))
    qd, sd = upload_weights(q, s)
    t = torch()
    ws = t.empty(native.q8_proj_fused_workspace(mode, 1, k), dtype=t.uint8, device="cuda")
    y = t.empty((1, n), dtype=t.float32, device="cuda")
    native.q8_proj_fused(mode, qd, sd, dev(h), y, ws, gain=dev(g), eps=1e-5)
    check_close(mode, host(y), y_o, norm, what=f"fused {mode} K={k}")
    xq, xd = native.activation_buffers(mode, 1, k, device="cuda")
    native.act_quant(mode, dev(h), xq, xd, norm=True, gain=dev(g), eps=1e-5)
    y2 = t.empty((1, n), dtype=t.float32, device="cuda")
    native.q8_proj(mode, qd, sd, xq, xd, 1, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))
    no_device_error()


@pytest.mark.parametrize("mode", MODES)
def test_proj_deterministic_and_zero(mode):
    rng = np.random.default_rng(77)
    n, k, rows = 500, 4096, 4
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    x[1] = 0.0
    act = orc.quantize(mode, x)
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    t = torch()
    y1 = t.empty((rows, n), dtype=t.float32, device="cuda")
    y2 = t.empty_like(y1)
    native.q8_proj(mode, qd, sd, xq, xd, rows, y1)
    native.q8_proj(mode, qd, sd, xq, xd, rows, y2)
    a, b = host(y1), host(y2)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.all(a[1] == 0)


# ----------------------------------------------------------- fused producer

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k,rows", [(300, 4096, 1), (100, 14336, 2), (64, 1024, 16),
                                      (50, 16384, 1), (40, 16416, 1), (37, 96, 1), (7, 14336, 1),
                                      # rows of one slice above 4096 values, a ragged part, and
                                      # two slices with a ragged last one (the f32 kernel keeps
                                      # the converted activation after its weight ring there)
                                      (77, 4128, 1), (61, 5120, 1), (45, 8224, 1), (33, 11008, 1)])
def test_fused_matches_oracle_and_composition(mode, n, k, rows):
    rng = np.random.default_rng(5 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    h = synth.activations(rng, rows, k)
    g = synth.gain(rng, k)
    x, _ = orc.rmsnorm(h, g, 1e-5)
    y_o, norm = orc.project(mode, q, s, orc.quantize(mode, x))
    qd, sd = upload_weights(q, s)
    t = torch()
    hd, gd = dev(h), dev(g)
    ws = t.empty(native.q8_proj_fused_workspace(mode, rows, k), dtype=t.uint8, device="cuda")
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    native.q8_proj_fused(mode, qd, sd, hd, y, ws, gain=gd, eps=1e-5)
    check_close(mode, host(y), y_o, norm, what=f"fused {mode}")
    # the fused call computes exactly what its two unfused parts compute
    xq, xd = native.activation_buffers(mode, rows, k)
    native.act_quant(mode, hd, xq, xd, norm=True, gain=gd, eps=1e-5)
    y2 = t.empty_like(y)
    native.q8_proj(mode, qd, sd, xq, xd, rows, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


# ------------------------------------------- residual added before the norm

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("rows,k", [(1, 96), (1, 4096), (3, 4128), (2, 14336), (17, 1024)])
@pytest.mark.parametrize("with_gain", [False, True])
def test_act_quant_residual_bit_exact(mode, rows, k, with_gain):
    # s = h + r (one f32 rounding) written back, then the producer on s
    rng = np.random.default_rng(40 + rows * 3 + k + (1 if with_gain else 0))
    h = synth.activations(rng, rows, k)
    r = synth.activations(rng, rows, k)
    r[0, :QK] = -h[0, :QK]                      # a block that cancels to zero
    g = synth.gain(rng, k) if with_gain else None
    s_o = orc.residual_add(h, r)
    x_o, rs = orc.rmsnorm(s_o, g, 1e-5)
    act_o = orc.quantize(mode, x_o)
    t = torch()
    xq, xd = native.activation_buffers(mode, rows, k)
    s_out = t.empty((rows, k), dtype=t.float32, device="cuda")
    native.act_quant_residual(mode, dev(h), dev(r), xq, xd, s_out=s_out,
                              gain=dev(g) if g is not None else None, eps=1e-5)
    assert np.array_equal(host(s_out).view(np.uint32), s_o.view(np.uint32))
    assert_codes_match(act_to_numpy(mode, xq, xd), act_o, rs, what=f"residual {mode} {rows}x{k}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k,rows", [(300, 4096, 1), (7, 14336, 1), (37, 96, 1), (100, 4096, 3),
                                      (50, 5120, 1), (29, 11008, 1)])
def test_fused_residual_matches_oracle_and_composition(mode, n, k, rows):
    rng = np.random.default_rng(60 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    h = synth.activations(rng, rows, k)
    r = synth.activations(rng, rows, k)
    g = synth.gain(rng, k)
    s_o = orc.residual_add(h, r)
    y_o, norm = orc.project(mode, q, s, orc.quantize(mode, orc.rmsnorm(s_o, g, 1e-5)[0]))
    qd, sd = upload_weights(q, s)
    t = torch()
    hd, rd, gd = dev(h), dev(r), dev(g)
    ws = t.empty(native.q8_proj_fused_workspace(mode, rows, k), dtype=t.uint8, device="cuda")
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    s_out = t.full((rows, k), float("nan"), dtype=t.float32, device="cuda")
    native.q8_proj_fused_residual(mode, qd, sd, hd, rd, y, ws, s_out=s_out, gain=gd, eps=1e-5)
    check_close(mode, host(y), y_o, norm, what=f"fused residual {mode}")
    assert np.array_equal(host(s_out).view(np.uint32), s_o.view(np.uint32))
    # bitwise what the residual producer followed by the projection computes,
    # and what the plain fused call computes on s
    xq, xd = native.activation_buffers(mode, rows, k)
    native.act_quant_residual(mode, hd, rd, xq, xd, gain=gd, eps=1e-5)
    y2 = t.empty_like(y)
    native.q8_proj(mode, qd, sd, xq, xd, rows, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))
    y3 = t.empty_like(y)
    native.q8_proj_fused(mode, qd, sd, dev(s_o), y3, ws, gain=gd, eps=1e-5)
    assert np.array_equal(host(y).view(np.uint32), host(y3).view(np.uint32))
    # without s_out nothing else changes
    y4 = t.empty_like(y)
    native.q8_proj_fused_residual(mode, qd, sd, hd, rd, y4, ws, gain=gd, eps=1e-5)
    assert np.array_equal(host(y).view(np.uint32), host(y4).view(np.uint32))


# ------------------------------------------------ SwiGLU producer of down

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("rows,k", [(1, 96), (1, 14336), (3, 4128), (2, 1024), (17, 512)])
def test_act_quant_swiglu_bit_exact(mode, rows, k):
    rng = np.random.default_rng(80 + rows + k)
    gu = (synth.activations(rng, rows, 2 * k) * 3.0).astype(np.float32)
    gu[0, :QK] = 0.0                            # a gate block of zeros: x = 0
    gu[-1, 1] = -120.0                          # e^120 overflows: silu -> -0
    act_o = orc.quantize(mode, orc.swiglu(gu))
    xq, xd = native.activation_buffers(mode, rows, k)
    native.act_quant_swiglu(mode, dev(gu), xq, xd)
    for a, b in zip(act_to_numpy(mode, xq, xd), act_o):
        assert np.array_equal(a.view(np.uint8) if a.dtype != np.float32 else a.view(np.uint32),
                              b.view(np.uint8) if b.dtype != np.float32 else b.view(np.uint32))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k,rows", [(300, 14336, 1), (64, 4096, 1), (37, 96, 1), (100, 1024, 3),
                                      (31, 4128, 1), (40, 8224, 1), (20, 16384, 1)])
def test_fused_swiglu_matches_oracle_and_composition(mode, n, k, rows):
    rng = np.random.default_rng(90 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    gu = (synth.activations(rng, rows, 2 * k) * 3.0).astype(np.float32)
    y_o, norm = orc.project(mode, q, s, orc.quantize(mode, orc.swiglu(gu)))
    qd, sd = upload_weights(q, s)
    t = torch()
    gud = dev(gu)
    ws = t.empty(native.q8_proj_fused_workspace(mode, rows, k), dtype=t.uint8, device="cuda")
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    native.q8_proj_fused_swiglu(mode, qd, sd, gud, y, ws)
    check_close(mode, host(y), y_o, norm, what=f"fused swiglu {mode}")
    # bitwise what the SwiGLU producer followed by the projection computes
    xq, xd = native.activation_buffers(mode, rows, k)
    native.act_quant_swiglu(mode, gud, xq, xd)
    y2 = t.empty_like(y)
    native.q8_proj(mode, qd, sd, xq, xd, rows, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


# ------------------------------------------------------- KV-row epilogue

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("rows,pos", [(1, [3]), (1, [0]), (3, [0, 4, 2]), (9, [4, 0, 1, 2, 3, 4, 0, 1, 2])])
def test_fused_kv_rows(mode, rows, pos):
    # a QKV projection of N = 384 (q 256, K 64, V 64) into caches of 5 rows
    n, k, kv_col, d, n_pos = 384, 1024, 256, 64, 5
    rng = np.random.default_rng(100 + rows + pos[0])
    q, s = synth.q8_weights(rng, n, k)
    h = synth.activations(rng, rows, k)
    g = synth.gain(rng, k)
    y_o, norm = orc.project(mode, q, s, orc.quantize(mode, orc.rmsnorm(h, g, 1e-5)[0]))
    qd, sd = upload_weights(q, s)
    t = torch()
    ws = t.empty(native.q8_proj_fused_workspace(mode, rows, k), dtype=t.uint8, device="cuda")
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    kc = t.full((rows, n_pos, d), float("nan"), dtype=t.float32, device="cuda")
    vc = t.full((rows, n_pos, d), float("nan"), dtype=t.float32, device="cuda")
    posd = t.tensor(pos, dtype=t.int32, device="cuda")
    native.q8_proj_fused_kv(mode, qd, sd, dev(h), y, ws, posd, kv_col, kc, vc, gain=dev(g), eps=1e-5)
    yh = host(y)
    check_close(mode, yh, y_o, norm, what=f"fused kv {mode}")
    kc_o = np.full((rows, n_pos, d), np.nan, np.float32)
    vc_o = np.full((rows, n_pos, d), np.nan, np.float32)
    assert orc.kv_write(yh, pos, kv_col, d, kc_o, vc_o) == 0
    assert np.array_equal(host(kc).view(np.uint32), kc_o.view(np.uint32))
    assert np.array_equal(host(vc).view(np.uint32), vc_o.view(np.uint32))
    # y is what the plain fused call computes
    y2 = t.empty_like(y)
    native.q8_proj_fused(mode, qd, sd, dev(h), y2, ws, gain=dev(g), eps=1e-5)
    assert np.array_equal(yh.view(np.uint32), host(y2).view(np.uint32))


@pytest.mark.parametrize("rows", [1, 3])
@pytest.mark.parametrize("k", [512, 1024])
def test_fused_kv_position_out_of_range(rows, k):
    # K = 1024: the row-per-lane kernel's KV epilogue at rows = 1
    n, kv_col, d, n_pos = 256, 128, 32, 4
    rng = np.random.default_rng(7 + rows)
    q, s = synth.q8_weights(rng, n, k)
    h = synth.activations(rng, rows, k)
    qd, sd = upload_weights(q, s)
    t = torch()
    ws = t.empty(native.q8_proj_fused_workspace("i8", rows, k), dtype=t.uint8, device="cuda")
    y = t.empty((rows, n), dtype=t.float32, device="cuda")
    kc = t.full((rows, n_pos, d), 7.0, dtype=t.float32, device="cuda")
    vc = t.full((rows, n_pos, d), 7.0, dtype=t.float32, device="cuda")
    bad = [n_pos] + [-1] * (rows - 1)
    native.q8_proj_fused_kv("i8", qd, sd, dev(h), y, ws, t.tensor(bad, dtype=t.int32, device="cuda"),
                            kv_col, kc, vc)
    assert native.q8_device_error() == 2          # reported, and cleared by the read
    assert np.all(host(kc) == 7.0) and np.all(host(vc) == 7.0)


def test_residual_argument_errors():
    t = torch()
    k, n = 64, 8
    q = t.zeros((n, k), dtype=t.int8, device="cuda")
    s = t.zeros((n, k // QK), dtype=t.int16, device="cuda")
    h = t.zeros((1, k), dtype=t.float32, device="cuda")
    r = t.zeros((1, k), dtype=t.float32, device="cuda")
    y = t.empty((1, n), dtype=t.float32, device="cuda")
    ws = t.empty(native.q8_proj_fused_workspace("i8", 1, k), dtype=t.uint8, device="cuda")
    xq, xd = native.activation_buffers("i8", 1, k)
    with pytest.raises(native.Q8Error, match="Q8_ERR_ARG"):   # no residual
        native.act_quant_residual("i8", h, None, xq, xd)
    with pytest.raises(native.Q8Error, match="Q8_ERR_ARG"):   # s_out overlaps h
        native.q8_proj_fused_residual("i8", q, s, h, r, y, ws, s_out=h)
    with pytest.raises(native.Q8Error, match="Q8_ERR_ARG"):   # s_out overlaps r
        native.act_quant_residual("i8", h, r, xq, xd, s_out=r)


# ------------------------------------------------------------- LM head

def _planted_head(n, k, rows, seed):
    return synth.planted_head(seed, n, k, rows)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n,k,rows", [(20000, 1024, 1), (20000, 1024, 3), (20000, 1024, 6),
                                      (20000, 2048, 8), (20000, 1024, 16), (5000, 4096, 20),
                                      (8, 256, 1)])
def test_head_argmax_planted(mode, n, k, rows):
    q, s, h, pos = _planted_head(n, k, rows, seed=n + k + rows)
    x, _ = orc.rmsnorm(h)
    act = orc.quantize(mode, x)
    tok_o, best_o, y_o = orc.head_argmax(mode, q, s, act)
    assert np.array_equal(tok_o, pos[np.arange(rows) % 8])
    t = torch()
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    ws = native.argmax_workspace(rows)
    tok = t.empty(rows, dtype=t.int32, device="cuda")
    mx = t.empty(rows, dtype=t.float64, device="cuda")
    logits = t.empty((rows, n), dtype=t.float64 if mode == "f32" else t.float32, device="cuda")
    for _ in range(2):  # the workspace counter must come back to zero
        native.head_argmax(mode, qd, sd, xq, xd, rows, tok, ws, maxval=mx, logits=logits)
        assert np.array_equal(host(tok), tok_o)
    _, norm = orc.project(mode, q, s, act)
    check_close(mode, host(logits), y_o, norm, out_f64=True, what="head logits")
    rowsel = np.arange(rows)
    check_close(mode, host(mx), best_o, norm[rowsel, tok_o], out_f64=True, what="head max")
    assert int(host(ws[:4].view(t.int32))[0]) == 0


@pytest.mark.parametrize("mode", MODES)
def test_head_argmax_equals_argmax_of_projection(mode):
    # unplanted random head: the fused arg-max picks the same index as the
    # arg-max of the library's own projection output
    rng = np.random.default_rng(31)
    n, k, rows = 30011, 1024, 5
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    act = orc.quantize(mode, x)
    t = torch()
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    y = t.empty((rows, n), dtype=t.float64 if mode == "f32" else t.float32, device="cuda")
    native.q8_proj(mode, qd, sd, xq, xd, rows, y, out_f64=(mode == "f32"))
    tok = t.empty(rows, dtype=t.int32, device="cuda")
    native.head_argmax(mode, qd, sd, xq, xd, rows, tok, native.argmax_workspace(rows))
    tok_ref, _ = orc.argmax(host(y))
    assert np.array_equal(host(tok), tok_ref)


def _tie_head(n, k, rows, pairs, seed):
    """A random Q8_0 head where activation row m's winner is planted at the
    two indices pairs[m % 8] (identical rows, so their logits are equal
    bit for bit): the arg-max must return the lower index."""
    rng = np.random.default_rng(seed)
    q, s = synth.q8_weights(rng, n, k)
    h, base = synth.head_activations(rng, rows, k)
    for j, (a, b) in enumerate(pairs):
        synth.plant_head_rows(q, s, base[j:j + 1], np.array([a]))
        q[b], s[b] = q[a], s[a]
    return q, s, h


TIE_PAIRS = [(0, 19999), (1000, 1001), (5000, 5003), (7, 12000), (19990, 19998), (2, 3),
             (9000, 9100), (15000, 15001)]


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("rows", [1, 16])
@pytest.mark.parametrize("noalloc", [False, True])
def test_head_argmax_exact_ties(mode, rows, noalloc):
    """Exact ties between identical head rows, inside one CTA's rows and in
    different CTAs (n = 0 with n = N-1): the lowest index wins."""
    n, k = 20000, 1024
    q, s, h = _tie_head(n, k, rows, TIE_PAIRS, seed=rows + 3)
    x, _ = orc.rmsnorm(h)
    act = orc.quantize(mode, x)
    tok_o, _, y_o = orc.head_argmax(mode, q, s, act)
    want = np.array([min(TIE_PAIRS[m % 8]) for m in range(rows)])
    assert np.array_equal(tok_o, want)
    rowsel = np.arange(rows)
    assert np.array_equal(y_o[rowsel, want], y_o[rowsel, [max(TIE_PAIRS[m % 8]) for m in range(rows)]])
    t = torch()
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    tok = t.full((rows,), -7, dtype=t.int32, device="cuda")
    if noalloc:
        native.head_argmax_noalloc(mode, qd, sd, xq, xd, rows, tok)
    else:
        native.head_argmax(mode, qd, sd, xq, xd, rows, tok, native.argmax_workspace(rows))
    assert np.array_equal(host(tok), want)


@pytest.mark.parametrize("mode", ["i8", "i8x2"])
@pytest.mark.parametrize("rows", [1, 3, 16])
@pytest.mark.parametrize("k", [256, 1024])
def test_head_argmax_nan_and_infinite_logits(mode, rows, k):
    """NaN logits are never the maximum; a row of -inf gives index 0; a row of
    NaN gives index 0 and the value NaN (infinite binary16 scales: 0 * inf is
    NaN, a negative block dot times inf is -inf).  K = 1024: the row-per-lane
    kernel's arg-max; K = 256: the decode kernel's."""
    n = 3000
    rng = np.random.default_rng(77 + rows + k)
    q, s = synth.q8_weights(rng, n, k)
    h, base = synth.head_activations(rng, rows, k)
    pos = np.array([5, 2999, 1, 700, 1500, 2000, 2500, 2998])
    synth.plant_head_rows(q, s, base, pos)
    inf16 = np.uint16(0x7C00)
    q[0], s[0] = 0, inf16                       # logit NaN at n = 0
    x, _ = orc.rmsnorm(h)
    act = orc.quantize(mode, x)
    tok_o, _, _ = orc.head_argmax(mode, q, s, act)
    assert np.array_equal(tok_o, pos[np.arange(rows) % 8])
    t = torch()
    xq, xd = upload_act(mode, act, rows, k)
    tok = t.full((rows,), -7, dtype=t.int32, device="cuda")
    mx = t.empty(rows, dtype=t.float64, device="cuda")
    qd, sd = upload_weights(q, s)
    native.head_argmax(mode, qd, sd, xq, xd, rows, tok, native.argmax_workspace(rows), maxval=mx)
    assert np.array_equal(host(tok), tok_o)
    # every logit -inf: weights -1 with infinite scales, activation codes > 0
    hp = np.abs(h) + np.float32(0.5)
    actp = orc.quantize(mode, orc.rmsnorm(hp)[0])
    qn = np.full((n, k), -1, np.int8)
    sn = np.full((n, k // QK), inf16, np.uint16)
    tok_o, best_o, _ = orc.head_argmax(mode, qn, sn, actp)
    assert np.all(tok_o == 0) and np.all(best_o == -np.inf)
    xq, xd = upload_act(mode, actp, rows, k)
    qd, sd = upload_weights(qn, sn)
    native.head_argmax(mode, qd, sd, xq, xd, rows, tok, native.argmax_workspace(rows), maxval=mx)
    assert np.all(host(tok) == 0) and np.all(host(mx) == -np.inf)
    # every logit NaN: zero weights with infinite scales
    qd, sd = upload_weights(np.zeros((n, k), np.int8), sn)
    tok.fill_(-7)
    native.head_argmax(mode, qd, sd, xq, xd, rows, tok, native.argmax_workspace(rows), maxval=mx)
    assert np.all(host(tok) == 0) and np.all(np.isnan(host(mx)))


# --------------------------------------------------- full-size workloads

@pytest.mark.parametrize("mode", MODES)
def test_decode_layer_full_size_sampled(mode):
    """The d=4096 layer's four projections at full size, rows = 1, activation
    RMSNorm(N(0,1)) quantized in the producer; sampled output rows are checked
    against the oracle one by one."""
    t = torch()
    rng = np.random.default_rng(0)
    for name, n, k in synth.LAYER_D4096:
        q, s = synth.q8_weights(rng, n, k)
        h = synth.activations(rng, 1, k)
        qd, sd = upload_weights(q, s)
        ws = t.empty(native.q8_proj_fused_workspace(mode, 1, k), dtype=t.uint8, device="cuda")
        y = t.empty((1, n), dtype=t.float32, device="cuda")
        native.q8_proj_fused(mode, qd, sd, dev(h), y, ws)
        idx = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 200)]))
        x, _ = orc.rmsnorm(h)
        y_o, norm = orc.project(mode, q[idx], s[idx], orc.quantize(mode, x))
        check_close(mode, host(y)[:, idx], y_o, norm, what=f"{name} {mode}")


@pytest.mark.parametrize("mode,rows", [("i8", 1), ("i8", 16), ("f32", 1)])
def test_head_full_size(mode, rows):
    n, k = synth.HEAD_SHAPE
    q, s, h, pos = _planted_head(n, k, rows, seed=4)
    x, _ = orc.rmsnorm(h)
    act = orc.quantize(mode, x)
    t = torch()
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, rows, k)
    tok = t.empty(rows, dtype=t.int32, device="cuda")
    mx = t.empty(rows, dtype=t.float64, device="cuda")
    native.head_argmax(mode, qd, sd, xq, xd, rows, tok, native.argmax_workspace(rows), maxval=mx)
    want = pos[np.arange(rows) % 8]
    assert np.array_equal(host(tok), want)
    y_o, norm = orc.project(mode, q[want], s[want], act)
    rowsel = np.arange(rows)
    check_close(mode, host(mx), y_o[rowsel, rowsel], norm[rowsel, rowsel], out_f64=True,
                what="head max value")


# ------------------------------------------------------- tensor-core chunk path

@pytest.mark.parametrize("mode", ["i8", "i8x2"])
@pytest.mark.parametrize("n,k,t", [(300, 1024, 16), (129, 4096, 33), (257, 1024, 128),
                                   (130, 4096, 129), (64, 14336, 48), (1000, 1024, 256),
                                   (77, 2048, 5), (128, 3328, 20), (2000, 4096, 64),
                                   (96, 1280, 97)])
def test_chunk_tensor_core_parity(mode, n, k, t):
    rng = np.random.default_rng(3000 + n + k + t)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, t, k)
    act = orc.quantize(mode, x)
    y_o, norm = orc.project(mode, q, s, act)
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, t, k)
    tt = torch()
    y = tt.empty((t, n), dtype=tt.float32, device="cuda")
    native.q8_proj_chunk(mode, qd, sd, xq, xd, t, y)
    check_close(mode, host(y), y_o, norm, what=f"chunk {mode} {n}x{k} T={t}")
    y2 = tt.empty_like(y)
    native.q8_proj_chunk(mode, qd, sd, xq, xd, t, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


# Shapes with more 128 x TT tiles than clusters that fit, so that the clusters
# run in several waves: K unsplit (256), and split over a cluster of CTAs whose
# partials meet in distributed shared memory (K = 2304: 9 groups of 8 blocks
# split 5 + 4; a ragged last tile at N = 20000).
WAVE_SHAPES = [("i8", 16, 40000, 256), ("i8", 16, 20000, 2048), ("i8", 5, 20000, 6144),
               ("i8", 16, 20000, 8192), ("i8", 32, 20000, 12288), ("i8", 40, 20000, 8192),
               ("i8x2", 16, 25600, 2304), ("i8x2", 32, 20000, 2048)]


@pytest.mark.parametrize("mode,t,n,k", WAVE_SHAPES)
def test_chunk_many_tiles_sampled(mode, t, n, k):
    plan = native.q8_debug_chunk_plan(mode, n, k, t)
    assert plan["waves"] > 1 and plan["tiles"] > plan["clusters"], plan
    assert plan["ks"] & (plan["ks"] - 1) == 0, plan   # splits are powers of two
    rng = np.random.default_rng(6000 + t + n + k)
    q, s = synth.q8_weights(rng, n, k)
    act = orc.quantize(mode, synth.activations(rng, t, k))
    qd, sd = upload_weights(q, s)
    xq, xd = upload_act(mode, act, t, k)
    tt = torch()
    y = tt.empty((t, n), dtype=tt.float32, device="cuda")
    native.q8_proj_chunk(mode, qd, sd, xq, xd, t, y)
    # the first and the last tile whole (every row slice of the split), the
    # rows around a tile boundary in mid-matrix, and random rows
    mid = (n // 256) * 128
    idx = np.unique(np.concatenate([np.arange(128), np.arange((n - 1) // 128 * 128, n),
                                    np.arange(mid - 3, mid + 3), rng.integers(0, n, 300)]))
    y_o, norm = orc.project(mode, q[idx], s[idx], act)
    check_close(mode, host(y)[:, idx], y_o, norm, what=f"chunk {mode} {n}x{k} T={t} {plan}")
    # the split-K sums are added in rank order: the same bits every time
    y2 = tt.empty_like(y)
    native.q8_proj_chunk(mode, qd, sd, xq, xd, t, y2)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))


def test_head_plan():
    """The 16-row LM head on the tensor cores: 1002 tiles of 128 x 16, K
    unsplit (the arg-max needs whole dots), one CTA per SM at a time."""
    plan = native.q8_debug_chunk_plan("i8", *synth.HEAD_SHAPE, 16, argmax=True)
    assert plan["ks"] == 1 and plan["tiles"] == 1002 and plan["TT"] == 16, plan
    sms = torch().cuda.get_device_properties(0).multi_processor_count
    assert plan["clusters"] == sms and plan["waves"] == -(-1002 // sms), plan


def test_f32_chunk_plan():
    """The f32 mode's tensor-core plan: tiles of 16 or 32 activation rows (four
    byte planes make the MMA's N), the head's K unsplit, and K split over a
    cluster where a projection has few tiles."""
    head = native.q8_debug_chunk_plan("f32", *synth.HEAD_SHAPE, 16, argmax=True)
    assert head["TT"] == 16 and head["ks"] == 1 and head["tiles"] == 1002, head
    wo = native.q8_debug_chunk_plan("f32", 4096, 4096, 8)
    assert wo["TT"] == 16 and wo["tiles"] == 32 and wo["ks"] > 1, wo
    big = native.q8_debug_chunk_plan("f32", 4096, 4096, 40)
    assert big["TT"] == 32 and big["tiles"] == 64, big


@pytest.mark.parametrize("mode", ["i8", "i8x2"])
@pytest.mark.parametrize("n,k,t", [(129, 1024, 16), (64, 4096, 130), (40, 512, 3), (130, 768, 64)])
def test_chunk_block_dots_exact(mode, n, k, t):
    """The tensor-core per-block accumulators are the exact integer block dots."""
    rng = np.random.default_rng(4000 + n + k + t)
    q, _ = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, t, k)
    act = orc.quantize(mode, x)
    isum_o = orc.block_dots(q, act[0], act[1] if mode == "i8x2" else None)
    tt = torch()
    xq, _ = upload_act(mode, act, t, k)
    isum = tt.empty((t, n, k // QK), dtype=tt.int32, device="cuda")
    native.q8_debug_block_dots(mode, dev(q), xq, t, isum, path=1)
    assert np.array_equal(host(isum), isum_o)


@pytest.mark.parametrize("mode", ["i8", "i8x2"])
def test_prefill_chunk_full_size_sampled(mode):
    """A 256-row prefill chunk through the d=4096 layer's matrices at full size,
    each row RMSNorm(N(0,1)) quantized in the producer; sampled output columns
    are checked against the oracle."""
    tt = torch()
    rng = np.random.default_rng(5)
    T = 256
    for name, n, k in synth.LAYER_D4096:
        q, s = synth.q8_weights(rng, n, k)
        h = synth.activations(rng, T, k)
        qd, sd = upload_weights(q, s)
        xq, xd = native.activation_buffers(mode, T, k)
        native.act_quant(mode, dev(h), xq, xd, norm=True)
        y = tt.empty((T, n), dtype=tt.float32, device="cuda")
        native.q8_proj_chunk(mode, qd, sd, xq, xd, T, y)
        idx = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 64)]))
        x, r = orc.rmsnorm(h)
        act = orc.quantize(mode, x)
        assert_codes_match(act_to_numpy(mode, xq, xd), act, r, what=f"{name} {mode} T={T}")
        y_o, norm = orc.project(mode, q[idx], s[idx], act)
        check_close(mode, host(y)[:, idx], y_o, norm, what=f"{name} {mode} T={T}")

"""Helpers for the GPU parity tests: upload seeded numpy inputs, run the
library through its C ABI binding, and compare with the oracle."""
import numpy as np
import pytest

from q8_quantized_projection_gb300 import native

QK = 32
RTOL_Q = 1e-5     # one-word / two-word modes, f32 outputs, norm-relative
RTOL_F64 = 1e-9   # f32 activations with f64 sums, norm-relative


def torch():
    import torch as _t
    return _t


def dev(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a)).to("cuda")


def host(t):
    torch().cuda.synchronize()
    return t.cpu().numpy()


def upload_weights(q, s):
    return dev(q), dev(s.view(np.int16))


def upload_act(mode, act, rows, k):
    """Oracle producer output -> device tensors in the library's layout."""
    t = torch()
    if mode == "f32":
        return dev(act[0]), None
    if mode == "i8":
        return dev(act[0]), dev(act[1])
    xh, xl, xd = act
    return dev(np.stack([xh, xl])), dev(xd)


def act_to_numpy(mode, xq, xd):
    """Library activation tensors -> oracle tuple."""
    if mode == "f32":
        return (host(xq),)
    if mode == "i8":
        return host(xq), host(xd)
    both = host(xq)
    return both[0], both[1], host(xd)


def check_close(mode, y, y_o, norm, out_f64=False, what=""):
    """Norm-relative comparison; returns the worst error in units of the tolerance."""
    y = np.asarray(y, dtype=np.float64)
    y_o = np.asarray(y_o, dtype=np.float64)
    if mode == "f32":
        tol = RTOL_F64 * norm
        if not out_f64:
            tol = tol + np.spacing(np.abs(y_o).astype(np.float32)).astype(np.float64)
    else:
        tol = RTOL_Q * norm
    tol = tol + 1e-300
    err = np.abs(y - y_o)
    worst = float(np.max(err / tol)) if err.size else 0.0
    assert np.all(err <= tol), f"{what}: worst error {worst:.3g} x tolerance"
    return worst


def no_device_error():
    assert native.q8_device_error() == 0


def _bits(a):
    return a.view(np.uint8) if a.dtype != np.float32 else a.view(np.uint32)


def assert_codes_match(got, want, r=None, what=""):
    """Producer outputs (codes and scales, or f32 x) bit for bit.  With the
    rows' f64 RMS scales r (the oracle's), a mismatching row is classified:
    one whose r lies near an f32 rounding boundary (oracle.near_tie) may
    round rf the other way under another correct evaluation; such a row is
    reported as an expected failure, never passed silently; any other
    mismatch fails."""
    from oracle import oracle as orc
    bad_rows = set()
    for a, b in zip(got, want):
        a2, b2 = _bits(a), _bits(b)
        if a2.shape != b2.shape:
            raise AssertionError(f"{what}: shape {a2.shape} != {b2.shape}")
        if not np.array_equal(a2, b2):
            rows = np.nonzero(np.any((a2 != b2).reshape(a2.shape[0], -1), axis=1))[0]
            bad_rows.update(int(m) for m in rows)
    if not bad_rows:
        return
    rows = sorted(bad_rows)
    if r is None:
        raise AssertionError(f"{what}: codes differ in rows {rows[:8]}")
    near = orc.near_tie(np.asarray(r)[rows])
    if not np.all(near):
        far = [m for m, f in zip(rows, near) if not f]
        raise AssertionError(f"{what}: codes differ in rows {far[:8]}, not near an f32 tie")
    pytest.xfail(f"{what}: codes differ only in near-tie rows {rows[:8]} "
                 f"(r within {orc.NEAR_TIE_REL:.1e} of an f32 rounding boundary)")

"""Helpers for the GPU parity tests: upload seeded numpy inputs, run the
library through its C ABI binding, and compare with the oracle."""
import numpy as np

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

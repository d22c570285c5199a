"""Thin ctypes binding of libq8proj.so (the C ABI in include/q8proj.h).

Every function here has the C entry point's name and only marshals arguments:
torch tensors become device pointers, the current torch stream becomes the
cudaStream_t, and a non-zero status becomes a Q8Error.  All computation runs
in the library's CUDA kernels; there is no other path.  If the library is
missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libq8proj.so")

Q8_ACT_F32, Q8_ACT_I8, Q8_ACT_I8X2 = 0, 1, 2
MODES = {"f32": Q8_ACT_F32, "i8": Q8_ACT_I8, "i8x2": Q8_ACT_I8X2}
Q8_MAX_ROWS = 256

_STATUS = ["Q8_OK", "Q8_ERR_ARG", "Q8_ERR_SHAPE", "Q8_ERR_ALIGN", "Q8_ERR_MODE",
           "Q8_ERR_CUDA", "Q8_ERR_UNSUPPORTED", "Q8_ERR_WORKSPACE"]

# Every symbol the header declares, with (restype, argtypes).
_i64, _vp, _int, _sz = C.c_int64, C.c_void_p, C.c_int, C.c_size_t
SIGNATURES = {
    "q8_status_str": (C.c_char_p, [_int]),
    "q8_version": (_int, []),
    "q8_last_cuda_error": (_int, []),
    "q8_device_error": (_int, [_vp, _vp]),
    "q8_set_pdl": (None, [_int]),
    "q8_pack": (_int, [_vp, _i64, _i64, _vp, _vp, _vp, _vp]),
    "act_quant": (_int, [_int, _vp, _i64, _i64, _int, _vp, C.c_float, _vp, _vp, _vp]),
    "act_quant_residual": (_int, [_int, _vp, _vp, _vp, _i64, _i64, _vp, C.c_float, _vp, _vp, _vp]),
    "act_quant_swiglu": (_int, [_int, _vp, _i64, _i64, _vp, _vp, _vp]),
    "q8_proj": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _int, _vp]),
    "q8_proj_chunk": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp]),
    "q8_proj_fused": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _i64, _vp, C.c_float, _vp, _int,
                             _vp, _sz, _vp]),
    "q8_proj_fused_workspace": (_sz, [_int, _i64, _i64]),
    "q8_proj_fused_residual": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _i64, _vp, C.c_float,
                                      _vp, _int, _vp, _sz, _vp]),
    "q8_proj_fused_swiglu": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _i64, _vp, _int, _vp, _sz, _vp]),
    "q8_proj_fused_kv": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _i64, _vp, C.c_float, _vp, _vp, _i64,
                                _i64, _vp, _vp, _i64, _vp, _sz, _vp]),
    "head_argmax": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _sz,
                           _vp]),
    "head_argmax_workspace": (_sz, [_i64]),
    "q8_debug_block_dots": (_int, [_int, _vp, _vp, _i64, _i64, _i64, _vp, _int, _vp]),
    "q8_debug_row_geometry": (_int, [_int, _i64, _i64, _i64, _int, _int, _vp]),
    "q8_debug_row_geometry_fused": (_int, [_int, _int, _i64, _i64, _int, _int, _vp]),
    "q8_debug_chunk_plan": (_int, [_int, _i64, _i64, _i64, _int, _vp]),
    "head_argmax_noalloc": (_int, [_int, _vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp, _vp,
                                   _vp]),
    "head_argmax_noalloc_scratch_bytes": (_sz, []),
}


class Q8Error(RuntimeError):
    def __init__(self, status: int, where: str, cuda_err: int = 0):
        name = _STATUS[status] if 0 <= status < len(_STATUS) else f"status {status}"
        msg = f"{where}: {name}" + (f" (cuda error {cuda_err})" if cuda_err else "")
        super().__init__(msg)
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libq8proj.so (raises OSError when it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise OSError(f"libq8proj.so not found at {p}; build it with "
                              "q8_quantized_projection_gb300.build.build()")
            lib = C.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise Q8Error(status, where, load().q8_last_cuda_error() if status == 5 else 0)


def _mode(mode) -> int:
    return MODES[mode] if isinstance(mode, str) else int(mode)


def q8_version() -> int:
    return load().q8_version()


def q8_set_pdl(enable: bool) -> None:
    load().q8_set_pdl(1 if enable else 0)


def q8_device_error(stream=None) -> int:
    code = C.c_int32(0)
    _check(load().q8_device_error(C.byref(code), _stream(stream)), "q8_device_error")
    return code.value


def q8_pack(w, q, s, overflow=None, stream=None):
    n, k = w.shape
    _check(load().q8_pack(_ptr(w), n, k, _ptr(q), _ptr(s), _ptr(overflow), _stream(stream)),
           "q8_pack")


def act_quant(mode, h, xq, xd, norm=False, gain=None, eps=1e-5, stream=None):
    rows, k = h.shape
    _check(load().act_quant(_mode(mode), _ptr(h), rows, k, 1 if norm else 0, _ptr(gain),
                            float(eps), _ptr(xq), _ptr(xd), _stream(stream)), "act_quant")


def act_quant_residual(mode, h, r, xq, xd, s_out=None, gain=None, eps=1e-5, stream=None):
    rows, k = h.shape
    _check(load().act_quant_residual(_mode(mode), _ptr(h), _ptr(r), _ptr(s_out), rows, k, _ptr(gain),
                                     float(eps), _ptr(xq), _ptr(xd), _stream(stream)),
           "act_quant_residual")


def act_quant_swiglu(mode, gu, xq, xd, stream=None):
    rows, k2 = gu.shape
    _check(load().act_quant_swiglu(_mode(mode), _ptr(gu), rows, k2 // 2, _ptr(xq), _ptr(xd),
                                   _stream(stream)), "act_quant_swiglu")


def q8_proj(mode, q, s, xq, xd, rows, y, out_f64=False, stream=None):
    n, k = q.shape
    _check(load().q8_proj(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(xq), _ptr(xd), rows, _ptr(y),
                          1 if out_f64 else 0, _stream(stream)), "q8_proj")


def q8_proj_chunk(mode, q, s, xq, xd, T, y, stream=None):
    n, k = q.shape
    _check(load().q8_proj_chunk(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(xq), _ptr(xd), T,
                                _ptr(y), _stream(stream)), "q8_proj_chunk")


def q8_proj_fused_workspace(mode, rows, k) -> int:
    return int(load().q8_proj_fused_workspace(_mode(mode), rows, k))


def q8_proj_fused(mode, q, s, h, y, workspace, gain=None, eps=1e-5, out_f64=False, stream=None):
    n, k = q.shape
    rows = h.shape[0]
    _check(load().q8_proj_fused(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(h), rows, _ptr(gain),
                                float(eps), _ptr(y), 1 if out_f64 else 0, _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)),
           "q8_proj_fused")


def q8_proj_fused_residual(mode, q, s, h, r, y, workspace, s_out=None, gain=None, eps=1e-5,
                           out_f64=False, stream=None):
    n, k = q.shape
    rows = h.shape[0]
    _check(load().q8_proj_fused_residual(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(h), _ptr(r),
                                         _ptr(s_out), rows, _ptr(gain), float(eps), _ptr(y),
                                         1 if out_f64 else 0, _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream)),
           "q8_proj_fused_residual")


def q8_proj_fused_swiglu(mode, q, s, gu, y, workspace, out_f64=False, stream=None):
    n, k = q.shape
    rows = gu.shape[0]
    if gu.shape[1] != 2 * k:
        raise ValueError("gate+up rows must hold 2K values")
    _check(load().q8_proj_fused_swiglu(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(gu), rows, _ptr(y),
                                       1 if out_f64 else 0, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "q8_proj_fused_swiglu")


def q8_proj_fused_kv(mode, q, s, h, y, workspace, pos, kv_col, k_cache, v_cache, gain=None,
                     eps=1e-5, stream=None):
    """k_cache, v_cache: [rows, n_pos, kv_dim] float32; pos: int32 [rows] on the device."""
    n, k = q.shape
    rows = h.shape[0]
    _, n_pos, kv_dim = k_cache.shape
    _check(load().q8_proj_fused_kv(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(h), rows, _ptr(gain),
                                   float(eps), _ptr(y), _ptr(pos), kv_col, kv_dim, _ptr(k_cache),
                                   _ptr(v_cache), n_pos, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "q8_proj_fused_kv")


def head_argmax_workspace(rows) -> int:
    return int(load().head_argmax_workspace(rows))


def head_argmax(mode, q, s, xq, xd, rows, tok, workspace, maxval=None, logits=None, stream=None):
    n, k = q.shape
    _check(load().head_argmax(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(xq), _ptr(xd), rows,
                              _ptr(tok), _ptr(maxval), _ptr(logits), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)),
           "head_argmax")


def head_argmax_noalloc(mode, q, s, xq, xd, rows, tok, maxval=None, logits=None, stream=None):
    """head_argmax with the library's own fixed scratch (no workspace, no allocation)."""
    n, k = q.shape
    _check(load().head_argmax_noalloc(_mode(mode), _ptr(q), _ptr(s), n, k, _ptr(xq), _ptr(xd),
                                      rows, _ptr(tok), _ptr(maxval), _ptr(logits),
                                      _stream(stream)), "head_argmax_noalloc")


def q8_debug_block_dots(mode, q, xq, rows, isum, path=0, stream=None):
    n, k = q.shape
    _check(load().q8_debug_block_dots(_mode(mode), _ptr(q), _ptr(xq), n, k, rows, _ptr(isum),
                                      int(path), _stream(stream)), "q8_debug_block_dots")


ROW_GEOMETRY_FIELDS = ("R", "KS", "nks", "PB", "npr", "nprr", "RS", "rpw", "items", "stride",
                       "stage_bytes", "nstages", "r0", "r1", "sbrows", "ep_off", "ring_bytes",
                       "psum_bytes", "psum_row_unit", "cpl", "warps")


def q8_debug_row_geometry(mode, rows, n, k, grid, cta):
    """The decode kernel's stage geometry for one CTA (host only), as a dict;
    None when the projection would run its slice-major kernel instead."""
    out = (C.c_int64 * len(ROW_GEOMETRY_FIELDS))()
    st = load().q8_debug_row_geometry(_mode(mode), int(rows), int(n), int(k), int(grid), int(cta),
                                      C.cast(out, C.c_void_p))
    if st == 6:   # Q8_ERR_UNSUPPORTED
        return None
    _check(st, "q8_debug_row_geometry")
    return dict(zip(ROW_GEOMETRY_FIELDS, list(out)))


FUSED_PRODUCERS = {"plain": 0, "residual": 1, "swiglu": 2}


def q8_debug_row_geometry_fused(mode, prod, n, k, grid, cta):
    """The same fields for a fused call's decode launch (rows = 1), prod one of
    FUSED_PRODUCERS; None when the fused producer does not take K."""
    out = (C.c_int64 * len(ROW_GEOMETRY_FIELDS))()
    st = load().q8_debug_row_geometry_fused(_mode(mode), FUSED_PRODUCERS[prod], int(n), int(k),
                                            int(grid), int(cta), C.cast(out, C.c_void_p))
    if st == 6:   # Q8_ERR_UNSUPPORTED
        return None
    _check(st, "q8_debug_row_geometry_fused")
    return dict(zip(ROW_GEOMETRY_FIELDS, list(out)))


CHUNK_PLAN_FIELDS = ("TT", "ks", "tiles", "clusters", "waves", "stages")


def q8_debug_chunk_plan(mode, n, k, t, argmax=False):
    """The tensor-core path's launch plan for a projection of t rows (host
    side, the current device's occupancy), as a dict."""
    out = (C.c_int64 * len(CHUNK_PLAN_FIELDS))()
    st = load().q8_debug_chunk_plan(_mode(mode), int(n), int(k), int(t), int(bool(argmax)),
                                    C.cast(out, C.c_void_p))
    _check(st, "q8_debug_chunk_plan")
    return dict(zip(CHUNK_PLAN_FIELDS, list(out)))


# ------------------------------------------------------------ buffer helpers

def activation_buffers(mode, rows, k, device="cuda"):
    """Allocate (xq, xd) device tensors in the mode's activation layout."""
    import torch
    m = _mode(mode)
    if m == Q8_ACT_F32:
        return torch.empty((rows, k), dtype=torch.float32, device=device), None
    planes = 1 if m == Q8_ACT_I8 else 2
    xq = torch.empty((planes, rows, k), dtype=torch.int8, device=device)
    xd = torch.empty((rows, k // 32), dtype=torch.float32, device=device)
    return (xq[0] if planes == 1 else xq), xd


def argmax_workspace(rows, device="cuda"):
    """A zeroed head_argmax workspace (the counter word must start at zero)."""
    import torch
    nbytes = head_argmax_workspace(rows)
    return torch.zeros((nbytes + 15) // 16 * 16, dtype=torch.uint8, device=device)

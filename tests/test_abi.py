"""Host-side checks of the C ABI: every declared symbol is exported and bound,
and argument validation answers before anything touches a GPU."""
import ctypes as C
import os
import re

import pytest

from q8_quantized_projection_gb300 import build, native

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "q8proj.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text,
                       flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return native.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("q8_pack", "act_quant", "q8_proj", "q8_proj_chunk", "q8_proj_fused",
               "head_argmax", "q8_debug_block_dots"):
        assert fn in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert set(names) == set(native.SIGNATURES), set(names) ^ set(native.SIGNATURES)
    for n in names:
        assert hasattr(lib, n), n


def test_status_names_and_version(lib):
    assert lib.q8_version() == 106
    for i, name in enumerate(native._STATUS):
        assert lib.q8_status_str(i).decode() == name
    assert lib.q8_status_str(99).decode() == "Q8_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    assert lib.q8_proj_fused_workspace(0, 1, 4096) == 16384 + 512
    assert lib.q8_proj_fused_workspace(1, 3, 4096) == 12288 + 1536
    assert lib.q8_proj_fused_workspace(2, 3, 4096) == 24576 + 1536
    assert lib.q8_proj_fused_workspace(7, 3, 4096) == 0
    # tensor-core ticket + one key per row (up to 256 rows) + the CUDA-core
    # path's ticket and one candidate per CTA (up to 1024) and row of a group
    assert lib.head_argmax_workspace(1) == 256 + 8 * 256 + 256 + 1024 * 16
    assert lib.head_argmax_workspace(40) == 256 + 8 * 256 + 256 + 1024 * 16 * 16
    assert lib.head_argmax_workspace(0) == 0
    assert lib.head_argmax_noalloc_scratch_bytes() == lib.head_argmax_workspace(256)


A = C.c_void_p(4096)          # a 16-byte aligned non-null placeholder (never dereferenced)
U = C.c_void_p(4096 + 4)      # misaligned placeholder


@pytest.mark.parametrize("args,status", [
    ((0, None, A, 8, 64, A, A, 1, A, 0, None), 1),      # null q
    ((0, A, A, 8, 60, A, A, 1, A, 0, None), 2),         # K not a multiple of 32
    ((0, A, A, 0, 64, A, A, 1, A, 0, None), 2),         # N = 0
    ((1, A, A, 8, 64, A, A, 0, A, 0, None), 2),         # rows = 0
    ((1, A, A, 8, 64, A, A, 257, A, 0, None), 2),       # rows above the maximum
    ((1, U, A, 8, 64, A, A, 1, A, 0, None), 3),         # misaligned q
    ((3, A, A, 8, 64, A, A, 1, A, 0, None), 4),         # unknown mode
    ((1, A, A, 8, 64, A, A, 1, A, 1, None), 4),         # f64 output outside the f32 mode
    ((1, A, A, 8, 64, A, None, 1, A, 0, None), 1),      # one-word mode needs scales
])
def test_q8_proj_rejects_bad_arguments(lib, args, status):
    assert lib.q8_proj(*args) == status


def test_other_entry_points_reject_bad_arguments(lib):
    assert lib.q8_pack(None, 4, 64, A, A, None, None) == 1
    assert lib.q8_pack(A, 4, 48, A, A, None, None) == 2
    assert lib.act_quant(1, A, 1, 64, 2, None, 1e-5, A, A, None) == 1
    assert lib.act_quant(1, A, 1, 64, 1, None, -1.0, A, A, None) == 1
    assert lib.act_quant(5, A, 1, 64, 1, None, 1e-5, A, A, None) == 4
    assert lib.q8_proj_chunk(1, A, A, 8, 64, A, A, 300, A, None) == 2
    assert lib.q8_proj_fused(1, A, A, 8, 64, A, 1, None, 1e-5, A, 0, None, 0, None) == 7
    assert lib.q8_proj_fused(1, A, A, 8, 64, A, 1, None, 1e-5, A, 0, A, 16, None) == 7
    assert lib.head_argmax(1, A, A, 8, 64, A, A, 1, A, None, None, A, 16, None) == 7
    assert lib.head_argmax(1, A, A, 8, 64, A, A, 1, None, None, None, A, 1 << 20, None) == 1
    assert lib.q8_debug_block_dots(0, A, A, 8, 64, 1, A, 0, None) == 4
    assert lib.q8_debug_block_dots(1, A, A, 1 << 20, 4096, 256, A, 0, None) == 2


def test_widened_entry_points_reject_bad_arguments(lib):
    # residual before the norm: r required, s_out aligned and disjoint from h and r
    f = lib.act_quant_residual
    assert f(1, A, None, None, 1, 64, None, 1e-5, A, A, None) == 1
    assert f(1, A, U, None, 1, 64, None, 1e-5, A, A, None) == 3
    assert f(1, A, C.c_void_p(8192), A, 1, 64, None, 1e-5, A, A, None) == 1   # s_out == h
    assert f(5, A, C.c_void_p(8192), None, 1, 64, None, 1e-5, A, A, None) == 4
    g = lib.q8_proj_fused_residual
    assert g(1, A, A, 8, 64, None, A, None, 1, None, 1e-5, A, 0, A, 1 << 20, None) == 1
    assert g(1, A, A, 8, 64, A, A, None, 0, None, 1e-5, A, 0, A, 1 << 20, None) == 2
    assert g(1, A, A, 8, 64, A, None, None, 1, None, 1e-5, A, 0, A, 1 << 20, None) == 1
    # SwiGLU producer
    assert lib.act_quant_swiglu(5, A, 1, 64, A, A, None) == 4
    assert lib.act_quant_swiglu(1, U, 1, 64, A, A, None) == 3
    assert lib.q8_proj_fused_swiglu(1, A, A, 8, 64, A, 1, A, 0, None, 0, None) == 7
    # KV-cache-row epilogue
    kv = lib.q8_proj_fused_kv
    ok = dict(pos=A, col=0, dim=2, kc=C.c_void_p(1 << 20), vc=C.c_void_p(1 << 21), npos=16)

    def call(N=8, K=64, rows=1, **over):
        a = dict(ok, **over)
        return kv(1, A, A, N, K, A, rows, None, 1e-5, A, a["pos"], a["col"], a["dim"], a["kc"],
                  a["vc"], a["npos"], A, 1 << 20, None)

    assert call(pos=None) == 1
    assert call(kc=None) == 1
    assert call(rows=0) == 2
    assert call(dim=0) == 2
    assert call(col=5, dim=2) == 2                 # V slice past N
    assert call(col=-1) == 2
    assert call(dim=1 << 62) == 2                  # no overflow in the range check
    assert call(npos=0) == 2
    assert call(npos=1 << 31) == 2                 # positions are int32
    assert call(N=1 << 20, dim=1 << 18, npos=(1 << 31) - 1) == 2   # a cache beyond 2^40 bytes
    assert call(K=16416) == 6                      # the decode kernel's K
    assert call(pos=U) == 3
    assert call(vc=C.c_void_p((1 << 20) + 16)) == 1   # K and V caches overlap

def test_chunk_plan_host_errors(lib):
    """q8_debug_chunk_plan checks its arguments before touching a device."""
    import ctypes as C
    out = (C.c_int64 * 6)()
    assert lib.q8_debug_chunk_plan(3, 128, 4096, 16, 0, C.cast(out, C.c_void_p)) == 4     # mode
    assert lib.q8_debug_chunk_plan(1, 128, 4100, 16, 0, C.cast(out, C.c_void_p)) == 2     # K % 256
    assert lib.q8_debug_chunk_plan(1, 128, 4096, 0, 0, C.cast(out, C.c_void_p)) == 2      # T
    assert lib.q8_debug_chunk_plan(1, 128, 4096, 257, 0, C.cast(out, C.c_void_p)) == 2    # T > max
    assert lib.q8_debug_chunk_plan(1, 128, 4096, 16, 0, None) == 1                         # out

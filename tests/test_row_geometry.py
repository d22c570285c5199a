"""Host-side checks of the decode kernel's stage geometry (no GPU needed).

The geometry comes from the library itself (q8_debug_row_geometry runs the
same host/device function the kernel evaluates per CTA); these tests check the
invariants the kernel's indexing relies on: every stage fits its ring slot,
the slots fit the ring, a stage's (row, part) pairs are served by whole warp
groups, the parts tile each slice, the part sums of a super-block fit their
area, and every CTA owns a contiguous share of the rows.
"""
import pytest

from q8_quantized_projection_gb300 import build, native

# K values: the configs' rows, powers of two, and lengths that leave ragged
# parts, ragged chunk columns and ragged slices
KS = [32, 64, 96, 160, 512, 992, 1024, 1056, 2048, 3104, 4096, 4128, 5120, 8192, 8224,
      11008, 14336, 16384, 16416, 24576, 32768, 65536]
KINDS = [("f32", 1), ("i8", 1), ("i8", 2), ("i8", 4), ("i8", 8), ("i8x2", 1), ("i8x2", 2),
         ("i8x2", 4)]
STAGE = 32768          # weight bytes of one stage at most
MAX_STAGES = 16


@pytest.fixture(scope="module")
def lib():
    build.build()
    return native.load()


def geometry(mode, rows, n, k, grid, cta):
    return native.q8_debug_row_geometry(mode, rows, n, k, grid, cta)


def check_invariants(mode, rows, n, k, grid, cta, g):
    where = f"{mode} rows={rows} N={n} K={k} cta={cta}/{grid}: {g}"
    R, KS, nks, PB, npr, nprr = g["R"], g["KS"], g["nks"], g["PB"], g["npr"], g["nprr"]
    RS, rpw, items, stride = g["RS"], g["rpw"], g["items"], g["stride"]
    assert R >= rows and R in (1, 2, 4, 8), where
    # slices tile the row; parts tile the slice
    assert KS % 32 == 0 and KS * (nks - 1) < k <= KS * nks, where
    assert npr & (npr - 1) == 0 and 1 <= nprr <= npr <= g["warps"], where
    assert PB % 32 == 0 and PB <= 512 * g["cpl"], where
    assert PB * (nprr - 1) < KS <= PB * nprr, where
    last = k - KS * (nks - 1)
    assert last % 32 == 0 and 0 < last <= KS, where
    # a stage: RS whole row-slices in one slot; its pairs served by warp groups
    assert RS & (RS - 1) == 0 and RS * KS <= STAGE, where
    assert items * rpw == RS * npr and g["warps"] % items == 0, where
    assert stride == g["warps"] // items, where
    assert g["stage_bytes"] % 1024 == 0 and g["stage_bytes"] >= RS * KS, where
    # every warp group owns at least one ring slot; the slots fit the ring
    assert stride <= g["nstages"] <= MAX_STAGES, where
    assert g["nstages"] * g["stage_bytes"] <= g["ring_bytes"], where
    # part sums of a super-block fit their area
    assert g["sbrows"] >= RS and g["sbrows"] % RS == 0, where
    assert g["sbrows"] * nks * nprr * g["psum_row_unit"] <= g["psum_bytes"], where
    # the CTA's rows
    assert g["r0"] == n * cta // grid and g["r1"] == n * (cta + 1) // grid, where
    if mode == "f32":
        # a lane owns one 32-value block: a part is 32 lanes x 32 bytes, and a
        # warp serves four rows RS/4 apart
        assert R == 1 and PB == 1024 and rpw == 4 and RS % 4 == 0, where
        # each (slice, part) keeps its binade beside the part sums
        assert g["ep_off"] == g["psum_bytes"] and nks * nprr * 2 <= 1024, where
        if nks == 1 and k <= 4096:
            # the shared block conversion: 128 bytes a block in the part-sum
            # area, the blocks' binades after the parts' binades
            assert (k // 32) * 128 <= g["psum_bytes"], where
            assert 4 * k <= g["psum_bytes"], where   # the fused RMS pass's staged input
        if k <= 16384:
            # the blocks' binades of a shared block conversion (up to the fused
            # producer's 16384 values) follow the parts' 1024 bytes
            assert nprr * nks * 2 <= 1024 and 1024 + (k // 32) * 2 <= 2048, where
            # warp w converts the w-th 1024 values: slices of whole parts
            assert nks == 1 or KS % PB == 0, where
    else:
        assert rpw in (1, 2) and rpw <= RS, where


@pytest.mark.parametrize("mode,rows", KINDS)
def test_decode_geometry_invariants(lib, mode, rows):
    served = 0
    for k in KS:
        for n in (1, 7, 152, 4096, 28672):
            grid = min(152, n)
            for cta in sorted({0, grid // 2, grid - 1}):
                g = geometry(mode, rows, n, k, grid, cta)
                if g is None:
                    continue
                served += 1
                check_invariants(mode, rows, n, k, grid, cta, g)
    assert served > 0


@pytest.mark.parametrize("mode,rows", KINDS)
def test_decode_kernel_serves_the_configs(lib, mode, rows):
    # every K of the layer configs and the decode kernel's fused-producer limit
    for k in (1024, 4096, 14336, 16384):
        assert geometry(mode, rows, 4096, k, 152, 0) is not None, (mode, rows, k)


def test_rows_of_all_ctas_partition_the_matrix(lib):
    for n in (1, 5, 151, 152, 153, 4096, 6144):
        grid = min(152, n)
        spans = [geometry("i8", 1, n, 4096, grid, c) for c in range(grid)]
        assert spans[0]["r0"] == 0 and spans[-1]["r1"] == n
        for a, b in zip(spans, spans[1:]):
            assert a["r1"] == b["r0"] and a["r1"] > a["r0"]


def test_geometry_argument_errors(lib):
    out = (native.C.c_int64 * 21)()
    f = lib.q8_debug_row_geometry
    assert f(1, 1, 100, 4096, 10, 0, None) == 1          # no output buffer
    assert f(9, 1, 100, 4096, 10, 0, out) == 4           # mode
    assert f(1, 1, 100, 4100, 10, 0, out) == 2           # K % 32
    assert f(1, 0, 100, 4096, 10, 0, out) == 2           # rows
    assert f(1, 1, 100, 4096, 10, 10, out) == 1          # cta outside the grid
    assert f(1, 1, 5, 4096, 10, 0, out) == 1             # more CTAs than rows
    assert f(0, 2, 100, 4096, 10, 0, out) == 6           # f32 decodes one row a launch
    assert f(1, 9, 100, 4096, 10, 0, out) == 6           # one-word: 8 rows a pass at most


def test_f32_two_slice_rows_take_the_slice_inner_order(lib):
    # rows of 8,192 < K <= 16,384 values run in two slices; with two warp groups
    # and an even ring each group's slots then always carry one slice (the
    # kernel's slice-inner stage order, taken by the unfused f32 launches)
    for k in (8224, 11008, 14336, 16384):
        g = geometry("f32", 1, 4096, k, 152, 0)
        assert g["nks"] == 2 and g["stride"] % g["nks"] == 0, g
        assert g["nstages"] % g["stride"] == 0, g


@pytest.mark.parametrize("mode", ["f32", "i8", "i8x2"])
@pytest.mark.parametrize("prod", ["plain", "residual", "swiglu"])
def test_fused_decode_geometry(lib, mode, prod):
    # a fused call's decode launch (rows = 1, up to the producer's 16384
    # values): the same invariants; in f32 mode the residual and SwiGLU
    # producers above 4096 values give up the ring's last 4K bytes (rounded up
    # to 1 KB) to the converted activation, and the stages fit what is left
    full = 196608 if mode == "f32" else 163840
    for k in [kk for kk in KS if kk <= 16384]:
        for n in (7, 4096, 28672):
            grid = min(152, n)
            for cta in sorted({0, grid - 1}):
                g = native.q8_debug_row_geometry_fused(mode, prod, n, k, grid, cta)
                assert g is not None, (mode, n, k)
                check_invariants(mode, 1, n, k, grid, cta, g)
                shorter = mode == "f32" and prod != "plain" and k > 4096
                planes = (4 * k + 1023) // 1024 * 1024 if shorter else 0
                assert g["ring_bytes"] == full - planes, (mode, k, g)
                if planes:
                    # the converting warps: one a (slice, part), all 16 at most
                    assert g["nks"] * g["nprr"] <= g["warps"], (k, g)
                    assert g["nstages"] >= 3, (k, g)
                else:
                    assert g == native.q8_debug_row_geometry(mode, 1, n, k, grid, cta)
    assert native.q8_debug_row_geometry_fused(mode, prod, 4096, 16416, 152, 0) is None


def test_fused_geometry_argument_errors(lib):
    out = (native.C.c_int64 * 21)()
    f = lib.q8_debug_row_geometry_fused
    assert f(0, 0, 100, 4096, 10, 0, None) == 1          # no output buffer
    assert f(0, 3, 100, 4096, 10, 0, out) == 1           # producer kind
    assert f(9, 0, 100, 4096, 10, 0, out) == 4           # mode
    assert f(0, 1, 100, 4100, 10, 0, out) == 2           # K % 32
    assert f(0, 2, 100, 4096, 10, 10, out) == 1          # cta outside the grid
    assert f(0, 1, 100, 16416, 10, 0, out) == 6          # beyond the fused producer's row

// geometry.cu -- the decode kernel's stage geometry seen from the host, so that
// its invariants (ring, scale ring and part-sum bounds, rows a warp, the warp
// groups' slot ownership) can be checked without a GPU.  Nothing here touches
// a device.
#include "gemv_row.cuh"
#include "q8proj.h"

namespace q8 {
namespace {

constexpr int kGeoFields = 21;

// One CTA's geometry for a kernel instantiated with R activation rows, in the
// order q8proj.h documents; false when the decode kernel does not take K.
template <int MODE, int R, bool FUSE = false, int PROD = kProdPlain>
bool row_geometry_of(int64_t N, int64_t K, int grid, int cta, int64_t* out) {
    if (!row_kernel_fits<MODE, R>(K)) return false;
    using A = typename AccT<MODE>::T;
    const int ring = row_ring_of<MODE, FUSE, PROD>(K);
    const RowGeo g = row_geo(N, K, grid, cta, row_cpl<MODE, R>(), int(R * sizeof(A)),
                             row_rpw<MODE, R>(), ring, row_part_extra<MODE, R>());
    const int64_t v[kGeoFields] = {R,          g.KS,          g.nks,      g.PB,
                                   g.npr,      g.nprr,        g.RS,       g.rpw,
                                   g.items,    g.stride,      g.stage_bytes, g.nstages,
                                   g.r0,       g.r1,          g.sbrows,   g.ep_off,
                                   ring,       kRowPsumBytes, int64_t(R * sizeof(A)),
                                   row_cpl<MODE, R>(), kRowWarps};
    for (int i = 0; i < kGeoFields; ++i) out[i] = v[i];
    return true;
}

}  // namespace
}  // namespace q8

extern "C" q8_status q8_debug_row_geometry(int mode, int64_t rows, int64_t N, int64_t K, int grid,
                                           int cta, int64_t* out) {
    using namespace q8;
    if (!out) return Q8_ERR_ARG;
    if (mode < Q8_ACT_F32 || mode > Q8_ACT_I8X2) return Q8_ERR_MODE;
    if (N < 1 || K < Q8_QK || K % Q8_QK != 0 || K > (int64_t(1) << 24) || rows < 1)
        return Q8_ERR_SHAPE;
    if (grid < 1 || cta < 0 || cta >= grid || int64_t(grid) > N) return Q8_ERR_ARG;
    // the same choice of kernel as the projection's dispatch: the first
    // instantiation with at least `rows` rows whose part sums fit
    bool ok = false;
    switch (mode) {
        case Q8_ACT_F32:
            ok = rows <= 1 && row_geometry_of<0, 1>(N, K, grid, cta, out);
            break;
        case Q8_ACT_I8:
            ok = (rows <= 1 && row_geometry_of<1, 1>(N, K, grid, cta, out)) ||
                 (rows <= 2 && row_geometry_of<1, 2>(N, K, grid, cta, out)) ||
                 (rows <= 4 && row_geometry_of<1, 4>(N, K, grid, cta, out)) ||
                 (rows <= 8 && row_geometry_of<1, 8>(N, K, grid, cta, out));
            break;
        default:
            ok = (rows <= 1 && row_geometry_of<2, 1>(N, K, grid, cta, out)) ||
                 (rows <= 2 && row_geometry_of<2, 2>(N, K, grid, cta, out)) ||
                 (rows <= 4 && row_geometry_of<2, 4>(N, K, grid, cta, out));
            break;
    }
    return ok ? Q8_OK : Q8_ERR_UNSUPPORTED;
}

extern "C" q8_status q8_debug_row_geometry_fused(int mode, int prod, int64_t N, int64_t K, int grid,
                                                 int cta, int64_t* out) {
    using namespace q8;
    if (!out) return Q8_ERR_ARG;
    if (mode < Q8_ACT_F32 || mode > Q8_ACT_I8X2) return Q8_ERR_MODE;
    if (prod < kProdPlain || prod > kProdSwiglu) return Q8_ERR_ARG;
    if (N < 1 || K < Q8_QK || K % Q8_QK != 0 || K > (int64_t(1) << 24)) return Q8_ERR_SHAPE;
    if (grid < 1 || cta < 0 || cta >= grid || int64_t(grid) > N) return Q8_ERR_ARG;
    if (K > kFusedMaxK) return Q8_ERR_UNSUPPORTED;   // the producer's row
    bool ok = false;
    switch (mode) {
        case Q8_ACT_F32:
            ok = prod == kProdPlain      ? row_geometry_of<0, 1, true, kProdPlain>(N, K, grid, cta, out)
                 : prod == kProdResidual ? row_geometry_of<0, 1, true, kProdResidual>(N, K, grid, cta, out)
                                         : row_geometry_of<0, 1, true, kProdSwiglu>(N, K, grid, cta, out);
            break;
        case Q8_ACT_I8: ok = row_geometry_of<1, 1, true>(N, K, grid, cta, out); break;
        default: ok = row_geometry_of<2, 1, true>(N, K, grid, cta, out); break;
    }
    return ok ? Q8_OK : Q8_ERR_UNSUPPORTED;
}

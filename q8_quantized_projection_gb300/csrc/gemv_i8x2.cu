// gemv_i8x2.cu -- instantiations of the CUDA-core projection for activation
// mode 2: the row-per-lane kernel (gemv_rpl.cuh) for 1-4 rows with K % 1024 ==
// 0 (plain projections, the LM head's arg-max and fused decode steps), else
// the decode kernel (gemv_row.cuh: other K); the slice-major kernel (gemv.cuh)
// for more rows.  One file per mode so the build runs in parallel.
#include "gemv_row.cuh"
#include "gemv_rpl.cuh"

namespace q8 {

template <bool ARGMAX>
static cudaError_t dispatch_rows(const GemvArgs& a, const LaunchCtx& ctx) {
    // a weight row a lane (K % 1024 == 0), plain or with the arg-max
    if (a.rows <= 1 && rpl_fits(a)) return launch_gemv_rpl_t<2, 1, false, kProdPlain, false, ARGMAX>(a, ctx);
    if (a.rows <= 2 && rpl_fits(a)) return launch_gemv_rpl_t<2, 2, false, kProdPlain, false, ARGMAX>(a, ctx);
    if (a.rows <= 4 && rpl_fits(a)) return launch_gemv_rpl_t<2, 4, false, kProdPlain, false, ARGMAX>(a, ctx);
    if (a.rows <= 1 && row_kernel_fits<2, 1>(a.K)) return launch_gemv_row_t<2, 1, ARGMAX>(a, ctx);
    if (a.rows <= 2 && row_kernel_fits<2, 2>(a.K)) return launch_gemv_row_t<2, 2, ARGMAX>(a, ctx);
    if (a.rows <= 4 && row_kernel_fits<2, 4>(a.K)) return launch_gemv_row_t<2, 4, ARGMAX>(a, ctx);
    if (a.rows <= 4) return launch_gemv_t<2, 4, ARGMAX>(a, ctx);
    if (a.rows <= 8) return launch_gemv_t<2, 8, ARGMAX>(a, ctx);
    return launch_gemv_t<2, 16, ARGMAX>(a, ctx);
}

cudaError_t launch_gemv_mode2(const GemvArgs& a, const LaunchCtx& ctx) {
    return a.tok ? dispatch_rows<true>(a, ctx) : dispatch_rows<false>(a, ctx);
}

cudaError_t launch_gemv_fused_mode2(const GemvArgs& a, const LaunchCtx& ctx) {
    if (rpl_fits_fused(a)) {
        // a weight row a lane, the produced row in shared memory
        if (a.k_cache) return launch_gemv_rpl_t<2, 1, true, kProdPlain, true>(a, ctx);
        if (a.prod == kProdResidual) return launch_gemv_rpl_t<2, 1, true, kProdResidual>(a, ctx);
        if (a.prod == kProdSwiglu) return launch_gemv_rpl_t<2, 1, true, kProdSwiglu>(a, ctx);
        return launch_gemv_rpl_t<2, 1, true>(a, ctx);
    }
    if (a.k_cache) return launch_gemv_row_t<2, 1, false, true, kProdPlain, true>(a, ctx);
    if (a.prod == kProdResidual) return launch_gemv_row_t<2, 1, false, true, kProdResidual>(a, ctx);
    if (a.prod == kProdSwiglu) return launch_gemv_row_t<2, 1, false, true, kProdSwiglu>(a, ctx);
    return launch_gemv_row_t<2, 1, false, true>(a, ctx);
}

}  // namespace q8

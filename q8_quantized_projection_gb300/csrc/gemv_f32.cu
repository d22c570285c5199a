// gemv_f32.cu -- instantiations of the CUDA-core projection for activation
// mode 0: the row-per-lane kernel (gemv_rpl.cuh) for K % 1024 == 0, one row
// up to 16384 values or a pair of rows up to 8192 (plain projections, the LM
// head's arg-max and fused decode steps), else the decode kernel
// (gemv_row.cuh: other K; one row a launch, the mode being bound by
// instruction issue), and the slice-major kernel (gemv.cuh) for K beyond the
// decode kernel's part sums.  One file per mode so the build runs in parallel.
#include "gemv_row.cuh"
#include "gemv_rpl.cuh"

namespace q8 {

template <bool ARGMAX>
static cudaError_t dispatch_rows(const GemvArgs& a, const LaunchCtx& ctx) {
    // a weight row a lane (K % 1024 == 0), plain or with the arg-max
    if (a.rows <= 1 && rpl_fits(a)) return launch_gemv_rpl_t<0, 1, false, kProdPlain, false, ARGMAX>(a, ctx);
    if (a.rows == 2 && rpl_fits(a)) return launch_gemv_rpl_t<0, 2, false, kProdPlain, false, ARGMAX>(a, ctx);
    if (a.rows <= 1 && row_kernel_fits<0, 1>(a.K)) return launch_gemv_row_t<0, 1, ARGMAX>(a, ctx);
    return launch_gemv_t<0, 4, ARGMAX>(a, ctx);
}

cudaError_t launch_gemv_mode0(const GemvArgs& a, const LaunchCtx& ctx) {
    return a.tok ? dispatch_rows<true>(a, ctx) : dispatch_rows<false>(a, ctx);
}

cudaError_t launch_gemv_fused_mode0(const GemvArgs& a, const LaunchCtx& ctx) {
    if (rpl_fits_fused(a)) {
        // a weight row a lane, the row's fixed-point planes in shared memory
        if (a.k_cache) return launch_gemv_rpl_t<0, 1, true, kProdPlain, true>(a, ctx);
        if (a.prod == kProdResidual) return launch_gemv_rpl_t<0, 1, true, kProdResidual>(a, ctx);
        if (a.prod == kProdSwiglu) return launch_gemv_rpl_t<0, 1, true, kProdSwiglu>(a, ctx);
        return launch_gemv_rpl_t<0, 1, true>(a, ctx);
    }
    if (a.k_cache) return launch_gemv_row_t<0, 1, false, true, kProdPlain, true>(a, ctx);
    if (a.prod == kProdResidual) return launch_gemv_row_t<0, 1, false, true, kProdResidual>(a, ctx);
    if (a.prod == kProdSwiglu) return launch_gemv_row_t<0, 1, false, true, kProdSwiglu>(a, ctx);
    return launch_gemv_row_t<0, 1, false, true>(a, ctx);
}

}  // namespace q8

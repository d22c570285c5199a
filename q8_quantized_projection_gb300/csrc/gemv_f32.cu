// gemv_f32.cu -- instantiations of the CUDA-core projection for activation
// mode 0: the decode kernel (gemv_row.cuh), one activation row per launch (the
// mode is bound by instruction issue, not HBM, so a row per pass over the
// weights is faster than sharing a pass), and the slice-major kernel
// (gemv.cuh) for K beyond the decode kernel's part sums.  One file per mode so
// the build runs in parallel.
#include "gemv_row.cuh"

namespace q8 {

template <bool ARGMAX>
static cudaError_t dispatch_rows(const GemvArgs& a, const LaunchCtx& ctx) {
    if (a.rows <= 1 && row_kernel_fits<0, 1>(a.K)) return launch_gemv_row_t<0, 1, ARGMAX>(a, ctx);
    return launch_gemv_t<0, 4, ARGMAX>(a, ctx);
}

cudaError_t launch_gemv_mode0(const GemvArgs& a, const LaunchCtx& ctx) {
    return a.tok ? dispatch_rows<true>(a, ctx) : dispatch_rows<false>(a, ctx);
}

cudaError_t launch_gemv_fused_mode0(const GemvArgs& a, const LaunchCtx& ctx) {
    if (a.k_cache) return launch_gemv_row_t<0, 1, false, true, kProdPlain, true>(a, ctx);
    if (a.prod == kProdResidual) return launch_gemv_row_t<0, 1, false, true, kProdResidual>(a, ctx);
    if (a.prod == kProdSwiglu) return launch_gemv_row_t<0, 1, false, true, kProdSwiglu>(a, ctx);
    return launch_gemv_row_t<0, 1, false, true>(a, ctx);
}

}  // namespace q8

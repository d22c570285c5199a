// gemv_i8x2.cu -- instantiations of the CUDA-core projection for activation
// mode 2 (see gemv.cuh), split per mode so the build compiles in parallel.
#include "gemv.cuh"

namespace q8 {

template <bool ARGMAX>
static cudaError_t dispatch_rows(const GemvArgs& a, const LaunchCtx& ctx) {
    if (a.rows <= 1) return launch_gemv_t<2, 1, 4, ARGMAX>(a, ctx);
    if (a.rows <= 2) return launch_gemv_t<2, 2, 4, ARGMAX>(a, ctx);
    if (a.rows <= 4) return launch_gemv_t<2, 4, 2, ARGMAX>(a, ctx);
    if (a.rows <= 8) return launch_gemv_t<2, 8, 1, ARGMAX>(a, ctx);
    return launch_gemv_t<2, 16, 1, ARGMAX>(a, ctx);
}

cudaError_t launch_gemv_mode2(const GemvArgs& a, const LaunchCtx& ctx) {
    return a.tok ? dispatch_rows<true>(a, ctx) : dispatch_rows<false>(a, ctx);
}

}  // namespace q8

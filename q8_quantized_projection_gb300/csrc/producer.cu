// producer.cu -- weight pack, the stand-alone activation producer (RMSNorm ->
// quant, one CTA per row) and the debug block-dot kernel.
#include "common.cuh"
#include "launch.h"
#include "rmsnorm.cuh"

namespace q8 {

int pdl_attrs(const LaunchCtx& ctx, cudaLaunchAttribute* attrs) {
    if (!ctx.pdl) return 0;
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    return 1;
}

// ------------------------------------------------------------------ pack

// Q8_0 pack, one warp per 32-value block: s = binary16(amax/127),
// q = round_half_away(w/s) in [-127, 127], 0 where s == 0 or w/s is NaN.
__global__ void __launch_bounds__(256) pack_kernel(const float* __restrict__ w, int64_t N,
                                                   int64_t K, int8_t* __restrict__ q,
                                                   uint16_t* __restrict__ s, int32_t* overflow) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / Q8_QK, total = N * nb;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t blk = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); blk < total;
         blk += warps) {
        const int64_t n = blk / nb, b = blk % nb;
        const int64_t idx = n * K + b * Q8_QK + lane;
        const float v = w[idx];
        float a = fabsf(v);
        a = (a > 0.0f) ? a : 0.0f;  // a NaN never becomes the block maximum
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const float d = __fdiv_rn(a, 127.0f);
        const __half hs = __float2half_rn(d);
        const float sf = __half2float(hs);
        if (lane == 0) {
            s[n * nb + b] = __half_as_ushort(hs);
            if (overflow && isinf(sf)) atomicAdd(overflow, 1);
        }
        float r = 0.0f;
        if (sf != 0.0f) {
            r = roundf(__fdiv_rn(v, sf));
            r = isnan(r) ? 0.0f : fminf(fmaxf(r, -127.0f), 127.0f);
        }
        q[idx] = static_cast<int8_t>(static_cast<int>(r));
    }
}

cudaError_t launch_pack(const float* w, int64_t N, int64_t K, int8_t* q, uint16_t* s,
                        int32_t* overflow, const LaunchCtx& ctx) {
    const int64_t blocks = N * (K / Q8_QK);
    int64_t grid = (blocks + 7) / 8;
    const int64_t cap = int64_t(ctx.num_sms) * 8;
    if (grid > cap) grid = cap;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[1];
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(256);
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, pack_kernel, w, N, K, q, s, overflow);
}

// ------------------------------------------------------- activation producer

struct AqParams {
    const float* h;
    const float* res;   // residual added before the norm, or NULL
    float* s_out;       // h + res written back, or NULL
    const float* gain;
    float eps;
    int64_t rows, K;
    void* out;
    float* xd;
};

// One CTA of kProdThreads threads per activation row (rmsnorm.cuh holds the
// arithmetic, shared with the decode projection's fused producer).
// PROD: kProdPlain, kProdResidual (h + r before the norm) or kProdSwiglu (h is
// the fused gate+up output, rows of 2K values).
template <int MODE, bool NORM, int PROD>
__global__ void __launch_bounds__(kProdThreads) act_quant_kernel(const AqParams p) {
    __shared__ float2 s_pair[kProdWarps];
    __shared__ float s_rf;
    const int tid = threadIdx.x;
    const int64_t m = blockIdx.x;
    const int64_t K = p.K, nb = K / Q8_QK;
    const float* h = p.h + m * K * (PROD == kProdSwiglu ? 2 : 1);

    pdl_wait();
    pdl_launch_dependents();

    void* out;
    if constexpr (MODE == 0)
        out = reinterpret_cast<float*>(p.out) + m * K;
    else
        out = reinterpret_cast<int8_t*>(p.out) + m * K;
    constexpr bool RES = PROD == kProdResidual;
    row_produce<MODE, NORM, PROD>(h, RES ? p.res + m * K : nullptr,
                                  RES && p.s_out ? p.s_out + m * K : nullptr, p.gain, p.eps, K, tid,
                                  1, s_pair, &s_rf, out, p.rows * K,
                            MODE == 0 ? nullptr : p.xd + m * nb);
}

template <int MODE, bool NORM, int PROD = kProdPlain>
static cudaError_t launch_aq_t(const AqParams& p, const LaunchCtx& ctx) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[1];
    cfg.gridDim = dim3(unsigned(p.rows));
    cfg.blockDim = dim3(kProdThreads);
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, act_quant_kernel<MODE, NORM, PROD>, p);
}

cudaError_t launch_act_quant(int mode, int prod, const float* h, const float* res, float* s_out,
                             int64_t rows, int64_t K, int norm, const float* gain, float eps, void* xq,
                             float* xd, const LaunchCtx& ctx) {
    AqParams p{h, res, s_out, gain, eps, rows, K, xq, xd};
    if (prod == kProdResidual) {   // the residual comes with the norm
        if (mode == 0) return launch_aq_t<0, true, kProdResidual>(p, ctx);
        if (mode == 1) return launch_aq_t<1, true, kProdResidual>(p, ctx);
        return launch_aq_t<2, true, kProdResidual>(p, ctx);
    }
    if (prod == kProdSwiglu) {     // no norm
        if (mode == 0) return launch_aq_t<0, false, kProdSwiglu>(p, ctx);
        if (mode == 1) return launch_aq_t<1, false, kProdSwiglu>(p, ctx);
        return launch_aq_t<2, false, kProdSwiglu>(p, ctx);
    }
    if (norm) {
        if (mode == 0) return launch_aq_t<0, true>(p, ctx);
        if (mode == 1) return launch_aq_t<1, true>(p, ctx);
        return launch_aq_t<2, true>(p, ctx);
    }
    if (mode == 0) return launch_aq_t<0, false>(p, ctx);
    if (mode == 1) return launch_aq_t<1, false>(p, ctx);
    return launch_aq_t<2, false>(p, ctx);
}

// -------------------------------------------------------- KV-row scatter

// The KV-row epilogue for batches: row m's K/V slices of y [rows][N] into
// cache row pos[m] of its sequence (caches [rows][n_pos][kv_dim]).  One CTA
// per (row, 256 cache entries of K then V); a position outside the cache
// writes nothing and sets the device error word.
__global__ void kv_scatter_kernel(const float* y, int64_t N, const int32_t* pos, int64_t kv_col,
                                  int64_t kv_dim, int64_t n_pos, float* k_cache, float* v_cache,
                                  int* err) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t m = blockIdx.y;
    const int ps = pos[m];
    if (ps < 0 || ps >= n_pos) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicExch(err, Q8_DEVERR_POSITION);
        return;
    }
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;   // [0, 2*kv_dim)
    if (i >= 2 * kv_dim) return;
    const float v = y[m * N + kv_col + i];
    float* cache = i < kv_dim ? k_cache : v_cache;
    cache[(m * n_pos + ps) * kv_dim + (i < kv_dim ? i : i - kv_dim)] = v;
}

cudaError_t launch_kv_scatter(const float* y, int64_t rows, int64_t N, const int32_t* pos, int64_t kv_col,
                              int64_t kv_dim, int64_t n_pos, float* k_cache, float* v_cache,
                              const LaunchCtx& ctx) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[1];
    cfg.gridDim = dim3(unsigned((2 * kv_dim + 255) / 256), unsigned(rows));
    cfg.blockDim = dim3(256);
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kv_scatter_kernel, y, N, pos, kv_col, kv_dim, n_pos, k_cache,
                              v_cache, ctx.dev_err);
}

// ----------------------------------------------------------- debug block dots

// isum[m][n][b] from the same 16-value dot helpers the GEMV kernels use.
template <int MODE>
__global__ void __launch_bounds__(256) debug_dots_kernel(const int8_t* __restrict__ q,
                                                         const int8_t* __restrict__ xq, int64_t N,
                                                         int64_t K, int64_t rows,
                                                         int32_t* __restrict__ isum) {
    pdl_wait();
    const int64_t nb = K / Q8_QK, total = rows * N * nb;
    for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += int64_t(gridDim.x) * blockDim.x) {
        const int64_t b = t % nb, n = (t / nb) % N, m = t / (nb * N);
        const int8_t* wp = q + n * K + b * Q8_QK;
        const int8_t* ap = xq + m * K + b * Q8_QK;
        int v;
        if constexpr (MODE == 1) {
            v = dot16_i8(ldg_nc_v4(wp), ldg_nc_v4(ap)) + dot16_i8(ldg_nc_v4(wp + 16), ldg_nc_v4(ap + 16));
        } else {
            const int8_t* lp = ap + rows * K;
            v = dot16_i8x2(ldg_nc_v4(wp), ldg_nc_v4(ap), ldg_nc_v4(lp)) +
                dot16_i8x2(ldg_nc_v4(wp + 16), ldg_nc_v4(ap + 16), ldg_nc_v4(lp + 16));
        }
        isum[t] = v;
    }
}

cudaError_t launch_debug_dots(int mode, const int8_t* q, const void* xq, int64_t N, int64_t K,
                              int64_t rows, int32_t* isum, const LaunchCtx& ctx) {
    const int64_t total = rows * N * (K / Q8_QK);
    int64_t grid = (total + 255) / 256;
    if (grid > int64_t(ctx.num_sms) * 16) grid = int64_t(ctx.num_sms) * 16;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[1];
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(256);
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    const int8_t* a = reinterpret_cast<const int8_t*>(xq);
    if (mode == 1) return cudaLaunchKernelEx(&cfg, debug_dots_kernel<1>, q, a, N, K, rows, isum);
    return cudaLaunchKernelEx(&cfg, debug_dots_kernel<2>, q, a, N, K, rows, isum);
}

}  // namespace q8

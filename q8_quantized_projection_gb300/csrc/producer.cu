// producer.cu -- weight pack, the activation producer (RMSNorm -> quant) and
// the debug block-dot kernel.
//
// The producer is tiny in bytes but sits on the decode step's critical path,
// so it is spread wide: a row's K is split over a thread-block cluster (up to
// 16 CTAs), each CTA folds its slice's sum of squares in f64, the partial sums
// are exchanged through distributed shared memory and every CTA adds them in
// rank order (so all agree bit for bit), then each CTA normalises and
// quantises its own blocks, one warp per 32-value block.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"

namespace cg = cooperative_groups;

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
    const float* gain;
    float eps;
    int64_t rows, K;
    void* out;
    float* xd;
};

template <int MODE, bool NORM>
__global__ void __launch_bounds__(256) act_quant_kernel(const AqParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = gridDim.x, c = blockIdx.x;
    const int64_t m = blockIdx.y;
    const int64_t K = p.K, nb = K / Q8_QK;
    const int64_t bpc = (nb + C - 1) / C;
    const int64_t b0 = int64_t(c) * bpc, b1 = min(nb, b0 + bpc);
    const float* h = p.h + m * K;

    pdl_wait();
    pdl_launch_dependents();

    float rf = 1.0f;
    if constexpr (NORM) {
        __shared__ double warp_ss[8];
        __shared__ double cta_ss;
        __shared__ float s_rf;
        double ss = 0.0;
        for (int64_t b = b0 + warp; b < b1; b += 8) {
            const double v = double(h[b * Q8_QK + lane]);
            ss = fma(v, v, ss);  // v*v is exact in f64
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) warp_ss[warp] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            double t = 0.0;
            for (int w2 = 0; w2 < 8; ++w2) t += warp_ss[w2];
            cta_ss = t;
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (threadIdx.x == 0) {
            double tot = 0.0;
            for (int r = 0; r < C; ++r) tot += *cluster.map_shared_rank(&cta_ss, r);
            const double mean = __ddiv_rn(tot, double(K));
            const double r = __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(mean, double(p.eps))));
            s_rf = __double2float_rn(r);
        }
        cluster.sync();  // no CTA leaves while a peer still reads its partial
        rf = s_rf;
    }

    for (int64_t b = b0 + warp; b < b1; b += 8) {
        const int64_t k = b * Q8_QK + lane;
        float x = h[k];
        if constexpr (NORM) {
            x = __fmul_rn(x, rf);
            if (p.gain) x = __fmul_rn(x, p.gain[k]);
        }
        if constexpr (MODE == 0) {
            reinterpret_cast<float*>(p.out)[m * K + k] = x;
        } else {
            float a = fabsf(x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            const float lim = (MODE == 1) ? 127.0f : 8191.0f;
            const float d = __fdiv_rn(a, lim);
            const int code = quantize_code(x, d, lim);
            int8_t* out = reinterpret_cast<int8_t*>(p.out);
            if constexpr (MODE == 1) {
                out[m * K + k] = static_cast<int8_t>(code);
            } else {
                const int lo = ((code + 64) & 127) - 64;  // Euclidean residue, centred
                const int hi = (code - lo) >> 7;          // exact: code - lo is a multiple of 128
                out[m * K + k] = static_cast<int8_t>(hi);
                out[p.rows * K + m * K + k] = static_cast<int8_t>(lo);
            }
            if (lane == 0) p.xd[m * nb + b] = d;
        }
    }
}

template <int MODE, bool NORM>
static cudaError_t launch_aq_t(const AqParams& p, int C, const LaunchCtx& ctx) {
    auto kern = act_quant_kernel<MODE, NORM>;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[2];
    int na = pdl_attrs(ctx, attrs);
    if (NORM) {
        static bool configured = false;
        if (!configured) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            configured = true;
        }
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = unsigned(C);
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.gridDim = dim3(unsigned(C), unsigned(p.rows));
    cfg.blockDim = dim3(256);
    cfg.stream = ctx.stream;
    cfg.numAttrs = unsigned(na);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

cudaError_t launch_act_quant(int mode, const float* h, int64_t rows, int64_t K, int norm,
                             const float* gain, float eps, void* xq, float* xd,
                             const LaunchCtx& ctx) {
    AqParams p{h, gain, eps, rows, K, xq, xd};
    const int64_t nb = K / Q8_QK;
    int C;
    if (norm) {
        C = int(nb < 16 ? nb : 16);  // cluster over the row (16 = non-portable maximum)
    } else {
        const int64_t c = (nb + 15) / 16;
        C = int(c > 64 ? 64 : c);
    }
    if (norm) {
        if (mode == 0) return launch_aq_t<0, true>(p, C, ctx);
        if (mode == 1) return launch_aq_t<1, true>(p, C, ctx);
        return launch_aq_t<2, true>(p, C, ctx);
    }
    if (mode == 0) return launch_aq_t<0, false>(p, C, ctx);
    if (mode == 1) return launch_aq_t<1, false>(p, C, ctx);
    return launch_aq_t<2, false>(p, C, ctx);
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

// rmsnorm.cuh -- the activation producer's row arithmetic, shared by the
// stand-alone producer kernel (producer.cu) and the decode projection with the
// producer fused in (gemv_row.cuh), so both compute bit-identical codes.
//
// Both run it on exactly kProdThreads threads with a fixed assignment:
// thread t owns the float4 groups t, t + kProdThreads, ... of the row.
//  * Sum of squares: each square is split exactly by an FMA and accumulated
//    as an f32 pair (error-free transforms, ~48 bits), reduced over the warp
//    in a fixed xor order, then the warp sums are added in warp order in f64
//    (f64 arithmetic and f32<->f64 conversions are slow on this part, so only
//    one value per warp goes to f64).  r = 1/sqrt(ss/K + eps) in f64 with
//    IEEE division and square root; rf = float(r).
//  * Quantisation: a 32-value block is 8 consecutive float4 groups, held by 8
//    consecutive lanes; amax is an exact max over 3 shuffles, the scale is
//    d = amax / lim (IEEE division) and every code is round_half_away(x / d).
#pragma once

#include "common.cuh"

namespace q8 {

constexpr int kProdThreads = 512;
constexpr int kProdWarps = kProdThreads / 32;

__device__ __forceinline__ void pair_add(float& sh, float& sl, float v) {
    const float s = __fadd_rn(sh, v);
    const float bb = __fsub_rn(s, sh);
    const float e = __fadd_rn(__fsub_rn(sh, __fsub_rn(s, bb)), __fsub_rn(v, bb));
    sh = s;
    sl = __fadd_rn(sl, e);
}

__device__ __forceinline__ void pair_add_sq(float& sh, float& sl, float v) {
    const float p = __fmul_rn(v, v);
    const float pe = __fmaf_rn(v, v, -p);   // exact low part of v*v
    pair_add(sh, sl, p);
    sl = __fadd_rn(sl, pe);
}

// rf = float(1 / sqrt(sum(h^2)/K + eps)) for one row.  All kProdThreads
// threads call it; `bar` is a named-barrier id over exactly those threads.
// s_warp: kProdWarps doubles of shared scratch; s_rf: one float.
__device__ __forceinline__ float row_rms_scale(const float* h, int64_t K, float eps, int tid,
                                               int bar, double* s_warp, float* s_rf) {
    float sh = 0.0f, sl = 0.0f;
    const int64_t groups = K >> 2;
    for (int64_t gi = tid; gi < groups; gi += kProdThreads) {
        const int4 v = ldg_nc_v4(h + 4 * gi);
        pair_add_sq(sh, sl, __int_as_float(v.x));
        pair_add_sq(sh, sl, __int_as_float(v.y));
        pair_add_sq(sh, sl, __int_as_float(v.z));
        pair_add_sq(sh, sl, __int_as_float(v.w));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float rh = __shfl_xor_sync(0xffffffffu, sh, o);
        const float rl = __shfl_xor_sync(0xffffffffu, sl, o);
        pair_add(sh, sl, rh);
        sl = __fadd_rn(sl, rl);
    }
    if ((tid & 31) == 0) s_warp[tid >> 5] = double(sh) + double(sl);
    named_bar(bar, kProdThreads);
    if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < kProdWarps; ++w) t += s_warp[w];
        const double mean = __ddiv_rn(t, double(K));
        const double r = __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(mean, double(eps))));
        *s_rf = __double2float_rn(r);
    }
    named_bar(bar, kProdThreads);
    return *s_rf;
}

// Normalises (when rf is given) and quantises one row in the mode's layout.
// MODE 0 writes f32 x; MODE 1 one int8 code plane; MODE 2 the hi plane at
// out and the lo plane at out + plane.  xd receives one scale per block.
// Every thread of the kProdThreads calls it (block lanes meet in shuffles).
template <int MODE, bool NORM>
__device__ __forceinline__ void row_quantize(const float* h, const float* gain, float rf,
                                             int64_t K, int tid, void* out, int64_t plane,
                                             float* xd) {
    const int64_t groups = K >> 2;
    // Every lane of a warp runs the same number of iterations (groups is a
    // multiple of 8 and the stride a multiple of 32), so shuffles stay full.
    for (int64_t gi = tid; gi < ((groups + 31) & ~int64_t(31)); gi += kProdThreads) {
        const bool live = gi < groups;
        float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (live) {
            const int4 v = ldg_nc_v4(h + 4 * gi);
            x[0] = __int_as_float(v.x);
            x[1] = __int_as_float(v.y);
            x[2] = __int_as_float(v.z);
            x[3] = __int_as_float(v.w);
            if constexpr (NORM) {
                int4 g4 = make_int4(0x3f800000, 0x3f800000, 0x3f800000, 0x3f800000);
                if (gain) g4 = ldg_nc_v4(gain + 4 * gi);
                const float gv[4] = {__int_as_float(g4.x), __int_as_float(g4.y),
                                     __int_as_float(g4.z), __int_as_float(g4.w)};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    x[e] = __fmul_rn(x[e], rf);
                    if (gain) x[e] = __fmul_rn(x[e], gv[e]);
                }
            }
        }
        if constexpr (MODE == 0) {
            if (live)
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + 4 * gi) =
                    make_float4(x[0], x[1], x[2], x[3]);
        } else {
            float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            if (live) {
                const float lim = (MODE == 1) ? 127.0f : 8191.0f;
                const float d = __fdiv_rn(a, lim);
                int code[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) code[e] = quantize_code(x[e], d, lim);
                int8_t* o = reinterpret_cast<int8_t*>(out);
                if constexpr (MODE == 1) {
                    const unsigned w = (unsigned(code[0]) & 0xffu) | ((unsigned(code[1]) & 0xffu) << 8) |
                                       ((unsigned(code[2]) & 0xffu) << 16) | (unsigned(code[3]) << 24);
                    *reinterpret_cast<unsigned*>(o + 4 * gi) = w;
                } else {
                    unsigned wh = 0, wl = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int lo = ((code[e] + 64) & 127) - 64;   // Euclidean residue, centred
                        const int hi = (code[e] - lo) >> 7;           // exact
                        wh |= (unsigned(hi) & 0xffu) << (8 * e);
                        wl |= (unsigned(lo) & 0xffu) << (8 * e);
                    }
                    *reinterpret_cast<unsigned*>(o + 4 * gi) = wh;
                    *reinterpret_cast<unsigned*>(o + plane + 4 * gi) = wl;
                }
                if ((gi & 7) == 0) xd[gi >> 3] = d;
            }
        }
    }
}

}  // namespace q8

// rmsnorm.cuh -- the activation producer's row arithmetic, shared by the
// stand-alone producer kernel (producer.cu) and the decode projection with the
// producer fused in (gemv_row.cuh), so both compute bit-identical codes.
//
// Both run it on exactly kProdThreads threads with a fixed assignment:
// thread t owns the float4 groups t, t + kProdThreads, ... of the row.
//  * Sum of squares: each square is split exactly by an FMA and accumulated
//    as an f32 pair (error-free transforms, ~48 bits), reduced over the warp
//    and then over the warps in fixed orders.  rf = float(1/sqrt(ss/K + eps))
//    is evaluated in f32 pairs to ~2^-44 relative before its final rounding
//    (the part's FP64 latency would dominate the producer).
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

// Float4 groups of the row a thread keeps in registers between the two
// passes (K <= kProdThreads * 4 * kProdCache = 16384); longer rows reload
// the groups beyond from global memory.
constexpr int kProdCache = 8;

// f32 pair arithmetic for the one scalar chain of the row (the part's FP64
// rate and f32<->f64 conversions are far too slow for a latency path).
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// rf = float(1 / sqrt(S/K + eps)) for S = sh + sl, to about 2^-44 relative
// before the final rounding: the quotient S/K with its exact FMA remainder,
// then one Newton step on the hardware reciprocal square root evaluated in
// f32 pairs.
__device__ __forceinline__ float rms_scale_from_sum(float sh, float sl, int64_t K, float eps) {
    const float kf = float(K);   // exact for K < 2^24
    const float q1 = __fdiv_rn(sh, kf);
    const float rem = __fmaf_rn(-q1, kf, sh);   // sh - q1*K exactly
    const float q2 = __fdiv_rn(__fadd_rn(rem, sl), kf);
    float mh, ml;
    fast_two_sum(q1, q2, mh, ml);
    float vh, vl;   // v = mean + eps
    {
        float s, e;
        const float bb = __fadd_rn(mh, eps);
        s = bb;
        const float z = __fsub_rn(s, mh);
        e = __fadd_rn(__fsub_rn(mh, __fsub_rn(s, z)), __fsub_rn(eps, z));
        fast_two_sum(s, __fadd_rn(e, ml), vh, vl);
    }
    if (!(vh > 0.0f)) return vh == 0.0f ? INFINITY : __int_as_float(0x7fc00000);
    if (isinf(vh)) return 0.0f;
    const float y0 = rsqrtf(vh);
    // t = v*y0^2 - 1, with y0^2 and v*y0^2 split exactly by FMAs
    const float ph = __fmul_rn(y0, y0);
    const float pl = __fmaf_rn(y0, y0, -ph);
    const float ah = __fmul_rn(vh, ph);
    float al = __fmaf_rn(vh, ph, -ah);
    al = __fmaf_rn(vh, pl, al);
    al = __fmaf_rn(vl, ph, al);
    const float tt = __fadd_rn(__fsub_rn(ah, 1.0f), al);   // ah - 1 is exact (ah ~ 1)
    const float corr = __fmul_rn(__fmul_rn(-0.5f, y0), tt);
    float rh, rl;
    fast_two_sum(y0, corr, rh, rl);
    return __fadd_rn(rh, rl);
}

// 1/d to within one ulp: the hardware reciprocal estimate refined by one
// Newton step, r1 = r0 + r0*(1 - d*r0), evaluated with FMAs.
__device__ __forceinline__ float recip_refined(float d) {
    float r0;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r0) : "f"(d));
    const float e = __fmaf_rn(-d, r0, 1.0f);
    return __fmaf_rn(r0, e, r0);
}

// The 4 codes round_half_away(x / d), clamped to [-lim, lim] (d > 0), of one
// float4 group.  qa = x*(1/d) with 1/d within one ulp is within 2^-22
// (relative) of the IEEE quotient x/d, so qa and x/d round alike unless |qa|
// lies within 2^-21*|qa| of a half-integer; only those values take the IEEE
// division (a divergent branch, about 2^-20*|q| of the codes).  Away from
// ties, rounding |qa| < 2^22 to the nearest integer is exact by adding and
// subtracting 1.5*2^23, whose low bits then hold the integer: no conversion
// instruction (a narrow pipe on this part) on the common path.
__device__ __forceinline__ void quantize4(const float (&x)[4], float d, float lim, int (&code)[4]) {
    constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23
    const float rcp = recip_refined(d);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float aq = fabsf(__fmul_rn(x[e], rcp));
        const float t = __fadd_rn(fminf(aq, lim + 1.0f), kMagic);
        const float vf = __fsub_rn(t, kMagic);                     // nearest integer, exact
        int c = __float_as_int(t) - __float_as_int(kMagic);
        const float dist = fabsf(__fsub_rn(aq, vf));              // to the nearest integer
        if (dist > __fmaf_rn(-aq, 0x1p-21f, 0.5f))
            c = static_cast<int>(fabsf(roundf(__fdiv_rn(x[e], d))));   // near a tie: IEEE decides
        c = min(c, static_cast<int>(lim));
        code[e] = x[e] < 0.0f ? -c : c;
    }
}

// One float4 group of the row: normalise, then store (MODE 0) or quantise
// with its block (MODE 1, 2).  All lanes of the warp call it together.
template <int MODE, bool NORM>
__device__ __forceinline__ void produce_group(float (&x)[4], const float (&gg)[4], bool has_gain,
                                              float rf, int64_t gi, bool live, void* out,
                                              int64_t plane, float* xd) {
    if constexpr (NORM) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[e] = __fmul_rn(x[e], rf);
            if (has_gain) x[e] = __fmul_rn(x[e], gg[e]);
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
            int code[4] = {0, 0, 0, 0};
            quantize4(x, d == 0.0f ? 1.0f : d, lim, code);   // d == 0: every x is 0
            if (d == 0.0f) code[0] = code[1] = code[2] = code[3] = 0;
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

// The thread partials (sh, sl) of the sum of squares -> rf, shared by every
// producer: the warp reduction in a fixed xor order, then the warps' pairs in
// a fixed tree, then the scale (rms_scale_from_sum).  All kProdThreads threads
// call it; `bar` is a named-barrier id over exactly those threads.
__device__ __forceinline__ float rms_scale_reduce(float sh, float sl, int64_t K, float eps, int tid,
                                                  int bar, float2* s_pair, float* s_rf) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float rh = __shfl_xor_sync(0xffffffffu, sh, o);
        const float rl = __shfl_xor_sync(0xffffffffu, sl, o);
        pair_add(sh, sl, rh);
        sl = __fadd_rn(sl, rl);
    }
    if ((tid & 31) == 0) s_pair[tid >> 5] = make_float2(sh, sl);
    named_bar(bar, kProdThreads);
    if (tid < 32) {
        float2 v = tid < kProdWarps ? s_pair[tid] : make_float2(0.0f, 0.0f);
        sh = v.x;
        sl = v.y;
#pragma unroll
        for (int o = kProdWarps / 2; o > 0; o >>= 1) {
            const float rh = __shfl_xor_sync(0xffffffffu, sh, o);
            const float rl = __shfl_xor_sync(0xffffffffu, sl, o);
            pair_add(sh, sl, rh);
            sl = __fadd_rn(sl, rl);
        }
        if (tid == 0) *s_rf = rms_scale_from_sum(sh, sl, K, eps);
    }
    named_bar(bar, kProdThreads);
    return *s_rf;
}

// Kinds of producer input: h as given (optionally normalised), the residual
// sum h + r (normalised), or the SwiGLU of a fused gate+up row (not
// normalised).
constexpr int kProdPlain = 0;
constexpr int kProdResidual = 1;
constexpr int kProdSwiglu = 2;

// e^x in binary32 by one fixed method, so that a producer's codes are
// reproducible from its definition: Cody and Waite's reduction x = k*ln2 + r,
// k = rint(x/ln2), |r| <= ln2/2, with ln2 as a 16-bit head (k*head exact for
// |k| <= 2^8) plus its binary32 remainder; e^r by its Taylor series to degree
// 7 (coefficients 1/i! rounded to binary32) in Horner form with fused
// multiply-adds; then 2^k in two exact power-of-two steps.  Within one ulp of
// the correctly rounded e^x on [-104, 88.7].
__device__ __forceinline__ float exp_cw(float x) {
    if (x != x) return x;
    if (x > 88.75f) return __int_as_float(0x7f800000);
    if (x < -104.0f) return 0.0f;
    const float magic = 12582912.0f;   // 1.5*2^23: rint by addition
    const float t = __fmaf_rn(x, 0x1.715476p+0f, magic);
    const float kf = __fsub_rn(t, magic);
    const int k = __float_as_int(t) - 0x4B400000;
    float r = __fmaf_rn(-kf, 0x1.62e4p-1f, x);
    r = __fmaf_rn(-kf, 0x1.7f7d1cp-20f, r);
    float q = 0x1.a01a02p-13f;              // 1/7!
    q = __fmaf_rn(q, r, 0x1.6c16c2p-10f);   // 1/6!
    q = __fmaf_rn(q, r, 0x1.111112p-7f);    // 1/5!
    q = __fmaf_rn(q, r, 0x1.555556p-5f);    // 1/4!
    q = __fmaf_rn(q, r, 0x1.555556p-3f);    // 1/3!
    q = __fmaf_rn(q, r, 0.5f);
    q = __fmaf_rn(q, r, 1.0f);
    q = __fmaf_rn(q, r, 1.0f);
    const int k1 = k >> 1, k2 = k - k1;     // each in [-76, 64]
    return __fmul_rn(__fmul_rn(q, __int_as_float((k1 + 127) << 23)), __int_as_float((k2 + 127) << 23));
}

// silu(g) * u = g / (1 + e^-g) * u, each step one binary32 rounding.
__device__ __forceinline__ float swiglu1(float g, float u) {
    return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, exp_cw(-g))), u);
}

// Float4 group gi of a SwiGLU producer's input: gate = gu[0..F), up =
// gu[F..2F) of the fused gate+up row.
__device__ __forceinline__ float4 load_swiglu4(const float* gu, int64_t F, int64_t gi) {
    const int4 g = ldg_nc_v4(gu + 4 * gi);
    const int4 u = ldg_nc_v4(gu + F + 4 * gi);
    return make_float4(swiglu1(__int_as_float(g.x), __int_as_float(u.x)),
                       swiglu1(__int_as_float(g.y), __int_as_float(u.y)),
                       swiglu1(__int_as_float(g.z), __int_as_float(u.z)),
                       swiglu1(__int_as_float(g.w), __int_as_float(u.w)));
}

// Float4 group gi of the producer's input: h, or with a residual r the sum
// s = h + r (one f32 rounding, the residual added before the norm), stored to
// s_out when it is set (the updated residual stream).
__device__ __forceinline__ float4 load_input4(const float* h, const float* r, float* s_out, int64_t gi) {
    const int4 v = ldg_nc_v4(h + 4 * gi);
    float4 s = make_float4(__int_as_float(v.x), __int_as_float(v.y), __int_as_float(v.z),
                           __int_as_float(v.w));
    if (r) {
        const int4 w = ldg_nc_v4(r + 4 * gi);
        s.x = __fadd_rn(s.x, __int_as_float(w.x));
        s.y = __fadd_rn(s.y, __int_as_float(w.y));
        s.z = __fadd_rn(s.z, __int_as_float(w.z));
        s.w = __fadd_rn(s.w, __int_as_float(w.w));
    }
    if (s_out) *reinterpret_cast<float4*>(s_out + 4 * gi) = s;
    return s;
}

// rf alone (the f32 mode's fused producer, whose consumers form x = (h*rf)*g
// themselves): the same per-thread order of squares as row_produce, so the
// same rf.
// With a residual r the input is s = h + r, stored to s_out when it is set;
// with `stage` (shared memory, K floats) the input is also kept there.
__device__ __forceinline__ float row_rms_scale(const float* h, const float* r, float* s_out, int64_t K,
                                               float eps, int tid, int bar, float2* s_pair,
                                               float* s_rf, float* stage = nullptr) {
    float sh = 0.0f, sl = 0.0f;
    for (int64_t gi = tid; gi < (K >> 2); gi += kProdThreads) {
        const float4 v = load_input4(h, r, s_out, gi);
        if (stage) *reinterpret_cast<float4*>(stage + 4 * gi) = v;
        pair_add_sq(sh, sl, v.x);
        pair_add_sq(sh, sl, v.y);
        pair_add_sq(sh, sl, v.z);
        pair_add_sq(sh, sl, v.w);
    }
    return rms_scale_reduce(sh, sl, K, eps, tid, bar, s_pair, s_rf);
}

// The producer of one row: optional RMSNorm (x = (h * rf) * g), then the
// mode's quantisation (MODE 0 writes f32 x; MODE 1 one int8 code plane;
// MODE 2 the hi plane at out and the lo plane at out + plane; xd receives one
// scale per block).  Every one of the kProdThreads threads calls it; `bar` is
// a named-barrier id over exactly those threads.  s_pair: kProdWarps float2
// of shared scratch; s_rf: one float.
//  * Sum of squares: each square is split exactly by an FMA and accumulated
//    as an f32 pair (error-free transforms, ~48 bits), reduced over the warp
//    in a fixed xor order, then over the warps in a fixed tree.
//  * Quantisation: a 32-value block is 8 consecutive float4 groups, held by 8
//    consecutive lanes; amax is an exact max over 3 shuffles, the scale is
//    d = amax / lim (IEEE division) and every code is round_half_away(x / d).
// With a residual r (the residual added before the norm) the input is
// s = h + r, one rounding, stored to s_out when it is set.  PROD ==
// kProdSwiglu: h is the fused gate+up row (2K values) and the input is its
// SwiGLU (NORM is then false).
template <int MODE, bool NORM, int PROD = kProdPlain>
__device__ __forceinline__ void row_produce(const float* h, const float* r, float* s_out,
                                            const float* gain, float eps, int64_t K, int tid,
                                            int bar, float2* s_pair, float* s_rf, void* out,
                                            int64_t plane, float* xd) {
    const int64_t groups = K >> 2;
    // every lane of a warp runs the same iterations (groups is a multiple of 8
    // and the stride a multiple of 32), so the block shuffles stay full
    const int iters = int((groups + kProdThreads - 1) / kProdThreads);
    float4 hv[kProdCache], gv[kProdCache];
#pragma unroll
    for (int j = 0; j < kProdCache; ++j) {
        const int64_t gi = tid + int64_t(j) * kProdThreads;
        hv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        gv[j] = make_float4(1.f, 1.f, 1.f, 1.f);
        if (j < iters && gi < groups) {
            hv[j] = PROD == kProdSwiglu ? load_swiglu4(h, K, gi) : load_input4(h, r, s_out, gi);
            if (NORM && gain) {
                const int4 g4 = ldg_nc_v4(gain + 4 * gi);
                gv[j] = make_float4(__int_as_float(g4.x), __int_as_float(g4.y),
                                    __int_as_float(g4.z), __int_as_float(g4.w));
            }
        }
    }
    float rf = 1.0f;
    if constexpr (NORM) {
        float sh = 0.0f, sl = 0.0f;
#pragma unroll
        for (int j = 0; j < kProdCache; ++j) {
            pair_add_sq(sh, sl, hv[j].x);
            pair_add_sq(sh, sl, hv[j].y);
            pair_add_sq(sh, sl, hv[j].z);
            pair_add_sq(sh, sl, hv[j].w);
        }
        for (int64_t gi = tid + int64_t(kProdCache) * kProdThreads; gi < groups; gi += kProdThreads) {
            const float4 v = load_input4(h, r, nullptr, gi);   // stored in the pass below
            pair_add_sq(sh, sl, v.x);
            pair_add_sq(sh, sl, v.y);
            pair_add_sq(sh, sl, v.z);
            pair_add_sq(sh, sl, v.w);
        }
        rf = rms_scale_reduce(sh, sl, K, eps, tid, bar, s_pair, s_rf);
    }
    // cached groups: unrolled, so independent groups overlap their latencies
#pragma unroll
    for (int j = 0; j < kProdCache; ++j) {
        if (j < iters) {
            const int64_t gi = tid + int64_t(j) * kProdThreads;
            float x[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
            const float gg[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
            produce_group<MODE, NORM>(x, gg, gain != nullptr, rf, gi, gi < groups, out, plane, xd);
        }
    }
    for (int j = kProdCache; j < iters; ++j) {
        const int64_t gi = tid + int64_t(j) * kProdThreads;
        const bool live = gi < groups;
        float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float gg[4] = {1.0f, 1.0f, 1.0f, 1.0f};
        if (live) {
            const float4 v = PROD == kProdSwiglu ? load_swiglu4(h, K, gi) : load_input4(h, r, s_out, gi);
            x[0] = v.x;
            x[1] = v.y;
            x[2] = v.z;
            x[3] = v.w;
            if (NORM && gain) {
                const int4 g4 = ldg_nc_v4(gain + 4 * gi);
                gg[0] = __int_as_float(g4.x);
                gg[1] = __int_as_float(g4.y);
                gg[2] = __int_as_float(g4.z);
                gg[3] = __int_as_float(g4.w);
            }
        }
        produce_group<MODE, NORM>(x, gg, gain != nullptr, rf, gi, live, out, plane, xd);
    }
}

}  // namespace q8

// gemv.cuh -- CUDA-core Q8_0 projection for few activation rows (decode step,
// small batches, the LM head), sm_103a.
//
// At rows = 1..16 the projection is bound by HBM: every weight byte is read
// once per step (34 bytes per 32 weights) and the arithmetic per byte is a
// fraction of a dp4a.  Design:
//
//  * Persistent grid, one CTA per SM.  CTA c owns the contiguous weight rows
//    [N*c/G, N*(c+1)/G), so the imbalance between CTAs is at most one row.
//  * K is cut into slices of SLB = 512*CPL bytes (the last one shorter).  Work
//    runs slice-major: for a slice, all of the CTA's rows stream through a
//    shared-memory ring fed by the bulk-copy (TMA) engine, NW*RPW rows a stage
//    (NW = 8 or 16 consumer warps), 128 KB in flight per SM.  Weights never depend on the previous kernel,
//    so the producer warp starts before griddepcontrol.wait (programmatic
//    dependent launch); consumers wait before touching activations.
//  * Consumer warp w owns rows w, w+NW, ... of every stage; lane l owns the
//    16-byte chunks l + 32c (c < CPL) of the slice, so its activation chunks
//    stay in registers for the whole slice.  A row costs each lane CPL shared
//    loads, the dots, and one warp-shuffle reduction; a row's running sum
//    across slices lives in shared memory and is touched only by its warp, so
//    consumer warps never synchronise with each other.
//  * One-word mode: 4 dp4a per 16 weights; two-word: 8 dp4a (hi and lo
//    planes) combined as 128*hi + lo exactly in int32.  f32 mode: each lane
//    writes its 16 activations of a chunk as 31-bit fixed point relative to
//    their own binade (4 int8 planes), so a chunk's dot with the int8 weights
//    is an exact int64 from 16 dp4a; chunk values are scaled and summed as f32
//    pairs (error-free transforms, ~48 bits), because the GB300's FP64 rate
//    and f32<->f64 conversions are far below one operation per weight.
//  * Optional arg-max epilogue for the LM head: per-CTA best (value, lowest
//    index), then the last CTA to take a ticket reduces all candidates.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace q8 {

constexpr int kGemvMaxConsumerWarps = 16;
constexpr int kGemvRing = 131072;       // weight bytes in flight per CTA
constexpr int kGemvStageMax = 32768;    // weight bytes of one stage, upper bound
constexpr int kGemvMaxStages = 16;
constexpr int kGemvYaccBytes = 32768;   // row accumulators of one super-block

struct GemvParams {
    const int8_t* q;
    const uint16_t* s;
    int64_t N, K;
    const void* act;
    const float* xd;
    int64_t plane;
    int rows;
    void* y;
    int out_f64;
    int32_t* tok;
    double* maxval;
    unsigned char* ws;
    int* err;
    const float* h;      // fused producer input (decode kernel only)
    const float* res;    // residual added before the norm, or NULL
    float* s_out;        // h + res written back (by CTA 0), or NULL
    const float* gain;
    float eps;
    // KV-row epilogue (decode kernel only): columns [kv_col, kv_col + kv_dim)
    // of row m also go to k_cache row pos[m], the next kv_dim to v_cache;
    // caches [rows][n_pos][kv_dim].  k_cache NULL: none.
    const int32_t* pos;
    int64_t kv_col, kv_dim, n_pos;
    float* k_cache;
    float* v_cache;
};

// Chunks (16 bytes of K) each lane owns per slice, and consumer warps per
// CTA, for the slice-major kernel (4 to 16 activation rows).
template <int MODE, int R>
__host__ __device__ constexpr int gemv_cpl() {
    return MODE == 0 ? (R == 1 ? 4 : (R == 2 ? 2 : 1)) : (R <= 8 ? 8 / R : 1);
}
template <int MODE, int R>
__host__ __device__ constexpr int gemv_warps() {
    return 8;
}

// ------------------------------------------------------------ f32 pairs

// Unevaluated f32 pair hi + lo (about 48 significant bits), added with
// error-free transforms.
struct DF {
    float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    return DF{s, __fadd_rn(__fadd_rn(a.lo, b.lo), e)};
}

template <int MODE>
struct AccT {
    using T = float;
};
template <>
struct AccT<0> {
    using T = DF;
};

__device__ __forceinline__ float acc_zero(float) { return 0.0f; }
__device__ __forceinline__ DF acc_zero(DF) { return DF{0.0f, 0.0f}; }
__device__ __forceinline__ float acc_add(float a, float b) { return a + b; }
__device__ __forceinline__ DF acc_add(DF a, DF b) { return df_add(a, b); }
__device__ __forceinline__ double acc_value(float a) { return double(a); }
__device__ __forceinline__ double acc_value(DF a) { return double(a.hi) + double(a.lo); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ DF warp_sum(DF v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const DF r{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
        v = df_add(v, r);
    }
    return v;
}

// ------------------------------------------------------------ f32-mode math

__device__ __forceinline__ int dp4a_su(int a_signed, unsigned b_unsigned, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_signed), "r"(b_unsigned), "r"(c));
    return d;
}

// Binade bound: |x| < 2^e (subnormals and zero give -126).
__device__ __forceinline__ int binade(float a) {
    const int eb = (__float_as_int(a) >> 23) & 0xff;
    return eb == 0 ? -126 : eb - 126;
}

// 2^n as a float for -126 <= n <= 127, from its bit pattern.
__device__ __forceinline__ float pow2i(int n) { return __int_as_float((n + 127) << 23); }

// The four byte planes of four int32 values: plane j holds byte j of v0..v3
// (v0 in the low byte), by two rounds of byte permutes.
__device__ __forceinline__ void byte_planes4(int v0, int v1, int v2, int v3, int& p0, int& p1,
                                             int& p2, int& p3) {
    unsigned t0, t1, t2, t3;
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(t0) : "r"(v0), "r"(v1));   // v0.b0 v1.b0 v0.b1 v1.b1
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(t1) : "r"(v2), "r"(v3));
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(t2) : "r"(v0), "r"(v1));   // v0.b2 v1.b2 v0.b3 v1.b3
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(t3) : "r"(v2), "r"(v3));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(p0) : "r"(t0), "r"(t1));
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(p1) : "r"(t0), "r"(t1));
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(p2) : "r"(t2), "r"(t3));
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(p3) : "r"(t2), "r"(t3));
}

// rint(t * s2) for |t * s2| <= 2^30, exactly and without a conversion
// instruction (those run on a narrow pipe): u = (3*2^30 + v) rounded, where
// floats are 2^8 apart, so vh = u - 3*2^30 is v rounded to a multiple of 2^8
// and its bits count those multiples; vl = v - vh (|vl| <= 2^7) is exact by
// a fused multiply-add, and rint(vl) is read from the bits of 1.5*2^23 + vl.
// rint(v) = vh + rint(vl), ties to even as vh is even.
__device__ __forceinline__ int rint_scaled30(float t, float s2) {
    const float C = 3221225472.0f;   // 3*2^30
    const float M = 12582912.0f;     // 1.5*2^23
    const float u = __fmaf_rn(t, s2, C);
    const float vh = __fsub_rn(u, C);
    const float vl = __fmaf_rn(t, s2, -vh);
    const float w = __fadd_rn(vl, M);
    return int((__float_as_uint(u) << 8) + __float_as_uint(w) - (0x4F400000u << 8) - 0x4B400000u);
}

// 16 f32 activations -> 4 byte planes of X = rint(x * 2^(30-E)), |X| <= 2^30,
// X = p3*2^24 + p2*2^16 + p1*2^8 + p0 (p3 signed, p2..p0 unsigned), and the
// chunk's binade E.  Plane j word u packs elements 4u..4u+3.
struct FixChunk {
    int p[4][4];
    int e;
};

__device__ __forceinline__ FixChunk fix_chunk(const float (&x)[16]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    FixChunk f;
    f.e = binade(amax);
    // x * 2^(30-E) as two multiplies by normal powers of two (see fix_chunk32)
    const int sh = 30 - f.e;
    const float s1 = pow2i(sh >> 1), s2 = pow2i(sh - (sh >> 1));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        int X[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) X[i] = rint_scaled30(__fmul_rn(x[4 * u + i], s1), s2);
        byte_planes4(X[0], X[1], X[2], X[3], f.p[0][u], f.p[1][u], f.p[2][u], f.p[3][u]);
    }
    return f;
}

// Exact chunk dot sum_e q_e * X_e as int64 (|.| < 2^42).
__device__ __forceinline__ long long fix_dot(const int4 w, const FixChunk& f) {
    const int wv[4] = {w.x, w.y, w.z, w.w};
    int P[4];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        int a = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) a = dp4a_su(wv[u], unsigned(f.p[j][u]), a);
        P[j] = a;
    }
    int a = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) a = __dp4a(wv[u], f.p[3][u], a);
    P[3] = a;
    const long long lo = (long long)P[1] * 256 + P[0];
    return ((long long)P[3] << 24) + ((long long)P[2] << 16) + lo;
}

// The same for a whole 32-value block (one binade for the block): plane j
// word u packs elements 4u..4u+3, u < 8.
struct FixChunk32 {
    int p[4][8];
    int e;
};

// v * 2^d for d <= 0 by two multiplies by normal powers of two (exact but in
// the subnormal range); a part more than 2^252 below the row's largest is
// dropped.
__device__ __forceinline__ float mul_pow2_neg(float v, int d) {
    if (d < -252) return 0.0f;
    return __fmul_rn(__fmul_rn(v, pow2i(d >> 1)), pow2i(d - (d >> 1)));
}

// 32 values -> X = rint(x * 2^(30-E)) in four byte planes, E the block's
// binade.  The scaling by 2^(30-E) (30-E in [-98, 156]) is two multiplies by
// normal powers of two: exact, except that an intermediate below 2^-126 can
// only arise when the product itself is below 2^-126, where X = 0 either way.
__device__ __forceinline__ FixChunk32 fix_chunk32(const float (&x)[32]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    FixChunk32 f;
    f.e = binade(amax);
    const int sh = 30 - f.e;
    const float s1 = pow2i(sh >> 1), s2 = pow2i(sh - (sh >> 1));
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        int X[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) X[i] = rint_scaled30(__fmul_rn(x[4 * u + i], s1), s2);
        byte_planes4(X[0], X[1], X[2], X[3], f.p[0][u], f.p[1][u], f.p[2][u], f.p[3][u]);
    }
    return f;
}

// Exact block dot sum_e q_e * X_e as int64 (|.| < 2^42): 32 weights as two
// 16-byte chunks.
__device__ __forceinline__ long long fix_dot32(const int4 w0, const int4 w1, const FixChunk32& f) {
    const int wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    int P[4];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        int a = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) a = dp4a_su(wv[u], unsigned(f.p[j][u]), a);
        P[j] = a;
    }
    int a = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) a = __dp4a(wv[u], f.p[3][u], a);
    P[3] = a;
    const long long lo = (long long)P[1] * 256 + P[0];
    return ((long long)P[3] << 24) + ((long long)P[2] << 16) + lo;
}

// The same block dot as fix_dot32, returned split for an exact conversion to
// f32 without 64-bit arithmetic: V = vh * 2^21 + vl with |vh| <= 2^22 and
// -2^21 <= vl < 2^21.  With L = P1*2^8 + P0 and H = P3*2^8 + P2 (so
// V = H*2^16 + L): L = (L >> 21)*2^21 + (L & (2^21-1)) and
// H*2^16 = (H >> 5)*2^21 + (H & 31)*2^16; one 2^21 moves from vl to vh to
// centre vl.  |V| <= 32*128*(2^31 - 2^7) < 2^43 - 2^18 keeps vh in range
// even for -128 weights.
__device__ __forceinline__ int2 fix_dot32_split(const int4 w0, const int4 w1, const FixChunk32& f) {
    const int wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    int P[4];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        int a = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) a = dp4a_su(wv[u], unsigned(f.p[j][u]), a);
        P[j] = a;
    }
    int a = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) a = __dp4a(wv[u], f.p[3][u], a);
    P[3] = a;
    const int L = P[1] * 256 + P[0];   // |P1| < 2^20, |P0| < 2^20
    const int H = P[3] * 256 + P[2];   // |P3| < 2^19, |P2| < 2^20
    return make_int2((H >> 5) + (L >> 21) + 1, (H & 31) * 65536 + (L & 0x1fffff) - 2097152);
}

// f * (vh * 2^21 + vl) exactly as an f32 pair, for fix_dot32_split's parts.
__device__ __forceinline__ DF scaled_pair_split(float f, int2 v) {
    const float fh = small_int_to_float(v.x) * 2097152.0f;   // exact: |vh| <= 2^22
    const float fl = small_int_to_float(v.y);                // exact: |vl| <= 2^21
    const float p1 = __fmul_rn(f, fh);
    const float e1 = __fmaf_rn(f, fh, -p1);
    const float p2 = __fmul_rn(f, fl);
    const float e2 = __fmaf_rn(f, fl, -p2);
    float s, e3;
    two_sum(p1, p2, s, e3);
    return DF{s, __fadd_rn(__fadd_rn(e1, e2), e3)};
}

// f * V exactly as an f32 pair (hi, lo), |lo| <~ 2^-23 |hi|.
__device__ __forceinline__ DF scaled_pair(float f, long long V) {
    const int vh = int(V >> 21);
    const int vl = int(V & 0x1fffff);
    const float fh = small_int_to_float(vh) * 2097152.0f;   // exact: |vh| < 2^21
    const float fl = small_int_to_float(vl);                // exact: 0 <= vl < 2^21
    const float p1 = __fmul_rn(f, fh);
    const float e1 = __fmaf_rn(f, fh, -p1);
    const float p2 = __fmul_rn(f, fl);
    const float e2 = __fmaf_rn(f, fl, -p2);
    float s, e3;
    two_sum(p1, p2, s, e3);
    return DF{s, __fadd_rn(__fadd_rn(e1, e2), e3)};
}

// --------------------------------------------------------------- geometry

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// The KV-row epilogue (decode and row-per-lane kernels): output column n of
// row m, when it falls in the K or V slice, also goes to cache row s_pos[m]
// of that row's sequence (-1: none).
__device__ __forceinline__ void kv_store(const GemvParams& p, const int* s_pos, int m, int64_t n,
                                         float v) {
    const int ps = s_pos[m];
    if (ps < 0) return;
    const int64_t d = n - p.kv_col;
    if (d < 0 || d >= 2 * p.kv_dim) return;
    float* cache = d < p.kv_dim ? p.k_cache : p.v_cache;
    const int64_t dd = d < p.kv_dim ? d : d - p.kv_dim;
    cache[(int64_t(m) * p.n_pos + ps) * p.kv_dim + dd] = v;
}
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

struct Geo {
    int64_t K;
    int slb;        // slice bytes (the last slice may be shorter)
    int nks;        // slices
    int RS;         // rows per stage (8 * rows per warp)
    int rpw;        // rows per consumer warp per stage
    int stage_bytes;
    int nstages;
    int64_t r0, r1; // CTA rows
    int64_t sbrows; // rows per super-block (multiple of RS)
    bool sl_inner = false;   // row block, then slice (the slices of a row block back to back)
};

// Walks the stages in the order producer and consumers share: super-block,
// then slice, then row block (or with sl_inner row block, then slice).
// Advancing never divides.
struct StageIter {
    int64_t sb0, sb_end, rb, ks;
    int sl, kl, slot;
    uint32_t phase;
    bool done;
};

__device__ __forceinline__ void stage_init(const Geo& g, StageIter& it) {
    it.sb0 = g.r0;
    it.sb_end = min64(g.r1, g.r0 + g.sbrows);
    it.rb = g.r0;
    it.ks = 0;
    it.sl = 0;
    it.kl = int(min64(g.slb, g.K));
    it.slot = 0;
    it.phase = 0;
    it.done = g.r0 >= g.r1;
}

__device__ __forceinline__ void stage_next(const Geo& g, StageIter& it) {
    if (g.sl_inner) {
        it.ks += it.kl;
        if (++it.sl == g.nks) {
            it.sl = 0;
            it.ks = 0;
            it.rb += g.RS;
            if (it.rb >= it.sb_end) {
                it.sb0 += g.sbrows;
                it.done = it.sb0 >= g.r1;
                it.sb_end = min64(g.r1, it.sb0 + g.sbrows);
                it.rb = it.sb0;
            }
        }
        it.kl = int(min64(g.slb, g.K - it.ks));
    } else if ((it.rb += g.RS) >= it.sb_end) {
        it.ks += it.kl;
        ++it.sl;
        if (it.sl == g.nks) {
            it.sb0 += g.sbrows;
            it.done = it.sb0 >= g.r1;
            it.sb_end = min64(g.r1, it.sb0 + g.sbrows);
            it.sl = 0;
            it.ks = 0;
        }
        it.kl = int(min64(g.slb, g.K - it.ks));
        it.rb = it.sb0;
    }
    if (++it.slot == g.nstages) {
        it.slot = 0;
        it.phase ^= 1u;
    }
}

template <int MODE, int R>
__host__ __device__ constexpr size_t gemv_smem_bytes() {
    return size_t(kGemvRing) + size_t(kGemvRing) / 16 + 2 * kGemvMaxStages * sizeof(uint64_t) +
           kGemvYaccBytes + size_t(kGemvMaxConsumerWarps) * R * sizeof(ArgmaxCand) + 64;
}

// The arg-max result of one activation row from its best (value, index)
// candidate: a row without any candidate (every logit NaN: NaN is never the
// maximum) gives index 0 and the value NaN.
__device__ __forceinline__ void argmax_store(const ArgmaxCand& b, int32_t* tok, double* maxval,
                                             int m) {
    const bool none = b.i == 0x7fffffffffffffffll;
    tok[m] = none ? 0 : int32_t(b.i);
    if (maxval) maxval[m] = none ? __longlong_as_double(0x7ff8000000000000ll) : b.v;
}

template <int NT>
__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

__device__ __forceinline__ void argmax_keep(double& bv, long long& bi, double v, long long i) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

// The last CTA's reduction of the grid's arg-max candidates (gc[c][rows],
// G CTAs) by all NT consumer threads: a strided share of the CTAs a thread,
// then the warp, then the warps in order (lowest index on ties).  The
// candidates are read from L2, which the ticket's fences made current, many
// at once (a single thread reading them one after another cost a round trip
// to L2 each, tens of microseconds for a grid of 152).  red: NT/32 entries of
// shared scratch.
template <int NT>
__device__ __forceinline__ void argmax_final(const ArgmaxCand* gc, int G, int rows, int tid,
                                             ArgmaxCand* red, int32_t* tok, double* maxval) {
    const int lane = tid & 31, warp = tid >> 5;
    for (int m = 0; m < rows; ++m) {
        double bv = -INFINITY;
        long long bi = 0x7fffffffffffffffll;
        for (int c2 = tid; c2 < G; c2 += NT) {
            const ArgmaxCand* src = gc + size_t(c2) * rows + m;
            argmax_keep(bv, bi, __ldcg(&src->v), __ldcg(&src->i));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const long long oi = __shfl_xor_sync(0xffffffffu, bi, o);
            argmax_keep(bv, bi, ov, oi);
        }
        if (lane == 0) red[warp] = {bv, bi};
        consumer_bar<NT>();
        if (tid == 0) {
            ArgmaxCand b = red[0];
            for (int w = 1; w < NT / 32; ++w) {
                double v = b.v;
                long long i = b.i;
                argmax_keep(v, i, red[w].v, red[w].i);
                b = {v, i};
            }
            argmax_store(b, tok, maxval, m);
        }
        consumer_bar<NT>();
    }
}

// --------------------------------------------------------------- the kernel

template <int MODE, int R, bool ARGMAX>
__global__ void __launch_bounds__(32 * (gemv_warps<MODE, R>() + 1), 1)
    gemv_kernel(const GemvParams p) {
    using A = typename AccT<MODE>::T;
    constexpr int CPL = gemv_cpl<MODE, R>();
    constexpr int kGemvConsumerWarps = gemv_warps<MODE, R>();
    constexpr int kGemvConsumers = 32 * kGemvConsumerWarps;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* wring = smem;
    unsigned char* sring = wring + kGemvRing;
    uint64_t* full = reinterpret_cast<uint64_t*>(sring + kGemvRing / 16);
    uint64_t* empty = full + kGemvMaxStages;
    A* yacc = reinterpret_cast<A*>(empty + kGemvMaxStages);              // [sbrows][R]
    ArgmaxCand* cand = reinterpret_cast<ArgmaxCand*>(reinterpret_cast<unsigned char*>(yacc) +
                                                     kGemvYaccBytes);   // [8][R]
    __shared__ float s_amax[kGemvConsumerWarps][R];
    __shared__ int s_emax[R];
    __shared__ unsigned int s_ticket;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;

    Geo g;
    g.K = p.K;
    g.slb = 512 * CPL;
    g.nks = int((p.K + g.slb - 1) / g.slb);
    {
        const int kmax = int(min64(p.K, g.slb));
        int rpw = (kGemvStageMax / kGemvConsumerWarps) / kmax;
        if (rpw * kGemvConsumerWarps * kmax > kGemvStageMax) rpw = 1;
        g.rpw = rpw < 1 ? 1 : (rpw > 16 ? 16 : rpw);
        g.RS = kGemvConsumerWarps * g.rpw;
        g.stage_bytes = (g.RS * kmax + 1023) & ~1023;
        const int ns = kGemvRing / g.stage_bytes;
        g.nstages = ns > kGemvMaxStages ? kGemvMaxStages : ns;
        g.r0 = p.N * c / G;
        g.r1 = p.N * (c + 1) / G;
        const int64_t yrows = kGemvYaccBytes / int64_t(R * sizeof(A));
        g.sbrows = (yrows / g.RS) * g.RS;
    }

    if (tid == 0) {
        for (int i = 0; i < g.nstages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kGemvConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    const bool scale_bulk = (p.K % 256) == 0;

    if (warp == kGemvConsumerWarps) {
        // -------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            const unsigned char* qsrc = reinterpret_cast<const unsigned char*>(p.q);
            const unsigned char* ssrc = reinterpret_cast<const unsigned char*>(p.s);
            int64_t issued = 0;
            StageIter it;
            stage_init(g, it);
            while (!it.done) {
                if (issued >= g.nstages && !mbar_wait(&empty[it.slot], it.phase ^ 1u, p.err)) break;
                const int nrows = int(min64(g.RS, it.sb_end - it.rb));
                const int kl = it.kl;
                uint32_t bytes = uint32_t(nrows) * kl;
                if (scale_bulk) bytes += uint32_t(nrows) * (kl / 16);
                mbar_arrive_expect_tx(&full[it.slot], bytes);
                unsigned char* wdst = wring + size_t(it.slot) * g.stage_bytes;
                unsigned char* sdst = sring + size_t(it.slot) * (g.stage_bytes / 16);
                if (kl == p.K) {
                    bulk_g2s_hint(wdst, qsrc + it.rb * p.K, uint32_t(nrows) * kl, &full[it.slot],
                                  policy);
                    if (scale_bulk)
                        bulk_g2s_hint(sdst, ssrc + it.rb * (p.K / 16), uint32_t(nrows) * (kl / 16),
                                      &full[it.slot], policy);
                } else {
                    const unsigned char* qrow = qsrc + it.rb * p.K + it.ks;
                    const unsigned char* srow = ssrc + it.rb * (p.K / 16) + it.ks / 16;
                    for (int j = 0; j < nrows; ++j) {
                        bulk_g2s_hint(wdst + size_t(j) * kl, qrow, uint32_t(kl), &full[it.slot],
                                      policy);
                        if (scale_bulk)
                            bulk_g2s_hint(sdst + size_t(j) * (kl / 16), srow, uint32_t(kl / 16),
                                          &full[it.slot], policy);
                        qrow += p.K;
                        srow += p.K / 16;
                    }
                }
                ++issued;
                stage_next(g, it);
            }
            // Never leave with copies in flight into this CTA's shared memory.
            for (int64_t i = max64(0, issued - g.nstages); i < issued; ++i)
                mbar_wait(&full[i % g.nstages], uint32_t((i / g.nstages) & 1), p.err);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    pdl_wait();   // activations and outputs belong to the previous kernel until here

    const int rows = p.rows;
    const int64_t K = p.K, N = p.N, nb = K / Q8_QK;
    const signed char* act8 = reinterpret_cast<const signed char*>(p.act);
    const float* actf = reinterpret_cast<const float*>(p.act);

    if constexpr (MODE == 0) {
        // Per activation row, the binade of its largest |x|: the common scale
        // of all chunk values (each chunk is relative to its own binade).
        float amax[R];
#pragma unroll
        for (int m = 0; m < R; ++m) amax[m] = 0.0f;
        for (int64_t k = int64_t(tid) * 4; k < K; k += 4 * kGemvConsumers) {
#pragma unroll
            for (int m = 0; m < R; ++m) {
                if (m < rows) {
                    const int4 t4 = ldg_nc_v4(actf + m * K + k);
                    amax[m] = fmaxf(amax[m], fmaxf(fmaxf(fabsf(__int_as_float(t4.x)),
                                                         fabsf(__int_as_float(t4.y))),
                                                   fmaxf(fabsf(__int_as_float(t4.z)),
                                                         fabsf(__int_as_float(t4.w)))));
                }
            }
        }
#pragma unroll
        for (int m = 0; m < R; ++m) {
            float a = amax[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            if (lane == 0) s_amax[warp][m] = a;
        }
        consumer_bar<kGemvConsumers>();
        if (tid < R) {
            float a = 0.0f;
            for (int w = 0; w < kGemvConsumerWarps; ++w) a = fmaxf(a, s_amax[w][tid]);
            s_emax[tid] = binade(a);
        }
    }

    // zero the row accumulators (a row's entry is only touched by its warp afterwards)
    for (int i = tid; i < g.sbrows * R; i += kGemvConsumers) yacc[i] = acc_zero(A{});
    consumer_bar<kGemvConsumers>();

    double best_v[ARGMAX ? R : 1];
    long long best_i[ARGMAX ? R : 1];
#pragma unroll
    for (int m = 0; m < (ARGMAX ? R : 1); ++m) {
        best_v[m] = -INFINITY;
        best_i[m] = 0x7fffffffffffffffll;
    }

    // activation chunk registers for the current slice
    int4 a1[CPL][R];
    int4 a2[CPL][R];
    float xdv[CPL][R];
    FixChunk fx[MODE == 0 ? CPL : 1][MODE == 0 ? R : 1];
    float p2s[CPL][R];
    int cur_sl = -1;

    bool ok = true;
    StageIter it;
    stage_init(g, it);
    for (; !it.done; stage_next(g, it)) {
        const int slot = it.slot;
        const int64_t rb = it.rb, ks = it.ks, sb0 = it.sb0;
        const int kl = it.kl, sl = it.sl;
        const int cpr = kl >> 4;
        const int nrows = int(min64(g.RS, it.sb_end - rb));

        if (sl != cur_sl) {
            // new slice: this lane's activation chunks
            cur_sl = sl;
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) {
                const int ch = lane + 32 * cc;
                if (ch < cpr) {
                    const int64_t k = ks + int64_t(ch) * 16;
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        if (m < rows) {
                            if constexpr (MODE == 0) {
                                float xs[16];
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const int4 t4 = ldg_nc_v4(actf + m * K + k + 4 * u);
                                    xs[4 * u + 0] = __int_as_float(t4.x);
                                    xs[4 * u + 1] = __int_as_float(t4.y);
                                    xs[4 * u + 2] = __int_as_float(t4.z);
                                    xs[4 * u + 3] = __int_as_float(t4.w);
                                }
                                fx[cc][m] = fix_chunk(xs);
                                p2s[cc][m] = ldexpf(1.0f, fx[cc][m].e - s_emax[m]);
                            } else {
                                a1[cc][m] = ldg_nc_v4(act8 + m * K + k);
                                if constexpr (MODE == 2)
                                    a2[cc][m] = ldg_nc_v4(act8 + p.plane + m * K + k);
                                xdv[cc][m] = __ldg(p.xd + m * nb + (k >> 5));
                            }
                        }
                    }
                }
            }
        }

        if (ok) ok = mbar_wait(&full[slot], it.phase, p.err);
        ok = __all_sync(0xffffffffu, ok);   // a timeout ends the whole warp's work together
        if (ok) {
            const uint32_t W = smem_u32(wring) + uint32_t(slot * g.stage_bytes);
            const uint32_t SC = smem_u32(sring) + uint32_t(slot * (g.stage_bytes / 16));
            const bool last = (sl == g.nks - 1);
            for (int jj = 0; jj < g.rpw; ++jj) {
                const int r = warp + kGemvConsumerWarps * jj;
                if (r >= nrows) break;
                A part[R];
#pragma unroll
                for (int m = 0; m < R; ++m) part[m] = acc_zero(A{});
                const uint32_t wrow = W + uint32_t(r * kl) + uint32_t(lane * 16);
                if (cpr == 32 * CPL) {
                    // full slice: every chunk valid, no predicates, so the
                    // CPL independent dots interleave
                    int4 w[CPL];
                    float sw[CPL];
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) w[cc] = lds128(wrow + 512 * cc);
                    if (scale_bulk) {
                        const uint32_t srow = SC + uint32_t(r * (kl >> 4)) + uint32_t((lane >> 1) * 2);
#pragma unroll
                        for (int cc = 0; cc < CPL; ++cc) sw[cc] = half_bits_to_float(lds16(srow + 32 * cc));
                    } else {
                        const uint16_t* srow = p.s + (rb + r) * nb + (ks >> 5) + (lane >> 1);
#pragma unroll
                        for (int cc = 0; cc < CPL; ++cc) sw[cc] = half_bits_to_float(__ldg(srow + 16 * cc));
                    }
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        if (m < rows) {
                            if constexpr (MODE == 0) {
                                DF d[CPL];
#pragma unroll
                                for (int cc = 0; cc < CPL; ++cc)
                                    d[cc] = scaled_pair(__fmul_rn(sw[cc], p2s[cc][m]),
                                                        fix_dot(w[cc], fx[cc][m]));
#pragma unroll
                                for (int cc = 0; cc < CPL; ++cc) part[m] = df_add(part[m], d[cc]);
                            } else {
                                float f[CPL];
#pragma unroll
                                for (int cc = 0; cc < CPL; ++cc) {
                                    const int isum = (MODE == 1) ? dot16_i8(w[cc], a1[cc][m])
                                                                 : dot16_i8x2(w[cc], a1[cc][m], a2[cc][m]);
                                    f[cc] = float(isum) * (sw[cc] * xdv[cc][m]);
                                }
#pragma unroll
                                for (int cc = 0; cc < CPL; ++cc) part[m] += f[cc];
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) {
                        const int ch = lane + 32 * cc;
                        if (ch < cpr) {
                            const int4 w = lds128(wrow + 512 * cc);
                            const float sw =
                                scale_bulk
                                    ? half_bits_to_float(lds16(SC + uint32_t(r * (kl >> 4)) + uint32_t((ch >> 1) * 2)))
                                    : half_bits_to_float(__ldg(p.s + (rb + r) * nb + (ks >> 5) + (ch >> 1)));
#pragma unroll
                            for (int m = 0; m < R; ++m) {
                                if (m < rows) {
                                    if constexpr (MODE == 0) {
                                        part[m] = df_add(part[m], scaled_pair(__fmul_rn(sw, p2s[cc][m]),
                                                                              fix_dot(w, fx[cc][m])));
                                    } else {
                                        const int isum = (MODE == 1) ? dot16_i8(w, a1[cc][m])
                                                                     : dot16_i8x2(w, a1[cc][m], a2[cc][m]);
                                        part[m] = fmaf(float(isum), sw * xdv[cc][m], part[m]);
                                    }
                                }
                            }
                        }
                    }
                }
                // one warp reduction per row, then the row's running sum
                const int64_t n = rb + r;
                A* yrow = yacc + int(n - sb0) * R;
#pragma unroll
                for (int m = 0; m < R; ++m) {
                    if (m < rows) {
                        const A tot = warp_sum(part[m]);
                        if (lane == 0) {
                            const A acc = acc_add(yrow[m], tot);
                            if (last) {
                                double val = acc_value(acc);
                                if constexpr (MODE == 0) val = ldexp(val, s_emax[m] - 30);
                                if (p.y) {
                                    if (MODE == 0 && p.out_f64)
                                        reinterpret_cast<double*>(p.y)[m * N + n] = val;
                                    else
                                        reinterpret_cast<float*>(p.y)[m * N + n] = float(val);
                                }
                                if constexpr (ARGMAX) {
                                    if (val > best_v[m] || (val == best_v[m] && n < best_i[m])) {
                                        best_v[m] = val;
                                        best_i[m] = n;
                                    }
                                }
                                yrow[m] = acc_zero(A{});
                            } else {
                                yrow[m] = acc;
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }

    if constexpr (ARGMAX) {
        // Per-CTA candidates, then the last CTA to take a ticket reduces the
        // whole grid's candidates.
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < R; ++m) cand[warp * R + m] = {best_v[m], best_i[m]};
        }
        consumer_bar<kGemvConsumers>();
        ArgmaxCand* gc = reinterpret_cast<ArgmaxCand*>(p.ws + kArgmaxHeader);
        unsigned int* counter = reinterpret_cast<unsigned int*>(p.ws);
        if (tid < rows) {
            ArgmaxCand b = cand[tid];
            for (int w2 = 1; w2 < kGemvConsumerWarps; ++w2) {
                const ArgmaxCand o = cand[w2 * R + tid];
                if (o.v > b.v || (o.v == b.v && o.i < b.i)) b = o;
            }
            gc[size_t(c) * rows + tid] = b;
            __threadfence();
        }
        consumer_bar<kGemvConsumers>();
        if (tid == 0) s_ticket = atomicAdd(counter, 1u);
        consumer_bar<kGemvConsumers>();
        if (s_ticket == unsigned(G - 1)) {
            __threadfence();
            argmax_final<kGemvConsumers>(gc, G, rows, tid, cand, p.tok, p.maxval);
            if (tid == 0) *counter = 0u;
        }
    }
}

template <int MODE, int R, bool ARGMAX>
cudaError_t launch_gemv_t(const GemvArgs& a, const LaunchCtx& ctx) {
    auto kern = gemv_kernel<MODE, R, ARGMAX>;
    constexpr size_t smem = gemv_smem_bytes<MODE, R>();
    static std::atomic<bool> configured[kMaxDevices];
    if (const cudaError_t e = set_smem_once(kern, size_t(smem), ctx.dev, configured); e != cudaSuccess)
        return e;
    GemvParams p{};
    p.q = a.q;
    p.s = a.s;
    p.N = a.N;
    p.K = a.K;
    p.act = a.act;
    p.xd = a.xd;
    p.plane = a.plane;
    p.rows = a.rows;
    p.y = a.y;
    p.out_f64 = a.out_f64;
    p.tok = a.tok;
    p.maxval = a.maxval;
    p.ws = reinterpret_cast<unsigned char*>(a.ws);
    p.err = ctx.dev_err;

    int grid = ctx.num_sms;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (int64_t(grid) > a.N) grid = int(a.N);

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[2];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * (gemv_warps<MODE, R>() + 1));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace q8

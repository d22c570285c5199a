// gemv.cuh -- CUDA-core Q8_0 projection for few activation rows (decode step,
// small batches, the LM head), sm_103a.
//
// The projection at rows = 1..16 is bound by HBM: every weight byte is read
// once per step (34 bytes per 32 weights) and the arithmetic per byte is a
// fraction of a dp4a.  Design:
//
//  * Persistent grid, one CTA per SM.  CTA c owns the contiguous weight rows
//    [N*c/G, N*(c+1)/G), so the imbalance between CTAs is at most one row.
//  * A producer warp streams the CTA's rows through a 4-stage shared-memory
//    ring with the bulk-copy (TMA) engine: a stage is 8*rpw rows by a K-slice
//    of at most 4096 bytes, one contiguous copy when whole rows fit, one copy
//    per row otherwise, plus the matching binary16 scales.  Up to 128 KB per
//    SM are in flight, which covers HBM latency without register pressure.
//  * The weights do not depend on the previous kernel on the stream, so the
//    producer starts before griddepcontrol.wait (programmatic dependent
//    launch); only the consumers wait before reading activations.
//  * Eight consumer warps each own whole weight rows of a stage; lanes walk
//    the row in 16-byte chunks (half a Q8_0 block), read the activation chunk
//    through the read-only path (it is shared by every warp of the SM and
//    stays in L1), and fold each half-block's exact int32 dot with the two
//    scales.  A row ends with one warp-shuffle reduction.
//  * Modes: one-word (4 dp4a per 16 weights), two-word (8 dp4a: hi and lo
//    planes, combined as 128*hi + lo exactly in int32), f32 (exact
//    TwoProduct/TwoSum double-float accumulation in f32 arithmetic, since
//    the GB300's FP64 rate is far below one add per weight at HBM speed).
//  * Optional arg-max epilogue for the LM head: per-CTA best (value, lowest
//    index), then the last CTA to take a ticket reduces all candidates.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace q8 {

constexpr int kGemvConsumerWarps = 8;
constexpr int kGemvThreads = 32 * (kGemvConsumerWarps + 1);
constexpr int kGemvStage = 32768;   // weight bytes per ring stage
constexpr int kGemvStages = 4;
constexpr int kGemvMaxRows = 16;

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
    int KS;          // K-slice bytes of a stage (multiple of 32)
    int nks;         // slices per row
    int rpw;         // rows per consumer warp per stage
    int scale_bulk;  // scales staged by bulk copy (K % 256 == 0)
    int32_t* tok;
    double* maxval;
    unsigned char* ws;
    int* err;
};

__host__ __device__ constexpr size_t gemv_smem_bytes() {
    return size_t(kGemvStages) * kGemvStage + size_t(kGemvStages) * (kGemvStage / 16) +
           2 * kGemvStages * sizeof(uint64_t) +
           size_t(kGemvConsumerWarps) * kGemvMaxRows * sizeof(ArgmaxCand) + 16;
}

__device__ __forceinline__ void consumer_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kGemvConsumerWarps) : "memory");
}

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Error-free transforms in f32 (no contraction: explicit _rn intrinsics).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Accumulates the 16 exact products sw*q_e*x_e of one chunk into (hi, lo).
__device__ __forceinline__ void f32_chunk(const int4 w, float sw, const float4* xv, float& hi,
                                          float& lo) {
    const int words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float xs[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float wv = __fmul_rn(sw, byte_as_float(words[u], j));  // exact: 11 x 7 bits
            const float p = __fmul_rn(wv, xs[j]);
            const float pe = __fmaf_rn(wv, xs[j], -p);                   // exact product error
            float s, e;
            two_sum(hi, p, s, e);
            hi = s;
            lo = __fadd_rn(lo, __fadd_rn(e, pe));
        }
    }
}

template <int MODE, int R, int RPWMAX, bool ARGMAX>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* wring = smem;
    unsigned char* sring = smem + size_t(kGemvStages) * kGemvStage;
    uint64_t* full = reinterpret_cast<uint64_t*>(sring + size_t(kGemvStages) * (kGemvStage / 16));
    uint64_t* empty = full + kGemvStages;
    ArgmaxCand* cand = reinterpret_cast<ArgmaxCand*>(empty + kGemvStages);
    __shared__ unsigned int s_ticket;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int64_t N = p.N, K = p.K, nb = K / Q8_QK;
    const int64_t r0 = N * c / G, r1 = N * (c + 1) / G;
    const int RS = 8 * p.rpw, KS = p.KS, nks = p.nks;
    const int64_t nrb = (r1 - r0 + RS - 1) / RS;
    const int64_t total = nrb * nks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kGemvStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kGemvConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kGemvConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            int64_t issued = 0;
            for (int64_t i = 0; i < total; ++i) {
                const int slot = int(i % kGemvStages);
                if (i >= kGemvStages) {
                    if (!mbar_wait(&empty[slot], uint32_t(((i / kGemvStages) - 1) & 1), p.err))
                        break;
                }
                const int64_t rb = r0 + (i / nks) * RS;
                const int nrows = int(min64(RS, r1 - rb));
                const int64_t ks = int64_t(i % nks) * KS;
                const int kl = int(min64(KS, K - ks));
                uint32_t bytes = uint32_t(nrows) * kl;
                if (p.scale_bulk) bytes += uint32_t(nrows) * (kl / 16);
                mbar_arrive_expect_tx(&full[slot], bytes);
                unsigned char* wdst = wring + size_t(slot) * kGemvStage;
                unsigned char* sdst = sring + size_t(slot) * (kGemvStage / 16);
                const unsigned char* qsrc = reinterpret_cast<const unsigned char*>(p.q);
                const unsigned char* ssrc = reinterpret_cast<const unsigned char*>(p.s);
                if (kl == K) {
                    bulk_g2s_hint(wdst, qsrc + rb * K, uint32_t(nrows) * kl, &full[slot], policy);
                    if (p.scale_bulk)
                        bulk_g2s_hint(sdst, ssrc + rb * (K / 16), uint32_t(nrows) * (kl / 16),
                                      &full[slot], policy);
                } else {
                    for (int j = 0; j < nrows; ++j) {
                        bulk_g2s_hint(wdst + size_t(j) * KS, qsrc + (rb + j) * K + ks, uint32_t(kl),
                                      &full[slot], policy);
                        if (p.scale_bulk)
                            bulk_g2s_hint(sdst + size_t(j) * (KS / 16),
                                          ssrc + (rb + j) * (K / 16) + ks / 16, uint32_t(kl / 16),
                                          &full[slot], policy);
                    }
                }
                ++issued;
            }
            // Never leave with copies in flight into this CTA's shared memory.
            for (int64_t i = max64(0, issued - kGemvStages); i < issued; ++i)
                mbar_wait(&full[i % kGemvStages], uint32_t((i / kGemvStages) & 1), p.err);
        }
        return;
    }

    // ------------------------------------------------------------- consumers
    pdl_wait();  // activations and outputs belong to the previous kernel until here

    const int rows = p.rows;
    const signed char* act8 = reinterpret_cast<const signed char*>(p.act);
    const float* actf = reinterpret_cast<const float*>(p.act);

    float acc[RPWMAX][R];
    float acc_lo[RPWMAX][R];  // f32 mode: low word of the double-float sum
#pragma unroll
    for (int jj = 0; jj < RPWMAX; ++jj)
#pragma unroll
        for (int m = 0; m < R; ++m) acc[jj][m] = acc_lo[jj][m] = 0.0f;

    double best_v[ARGMAX ? R : 1];
    long long best_i[ARGMAX ? R : 1];
#pragma unroll
    for (int m = 0; m < (ARGMAX ? R : 1); ++m) {
        best_v[m] = -INFINITY;
        best_i[m] = 0x7fffffffffffffffll;
    }

    bool ok = true;
    for (int64_t i = 0; i < total; ++i) {
        const int slot = int(i % kGemvStages);
        const int64_t rb = r0 + (i / nks) * RS;
        const int nrows = int(min64(RS, r1 - rb));
        const int sl = int(i % nks);
        const int64_t ks = int64_t(sl) * KS;
        const int kl = int(min64(KS, K - ks));
        if (ok) ok = mbar_wait(&full[slot], uint32_t((i / kGemvStages) & 1), p.err);
        if (ok) {
            const unsigned char* W = wring + size_t(slot) * kGemvStage;
            const uint16_t* SC = reinterpret_cast<const uint16_t*>(sring + size_t(slot) * (kGemvStage / 16));
            const int nch = kl / 16;
#pragma unroll
            for (int jj = 0; jj < RPWMAX; ++jj) {
                const int j = warp + 8 * jj;
                if (jj < p.rpw && j < nrows) {
                    const unsigned char* wrow = W + size_t(j) * KS;
                    for (int ch = lane; ch < nch; ch += 32) {
                        const int4 w = lds_v4(wrow + ch * 16);
                        const int64_t k = ks + ch * 16;
                        const int64_t blk = k >> 5;
                        const float sw =
                            p.scale_bulk ? half_bits_to_float(SC[j * (KS / 32) + (ch >> 1)])
                                         : half_bits_to_float(__ldg(p.s + (rb + j) * nb + blk));
#pragma unroll
                        for (int m = 0; m < R; ++m) {
                            if (m < rows) {
                                if constexpr (MODE == 0) {
                                    float4 xv[4];
                                    const float* xp = actf + m * K + k;
#pragma unroll
                                    for (int u = 0; u < 4; ++u) {
                                        const int4 t = ldg_nc_v4(xp + 4 * u);
                                        xv[u] = make_float4(__int_as_float(t.x), __int_as_float(t.y),
                                                            __int_as_float(t.z), __int_as_float(t.w));
                                    }
                                    f32_chunk(w, sw, xv, acc[jj][m], acc_lo[jj][m]);
                                } else {
                                    int isum;
                                    if constexpr (MODE == 1) {
                                        isum = dot16_i8(w, ldg_nc_v4(act8 + m * K + k));
                                    } else {
                                        isum = dot16_i8x2(w, ldg_nc_v4(act8 + m * K + k),
                                                          ldg_nc_v4(act8 + p.plane + m * K + k));
                                    }
                                    const float sc = sw * __ldg(p.xd + m * nb + blk);
                                    acc[jj][m] = fmaf(float(isum), sc, acc[jj][m]);
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        if (sl == nks - 1) {
            // Row block complete: reduce each owned row across the warp and emit.
#pragma unroll
            for (int jj = 0; jj < RPWMAX; ++jj) {
                const int j = warp + 8 * jj;
                if (jj < p.rpw && j < nrows) {
                    const int64_t n = rb + j;
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        if (m < rows) {
                            double v;
                            if constexpr (MODE == 0) {
                                v = warp_sum(double(acc[jj][m]) + double(acc_lo[jj][m]));
                            } else {
                                v = double(warp_sum(acc[jj][m]));
                            }
                            if (lane == 0) {
                                if (p.y) {
                                    if (MODE == 0 && p.out_f64)
                                        reinterpret_cast<double*>(p.y)[m * N + n] = v;
                                    else
                                        reinterpret_cast<float*>(p.y)[m * N + n] = float(v);
                                }
                                if constexpr (ARGMAX) {
                                    if (v > best_v[m] || (v == best_v[m] && n < best_i[m])) {
                                        best_v[m] = v;
                                        best_i[m] = n;
                                    }
                                }
                            }
                        }
                        acc[jj][m] = 0.0f;
                        acc_lo[jj][m] = 0.0f;
                    }
                }
            }
        }
    }

    if constexpr (ARGMAX) {
        // Per-CTA candidates, then the last CTA to finish reduces them all.
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < R; ++m) cand[warp * kGemvMaxRows + m] = {best_v[m], best_i[m]};
        }
        consumer_bar();
        ArgmaxCand* gc = reinterpret_cast<ArgmaxCand*>(p.ws + kArgmaxHeader);
        unsigned int* counter = reinterpret_cast<unsigned int*>(p.ws);
        if (threadIdx.x < rows) {
            const int m = threadIdx.x;
            ArgmaxCand b = cand[m];
            for (int w2 = 1; w2 < kGemvConsumerWarps; ++w2) {
                const ArgmaxCand o = cand[w2 * kGemvMaxRows + m];
                if (o.v > b.v || (o.v == b.v && o.i < b.i)) b = o;
            }
            gc[size_t(c) * rows + m] = b;
            __threadfence();
        }
        consumer_bar();
        if (threadIdx.x == 0) s_ticket = atomicAdd(counter, 1u);
        consumer_bar();
        if (s_ticket == unsigned(G - 1)) {
            __threadfence();
            if (threadIdx.x < rows) {
                const int m = threadIdx.x;
                ArgmaxCand b = {-INFINITY, 0x7fffffffffffffffll};
                for (int c2 = 0; c2 < G; ++c2) {
                    const volatile ArgmaxCand* src = gc + size_t(c2) * rows + m;
                    const ArgmaxCand o = {src->v, src->i};
                    if (o.v > b.v || (o.v == b.v && o.i < b.i)) b = o;
                }
                p.tok[m] = int32_t(b.i);
                if (p.maxval) p.maxval[m] = b.v;
            }
            if (threadIdx.x == 0) *counter = 0u;
        }
    }
}

// Stage geometry for a (mode, R) kernel and a given K.
inline void gemv_geometry(int64_t K, int rpwmax, GemvParams& p) {
    int rpw = 1;
    const int64_t per_warp_rows = kGemvStage / (8 * K);
    if (per_warp_rows >= 2) rpw = int(per_warp_rows >= rpwmax ? rpwmax : per_warp_rows);
    const int64_t ks_max = kGemvStage / (8 * rpw);
    p.rpw = rpw;
    p.KS = int(K <= ks_max ? K : ks_max);
    p.nks = int((K + p.KS - 1) / p.KS);
    p.scale_bulk = (K % 256 == 0) ? 1 : 0;
}

template <int MODE, int R, int RPWMAX, bool ARGMAX>
cudaError_t launch_gemv_t(const GemvArgs& a, const LaunchCtx& ctx) {
    auto kern = gemv_kernel<MODE, R, RPWMAX, ARGMAX>;
    static bool configured = false;  // per process; the attribute is per function
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(gemv_smem_bytes()));
        if (e != cudaSuccess) return e;
        configured = true;
    }
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
    gemv_geometry(a.K, RPWMAX, p);

    int grid = ctx.num_sms;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (int64_t(grid) > a.N) grid = int(a.N);

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[2];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = gemv_smem_bytes();
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace q8

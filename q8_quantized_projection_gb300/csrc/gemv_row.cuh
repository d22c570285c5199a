// gemv_row.cuh -- the decode-step projection (1 or 2 activation rows), sm_103a.
//
// The decode step is pure HBM streaming: 34 bytes per 32 weights, read once.
// This kernel keeps the memory side as simple as the bulk-copy engine likes
// it and the compute side free of synchronisation:
//
//  * Persistent grid, one CTA per SM; CTA c owns the contiguous weight rows
//    [N*c/G, N*(c+1)/G).
//  * A stage is RS whole rows of the weight matrix (RS*K <= 32 KB), so the
//    producer warp moves it with ONE contiguous bulk copy (plus one for its
//    binary16 scales).  Rows longer than 32 KB are cut into 32 KB slices, one
//    row-slice a stage.  Up to 128 KB per SM are in flight; the producer runs
//    ahead of griddepcontrol.wait because weights never depend on the
//    previous kernel on the stream.
//  * The 16 consumer warps split each stage's rows into parts of PB = 512*CPL
//    bytes of K: warp w always serves part w % NWR of row w / NWR, so its
//    lanes hold that part's activation chunks in registers for the whole
//    kernel (for K <= 32 KB), and every stage costs a lane CPL 16-byte
//    shared loads plus the dots.
//  * A row's parts meet through shared memory: each part's warp publishes its
//    sum, the row's warps meet on a named barrier of their own (2 warps for
//    K = 4096), and the part-0 warp adds the parts in part order (so the
//    result is bitwise reproducible) and emits the row.  No CTA-wide barrier
//    is needed while streaming.
//  * Numerics per mode are those of gemv.cuh (exact int32 block dots for the
//    int8 modes; exact fixed-point chunk dots and f32 pairs for f32).
#pragma once

#include "gemv.cuh"
#include "rmsnorm.cuh"

namespace q8 {

constexpr int kRowWarps = 16;
constexpr int kRowThreads = 32 * (kRowWarps + 1);
constexpr int kRowStage = 32768;
constexpr int kRowMaxRS = 64;

template <int MODE, int R>
__host__ __device__ constexpr int row_cpl() {
    return MODE == 0 ? (R == 1 ? 2 : 1) : (R == 1 ? 4 : 2);
}

// Shared bytes of the fused producer's activation: codes (two planes at most)
// and block scales of one row of up to kFusedMaxK values.
constexpr size_t kFusedActBytes = 2 * 16384 + (16384 / 32) * 4;

template <int MODE, int R, bool FUSE>
__host__ __device__ constexpr size_t row_smem_bytes() {
    using A = typename AccT<MODE>::T;
    return size_t(kGemvRing) + size_t(kGemvRing) / 16 + 2 * kGemvMaxStages * sizeof(uint64_t) +
           size_t(kGemvMaxStages) * kRowWarps * R * sizeof(A) +      // part sums
           kGemvYaccBytes + size_t(kRowWarps) * R * sizeof(ArgmaxCand) + 64 +
           (FUSE ? kFusedActBytes : 0);
}

struct RowGeo {
    int64_t K;
    int KS;          // bytes of K per stage (whole rows when KS == K)
    int nks;         // slices per row
    int RS;          // rows per stage
    int RPW;         // rows per warp per stage when a row has one part
    int NWR;         // warps (parts) per row
    int PB;          // part bytes
    int stage_bytes;
    int nstages;
    int64_t r0, r1;
    int64_t sbrows;  // rows per super-block of running sums (multiple of RS)
};

template <int MODE, int R, bool ARGMAX, bool FUSE>
__global__ void __launch_bounds__(kRowThreads, 1) gemv_row_kernel(const GemvParams p) {
    static_assert(!FUSE || (MODE != 0 && R == 1), "fused producer: int8 modes, one row");
    using A = typename AccT<MODE>::T;
    constexpr int CPL = row_cpl<MODE, R>();
    constexpr int NW = kRowWarps;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* wring = smem;
    unsigned char* sring = wring + kGemvRing;
    uint64_t* full = reinterpret_cast<uint64_t*>(sring + kGemvRing / 16);
    uint64_t* empty = full + kGemvMaxStages;
    A* psum = reinterpret_cast<A*>(empty + kGemvMaxStages);                 // [slot][warp][R]
    A* yacc = reinterpret_cast<A*>(psum + kGemvMaxStages * NW * R);         // [sbrows][R]
    ArgmaxCand* cand = reinterpret_cast<ArgmaxCand*>(reinterpret_cast<unsigned char*>(yacc) +
                                                     kGemvYaccBytes);       // [NW][R]
    __shared__ float s_amax[NW][R];
    __shared__ int s_emax[R];
    __shared__ unsigned int s_ticket;
    __shared__ double s_warp[kProdWarps];
    __shared__ float s_rf;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;

    RowGeo g;
    g.K = p.K;
    g.PB = 512 * CPL;
    {
        int64_t ks = p.K;
        if (ks > kRowStage) ks = kRowStage;
        if (ks > int64_t(NW) * g.PB) ks = int64_t(NW) * g.PB;
        g.KS = int(ks);
        g.nks = int((p.K + g.KS - 1) / g.KS);
        const int npr = (g.KS + g.PB - 1) / g.PB;
        if (npr == 1) {
            int rs = kRowStage / g.KS;
            if (rs > kRowMaxRS) rs = kRowMaxRS;
            rs = (rs / NW) * NW;
            g.RS = rs;
            g.RPW = rs / NW;
            g.NWR = 1;
        } else {
            int rs = kRowStage / g.KS;
            if (rs > NW / npr) rs = NW / npr;
            g.RS = rs < 1 ? 1 : rs;
            g.RPW = 1;
            g.NWR = npr;
        }
        g.stage_bytes = (g.RS * g.KS + 1023) & ~1023;
        const int ns = kGemvRing / g.stage_bytes;
        g.nstages = ns > kGemvMaxStages ? kGemvMaxStages : ns;
        g.r0 = p.N * c / G;
        g.r1 = p.N * (c + 1) / G;
        const int64_t yrows = kGemvYaccBytes / int64_t(R * sizeof(A));
        g.sbrows = (yrows / g.RS) * g.RS;
    }
    // Stage walk shared with gemv.cuh's iterator (RS rows x KS-byte slices).
    Geo sg;
    sg.K = g.K;
    sg.slb = g.KS;
    sg.nks = g.nks;
    sg.RS = g.RS;
    sg.rpw = g.RPW;
    sg.stage_bytes = g.stage_bytes;
    sg.nstages = g.nstages;
    sg.r0 = g.r0;
    sg.r1 = g.r1;
    sg.sbrows = g.sbrows;

    if (tid == 0) {
        for (int i = 0; i < g.nstages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    const bool scale_bulk = (p.K % 256) == 0;

    if (warp == NW) {
        // -------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t policy = policy_evict_first();
            const unsigned char* qsrc = reinterpret_cast<const unsigned char*>(p.q);
            const unsigned char* ssrc = reinterpret_cast<const unsigned char*>(p.s);
            int64_t issued = 0;
            StageIter it;
            stage_init(sg, it);
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
                stage_next(sg, it);
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
    const float* xdp = p.xd;
    int64_t plane = p.plane;
    if constexpr (FUSE) {
        // The producer, fused: RMSNorm -> quant of the one activation row into
        // shared memory, by the same code and thread layout as act_quant, while
        // the producer warp already streams weights.
        static_assert(32 * NW == kProdThreads, "fused producer needs kProdThreads consumers");
        unsigned char* sact = reinterpret_cast<unsigned char*>(cand + NW * R) + 64;
        float* sxd = reinterpret_cast<float*>(sact + 2 * kFusedMaxK);
        const float rf = row_rms_scale(p.h, K, p.eps, tid, 1, s_warp, &s_rf);
        row_quantize<MODE, true>(p.h, p.gain, rf, K, tid, sact, K, sxd);
        consumer_bar<32 * NW>();
        act8 = reinterpret_cast<const signed char*>(sact);
        xdp = sxd;
        plane = K;
    }
    // this warp's place in a stage
    const int rw = (g.NWR == 1) ? warp : warp / g.NWR;   // first row (NWR == 1: rows rw + NW*j)
    const int pw = (g.NWR == 1) ? 0 : warp % g.NWR;      // part
    const bool active = (g.NWR == 1) || (rw < g.RS);

    if constexpr (MODE == 0) {
        float amax[R];
#pragma unroll
        for (int m = 0; m < R; ++m) amax[m] = 0.0f;
        for (int64_t k = int64_t(tid) * 4; k < K; k += 4 * 32 * NW) {
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
        consumer_bar<32 * NW>();
        if (tid < R) {
            float a = 0.0f;
            for (int w = 0; w < NW; ++w) a = fmaxf(a, s_amax[w][tid]);
            s_emax[tid] = binade(a);
        }
    }
    for (int i = tid; i < g.sbrows * R; i += 32 * NW) yacc[i] = acc_zero(A{});
    consumer_bar<32 * NW>();

    double best_v[ARGMAX ? R : 1];
    long long best_i[ARGMAX ? R : 1];
#pragma unroll
    for (int m = 0; m < (ARGMAX ? R : 1); ++m) {
        best_v[m] = -INFINITY;
        best_i[m] = 0x7fffffffffffffffll;
    }

    int4 a1[CPL][R];
    int4 a2[CPL][R];
    float xdv[CPL][R];
    FixChunk fx[MODE == 0 ? CPL : 1][MODE == 0 ? R : 1];
    float p2s[CPL][R];
    int cur_sl = -1;
    int cpp = 0;   // chunks in this warp's part of the current slice

    bool ok = true;
    StageIter it;
    stage_init(sg, it);
    for (; !it.done; stage_next(sg, it)) {
        const int slot = it.slot;
        const int64_t rb = it.rb, ks = it.ks, sb0 = it.sb0;
        const int kl = it.kl, sl = it.sl;
        const int nrows = int(min64(g.RS, it.sb_end - rb));
        const int pbyte0 = pw * g.PB;   // this warp's part within the slice

        if (sl != cur_sl) {
            cur_sl = sl;
            const int pbytes = kl - pbyte0 < g.PB ? (kl - pbyte0 > 0 ? kl - pbyte0 : 0) : g.PB;
            cpp = pbytes >> 4;
#pragma unroll
            for (int cc = 0; cc < CPL; ++cc) {
                const int ch = lane + 32 * cc;
#pragma unroll
                for (int m = 0; m < R; ++m) {
                    a1[cc][m] = a2[cc][m] = make_int4(0, 0, 0, 0);
                    xdv[cc][m] = 0.0f;
                    p2s[cc][m] = 0.0f;
                    if constexpr (MODE == 0) fx[cc][m] = FixChunk{};
                }
                if (active && ch < cpp) {
                    const int64_t k = ks + pbyte0 + int64_t(ch) * 16;
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
                            } else if constexpr (FUSE) {
                                a1[cc][m] = lds_v4(act8 + m * K + k);
                                if constexpr (MODE == 2) a2[cc][m] = lds_v4(act8 + plane + m * K + k);
                                xdv[cc][m] = xdp[m * nb + (k >> 5)];
                            } else {
                                a1[cc][m] = ldg_nc_v4(act8 + m * K + k);
                                if constexpr (MODE == 2)
                                    a2[cc][m] = ldg_nc_v4(act8 + plane + m * K + k);
                                xdv[cc][m] = __ldg(xdp + m * nb + (k >> 5));
                            }
                        }
                    }
                }
            }
        }

        if (ok) ok = mbar_wait(&full[slot], it.phase, p.err);
        ok = __all_sync(0xffffffffu, ok);   // a timeout ends the whole warp's work together
        // rows this warp serves in this stage (it releases the slot after the
        // last of them is in registers, before any arithmetic)
        int nj = 0;
        if (active) {
            if (g.NWR == 1) {
                nj = (nrows - rw + NW - 1) / NW;
                if (nj > g.RPW) nj = g.RPW;
                if (nj < 0) nj = 0;
            } else {
                nj = rw < nrows ? 1 : 0;
            }
        }
        bool released = false;
        if (active) {
            const uint32_t W = smem_u32(wring) + uint32_t(slot * g.stage_bytes);
            const uint32_t SC = smem_u32(sring) + uint32_t(slot * (g.stage_bytes / 16));
            const bool last_slice = (sl == g.nks - 1);
            const bool full_part = (cpp == 32 * CPL);
            for (int j = 0; j < nj; ++j) {
                const int r = (g.NWR == 1) ? rw + NW * j : rw;
                A part[R];
#pragma unroll
                for (int m = 0; m < R; ++m) part[m] = acc_zero(A{});
                const uint32_t wrow = W + uint32_t(r * kl + pbyte0) + uint32_t(lane * 16);
                const int blk0 = pbyte0 >> 5;   // first block of the part within the slice
                // ---- loads: this row's weights and scales into registers
                int4 w[CPL];
                float sw[CPL];
                if (ok && full_part && scale_bulk) {
                    // common case: every chunk valid, scales staged with the weights
                    const uint32_t srow = SC + uint32_t(r * (kl >> 4)) + uint32_t((blk0 + (lane >> 1)) * 2);
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) w[cc] = lds128(wrow + 512 * cc);
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) sw[cc] = half_bits_to_float(lds16(srow + 32 * cc));
                } else {
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) {
                        const bool v = ok && (full_part || lane + 32 * cc < cpp);
                        const int blk = blk0 + (lane >> 1) + 16 * cc;
                        w[cc] = make_int4(0, 0, 0, 0);
                        sw[cc] = 0.0f;
                        if (v) {
                            w[cc] = lds128(wrow + 512 * cc);
                            sw[cc] = scale_bulk
                                         ? half_bits_to_float(lds16(SC + uint32_t(r * (kl >> 4)) + uint32_t(blk * 2)))
                                         : half_bits_to_float(__ldg(p.s + (rb + r) * nb + (ks >> 5) + blk));
                        }
                    }
                }
                if (j == nj - 1 && ok) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[slot]);
                    released = true;
                }
                // ---- arithmetic (invalid chunks hold zero weights and scales)
#pragma unroll
                for (int m = 0; m < R; ++m) {
                    if (m < rows) {
                        if constexpr (MODE == 0) {
                            DF d[CPL];
#pragma unroll
                            for (int cc = 0; cc < CPL; ++cc)
                                d[cc] = scaled_pair(__fmul_rn(sw[cc], p2s[cc][m]), fix_dot(w[cc], fx[cc][m]));
#pragma unroll
                            for (int cc = 0; cc < CPL; ++cc) part[m] = df_add(part[m], d[cc]);
                        } else {
#pragma unroll
                            for (int cc = 0; cc < CPL; ++cc) {
                                const int isum = (MODE == 1) ? dot16_i8(w[cc], a1[cc][m])
                                                             : dot16_i8x2(w[cc], a1[cc][m], a2[cc][m]);
                                part[m] = fmaf(float(isum), sw[cc] * xdv[cc][m], part[m]);
                            }
                        }
                    }
                }
                A tot[R];
#pragma unroll
                for (int m = 0; m < R; ++m) tot[m] = warp_sum(part[m]);
                // A row's parts meet through shared memory: every part's warp
                // publishes its sum, the row group syncs on its own named
                // barrier, and the part-0 warp adds the parts in order.
                bool finisher = true;
                if (g.NWR > 1) {
                    if (lane == 0) {
                        A* ps = psum + (slot * NW + warp) * R;
#pragma unroll
                        for (int m = 0; m < R; ++m) ps[m] = tot[m];
                    }
                    named_bar(2 + rw, 32 * g.NWR);
                    finisher = (pw == 0);
                    if (finisher && lane == 0) {
#pragma unroll
                        for (int m = 0; m < R; ++m) {
                            A s = psum[(slot * NW + rw * g.NWR) * R + m];
                            for (int q2 = 1; q2 < g.NWR; ++q2)
                                s = acc_add(s, psum[(slot * NW + rw * g.NWR + q2) * R + m]);
                            tot[m] = s;
                        }
                    }
                }
                if (finisher && lane == 0) {
                    const int64_t n = rb + r;
                    A* yrow = yacc + int(n - sb0) * R;
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        if (m < rows) {
                            const A acc = (g.nks > 1) ? acc_add(yrow[m], tot[m]) : tot[m];
                            if (last_slice) {
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
                                if (g.nks > 1) yrow[m] = acc_zero(A{});
                            } else {
                                yrow[m] = acc;
                            }
                        }
                    }
                }
            }
        }
        if (ok && !released) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }

    if constexpr (ARGMAX) {
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < R; ++m) cand[warp * R + m] = {best_v[m], best_i[m]};
        }
        consumer_bar<32 * NW>();
        ArgmaxCand* gc = reinterpret_cast<ArgmaxCand*>(p.ws + kArgmaxHeader);
        unsigned int* counter = reinterpret_cast<unsigned int*>(p.ws);
        if (tid < rows) {
            ArgmaxCand b = cand[tid];
            for (int w2 = 1; w2 < NW; ++w2) {
                const ArgmaxCand o = cand[w2 * R + tid];
                if (o.v > b.v || (o.v == b.v && o.i < b.i)) b = o;
            }
            gc[size_t(c) * rows + tid] = b;
            __threadfence();
        }
        consumer_bar<32 * NW>();
        if (tid == 0) s_ticket = atomicAdd(counter, 1u);
        consumer_bar<32 * NW>();
        if (s_ticket == unsigned(G - 1)) {
            __threadfence();
            if (tid < rows) {
                ArgmaxCand b = {-INFINITY, 0x7fffffffffffffffll};
                for (int c2 = 0; c2 < G; ++c2) {
                    const volatile ArgmaxCand* src = gc + size_t(c2) * rows + tid;
                    const ArgmaxCand o = {src->v, src->i};
                    if (o.v > b.v || (o.v == b.v && o.i < b.i)) b = o;
                }
                p.tok[tid] = int32_t(b.i);
                if (p.maxval) p.maxval[tid] = b.v;
            }
            if (tid == 0) *counter = 0u;
        }
    }
}

template <int MODE, int R, bool ARGMAX, bool FUSE = false>
cudaError_t launch_gemv_row_t(const GemvArgs& a, const LaunchCtx& ctx) {
    auto kern = gemv_row_kernel<MODE, R, ARGMAX, FUSE>;
    constexpr size_t smem = row_smem_bytes<MODE, R, FUSE>();
    static bool configured = false;  // per process; one device per process
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
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
    p.h = a.h;
    p.gain = a.gain;
    p.eps = a.eps;

    int grid = ctx.num_sms;
    if (grid > kMaxGrid) grid = kMaxGrid;
    if (int64_t(grid) > a.N) grid = int(a.N);

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[2];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace q8

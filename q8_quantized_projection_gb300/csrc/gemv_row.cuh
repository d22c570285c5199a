// gemv_row.cuh -- the decode-step projection (1 to 8 activation rows), sm_103a.
//
// The decode step is pure HBM streaming: 34 bytes per 32 weights, read once.
// The kernel keeps the memory side as simple as the bulk-copy engine likes it
// and the compute side free of synchronisation:
//
//  * Persistent grid, one CTA per SM; CTA c owns the contiguous weight rows
//    [N*c/G, N*(c+1)/G).
//  * A stage is RS whole rows of the weight matrix (RS*K <= 32 KB), moved by
//    ONE contiguous bulk copy (plus one for its binary16 scales); rows longer
//    than the stage are cut into slices, one row-slice a stage.  160 KB per SM
//    are in flight (192 KB in f32 mode); the producer warp runs ahead of
//    griddepcontrol.wait, since weights never depend on the previous kernel
//    on the stream.
//  * A row-slice is cut into npr parts of PB = 512*CPL bytes (npr a power of
//    two; trailing parts may be short or empty), so a stage holds RS*npr
//    (row, part) pairs, served as items = RS*npr/rpw items of rpw rows of one
//    part (rpw = 4 in f32 mode; 2 for one-word 4 and 8 rows and two-word 2
//    and 4 rows; else 1), items | 16.  Consumer warp w always
//    serves item w % items, in the stages whose ring slot is congruent to
//    w / items modulo 16/items (so every phase of a slot's barriers is seen by
//    the same warps): its part never changes, so its lanes hold that part's
//    activation chunks in registers for the whole kernel (one slice) and a
//    stage costs a lane CPL 16-byte shared loads plus the dots.  The slot is
//    released as soon as the weights are in registers.
//  * Each item's warp-reduced sum goes to a shared-memory slot of its own
//    (row, slice, part); at the end of a super-block of rows the consumers
//    meet once and add every row's parts in slice and part order, so the
//    result is bitwise reproducible.  Nothing synchronises consumer warps
//    while weights stream.
//  * Numerics: exact int32 block dots for the int8 modes; for f32 (one row a
//    launch) a lane owns a whole 32-value block: its 31-bit fixed-point copy
//    relative to the block's binade, an exact block dot, one f32-pair scaling,
//    each part's sums relative to the part's largest binade (rescaled to the
//    row's in the combine).
//  * Fused producer (FUSE): the consumers run RMSNorm -> quant (or, by PROD,
//    the residual added before the norm, or the SwiGLU of a gate+up row) in
//    the prologue while the producer warp streams weights; KV adds the
//    KV-cache-row epilogue to the combine.
#pragma once

#include "gemv.cuh"
#include "rmsnorm.cuh"

namespace q8 {

constexpr int kRowWarps = 16;
constexpr int kRowThreads = 32 * (kRowWarps + 1);
constexpr int kRowStage = 32768;       // weight bytes of one stage at most
constexpr int kRowRing = 163840;       // weight bytes in flight per CTA (int8 modes)
constexpr int kRowRingF32 = 196608;    // f32 mode: six 32 KB stages, so the two warp
                                       // groups of K = 4096 rows own three slots each

template <int MODE>
__host__ __device__ constexpr int row_ring() {
    return MODE == 0 ? kRowRingF32 : kRowRing;
}
constexpr int kRowPsumBytes = 16384;   // part sums of one super-block of rows
// f32 mode, beside the part sums: the (slice, part) binades in the first half,
// the 32-value blocks' binades of a shared block conversion (up to 16384
// values) in the second
constexpr int kRowEpBytes = 2048;
constexpr int kRowEpPartBytes = 1024;

// Weight-ring bytes of a launch.  f32 mode with a residual or SwiGLU producer
// fused and more than 4096 values a row: the converted activation (128 bytes
// of planes a 32-value block, 4K bytes; the residual producer stages its
// input s there first) stays in shared memory for the whole launch, in the
// ring's last 4K bytes (rounded up to 1 KB), which the stages give up.  K <=
// 16384 there, so at least 128 KB of stages remain.  (The plain RMSNorm
// producer keeps the full ring: its per-warp conversion is cheap, and in a
// chained layer the deeper ring measured faster than converting once.)
template <int MODE, bool FUSE, int PROD>
__host__ __device__ inline bool row_planes_after_ring(int64_t K) {
    return MODE == 0 && FUSE && PROD != kProdPlain && K > 4096;
}
template <int MODE, bool FUSE, int PROD>
__host__ __device__ inline int row_ring_of(int64_t K) {
    if (row_planes_after_ring<MODE, FUSE, PROD>(K))
        return row_ring<MODE>() - int((4 * K + 1023) & ~int64_t(1023));
    return row_ring<MODE>();
}

// 16-byte chunks a lane owns per part: the activation registers (R rows, one
// or two planes, or 17 words of fixed point in f32 mode) stay within ~32.
template <int MODE, int R>
__host__ __device__ constexpr int row_cpl() {
    return MODE == 1 ? 8 / R : MODE == 2 ? 4 / R : (R == 1 ? 2 : 1);
}

// Rows a warp serves per stage: the f32 mode's items are short (1 KB), so a
// warp takes up to four rows of its part (sharing its activation block): four
// independent dot chains, and one butterfly reduction for all of them.  The
// int8 modes with one or two chunks a lane (one-word 4 and 8 rows, two-word 2
// and 4) take two rows, so one butterfly over 2R values serves twice the
// weights.
template <int MODE, int R>
__host__ __device__ constexpr int row_rpw() {
    return (MODE == 0 && R == 1) ? 4
           : ((MODE == 1 && R >= 4) || (MODE == 2 && R >= 2)) ? 2
                                                              : 1;
}

// Bytes per (slice, part) kept beside the part sums: the f32 one-row path
// stores each part's activation binade there (its sums are relative to it).
template <int MODE, int R>
__host__ __device__ constexpr int row_part_extra() {
    return (MODE == 0 && R == 1) ? 2 : 0;
}

// Shared bytes of the fused producer's activation: codes (two planes at most)
// and block scales of one row of up to kFusedMaxK values.
constexpr size_t kFusedActBytes = 2 * 16384 + (16384 / 32) * 4;

template <int MODE, int R, bool FUSE>
__host__ __device__ constexpr size_t row_smem_bytes() {
    return size_t(row_ring<MODE>()) + size_t(row_ring<MODE>()) / 16 + 2 * kGemvMaxStages * sizeof(uint64_t) +
           kRowPsumBytes + (MODE == 0 ? kRowEpBytes : 0) + size_t(kRowWarps) * R * sizeof(ArgmaxCand) + 64 +
           (FUSE && MODE != 0 ? kFusedActBytes : 0);
}

struct RowGeo {
    int KS;          // bytes of K per slice (whole rows when KS == K)
    int nks;         // slices per row
    int PB;          // part bytes
    int npr;         // parts per slice: a power of two <= 16
    int nprr;        // parts that hold data (the rest are empty)
    int RS;          // rows per stage: a power of two
    int rpw;         // rows a warp serves per stage (its part of each)
    int items;       // RS * npr / rpw, a divisor of kRowWarps
    int stride;      // kRowWarps / items: warp groups, one per slot residue
    int stage_bytes;
    int nstages;
    int64_t r0, r1;
    int64_t sbrows;  // rows per super-block (a multiple of RS, >= RS when usable)
    int ep_off;      // byte offset of the per-(slice, part) binades in the part-sum area
};

__host__ __device__ inline RowGeo row_geo(int64_t N, int64_t K, int G, int c, int cpl,
                                          int psum_row_unit, int rpw_max, int ring,
                                          int part_extra) {
    RowGeo g;
    g.PB = 512 * cpl;
    int64_t ks = K;
    if (ks > kRowStage) ks = kRowStage;
    if (ks > int64_t(kRowWarps) * g.PB) ks = int64_t(kRowWarps) * g.PB;
    // rows of rpw_max within one stage: long rows are cut into slices
    if (rpw_max > 1 && ks > kRowStage / rpw_max) ks = kRowStage / rpw_max;
    g.KS = int(ks);
    g.nks = int((K + g.KS - 1) / g.KS);
    g.nprr = (g.KS + g.PB - 1) / g.PB;
    g.npr = 1;
    while (g.npr < g.nprr) g.npr <<= 1;
    const int rsmax = kRowStage / g.KS;
    g.RS = 1;
    while (g.RS * 2 <= rsmax && g.RS * 2 * g.npr <= kRowWarps * rpw_max) g.RS <<= 1;
    g.rpw = g.RS < rpw_max ? g.RS : rpw_max;
    while (g.RS * g.npr > kRowWarps * g.rpw) g.RS >>= 1;   // (never: kept as a guard)
    g.items = g.RS * g.npr / g.rpw;
    g.stride = kRowWarps / g.items;
    g.stage_bytes = (g.RS * g.KS + 1023) & ~1023;
    const int ns = ring / g.stage_bytes;
    g.nstages = ns > kGemvMaxStages ? kGemvMaxStages : ns;
    g.r0 = N * c / G;
    g.r1 = N * (c + 1) / G;
    const int64_t per_row = int64_t(g.nks) * g.nprr * psum_row_unit;
    const int64_t ep_bytes = (int64_t(g.nks) * g.nprr * part_extra + 15) & ~int64_t(15);
    g.ep_off = kRowPsumBytes;   // in an area of kRowEpBytes after the part sums
    g.sbrows = ep_bytes > kRowEpPartBytes ? 0 : ((kRowPsumBytes / per_row) / g.RS) * g.RS;
    return g;
}

// Whether the decode kernel handles this K (the part sums of RS rows fit).
template <int MODE, int R>
inline bool row_kernel_fits(int64_t K) {
    using A = typename AccT<MODE>::T;
    const RowGeo g = row_geo(1, K, 1, 0, row_cpl<MODE, R>(), int(R * sizeof(A)), row_rpw<MODE, R>(),
                             row_ring<MODE>(), row_part_extra<MODE, R>());
    // the f32 one-row items take four rows RS/4 apart (rows a stage >= 4, which
    // every K up to 2^20 gives: slices of at most 8192 values leave room for 4)
    if (MODE == 0 && R == 1 && (g.rpw != 4 || g.RS % 4 != 0)) return false;
    return g.sbrows >= g.RS;
}

// Whether the f32 one-row kernel runs K's stages row block, then slice: rows
// cut into slices whose count divides the warp groups, which divide the ring,
// so that each warp group's ring slots always carry the same slice and a warp
// converts its activation block once instead of at every slice change.
inline bool row_slices_inner(int64_t K) {
    const RowGeo g = row_geo(1, K, 1, 0, row_cpl<0, 1>(), int(sizeof(DF)), row_rpw<0, 1>(),
                             row_ring<0>(), row_part_extra<0, 1>());
    return g.nks > 1 && g.stride % g.nks == 0 && g.nstages % g.stride == 0;
}

// Sums each of R per-lane values over the warp with a butterfly that halves
// the rows at every exchange (log2(R) exchanges of R/2, R/4, ... values, then
// a plain reduction over the 32/R lanes left): lanes [r*32/R, (r+1)*32/R)
// end with row r's total.  Fixed order, so bitwise reproducible.
template <int R>
__device__ __forceinline__ float warp_sum_rows(const float (&v)[R], int lane) {
    float cur[R];
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i] = v[i];
#pragma unroll
    for (int step = 16, h = R / 2; h >= 1; step >>= 1, h >>= 1) {
        const bool upper = (lane & step) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = upper ? cur[i] : cur[i + h];
            const float keep = upper ? cur[i + h] : cur[i];
            cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, step);
        }
    }
    float s = cur[0];
#pragma unroll
    for (int o = 16 / R; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// The same butterfly for f32 pairs: lanes [r*32/R, (r+1)*32/R) end with row
// r's total, each exchange an error-free f32-pair addition.
template <int R>
__device__ __forceinline__ DF warp_sum_rows(const DF (&v)[R], int lane) {
    DF cur[R];
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i] = v[i];
#pragma unroll
    for (int step = 16, h = R / 2; h >= 1; step >>= 1, h >>= 1) {
        const bool upper = (lane & step) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const DF send = upper ? cur[i] : cur[i + h];
            const DF keep = upper ? cur[i + h] : cur[i];
            const DF got{__shfl_xor_sync(0xffffffffu, send.hi, step),
                         __shfl_xor_sync(0xffffffffu, send.lo, step)};
            cur[i] = df_add(keep, got);
        }
    }
    DF s = cur[0];
#pragma unroll
    for (int o = 16 / R; o > 0; o >>= 1) {
        const DF got{__shfl_xor_sync(0xffffffffu, s.hi, o), __shfl_xor_sync(0xffffffffu, s.lo, o)};
        s = df_add(s, got);
    }
    return s;
}

// A lane's 32-value block of f32-mode planes from shared memory (block b's
// 16-byte word group i in slot i ^ (b & 7) of its 128 bytes) and its binade.
__device__ __forceinline__ void load_planes_block(uint32_t planes_a, const short* pe, int blk,
                                                  FixChunk32& f) {
    const uint32_t base = planes_a + uint32_t(blk) * 128u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int4 v = lds128(base + uint32_t(((i ^ (blk & 7)) << 4)));
        f.p[i >> 1][4 * (i & 1) + 0] = v.x;
        f.p[i >> 1][4 * (i & 1) + 1] = v.y;
        f.p[i >> 1][4 * (i & 1) + 2] = v.z;
        f.p[i >> 1][4 * (i & 1) + 3] = v.w;
    }
    f.e = pe[blk];
}

// Four f32 activation values: read as they are, or (f32 mode with the
// producer fused) formed as x = (s*rf)*g with the producer's two roundings,
// s = h or, with a residual r, h + r rounded once.
// PROD == kProdSwiglu: h points into the fused gate+up row, whose up half
// starts K values later, and x is the SwiGLU of the two (no norm).
template <bool FUSE, int PROD = kProdPlain>
__device__ __forceinline__ void load_x4(const float* x, const float* h, const float* r, const float* g,
                                        float rf, float (&v)[4], int64_t K = 0) {
    if constexpr (FUSE && PROD == kProdSwiglu) {
        const float4 s = load_swiglu4(h, K, 0);
        v[0] = s.x;
        v[1] = s.y;
        v[2] = s.z;
        v[3] = s.w;
        return;
    }
    const int4 t4 = ldg_nc_v4(FUSE ? h : x);
    v[0] = __int_as_float(t4.x);
    v[1] = __int_as_float(t4.y);
    v[2] = __int_as_float(t4.z);
    v[3] = __int_as_float(t4.w);
    if constexpr (FUSE) {
        if (r) {
            const int4 r4 = ldg_nc_v4(r);
            v[0] = __fadd_rn(v[0], __int_as_float(r4.x));
            v[1] = __fadd_rn(v[1], __int_as_float(r4.y));
            v[2] = __fadd_rn(v[2], __int_as_float(r4.z));
            v[3] = __fadd_rn(v[3], __int_as_float(r4.w));
        }
        float gg[4] = {1.0f, 1.0f, 1.0f, 1.0f};
        if (g) {
            const int4 g4 = ldg_nc_v4(g);
            gg[0] = __int_as_float(g4.x);
            gg[1] = __int_as_float(g4.y);
            gg[2] = __int_as_float(g4.z);
            gg[3] = __int_as_float(g4.w);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[e] = __fmul_rn(v[e], rf);
            if (g) v[e] = __fmul_rn(v[e], gg[e]);
        }
    }
}

// PROD (fused producer only): kProdPlain (RMSNorm of h), kProdResidual (the
// residual added before the norm) or kProdSwiglu (the SwiGLU of the fused
// gate+up row h); each a separate instantiation, so the plain fused kernel
// carries none of the others.
// KV: the KV-row epilogue (the one-row fused decode launch only).
// SLI: stages run row block, then slice (the unfused f32 one-row kernel, rows
// cut into slices whose count divides the warp groups, which divide the ring:
// row_slices_inner).
template <int MODE, int R, bool ARGMAX, bool FUSE, int PROD = kProdPlain, bool KV = false,
          bool SLI = false, bool PLN = false>
__global__ void __launch_bounds__(kRowThreads, 1) gemv_row_kernel(const GemvParams p) {
    static_assert(!FUSE || R == 1, "fused producer: one row");
    static_assert(MODE != 0 || R == 1, "f32 mode: one row per launch");
    static_assert(PROD == kProdPlain || FUSE, "producer kinds belong to the fused producer");
    constexpr bool RES = PROD == kProdResidual;
    constexpr bool NORM = PROD != kProdSwiglu;
    // residual input and the updated residual stream (written by CTA 0 only)
    const float* const res = RES ? p.res : nullptr;
    float* const s_out = RES && blockIdx.x == 0 ? p.s_out : nullptr;
    using A = typename AccT<MODE>::T;
    constexpr int CPL = row_cpl<MODE, R>();
    constexpr int NW = kRowWarps;
    constexpr int NT = 32 * NW;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* wring = smem;
    constexpr int kRing = row_ring<MODE>();
    unsigned char* sring = wring + kRing;
    uint64_t* full = reinterpret_cast<uint64_t*>(sring + kRing / 16);
    uint64_t* empty = full + kGemvMaxStages;
    A* psum = reinterpret_cast<A*>(empty + kGemvMaxStages);   // [sbrows][nks][nprr][R]
    ArgmaxCand* cand = reinterpret_cast<ArgmaxCand*>(reinterpret_cast<unsigned char*>(psum) +
                                                     kRowPsumBytes +
                                                     (MODE == 0 ? kRowEpBytes : 0));   // [NW][R]
    __shared__ unsigned int s_ticket;
    __shared__ int s_pos[R];   // KV-row epilogue: each row's cache position
    __shared__ float2 s_pair[kProdWarps];
    __shared__ float s_rf;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    // PLN: the f32 planes' area after a shortened ring (row_planes_after_ring)
    static_assert(!PLN || (MODE == 0 && FUSE && PROD != kProdPlain),
                  "the planes after the ring serve the fused f32 residual and SwiGLU kernels");
    const int ring = PLN ? row_ring_of<MODE, FUSE, PROD>(p.K) : kRing;
    const RowGeo g = row_geo(p.N, p.K, G, c, CPL, int(R * sizeof(A)), row_rpw<MODE, R>(), ring,
                             row_part_extra<MODE, R>());
    // f32 mode, one row: a lane owns a whole 32-value block of its part (one
    // binade, one weight scale, one exact dot and one f32-pair scaling), and
    // each part's sums are relative to the part's own largest binade
    constexpr bool kBL = (MODE == 0 && R == 1 && CPL == 2);
    static_assert(!SLI || kBL, "the slice-inner order serves the f32 one-row kernel");
    short* s_ep = reinterpret_cast<short*>(reinterpret_cast<unsigned char*>(psum) + g.ep_off);

    if (tid == 0) {
        for (int i = 0; i < g.nstages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], g.items);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    const bool scale_bulk = (p.K % 256) == 0;

    if (warp == NW) {
        // -------------------------------------------------------------- producer
        if (lane == 0) {
            Geo sg;
            sg.K = p.K;
            sg.slb = g.KS;
            sg.nks = g.nks;
            sg.RS = g.RS;
            sg.rpw = 1;
            sg.stage_bytes = g.stage_bytes;
            sg.nstages = g.nstages;
            sg.r0 = g.r0;
            sg.r1 = g.r1;
            sg.sbrows = g.sbrows;
            sg.sl_inner = SLI;
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
    if (KV && tid < rows) {
        // positions belong to the previous kernel until griddepcontrol.wait;
        // one outside the cache writes nothing and is reported
        int ps = p.pos[tid];
        if (ps < 0 || ps >= p.n_pos) {
            atomicExch(p.err, Q8_DEVERR_POSITION);
            ps = -1;
        }
        s_pos[tid] = ps;
    }
    const signed char* act8 = reinterpret_cast<const signed char*>(p.act);
    const float* actf = reinterpret_cast<const float*>(p.act);
    const float* xdp = p.xd;
    int64_t plane = p.plane;
    float rf = 1.0f;   // f32 mode, fused: x = (h*rf)*g is formed where it is used
    if constexpr (FUSE && MODE == 0) {
        // f32: the consumers convert x into fixed-point planes themselves (no
        // code plane); with the norm only rf is computed here, and the RMS pass
        // keeps the input for the block conversion below: in the part-sum area
        // (not in use yet) up to 4096 values, else in the area after the ring
        float* const stage = PLN ? reinterpret_cast<float*>(wring + ring)
                                 : (g.nks == 1 && K <= 4096) ? reinterpret_cast<float*>(psum) : nullptr;
        if constexpr (NORM) rf = row_rms_scale(p.h, res, s_out, K, p.eps, tid, 1, s_pair, &s_rf, stage);
    } else if constexpr (FUSE) {
        static_assert(MODE != 0, "the shared-memory activation exists for the int8 modes only");
        // The producer, fused: RMSNorm -> quant of the one activation row into
        // shared memory, by the same code and thread layout as act_quant, while
        // the producer warp already streams weights.
        static_assert(NT == kProdThreads, "fused producer needs kProdThreads consumers");
        unsigned char* sact = reinterpret_cast<unsigned char*>(cand + NW * R) + 64;
        float* sxd = reinterpret_cast<float*>(sact + 2 * kFusedMaxK);
        // CTA 0 writes the updated residual stream, when asked
        row_produce<MODE, NORM, PROD>(p.h, res, s_out, p.gain, p.eps, K, tid, 1, s_pair, &s_rf, sact,
                                      K, sxd);
        consumer_bar<NT>();
        act8 = reinterpret_cast<const signed char*>(sact);
        xdp = sxd;
        plane = K;
    }

    if constexpr (ARGMAX) {
        // each warp's best (value, lowest index) per row, kept in shared
        // memory between super-blocks (out of the streaming loop's registers)
        if (tid < NW * R) cand[tid] = {-INFINITY, 0x7fffffffffffffffll};
    }

    // this warp's place in every stage it serves
    const int q = warp % g.items;
    const int jrow = q / g.npr;   // (first) row within the stage; the others RS/rpw apart
    const int pw = q % g.npr;     // part within the row-slice
    const int s_first = warp / g.items;

    int4 a1[CPL][R];
    int4 a2[CPL][R];
    float xdv[CPL][R];
    FixChunk32 fxb;
    float p2sb = 0.0f;
    bool validb = false;
    int cur_sl = -1;
    int ncc = 0, rag = 0;   // full 512-byte chunk columns of this part, lanes of the ragged one
    // f32 one-row kernel, the shared block conversion: each 32-value block is
    // converted once, by one thread, and every warp reads its blocks from
    // shared memory (a quarter of the conversions and of the activation's L2
    // traffic).  Block b's 32 words sit at b*128 bytes, 16-byte word group i in
    // slot i ^ (b & 7) (no bank conflicts); the blocks' binades follow the
    // parts' binades.  Rows of one slice up to 4096 values: warp w converts
    // part w into the part-sum area (not in use yet), and each warp keeps its
    // one block in registers for the launch.  PLN (a residual or SwiGLU
    // producer fused, more than 4096 values): warp w converts the w-th 1024 values (part w % nprr
    // of slice w / nprr: slices of whole parts) into the area after the ring,
    // where they stay, and a warp reloads its block at each change of slice.
    if constexpr (kBL) {
        if (PLN || (g.nks == 1 && K <= 4096)) {
            const uint32_t planes_a = smem_u32(PLN ? wring + ring : reinterpret_cast<unsigned char*>(psum));
            short* const pe = reinterpret_cast<short*>(reinterpret_cast<unsigned char*>(psum) + g.ep_off +
                                                       kRowEpPartBytes);   // block binades [K/32]
            // PLN: one warp a (slice, part), <= 16 (K <= 16384); the empty
            // parts of a ragged last slice record the binade of zero, which
            // the combine reads with the others
            if (warp < (PLN ? g.nks * g.nprr : g.npr)) {
                const int64_t k0 = int64_t(warp) * g.PB;
                const int pbytes = int(min64(max64(K - k0, 0), g.PB));
                const bool valid = lane < (pbytes >> 5);
                FixChunk32 f = FixChunk32{};
                f.e = -126;
                if (valid) {
                    const int64_t k = k0 + int64_t(lane) * 32;
                    float xs[32];
                    if constexpr (FUSE && NORM) {
                        // the RMS pass kept the input (h, or h + r) in this very
                        // block of the area: x = (s*rf)*g, then the planes in place
                        const float* sp = reinterpret_cast<const float*>(
                                              PLN ? wring + ring : reinterpret_cast<unsigned char*>(psum)) +
                                          k;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const float4 s4 = *reinterpret_cast<const float4*>(sp + 4 * u);
                            float gg[4] = {1.0f, 1.0f, 1.0f, 1.0f};
                            if (p.gain) {
                                const int4 g4 = ldg_nc_v4(p.gain + k + 4 * u);
                                gg[0] = __int_as_float(g4.x);
                                gg[1] = __int_as_float(g4.y);
                                gg[2] = __int_as_float(g4.z);
                                gg[3] = __int_as_float(g4.w);
                            }
                            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float v = __fmul_rn(sv[e], rf);
                                if (p.gain) v = __fmul_rn(v, gg[e]);
                                xs[4 * u + e] = v;
                            }
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            float xv[4];
                            load_x4<FUSE, PROD>(actf + k + 4 * u, p.h + k + 4 * u,
                                                RES ? res + k + 4 * u : nullptr,
                                                p.gain ? p.gain + k + 4 * u : nullptr, rf, xv, K);
                            xs[4 * u + 0] = xv[0];
                            xs[4 * u + 1] = xv[1];
                            xs[4 * u + 2] = xv[2];
                            xs[4 * u + 3] = xv[3];
                        }
                    }
                    f = fix_chunk32(xs);
                }
                const int ep = __reduce_max_sync(0xffffffffu, f.e);
                if constexpr (PLN) {
                    // the (slice, part) these values form
                    const int sl_w = int(k0 / g.KS);
                    const int pw_w = int((k0 - int64_t(sl_w) * g.KS) / g.PB);
                    if (lane == 0) s_ep[sl_w * g.nprr + pw_w] = short(ep);
                } else {
                    if (lane == 0 && warp < g.nprr) s_ep[warp] = short(ep);
                }
                if (valid) {
                    const int blk = warp * (g.PB >> 5) + lane;
                    const uint32_t base = planes_a + uint32_t(blk) * 128u;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        sts128(base + uint32_t(((i ^ (blk & 7)) << 4)), uint32_t(f.p[i >> 1][4 * (i & 1) + 0]),
                               uint32_t(f.p[i >> 1][4 * (i & 1) + 1]), uint32_t(f.p[i >> 1][4 * (i & 1) + 2]),
                               uint32_t(f.p[i >> 1][4 * (i & 1) + 3]));
                    pe[blk] = short(f.e);
                }
            }
            consumer_bar<NT>();
            if constexpr (!PLN) {
                // one slice: this warp's block into registers for the launch
                cur_sl = 0;
                const int pbytes = int(min64(max64(K - int64_t(pw) * g.PB, 0), g.PB));
                validb = lane < (pbytes >> 5);
                fxb = FixChunk32{};
                fxb.e = -126;
                if (validb) load_planes_block(planes_a, pe, pw * (g.PB >> 5) + lane, fxb);
                p2sb = validb ? ldexpf(1.0f, fxb.e - s_ep[pw]) : 0.0f;
                consumer_bar<NT>();   // the area holds part sums from here on
            }
        }
    }

    const uint32_t wring_a = smem_u32(wring), sring_a = smem_u32(sring);
    bool ok = true;
    int64_t gbase = 0;   // global index of the super-block's first stage
    for (int64_t sb0 = g.r0; sb0 < g.r1; sb0 += g.sbrows) {
        const int sbn = int(min64(g.sbrows, g.r1 - sb0));
        const int nrb = (sbn + g.RS - 1) / g.RS;
        const int nst_sb = g.nks * nrb;
        int sl = 0, rbi = 0;
        int slot = int(gbase % g.nstages);
        uint32_t phase = uint32_t((gbase / g.nstages) & 1);
        for (int t = 0; t < nst_sb && ok; ++t) {
            // a ring slot is always served by the same warps, so each of them
            // sees every phase of the slot's barriers
            if ((slot & (g.stride - 1)) != s_first) {
                if constexpr (SLI) {
                    if (++sl == g.nks) {
                        sl = 0;
                        ++rbi;
                    }
                } else if (++rbi == nrb) {
                    rbi = 0;
                    ++sl;
                }
                if (++slot == g.nstages) {
                    slot = 0;
                    phase ^= 1u;
                }
                continue;
            }
            const int64_t ks = int64_t(sl) * g.KS;
            const int kl = int(min64(g.KS, K - ks));
            if (sl != cur_sl) {
                // this part's activation chunks into registers
                cur_sl = sl;
                int pbytes = kl - pw * g.PB;
                pbytes = pbytes < 0 ? 0 : (pbytes > g.PB ? g.PB : pbytes);
                ncc = pbytes >> 9;
                rag = (pbytes & 511) >> 4;
                if constexpr (kBL) {
                    validb = lane < (pbytes >> 5);
                    fxb = FixChunk32{};
                    fxb.e = -126;   // the binade of zero: below every other
                    if constexpr (PLN) {
                        // the slice's block, converted in the prologue
                        const uint32_t planes_a = smem_u32(wring + ring);
                        const short* pe = reinterpret_cast<const short*>(reinterpret_cast<unsigned char*>(psum) +
                                                                         g.ep_off + kRowEpPartBytes);
                        if (validb) load_planes_block(planes_a, pe, int(ks >> 5) + pw * (g.PB >> 5) + lane, fxb);
                        p2sb = validb ? ldexpf(1.0f, fxb.e - s_ep[sl * g.nprr + pw]) : 0.0f;
                    } else if (validb) {
                        const int64_t k = ks + pw * g.PB + int64_t(lane) * 32;
                        float xs[32];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            float xv[4];
                            load_x4<FUSE, PROD>(actf + k + 4 * u, p.h + k + 4 * u,
                                                RES ? res + k + 4 * u : nullptr,
                                                p.gain ? p.gain + k + 4 * u : nullptr, rf, xv, K);
                            xs[4 * u + 0] = xv[0];
                            xs[4 * u + 1] = xv[1];
                            xs[4 * u + 2] = xv[2];
                            xs[4 * u + 3] = xv[3];
                        }
                        fxb = fix_chunk32(xs);
                    }
                    if constexpr (!PLN) {
                        // the part's largest binade; its sums are in units of 2^(ep-30)
                        const int ep = __reduce_max_sync(0xffffffffu, fxb.e);
                        p2sb = validb ? ldexpf(1.0f, fxb.e - ep) : 0.0f;
                        if (lane == 0 && pw < g.nprr) s_ep[sl * g.nprr + pw] = short(ep);
                    }
                }
#pragma unroll
                for (int cc = 0; cc < (kBL ? 0 : CPL); ++cc) {
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        a1[cc][m] = a2[cc][m] = make_int4(0, 0, 0, 0);
                        xdv[cc][m] = 0.0f;
                    }
                    if (cc < ncc || (cc == ncc && lane < rag)) {
                        const int64_t k = ks + pw * g.PB + int64_t(lane) * 16 + 512 * cc;
#pragma unroll
                        for (int m = 0; m < R; ++m) {
                            if (m < rows) {
                                if constexpr (FUSE) {
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

            if (ok) ok = mbar_wait(&full[slot], phase, p.err);
            ok = __all_sync(0xffffffffu, ok);   // a timeout ends the whole warp's work together
            const int row_sb = rbi * g.RS + jrow;   // row within the super-block
            const bool have = ok && row_sb < sbn && pw < g.nprr;
            // weights and scales of this item, at most 4 chunks (64 registers
            // worth) at a time; the slot goes back once the last group is loaded
            constexpr int GC = CPL < 4 ? CPL : 4;
            A part[R];
#pragma unroll
            for (int m = 0; m < R; ++m) part[m] = acc_zero(A{});
            const uint32_t wrow = wring_a + uint32_t(slot * g.stage_bytes + jrow * kl + pw * g.PB) +
                                  uint32_t(lane * 16);
            const int blk0 = (pw * g.PB) >> 5;   // first block of the part within the slice
            const uint32_t sbase = sring_a + uint32_t(slot * (g.stage_bytes / 16) + jrow * (kl >> 4));
            constexpr int RPW = row_rpw<MODE, R>();
            DF part2[RPW];   // f32 mode: this warp's rows of the stage
            unsigned have_rows = 0;   // f32 mode: bit i, row i of the item holds data
            // int8 modes, two rows of the part per stage (kMR)
            constexpr bool kMR = (MODE != 0 && RPW > 1);
            float pm[kMR ? RPW : 1][kMR ? R : 1];
            bool hvm[kMR ? RPW : 1];
            if constexpr (kMR) {
                const int rstep = g.RS / g.rpw;
                int4 wm[RPW][CPL];
                float swm[RPW][CPL];
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
                    const int rr = jrow + i * rstep;   // row within the stage
                    hvm[i] = have && i < g.rpw && rbi * g.RS + rr < sbn;
                    const uint32_t wr = wring_a + uint32_t(slot * g.stage_bytes + rr * kl + pw * g.PB) +
                                        uint32_t(lane * 16);
                    const uint32_t sr = sring_a + uint32_t(slot * (g.stage_bytes / 16) + rr * (kl >> 4));
                    const int64_t nrow = sb0 + rbi * g.RS + rr;
#pragma unroll
                    for (int cc = 0; cc < CPL; ++cc) {
                        wm[i][cc] = make_int4(0, 0, 0, 0);
                        swm[i][cc] = 0.0f;
                        if (hvm[i] && (cc < ncc || (cc == ncc && lane < rag))) {
                            const int blk = blk0 + (lane >> 1) + 16 * cc;
                            wm[i][cc] = lds128(wr + 512 * cc);
                            swm[i][cc] = scale_bulk ? half_bits_to_float(lds16(sr + uint32_t(blk * 2)))
                                                    : half_bits_to_float(__ldg(p.s + nrow * nb + (ks >> 5) + blk));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(&empty[slot]);
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        pm[i][m] = 0.0f;
#pragma unroll
                        for (int cc = 0; cc < CPL; ++cc) {
                            const int isum = (MODE == 1) ? dot16_i8(wm[i][cc], a1[cc][m])
                                                         : dot16_i8x2(wm[i][cc], a1[cc][m], a2[cc][m]);
                            const float fi = MODE == 1 ? small_int_to_float(isum) : float(isum);
                            pm[i][m] = fmaf(fi, swm[i][cc] * xdv[cc][m], pm[i][m]);
                        }
                    }
                }
            }
            if constexpr (kBL) {
                // each row's exact dot right after its weights are in
                // registers (one row's weights live at a time); the slot goes
                // back after the last row, then the f32-pair scalings.  Every
                // f32 one-row geometry serves four rows a warp (RS >= 4), rows
                // RS/4 apart.
                const int rstep = g.RS >> 2;
                int2 vb[RPW];
                uint16_t swh[RPW];
                unsigned rows_in = 0;   // bit i: the item's row i holds data
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
                    const int rr = jrow + i * rstep;   // row within the stage
                    const bool hr = have && rbi * g.RS + rr < sbn;
                    rows_in |= unsigned(hr) << i;
                    vb[i] = make_int2(0, 0);
                    swh[i] = 0;
                    if (hr && validb) {
                        // the lane's block; its scale sits at a sixteenth of the
                        // offset within the scale ring
                        const uint32_t o = uint32_t(slot * g.stage_bytes + rr * kl + pw * g.PB + lane * 32);
                        const int4 w0 = lds128(wring_a + o);
                        const int4 w1 = lds128(wring_a + o + 16u);
                        if (scale_bulk) swh[i] = lds16(sring_a + (o >> 4));
                        vb[i] = fix_dot32_split(w0, w1, fxb);
                    }
                }
                __syncwarp();
                if (lane == 0 && ok) mbar_arrive(&empty[slot]);
                if (!scale_bulk && validb) {
                    // scales not staged with the weights (K not a multiple of 256)
#pragma unroll
                    for (int i = 0; i < RPW; ++i)
                        if ((rows_in >> i) & 1u)
                            swh[i] = __ldg(p.s + (sb0 + rbi * g.RS + jrow + i * rstep) * nb + (ks >> 5) + blk0 + lane);
                }
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
                    part2[i] = DF{0.0f, 0.0f};
                    if (((rows_in >> i) & 1u) && validb)
                        part2[i] = scaled_pair_split(__fmul_rn(half_bits_to_float(swh[i]), p2sb), vb[i]);
                }
                have_rows = rows_in;
            }
#pragma unroll
            for (int c0 = 0; c0 < ((kBL || kMR) ? 0 : CPL); c0 += GC) {
                int4 w[GC];
                float sw[GC];
                if (have) {
                    if (ncc == CPL && scale_bulk) {
                        // common case: every chunk valid, scales staged with the weights
                        const uint32_t srow = sbase + uint32_t((blk0 + (lane >> 1)) * 2);
#pragma unroll
                        for (int cc = 0; cc < GC; ++cc) w[cc] = lds128(wrow + 512 * (c0 + cc));
#pragma unroll
                        for (int cc = 0; cc < GC; ++cc)
                            sw[cc] = half_bits_to_float(lds16(srow + 32 * (c0 + cc)));
                    } else {
                        const int64_t nrow = sb0 + row_sb;
#pragma unroll
                        for (int cc = 0; cc < GC; ++cc) {
                            const int ch = c0 + cc;
                            w[cc] = make_int4(0, 0, 0, 0);
                            sw[cc] = 0.0f;
                            if (ch < ncc || (ch == ncc && lane < rag)) {
                                const int blk = blk0 + (lane >> 1) + 16 * ch;
                                w[cc] = lds128(wrow + 512 * ch);
                                sw[cc] = scale_bulk ? half_bits_to_float(lds16(sbase + uint32_t(blk * 2)))
                                                    : half_bits_to_float(__ldg(p.s + nrow * nb + (ks >> 5) + blk));
                            }
                        }
                    }
                }
                if (c0 + GC >= CPL) {
                    // the weights are in registers: give the slot back
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(&empty[slot]);
                }
                if constexpr (MODE != 0) if (have) {
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        if (m < rows) {
                            {
#pragma unroll
                                for (int cc = 0; cc < GC; ++cc) {
                                    const int isum = (MODE == 1) ? dot16_i8(w[cc], a1[c0 + cc][m])
                                                                 : dot16_i8x2(w[cc], a1[c0 + cc][m], a2[c0 + cc][m]);
                                    // |isum| < 2^18 (one word) / 2^24 (two words)
                                    const float fi = MODE == 1 ? small_int_to_float(isum) : float(isum);
                                    part[m] = fmaf(fi, sw[cc] * xdv[c0 + cc][m], part[m]);
                                }
                            }
                        }
                    }
                }
            }
            if constexpr (kBL) {
                // one butterfly for the warp's rows: lanes [i*32/RPW, ...) end with row i
                const DF tot = warp_sum_rows<RPW>(part2, lane);
                const int i = lane / (32 / RPW);
                if ((lane & (32 / RPW - 1)) == 0 && ((have_rows >> i) & 1u)) {
                    const int rsb = rbi * g.RS + jrow + i * (g.RS >> 2);
                    psum[(size_t(rsb) * g.nks + sl) * g.nprr + pw] = reinterpret_cast<const A&>(tot);
                }
            } else if constexpr (kMR) {
                // one butterfly over the warp's RPW x R sums: lanes [v*32/V, ...)
                // end with sum v = i*R + m
                constexpr int V = RPW * R;
                float flat[V];
#pragma unroll
                for (int i = 0; i < RPW; ++i)
#pragma unroll
                    for (int m = 0; m < R; ++m) flat[i * R + m] = pm[i][m];
                const float tot = warp_sum_rows<V>(flat, lane);
                const int v = lane / (32 / V), i = v / R, m = v % R;
                bool hv = false;
#pragma unroll
                for (int k = 0; k < RPW; ++k)
                    if (k == i) hv = hvm[k];
                if ((lane & (32 / V - 1)) == 0 && hv) {
                    const int rsb = rbi * g.RS + jrow + i * (g.RS / g.rpw);
                    psum[((size_t(rsb) * g.nks + sl) * g.nprr + pw) * R + m] = tot;
                }
            } else if constexpr (MODE != 0) {
                if (have) {
                    A* ps = psum + ((size_t(row_sb) * g.nks + sl) * g.nprr + pw) * R;
                    const float tot = warp_sum_rows<R>(part, lane);
                    if ((lane & (32 / R - 1)) == 0) ps[lane / (32 / R)] = tot;
                }
            }
            if constexpr (SLI) {
                if (++sl == g.nks) {
                    sl = 0;
                    ++rbi;
                }
            } else if (++rbi == nrb) {
                rbi = 0;
                ++sl;
            }
            if (++slot == g.nstages) {
                slot = 0;
                phase ^= 1u;
            }
        }
        gbase += nst_sb;

        // every row of the super-block: its parts in slice and part order
        consumer_bar<NT>();
        if (ok) {
            const int nparts = g.nks * g.nprr;
            int E = -126;   // one row: the largest part binade is the row's
            if constexpr (kBL) {
                for (int u = 0; u < nparts; ++u) E = max(E, int(s_ep[u]));
            }
            // arg-max: this thread's rows all have activation row m = tid % R
            // (NT is a multiple of R)
            double bv = -INFINITY;
            long long bi = 0x7fffffffffffffffll;
            for (int i = tid; i < sbn * R; i += NT) {
                const int row_sb = i / R, m = i % R;
                if (m >= rows) continue;
                const A* ps = psum + size_t(row_sb) * nparts * R + m;
                A s = ps[0];
                const int64_t n = sb0 + row_sb;
                if constexpr (kBL) {
                    // each part rescaled to the row's binade (powers of two: exact
                    // but in the subnormal range), then added in order
                    s = DF{mul_pow2_neg(s.hi, s_ep[0] - E), mul_pow2_neg(s.lo, s_ep[0] - E)};
                    for (int u = 1; u < nparts; ++u) {
                        const A v = ps[size_t(u) * R];
                        const int d = s_ep[u] - E;
                        s = acc_add(s, DF{mul_pow2_neg(v.hi, d), mul_pow2_neg(v.lo, d)});
                    }
                    if (!ARGMAX && !p.out_f64) {
                        // f32 output: the pair rounded once, then scaled by 2^(E-30)
                        const int sc = E - 30;   // in [-156, 98]
                        const float yv =
                            __fmul_rn(__fmul_rn(__fadd_rn(s.hi, s.lo), pow2i(sc >> 1)), pow2i(sc - (sc >> 1)));
                        if (p.y) reinterpret_cast<float*>(p.y)[n] = yv;
                        if constexpr (KV) kv_store(p, s_pos, 0, n, yv);
                        continue;
                    }
                } else {
                    for (int u = 1; u < nparts; ++u) s = acc_add(s, ps[size_t(u) * R]);
                }
                double val = acc_value(s);
                if constexpr (kBL) {
                    val = ldexp(val, E - 30);
                }
                if (p.y) {
                    if (MODE == 0 && p.out_f64)
                        reinterpret_cast<double*>(p.y)[m * N + n] = val;
                    else
                        reinterpret_cast<float*>(p.y)[m * N + n] = float(val);
                }
                if constexpr (KV) kv_store(p, s_pos, m, n, float(val));
                if constexpr (ARGMAX) argmax_keep(bv, bi, val, n);
            }
            if constexpr (ARGMAX) {
                // over the warp's lanes of the same row m, then into the warp's
                // candidate of that row
#pragma unroll
                for (int o = 16; o >= R; o >>= 1) {
                    const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const long long oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    argmax_keep(bv, bi, ov, oi);
                }
                if (lane < R) {
                    ArgmaxCand& c = cand[warp * R + lane];
                    double cv = c.v;
                    long long ci = c.i;
                    argmax_keep(cv, ci, bv, bi);
                    c = {cv, ci};
                }
            }
        }
        consumer_bar<NT>();
    }

    if constexpr (ARGMAX) {
        // the warps' candidates (merged per super-block above), then per CTA,
        // then the last CTA to take a ticket reduces every CTA's candidate
        // (lowest index on ties)
        consumer_bar<NT>();
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
        consumer_bar<NT>();
        if (tid == 0) s_ticket = atomicAdd(counter, 1u);
        consumer_bar<NT>();
        if (s_ticket == unsigned(G - 1)) {
            __threadfence();
            argmax_final<NT>(gc, G, rows, tid, cand, p.tok, p.maxval);
            if (tid == 0) *counter = 0u;
        }
    }
}

template <int MODE, int R, bool ARGMAX, bool FUSE = false, int PROD = kProdPlain, bool KV = false>
cudaError_t launch_gemv_row_t(const GemvArgs& a, const LaunchCtx& ctx) {
    auto kern = gemv_row_kernel<MODE, R, ARGMAX, FUSE, PROD, KV, false, false>;
    bool sli = false;   // the kernel's variant: slice-inner order, or planes after the ring
    if constexpr (MODE == 0 && R == 1 && !FUSE) {
        // (measured: the fused launches run slower in this order, so they keep
        // the slice-outer one)
        sli = row_slices_inner(a.K);
        if (sli) kern = gemv_row_kernel<MODE, R, ARGMAX, FUSE, PROD, KV, true, false>;
    }
    if constexpr (MODE == 0 && R == 1 && FUSE && PROD != kProdPlain) {
        sli = row_planes_after_ring<MODE, FUSE, PROD>(a.K);
        if (sli) kern = gemv_row_kernel<MODE, R, ARGMAX, FUSE, PROD, KV, false, true>;
    }
    constexpr size_t smem = row_smem_bytes<MODE, R, FUSE>();
    static std::atomic<bool> configured[2][kMaxDevices];   // per kernel (order), per device
    if (const cudaError_t e = set_smem_once(kern, size_t(smem), ctx.dev, configured[sli ? 1 : 0]);
        e != cudaSuccess)
        return e;
    if (!row_kernel_fits<MODE, R>(a.K)) return cudaErrorInvalidValue;   // callers check first
    if (FUSE && a.K > kFusedMaxK) return cudaErrorInvalidValue;         // the producer's row
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
    p.res = a.res;
    p.s_out = a.s_out;
    p.gain = a.gain;
    p.eps = a.eps;
    p.pos = a.pos;
    p.kv_col = a.kv_col;
    p.kv_dim = a.kv_dim;
    p.n_pos = a.n_pos;
    p.k_cache = a.k_cache;
    p.v_cache = a.v_cache;

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

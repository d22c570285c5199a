// gemv_rpl.cuh -- the projection with a weight row a lane: the decode step
// (one row, with the RMSNorm -> quant producer and the KV-row epilogue fused or
// not), batches of up to 8 one-word or 4 two-word rows, f32 rows one or two at
// a time, and the LM head's arg-max; K % 1024 == 0.
//
// The decode kernel (gemv_row.cuh) gives each lane 16-byte chunks of a row's
// part and sums a row over the warp with a butterfly per item; with several
// activation rows that butterfly and the per-chunk scale products dominate its
// instruction count.  Here lane l of a warp owns weight row l of a group of 32
// rows: it
// reads its row's 32-value blocks and block scales from shared memory, each
// activation row's block (the same address for every lane: one broadcast
// load) and its scale, and keeps R running sums in registers.  No lane-to-lane
// reduction is left in the stream.
//
// A stage covers 32 weight rows x 1024 values of K (512 for one-row int8
// launches, see RplCfg):
//   - the weights as eight (four) tiles of 32 rows x 128 bytes, gathered by one
//     3-D TMA box (128-byte swizzle, so the 16-byte loads of 8 consecutive
//     lanes hit distinct bank groups);
//   - the rows' block scales, 32 rows x 64 bytes (64-byte swizzle, same
//     reason);
//   - the activation rows' codes (four tiles of R rows x 256 bytes a plane, one
//     3-D box) and block scales (R rows x 32), unless the rows are resident in
//     shared memory for the launch: the fused producer's row, and every f32
//     launch (fixed-point planes, see RplCfg).
// So a stage takes 4 TMA instructions (5 two-word): the producer's issue rate,
// which shares the memory-instruction queue with the consumers' shared-memory
// loads, kept up with HBM only once the eight weight tiles were one box.
// Weights and scales are issued before the wait on the previous kernel, with
// an evict-first L2 hint (read once per launch); activations after it.  A ring
// of four stages (eight half stages), the 16 consumer warps in four groups:
// group g takes stages t with t % 4 == g (from slots g, or g and g + 4, so
// each slot's phases are waited on by one group in order), and its warp q
// reduces quarter q of each (8 or 4 blocks) for every row of the group.  At the end of a row group the warps' sums go to shared
// memory and are added in warp order (fixed: results do not depend on timing):
// by a combining warp through two buffers (no consumer warp waits for
// another), or by the consumer warps themselves between two barriers.
//
// CTAs own whole 32-row groups (the ceil(N/32) groups split evenly over the
// grid): a tile never carries rows that another CTA reads as well.
//
// Requires K % 1024 == 0 (whole stages).  Every wait is bounded (device error
// word on time-out).
#pragma once

#include <cuda.h>

#include "gemv.cuh"
#include "gemv_row.cuh"
#include "rmsnorm.cuh"

namespace q8 {

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle sw);
bool make_map3(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t dims[3],
               const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle sw);

constexpr int kRplWarps = 16;                      // consumer warps
constexpr int kRplRows = 32;                       // weight rows a group: a lane each
constexpr int kRplGroups = 4;                      // consumer warp groups of four warps

// FUSE: one activation row, produced (RMSNorm -> quant, or by PROD the
// residual added before the norm, or the SwiGLU of a gate+up row) by the
// consumer warps into shared memory for the whole launch; the stages then
// carry weights and scales only.
// MODE 0 (f32 activations, one or two rows): the rows are converted once per
// CTA into shared memory, as 31-bit fixed-point byte planes of each 32-value
// block relative to the block's binade, with each block's factor 2^(E_b - E)
// to the row's largest binade E (fused or not).
template <int MODE, int R, bool FUSE = false, bool ARGMAX = false>
struct RplCfg {
    // A stage: 1024 values of K in a ring of four slots, one per warp group;
    // the one-row int8 launches (fused or not: the row is resident, so two TMA
    // instructions a stage) take 512 values in eight slots, warp group g
    // owning slots g and g + 4, so that a group's next stage loads while it
    // works on the current one (fused layer one-word 50.5 -> 47.5 us, two-word
    // 53.2 -> 49.8 us; launches that copy activations every stage lose at that
    // size: twice the TMA instructions a byte).  Fused and plain one-row
    // launches share the schedule, so their results stay bitwise equal.
    static constexpr bool kHalf = MODE != 0 && R == 1 && !ARGMAX;
    static constexpr int kKS = kHalf ? 512 : 1024;           // values of K a stage
    static constexpr int kSlots = kHalf ? 8 : 4;             // ring slots
    static constexpr int kBPW = kKS / Q8_QK / kRplGroups;    // blocks a warp takes of a stage
    // the row resident in shared memory: fused, f32, and one-row int8 (not the
    // LM head's arg-max, which keeps the 1024-value stages: 83.2 against
    // 84.3 us with half stages)
    static constexpr bool kResAct = FUSE || MODE == 0 || kHalf;
    static constexpr int kPlanes = MODE == 2 ? 2 : 1;
    static constexpr int kW = kRplRows * kKS;                // 8 tiles of [32][128]
    static constexpr int kS = kRplRows * (kKS / Q8_QK) * 2;  // [32][64] bytes of f16 scales
    static constexpr int kX = kResAct ? 0 : kPlanes * R * kKS;        // [plane][4 tiles][R][256]
    static constexpr int kXD = kResAct ? 0 : R * (kKS / Q8_QK) * 4;   // [R][32] f32
    // the resident rows: [plane][kMaxK] codes (int8 modes, one row) or
    // [R][kMaxK / 32][128] fixed-point planes (f32), then [R][kMaxK / 32]
    // block scales (int8) or block factors (f32), then (f32) [R][kMaxK / 32]
    // int16 block binades
    // the longest resident row: f32 pairs of rows up to 8192 values (both rows'
    // planes beside the ring), else kFusedMaxK
    static constexpr int kMaxK = (MODE == 0 && R == 2) ? 8192 : int(kFusedMaxK);
    static constexpr int kActBytes = MODE == 0 ? R * 4 * kMaxK : 2 * kMaxK;
    static constexpr int kAct = kResAct ? kActBytes + R * (kMaxK / Q8_QK) * (MODE == 0 ? 6 : 4) : 0;
    static constexpr int kStage = (kW + kS + kX + kXD + 1023) / 1024 * 1024;
    // The row group's partial sums are added by a combining warp through two
    // buffers where that pays (one-word 8 rows: 69.8 against 71.9 us a layer
    // of the four d = 4096 projections), else by the consumer warps between
    // two named barriers (4 rows: 56.5 against 57.6 us).
    static constexpr bool kComb = MODE == 1 && R >= 8 && !ARGMAX;
    static constexpr int kThreads = 32 * (kRplWarps + 1 + (kComb ? 1 : 0));
    // one buffer: [warp][R][lane], f32 (int8 modes) or f32 pairs (f32 mode)
    static constexpr int kPsum = kRplWarps * R * kRplRows * (MODE == 0 ? 8 : 4);
    static constexpr int kBufs = kComb ? 2 : 1;
    static constexpr size_t kSmem =
        size_t(kSlots) * kStage + kBufs * kPsum + (2 * kSlots + 4) * 8 + kAct + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory");
    static_assert(!FUSE || (R == 1 && !kComb), "fused producer: one row");
    static_assert(MODE != 0 || R <= 2, "f32 mode: one or two rows");
    static_assert(MODE != 0 || R == 1 || !FUSE, "f32 pairs: plain projections");
};

inline bool rpl_al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A plain projection in whole stages, with the 16-byte alignment the tensor
// maps need; anything else takes the decode kernel.
inline bool rpl_fits(const GemvArgs& a) {
    const auto al16 = rpl_al16;
    // f32 mode: one row up to kFusedMaxK values or a pair up to 8192, resident
    // in shared memory (f64 output allowed); int8: one row up to kFusedMaxK
    // values, resident
    const bool f32ok = a.mode != 0 ? (a.rows > 1 || a.K <= kFusedMaxK)
                                   : (a.rows == 1 && a.K <= kFusedMaxK) || (a.rows == 2 && a.K <= 8192);
    // y may be NULL for the arg-max (the LM head without logits)
    return f32ok && a.rows >= 1 && a.K >= 1024 && a.K % 1024 == 0 && a.N <= (int64_t(1) << 31) &&
           (a.y || a.tok) && (!a.out_f64 || a.mode == 0) && !a.h && !a.k_cache && al16(a.q) && al16(a.s) &&
           al16(a.act) && (a.mode == 0 || al16(a.xd)) && a.plane % 16 == 0 && (!a.tok || al16(a.ws));
}

// A fused decode step (one row, the producer in the kernel; with or without
// the KV-row epilogue) in whole stages, with its row in shared memory.
inline bool rpl_fits_fused(const GemvArgs& a) {
    return a.rows == 1 && a.h && a.K >= 1024 && a.K % 1024 == 0 && a.K <= kFusedMaxK &&
           a.N <= (int64_t(1) << 31) && a.y && (!a.out_f64 || a.mode == 0) && !a.tok && rpl_al16(a.q) &&
           rpl_al16(a.s) && rpl_al16(a.h);
}

__device__ __forceinline__ void rpl_tma2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void rpl_sts64(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ void rpl_tma3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void rpl_tma3d_ef(void* dst, const CUtensorMap* map, int x, int y, int z,
                                             uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void rpl_tma2d_ef(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                             uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

template <int MODE, int R, bool FUSE = false, int PROD = kProdPlain, bool KV = false, bool ARGMAX = false>
__global__ void __launch_bounds__(RplCfg<MODE, R, FUSE, ARGMAX>::kThreads, 1)
    gemv_rpl_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
                    const __grid_constant__ CUtensorMap tm_xh,
                    const __grid_constant__ CUtensorMap tm_xl, const __grid_constant__ CUtensorMap tm_xd,
                    const GemvParams p) {
    static_assert(MODE >= 0 && MODE <= 2, "activation mode");
    static_assert(PROD == kProdPlain || FUSE, "producer kinds belong to the fused producer");
    static_assert(!KV || (FUSE && PROD == kProdPlain), "the KV-row epilogue: fused plain decode step");
    static_assert(!FUSE || kRplWarps * 32 == kProdThreads, "fused producer needs kProdThreads consumers");
    static_assert(!ARGMAX || !FUSE, "the arg-max epilogue: plain projections");
    using C = RplCfg<MODE, R, FUSE, ARGMAX>;
    constexpr bool RES = PROD == kProdResidual;
    constexpr bool NORM = PROD != kProdSwiglu;
    __shared__ float2 s_pair[kProdWarps];
    __shared__ float s_rf;
    __shared__ int s_pos[1];   // KV-row epilogue: the row's cache position
    __shared__ int s_emax[R][kRplWarps + 1];   // f32 mode: the warps' largest block binades, then the row's
    __shared__ ArgmaxCand s_cand[R > 0 ? R : 1];   // arg-max: the CTA's best per activation row
    __shared__ ArgmaxCand s_red[kRplWarps];         // and the last CTA's reduction scratch
    __shared__ unsigned int s_ticket;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled weight tiles
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* psum = reinterpret_cast<float*>(smem + size_t(C::kSlots) * C::kStage);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(C::kSlots) * C::kStage + C::kBufs * C::kPsum);
    uint64_t* empty = full + C::kSlots;
    uint64_t* pfull = empty + C::kSlots;   // [2] a row group's partial sums written (kComb)
    uint64_t* pempty = pfull + 2;          // [2] and added up (kComb)
    unsigned char* sact = reinterpret_cast<unsigned char*>(pempty + 2);   // the resident row
    float* sxd = reinterpret_cast<float*>(sact + C::kActBytes);
    short* const seb = reinterpret_cast<short*>(sxd + R * (C::kMaxK / Q8_QK));   // f32: block binades
    // f32 rows longer than 4096 values (one row): the prologue forms x and the
    // block binades only, and the warp group that consumes a stage in the first
    // row group builds that stage's planes in place just before (`down`:
    // 18.4 -> 17.7 us; shorter rows convert faster in the prologue)
    const bool lazy = MODE == 0 && R == 1 && p.K > 4096;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int64_t N = p.N, K = p.K;
    // whole 32-row groups a CTA: a tile never holds another CTA's rows
    const int64_t ng_all = (N + kRplRows - 1) / kRplRows;
    const int64_t g0 = ng_all * c / G, g1 = ng_all * (c + 1) / G;
    const int64_t r0 = g0 * kRplRows, r1 = min64(N, g1 * kRplRows);
    const int ngroups = int(g1 - g0);
    const int nsl = int(K / C::kKS);
    const int64_t nst = int64_t(ngroups) * nsl;
    const int rows = p.rows;

    if (tid == 0) {
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 4);   // the slot's four warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&pfull[i], kRplWarps);   // lane 0 of each consumer warp
            mbar_init(&pempty[i], 1);          // lane 0 of the combining warp
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kRplWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            constexpr uint32_t kTx = uint32_t(C::kW + C::kS + C::kX + C::kXD);   // whole tiles, rows past the end zero
            // (a resident row: no activation copies; the weights never wait on
            // the previous kernel)
            auto acts = [&](int64_t t) {
                const int j = int(t % nsl), slot = int(t % C::kSlots);
                unsigned char* st = smem + size_t(slot) * C::kStage;
                // [4 chunks][R rows][256 bytes] a plane, one box each
                rpl_tma3d(st + C::kW + C::kS, &tm_xh, 0, 0, j * (C::kKS / 256), &full[slot]);
                if constexpr (MODE == 2)
                    rpl_tma3d(st + C::kW + C::kS + (C::kKS / 256) * R * 256, &tm_xl, 0, 0, j * (C::kKS / 256),
                              &full[slot]);
                rpl_tma2d(st + C::kW + C::kS + C::kX, &tm_xd, j * (C::kKS / Q8_QK), 0, &full[slot]);
            };
            const int64_t npre = nst < C::kSlots ? nst : C::kSlots;
            const uint64_t pol = policy_evict_first();
            int64_t issued = 0;
            for (int64_t t = 0; t < nst; ++t) {
                const int g = int(t / nsl), j = int(t % nsl), slot = int(t % C::kSlots);
                if (t >= C::kSlots &&
                    !mbar_wait(&empty[slot], uint32_t((t / C::kSlots) - 1) & 1u, p.err))
                    break;
                const int rg0 = int(r0 + int64_t(g) * kRplRows);
                mbar_arrive_expect_tx(&full[slot], kTx);
                unsigned char* st = smem + size_t(slot) * C::kStage;
                // [8 chunks][32 rows][128 bytes] in one box
                rpl_tma3d_ef(st, &tm_w, 0, rg0, j * (C::kKS / 128), &full[slot], pol);
                rpl_tma2d_ef(st + C::kW, &tm_s, j * (C::kKS / 16), rg0, &full[slot], pol);
                if constexpr (!C::kResAct) {
                    if (t == npre - 1) {
                        // the first stages' weights are on their way: the
                        // activations belong to the previous kernel until here
                        pdl_wait();
                        for (int64_t u = 0; u <= t; ++u) acts(u);
                    } else if (t >= npre) {
                        acts(t);
                    }
                }
                ++issued;
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int64_t t = issued > C::kSlots ? issued - C::kSlots : 0; t < issued; ++t)
                mbar_wait(&full[t % C::kSlots], uint32_t((t / C::kSlots) & 1), p.err);
        }
        return;
    }

    if (C::kComb && warp == kRplWarps + 1) {
        // ------------------------------------------------- combining warp
        // lane l adds row l's partial sums of the 16 warps in warp order
        pdl_wait();   // y belongs to the previous kernel until here
        bool okc = true;
        for (int g = 0; g < ngroups; ++g) {
            const int b = g & 1;
            const int64_t rg0 = r0 + int64_t(g) * kRplRows;
            const int nr = int(min64(kRplRows, r1 - rg0));
            if (okc) okc = mbar_wait(&pfull[b], uint32_t((g >> 1) & 1), p.err);
            if (okc && lane < nr) {
                // all R sums at once: every load is issued before the adds
                const float* ps = psum + b * (C::kPsum / 4);
                float sum[R];
#pragma unroll
                for (int m = 0; m < R; ++m) sum[m] = ps[m * kRplRows + lane];
#pragma unroll
                for (int w = 1; w < kRplWarps; ++w)
#pragma unroll
                    for (int m = 0; m < R; ++m) sum[m] += ps[(w * R + m) * kRplRows + lane];
#pragma unroll
                for (int m = 0; m < R; ++m)
                    if (m < rows) reinterpret_cast<float*>(p.y)[m * N + rg0 + lane] = sum[m];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[b]);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    if constexpr (!C::kComb) pdl_wait();   // h, y belong to the previous kernel until here
    if constexpr (KV) {
        if (tid == 0) {
            // the position belongs to the previous kernel until
            // griddepcontrol.wait; one outside the cache writes nothing and
            // is reported
            int ps = p.pos[0];
            if (ps < 0 || ps >= p.n_pos) {
                atomicExch(p.err, Q8_DEVERR_POSITION);
                ps = -1;
            }
            s_pos[0] = ps;
        }
    }
    if constexpr (MODE == 0) {
        // f32: x (read, or with the producer fused formed as the producer
        // forms it: x = (s*rf)*g, s = h or h + r, or the SwiGLU of a gate+up
        // row) converted into fixed-point planes, four lanes a block (8 values
        // each, 4 float4 groups of a block per lane pair); CTA 0 writes the
        // updated residual stream, when asked.  With the norm, the RMS pass
        // keeps s in the plane area (K floats: the planes' size), and each
        // block's planes are built in place.
        const float* const res = RES ? p.res : nullptr;
        float* const s_out = RES && blockIdx.x == 0 ? p.s_out : nullptr;
        constexpr bool STASH = FUSE && NORM;
        float* const stash = reinterpret_cast<float*>(sact);
        float rf = 1.0f;
        if constexpr (STASH) rf = row_rms_scale(p.h, res, s_out, K, p.eps, tid, 1, s_pair, &s_rf, stash);
        for (int m = 0; m < R; ++m) {
        // row m: planes at m * 4 * kMaxK, block factors at m * kMaxK / 32
        unsigned char* const plm = sact + size_t(m) * 4 * C::kMaxK;
        float* const sxm = sxd + m * (C::kMaxK / Q8_QK);
        const float* actf = static_cast<const float*>(p.act) + m * K;
        int* const se = reinterpret_cast<int*>(sxm);   // block binades until E is known
        int emax = -126;                                // the binade of zero
        // every lane of a warp runs the same iterations (K / 8 is a multiple
        // of 128), so the shuffles over a block's four lanes stay full
        for (int64_t t8 = tid; t8 < K / 8; t8 += kRplWarps * 32) {
            const int64_t k = t8 * 8;
            const int b = int(t8 >> 2), q = int(t8 & 3);   // block, eighth-of-32 within it
            float xs[8];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float xv[4];
                if constexpr (STASH) {
                    const float4 s4 = *reinterpret_cast<const float4*>(stash + k + 4 * u);
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
                        xv[e] = v;
                    }
                } else {
                    load_x4<FUSE, PROD>(actf + k + 4 * u, p.h + k + 4 * u, RES ? res + k + 4 * u : nullptr,
                                        p.gain ? p.gain + k + 4 * u : nullptr, rf, xv, K);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) xs[4 * u + e] = xv[e];
            }
            // the block's binade from its 32 values over the four lanes
            float amax = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(xs[e]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int eb = binade(amax);
            if (lazy) {
                // x in place of s (or written there), and the block's binade
                float* const xw = reinterpret_cast<float*>(plm) + k;
                *reinterpret_cast<float4*>(xw) = make_float4(xs[0], xs[1], xs[2], xs[3]);
                *reinterpret_cast<float4*>(xw + 4) = make_float4(xs[4], xs[5], xs[6], xs[7]);
                if (q == 0) seb[b] = short(eb);
            } else {
            // X = rint(x * 2^(30 - eb)) as in fix_chunk32, two words a plane
            const int sh = 30 - eb;
            const float s1 = pow2i(sh >> 1), s2 = pow2i(sh - (sh >> 1));
            int X[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) X[e] = rint_scaled30(__fmul_rn(xs[e], s1), s2);
            int pl[2][4];
            byte_planes4(X[0], X[1], X[2], X[3], pl[0][0], pl[0][1], pl[0][2], pl[0][3]);
            byte_planes4(X[4], X[5], X[6], X[7], pl[1][0], pl[1][1], pl[1][2], pl[1][3]);
            if constexpr (STASH) __syncwarp();   // the block's s read by its four lanes before the planes overwrite it
            // plane j words 2q, 2q+1: 16-byte group 2j + q / 2 (slot
            // (2j + q / 2) ^ (b & 7) of the block's 128 bytes), bytes 8 * (q % 2)
            const uint32_t base = smem_u32(plm) + uint32_t(b) * 128u + uint32_t(8 * (q & 1));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                rpl_sts64(base + uint32_t((((2 * j + (q >> 1)) ^ (b & 7)) << 4)), uint32_t(pl[0][j]),
                          uint32_t(pl[1][j]));
            }
            if (q == 0) se[b] = eb;
            emax = max(emax, eb);
        }
        emax = __reduce_max_sync(0xffffffffu, emax);
        if (lane == 0) s_emax[m][warp] = emax;
        consumer_bar<kRplWarps * 32>();
        int E = s_emax[m][0];
        for (int w = 1; w < kRplWarps; ++w) E = max(E, s_emax[m][w]);
        // each block's factor 2^(E_b - E): exact, or 0 far below the row's largest
        for (int b = tid; b < int(K / Q8_QK); b += kRplWarps * 32) sxm[b] = mul_pow2_neg(1.0f, se[b] - E);
        consumer_bar<kRplWarps * 32>();   // everyone has read s_emax
        if (tid == 0) s_emax[m][kRplWarps] = E;
        }
    }
    // the producer, fused (int8 modes): the RMS scale here, by act_quant's
    // reduction (CTA 0 writes the updated residual stream, when asked); the
    // quantisation, by act_quant's per-group code, a stage's 1024 values at a
    // time by the warp group that consumes that stage in the first row group,
    // just before it does (a row-group barrier later makes every stage's codes
    // visible to all groups)
    if constexpr (MODE != 0 && !FUSE && C::kResAct) {
        // one int8 row, plain: its codes (and lo plane) and block scales into
        // shared memory, where the fused launch keeps its produced row
        const unsigned char* src = static_cast<const unsigned char*>(p.act);
        for (int64_t i = tid; i < K / 16; i += kRplWarps * 32) {
            *reinterpret_cast<int4*>(sact + 16 * i) = ldg_nc_v4(src + 16 * i);
            if constexpr (MODE == 2) *reinterpret_cast<int4*>(sact + K + 16 * i) = ldg_nc_v4(src + p.plane + 16 * i);
        }
        for (int64_t i = tid; i < K / Q8_QK / 4; i += kRplWarps * 32)
            *reinterpret_cast<int4*>(sxd + 4 * i) = ldg_nc_v4(p.xd + 4 * i);
        consumer_bar<kRplWarps * 32>();
    }
    const float* const res_in = RES ? p.res : nullptr;
    float rf_in = 1.0f;
    if constexpr (FUSE && MODE != 0 && NORM) {
        float* const s_out = RES && blockIdx.x == 0 ? p.s_out : nullptr;
        rf_in = row_rms_scale(p.h, res_in, s_out, K, p.eps, tid, 1, s_pair, &s_rf);
    }
    const uint32_t sact_a = smem_u32(sact), sxd_a = smem_u32(sxd);
    const int wg = warp >> 2, qw = warp & 3;   // this warp's group and quarter of a stage
    bool ok = true;
    // arg-max: combine thread (m, l)'s best (value, lowest index) over the launch
    double bv = -INFINITY;
    long long bi = 0x7fffffffffffffffll;
    for (int g = 0; g < ngroups; ++g) {
        const int64_t rg0 = r0 + int64_t(g) * kRplRows;
        const int nr = int(min64(kRplRows, r1 - rg0));
        float acc[R];
#pragma unroll
        for (int m = 0; m < R; ++m) acc[m] = 0.0f;
        // f32 mode: each row's sum in units of 2^(E - 30), an f32 pair, as two
        // chains (even and odd blocks, added at the row group's end)
        DF accd[R][2];
#pragma unroll
        for (int m = 0; m < R; ++m) accd[m][0] = accd[m][1] = DF{0.0f, 0.0f};
        for (int j = 0; j < nsl; ++j) {
            const int64_t t = int64_t(g) * nsl + j;
            if (int(t % kRplGroups) != wg) continue;
            // (with one slot a group, the slot is the group: a constant)
            const int slot = C::kSlots == kRplGroups ? wg : int(t % C::kSlots);
            if constexpr (MODE == 0) {
                if (lazy && g == 0) {
                    // this stage's 32 blocks: X = rint(x * 2^(30 - E_b)) as in
                    // fix_chunk32, four lanes a block, in place of x (the
                    // block's lanes share a warp), then the group's barrier
                    const int tg = qw * 32 + lane;
                    if (tg < C::kKS / 8) {
                    const int b = j * (C::kKS / Q8_QK) + (tg >> 2), q = tg & 3;
                    const float* const xr = reinterpret_cast<const float*>(sact) + int64_t(b) * Q8_QK + 8 * q;
                    const float4 x0 = *reinterpret_cast<const float4*>(xr);
                    const float4 x1 = *reinterpret_cast<const float4*>(xr + 4);
                    const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    const int sh = 30 - int(seb[b]);
                    const float s1 = pow2i(sh >> 1), s2 = pow2i(sh - (sh >> 1));
                    int X[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) X[e] = rint_scaled30(__fmul_rn(xs[e], s1), s2);
                    int pl[2][4];
                    byte_planes4(X[0], X[1], X[2], X[3], pl[0][0], pl[0][1], pl[0][2], pl[0][3]);
                    byte_planes4(X[4], X[5], X[6], X[7], pl[1][0], pl[1][1], pl[1][2], pl[1][3]);
                    __syncwarp();   // the block's x read by its four lanes before the planes overwrite it
                    const uint32_t base = smem_u32(sact) + uint32_t(b) * 128u + uint32_t(8 * (q & 1));
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        rpl_sts64(base + uint32_t((((2 * i + (q >> 1)) ^ (b & 7)) << 4)), uint32_t(pl[0][i]),
                                  uint32_t(pl[1][i]));
                    }
                    asm volatile("bar.sync %0, 128;" ::"r"(2 + wg) : "memory");   // the group's four warps
                }
            }
            if constexpr (FUSE && MODE != 0) {
                if (g == 0) {
                    // this stage's 1024 values: 256 float4 groups, two a thread
                    // of the warp group (8 lanes a block, as in act_quant)
                    const int tg = qw * 32 + lane;
#pragma unroll
                    for (int i = 0; i < C::kKS / 512; ++i) {
                        const int64_t gi = int64_t(j) * (C::kKS / 4) + tg + 128 * i;
                        const float4 v = PROD == kProdSwiglu ? load_swiglu4(p.h, K, gi)
                                                             : load_input4(p.h, res_in, nullptr, gi);
                        float x[4] = {v.x, v.y, v.z, v.w};
                        float gg[4] = {1.0f, 1.0f, 1.0f, 1.0f};
                        if (NORM && p.gain) {
                            const int4 g4 = ldg_nc_v4(p.gain + 4 * gi);
                            gg[0] = __int_as_float(g4.x);
                            gg[1] = __int_as_float(g4.y);
                            gg[2] = __int_as_float(g4.z);
                            gg[3] = __int_as_float(g4.w);
                        }
                        produce_group<MODE, NORM>(x, gg, p.gain != nullptr, rf_in, gi, true, sact, K, sxd);
                    }
                    // the group's four warps (named barrier 2 + slot)
                    asm volatile("bar.sync %0, 128;" ::"r"(2 + wg) : "memory");
                }
            }
            if (ok) ok = mbar_wait(&full[slot], uint32_t((t / C::kSlots) & 1), p.err);
            ok = __all_sync(0xffffffffu, ok);
            if (ok && lane < nr) {
                const uint32_t st = smem_u32(smem + size_t(slot) * C::kStage);
                // the stage's activation codes and block scales: in the stage,
                // or (fused) at K offset j * kKS of the produced row
                const uint32_t xa = C::kResAct ? sact_a + uint32_t(j * C::kKS) : st + uint32_t(C::kW + C::kS);
                const uint32_t da = C::kResAct ? sxd_a + uint32_t((j * (C::kKS / Q8_QK) + qw * C::kBPW) * 4)
                                               : st + uint32_t(C::kW + C::kS + C::kX + qw * C::kBPW * 4);
                const uint32_t lo = C::kResAct ? uint32_t(K) : uint32_t((C::kKS / 256) * R * 256);   // the lo plane
                // the lane's row's block scales of this quarter: 16 bytes of a
                // 64-byte row, 64-byte swizzle (1024-value stages), or 8 bytes of
                // a 32-byte row, unswizzled (512-value stages)
                uint32_t sh[C::kBPW / 2];
                if constexpr (C::kKS == 1024) {
                    const int4 s8 = lds128(st + uint32_t(C::kW + lane * 64 + ((qw ^ ((lane >> 1) & 3)) << 4)));
                    sh[0] = uint32_t(s8.x);
                    sh[1] = uint32_t(s8.y);
                    sh[2] = uint32_t(s8.z);
                    sh[3] = uint32_t(s8.w);
                } else {
                    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                                 : "=r"(sh[0]), "=r"(sh[1])
                                 : "r"(st + uint32_t(C::kW + lane * (C::kKS / 16) + qw * 8)));
                }
                if constexpr (MODE == 0) {
                    // (two blocks in flight at one row; at two rows that spills)
#pragma unroll(R == 1 ? 2 : 1)
                    for (int b = 0; b < C::kBPW; ++b) {
                        const int B = qw * C::kBPW + b;
                        const uint32_t wr = st + uint32_t((B >> 2) * (kRplRows * 128) + lane * 128);
                        const int c0 = (B & 3) * 2;
                        const int4 w0 = lds128(wr + uint32_t(((c0 ^ (lane & 7)) << 4)));
                        const int4 w1 = lds128(wr + uint32_t((((c0 + 1) ^ (lane & 7)) << 4)));
                        const float sw =
                            half_bits_to_float(uint16_t((b & 1) ? (sh[b >> 1] >> 16) : (sh[b >> 1] & 0xFFFFu)));
                        // each row's planes of the block (the same address for
                        // every lane) and its factor to that row's binade
                        const int blk = j * (C::kKS / Q8_QK) + B;
#pragma unroll
                        for (int m = 0; m < R; ++m) {
                            FixChunk32 fx;
                            const uint32_t pb = sact_a + uint32_t(m * 4 * C::kMaxK) + uint32_t(blk) * 128u;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int4 v = lds128(pb + uint32_t(((i ^ (blk & 7)) << 4)));
                                fx.p[i >> 1][4 * (i & 1) + 0] = v.x;
                                fx.p[i >> 1][4 * (i & 1) + 1] = v.y;
                                fx.p[i >> 1][4 * (i & 1) + 2] = v.z;
                                fx.p[i >> 1][4 * (i & 1) + 3] = v.w;
                            }
                            const float f = __fmul_rn(
                                sw, __uint_as_float(lds32(sxd_a + uint32_t((m * (C::kMaxK / Q8_QK) + blk) * 4))));
                            // (one chain at two rows: the loop is not unrolled there)
                            constexpr int kMask = R == 1 ? 1 : 0;
                            accd[m][b & kMask] =
                                df_add(accd[m][b & kMask], scaled_pair_split(f, fix_dot32_split(w0, w1, fx)));
                        }
                    }
                } else {
#pragma unroll 2
                for (int b = 0; b < C::kBPW; ++b) {
                    const int B = qw * C::kBPW + b;   // block within the stage
                    // weight tile B / 4, row lane, 16-byte chunks (B % 4) * 2 and + 1, swizzled
                    const uint32_t wr = st + uint32_t((B >> 2) * (kRplRows * 128) + lane * 128);
                    const int c0 = (B & 3) * 2;
                    const int4 w0 = lds128(wr + uint32_t(((c0 ^ (lane & 7)) << 4)));
                    const int4 w1 = lds128(wr + uint32_t((((c0 + 1) ^ (lane & 7)) << 4)));
                    const float sw = half_bits_to_float(uint16_t((b & 1) ? (sh[b >> 1] >> 16) : (sh[b >> 1] & 0xFFFFu)));
                    // activation tile B / 8 (rows of 256 bytes), block B % 8; resident row: block B
                    const uint32_t xb =
                        C::kResAct ? xa + uint32_t(B * 32) : xa + uint32_t((B >> 3) * R * 256 + (B & 7) * 32);
#pragma unroll
                    for (int m = 0; m < R; ++m) {
                        const uint32_t xm = xb + uint32_t(m * 256);
                        const float xd = __uint_as_float(lds32(da + uint32_t(m * (C::kKS / Q8_QK) * 4 + 4 * b)));
                        float fi;
                        if constexpr (MODE == 1) {
                            // one dp4a chain started at the bits of 1.5 * 2^23:
                            // read as a float it is 1.5 * 2^23 + isum exactly
                            // (|isum| < 2^19), so one subtraction gives
                            // float(isum)
                            const int4 a0 = lds128(xm), a1 = lds128(xm + 16u);
                            int acc_i = 0x4B400000;
                            acc_i = __dp4a(w0.x, a0.x, acc_i);
                            acc_i = __dp4a(w0.y, a0.y, acc_i);
                            acc_i = __dp4a(w0.z, a0.z, acc_i);
                            acc_i = __dp4a(w0.w, a0.w, acc_i);
                            acc_i = __dp4a(w1.x, a1.x, acc_i);
                            acc_i = __dp4a(w1.y, a1.y, acc_i);
                            acc_i = __dp4a(w1.z, a1.z, acc_i);
                            acc_i = __dp4a(w1.w, a1.w, acc_i);
                            fi = __fsub_rn(__int_as_float(acc_i), 12582912.0f);
                        } else {
                            const uint32_t xl = xm + lo;
                            const int isum = dot16_i8x2(w0, lds128(xm), lds128(xl)) +
                                             dot16_i8x2(w1, lds128(xm + 16u), lds128(xl + 16u));
                            fi = float(isum);
                        }
                        acc[m] = fmaf(fi, sw * xd, acc[m]);
                    }
                }
                }
            }
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&empty[slot]);
        }
        if constexpr (C::kComb) {
            // the row group's sums to the combining warp, through one of two
            // buffers (free again once it has added the group before last)
            const int b = g & 1;
            if (ok && g >= 2) ok = mbar_wait(&pempty[b], uint32_t(((g >> 1) - 1) & 1), p.err);
            float* ps = psum + b * (C::kPsum / 4);
#pragma unroll
            for (int m = 0; m < R; ++m) ps[(warp * R + m) * kRplRows + lane] = acc[m];
            __syncwarp();   // the warp's writes before lane 0's release
            if (lane == 0) mbar_arrive(&pfull[b]);
        } else if constexpr (MODE == 0) {
            // the row group's f32-pair sums into shared memory; then thread
            // (m, l) adds row l's of activation row m over the 16 warps in warp
            // order and scales the pair, rounded once, by 2^(E_m - 30) (f32),
            // or the exact pair (f64)
            DF* const psd = reinterpret_cast<DF*>(psum);
#pragma unroll
            for (int m = 0; m < R; ++m) psd[(warp * R + m) * kRplRows + lane] = df_add(accd[m][0], accd[m][1]);
            consumer_bar<kRplWarps * 32>();
            if (ok && tid < kRplRows * R) {
                const int l = tid % kRplRows, m = tid / kRplRows;
                if (l < nr) {
                    DF sum = psd[m * kRplRows + l];
                    for (int w = 1; w < kRplWarps; ++w) sum = df_add(sum, psd[(w * R + m) * kRplRows + l]);
                    const int sc = s_emax[m][kRplWarps] - 30;   // in [-156, 98]
                    if (ARGMAX || p.out_f64) {
                        // exact: a power of two well inside the f64 range
                        const double val =
                            (double(sum.hi) + double(sum.lo)) * __longlong_as_double((long long)(sc + 1023) << 52);
                        if (p.y) {
                            if (p.out_f64)
                                reinterpret_cast<double*>(p.y)[m * N + rg0 + l] = val;
                            else
                                reinterpret_cast<float*>(p.y)[m * N + rg0 + l] = float(val);
                        }
                        if constexpr (ARGMAX) argmax_keep(bv, bi, val, rg0 + l);
                    } else {
                        const float yv = __fmul_rn(__fmul_rn(__fadd_rn(sum.hi, sum.lo), pow2i(sc >> 1)),
                                                   pow2i(sc - (sc >> 1)));
                        reinterpret_cast<float*>(p.y)[m * N + rg0 + l] = yv;
                        if constexpr (KV) kv_store(p, s_pos, 0, rg0 + l, yv);
                    }
                }
            }
            consumer_bar<kRplWarps * 32>();
        } else {
            // the row group's sums into shared memory; then thread (m, l) adds
            // row l's sums of activation row m over the 16 warps in warp order
#pragma unroll
            for (int m = 0; m < R; ++m) psum[(warp * R + m) * kRplRows + lane] = acc[m];
            consumer_bar<kRplWarps * 32>();
            if (ok && tid < kRplRows * R) {
                const int l = tid % kRplRows, m = tid / kRplRows;
                if (l < nr && m < rows) {
                    float sum = psum[m * kRplRows + l];
                    for (int w = 1; w < kRplWarps; ++w) sum += psum[(w * R + m) * kRplRows + l];
                    if (p.y) reinterpret_cast<float*>(p.y)[m * N + rg0 + l] = sum;
                    if constexpr (KV) kv_store(p, s_pos, m, rg0 + l, sum);
                    if constexpr (ARGMAX) argmax_keep(bv, bi, double(sum), rg0 + l);
                }
            }
            consumer_bar<kRplWarps * 32>();
        }
    }

    if constexpr (ARGMAX) {
        // warp m's lanes hold activation row m's candidates: the warp's best,
        // then per CTA into the workspace, and the last CTA to take a ticket
        // reduces every CTA's candidate (lowest index on ties)
        if (warp < R) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const long long oi = __shfl_xor_sync(0xffffffffu, bi, o);
                argmax_keep(bv, bi, ov, oi);
            }
            if (lane == 0) s_cand[warp] = {bv, bi};
        }
        consumer_bar<kRplWarps * 32>();
        ArgmaxCand* gc = reinterpret_cast<ArgmaxCand*>(p.ws + kArgmaxHeader);
        unsigned int* counter = reinterpret_cast<unsigned int*>(p.ws);
        if (tid < rows) {
            gc[size_t(c) * rows + tid] = s_cand[tid];
            __threadfence();
        }
        consumer_bar<kRplWarps * 32>();
        if (tid == 0) s_ticket = atomicAdd(counter, 1u);
        consumer_bar<kRplWarps * 32>();
        if (s_ticket == unsigned(G - 1)) {
            __threadfence();
            argmax_final<kRplWarps * 32>(gc, G, rows, tid, s_red, p.tok, p.maxval);
            if (tid == 0) *counter = 0u;
        }
    }
}

template <int MODE, int R, bool FUSE = false, int PROD = kProdPlain, bool KV = false, bool ARGMAX = false>
cudaError_t launch_gemv_rpl_t(const GemvArgs& a, const LaunchCtx& ctx) {
    using C = RplCfg<MODE, R, FUSE, ARGMAX>;
    auto kern = gemv_rpl_kernel<MODE, R, FUSE, PROD, KV, ARGMAX>;
    static std::atomic<bool> configured[kMaxDevices];
    if (const cudaError_t e = set_smem_once(kern, C::kSmem, ctx.dev, configured); e != cudaSuccess) return e;
    if (FUSE ? !rpl_fits_fused(a) : (!rpl_fits(a) || a.rows > R)) return cudaErrorInvalidValue;
    if (MODE == 0 && a.rows != R) return cudaErrorInvalidValue;   // f32: every resident row is used
    if (KV != (a.k_cache != nullptr)) return cudaErrorInvalidValue;
    if (ARGMAX != (a.tok != nullptr) || (ARGMAX && !a.ws)) return cudaErrorInvalidValue;
    alignas(64) CUtensorMap tw, ts, txh, txl, txd;
    const int8_t* xh = static_cast<const int8_t*>(a.act);
    // weights as (byte in a 128-byte chunk, row, chunk): a box of 8 chunks of
    // 32 rows lands as eight [32][128] tiles
    const uint64_t wd[3] = {128, uint64_t(a.N), uint64_t(a.K / 128)}, ws[2] = {uint64_t(a.K), 128};
    const uint32_t wb[3] = {128, kRplRows, C::kKS / 128};
    // activation codes as (byte in a 256-byte chunk, row, chunk)
    const uint64_t xdims[3] = {256, uint64_t(a.rows), uint64_t(a.K / 256)}, xs[2] = {uint64_t(a.K), 256};
    const uint32_t xb[3] = {256, uint32_t(R), C::kKS / 256};
    const bool okw =
        make_map3(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.q, wd, ws, wb, CU_TENSOR_MAP_SWIZZLE_128B) &&
        make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.s, a.K / 16, a.N, a.K / 16, C::kKS / 16, kRplRows,
                 C::kKS == 1024 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE);
    // a resident row: no activation copies (the unused maps repeat the weights')
    if (C::kResAct) txh = txl = txd = tw;
    const bool ok = okw && (C::kResAct ||
        (make_map3(&txh, CU_TENSOR_MAP_DATA_TYPE_UINT8, xh, xdims, xs, xb, CU_TENSOR_MAP_SWIZZLE_NONE) &&
        make_map3(&txl, CU_TENSOR_MAP_DATA_TYPE_UINT8, MODE == 2 ? xh + a.plane : xh, xdims, xs, xb,
                  CU_TENSOR_MAP_SWIZZLE_NONE) &&
        make_map(&txd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.xd, a.K / Q8_QK, a.rows, (a.K / Q8_QK) * 4,
                 C::kKS / Q8_QK, R, CU_TENSOR_MAP_SWIZZLE_NONE)));
    if (!ok) return cudaErrorInvalidValue;
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
    if (int64_t(grid) > (a.N + kRplRows - 1) / kRplRows) grid = int((a.N + kRplRows - 1) / kRplRows);
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[2];
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kern, tw, ts, txh, txl, txd, p);
}

}  // namespace q8

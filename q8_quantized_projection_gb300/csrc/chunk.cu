// chunk.cu -- the prefill-chunk / batched projection on the 5th-generation
// tensor cores (tcgen05, sm_103a): T activation rows at once, every weight
// byte read from HBM once per launch.
//
// Per Q8_0 block b the block dots of a 128-weight-row by TT-activation-row
// tile are one exact tensor-core product: int8 values are exact in f16, and
// 32 products of |q| <= 127 codes sum to < 2^24, so an f32 accumulator holds
// the integer isum exactly (two-word mode: one product per plane, then
// 128*hi + lo rounds once, exactly like float(isum)).  The scales do not fold
// into the product (they differ per block on both sides), so each block's
// product is read back and rescaled:  y[t][n] += isum * (s[n][b] * d[t][b]).
//
// CTA tile: 128 weight rows (MMA M) x TT activation rows (MMA N), over a
// range of K.  Warp roles, connected by mbarriers whose waits are bounded:
//   warp 0      producer: 2-D TMA tiles of weights (int8, 128-byte swizzle),
//               activation codes (one or two planes), activation scales and,
//               every 8 blocks, weight scales;
//   warp 1      owns TMEM; one thread issues the MMAs (kind::f16, K = 16, two
//               per block and activation plane) into one of NSLOT accumulator
//               slots, and commits them;
//   warps 2-5   converters (2-9: two groups of four taking alternate block
//               pairs), two blocks at a time: weights int8 -> f16 straight
//               into TMEM (the MMA's A operand, lane = weight row), activation
//               codes int8 -> f16 operand tiles in shared memory (K-major, no
//               swizzle), and both blocks' scales into the scale ring entries
//               of their accumulator slots;
//   next 8      epilogue: TMEM -> registers, rescale with packed f32x2 FMAs,
//               accumulate.
// A converted pair is freed by its MMAs' own completion (commit); an
// accumulator slot and its scale-ring entry by the epilogue.  TMEM columns
// 0..383 hold the accumulator slots, 384..511 four A pairs.
//
// Split K: when there are too few 128 x TT tiles to fill the GPU, KS CTAs (a
// thread-block cluster along z) share a tile, each over a contiguous range
// of 8-block groups; their partial sums meet in shared memory and each CTA
// adds up a slice of the tile over the cluster (distributed shared memory),
// in rank order, so results do not depend on timing.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace q8 {

constexpr int kCkM = 128;          // weight rows per tile
constexpr int kCkStageK = 128;     // bytes of K per TMA stage (4 blocks)
constexpr int kCkGroup = 8;        // blocks per weight-scale group (16 bytes of f16)
constexpr int kCkPairs = 4;        // converted block pairs in flight
constexpr int kCkAccCols = 384;    // TMEM columns for accumulator slots
constexpr int kCkEpiWarps = 8;
constexpr int kCkMaxSplit = 8;
constexpr int kCkSmemBudget = 227 * 1024;

template <int MODE, int TT>
struct CkCfg {
    static constexpr int kPlanes = (MODE == 2) ? 2 : 1;
    static constexpr int kSlotCols = TT * kPlanes;                    // TMEM columns per block
    static constexpr int kSlots = (kCkAccCols / kSlotCols) < 8 ? (kCkAccCols / kSlotCols) : 8;
    static constexpr int kTmemCols = 512;
    static constexpr int kW = kCkM * kCkStageK;                       // 16 KB
    static constexpr int kXPlane = TT * kCkStageK;
    static constexpr int kX = kXPlane * kPlanes;
    static constexpr int kXD = TT * 4 * 4;                            // [TT][4 blocks] f32
    static constexpr int kStage = (kW + kX + kXD + 1023) / 1024 * 1024;
    static constexpr int kSGroup = kCkM * kCkGroup * 2;               // [128][8 blocks] f16
    static constexpr int kSGroups = 4;
    static constexpr int kBPlane = TT * 64;                           // [TT][32] f16
    static constexpr int kBBlock = kBPlane * kPlanes;
    static constexpr int kOpPair = 2 * kBBlock;
    static constexpr int kScl = kCkM * 2 + TT * 4;                    // sw[128] f16, xd[TT] f32
    static constexpr int kCW = TT / 2;                                // columns per epilogue warp
    // Two converter groups take alternate block pairs when there are at
    // least 4 accumulator slots: a group then never waits on a slot barrier
    // more than one phase ahead of what it has seen (the parity would alias).
    static constexpr int kConvGroups = kSlots >= 4 ? 2 : 1;
    static constexpr int kEpiWarp0 = 2 + 4 * kConvGroups;
    static constexpr int kThreads = (kEpiWarp0 + kCkEpiWarps) * 32;
    static constexpr int kFixed = kSGroups * kSGroup + kCkPairs * kOpPair + kSlots * kScl +
                                  512 /*barriers*/ + 1024 /*alignment*/;
    static constexpr int kStages = (kCkSmemBudget - kFixed) / kStage < 8
                                       ? (kCkSmemBudget - kFixed) / kStage
                                       : 8;
    static constexpr size_t kSmem = size_t(kStages) * kStage + kFixed;
    static_assert(kStages >= 3, "TMA pipeline depth");
    static_assert(kStage % 1024 == 0, "swizzled TMA tiles need 1024-byte alignment");
    static_assert(kCkM * TT * 4 <= kStages * kStage, "split-K partial must fit the stages");
    static_assert(kSmem <= size_t(kCkSmemBudget), "shared memory");
    static_assert(kCW % 16 == 0, "epilogue columns");
    static_assert(kSlots >= 3, "accumulator slots");
};

struct CkParams {
    int64_t N, K, T;
    int groups_per_split;   // 8-block groups of K per CTA of a cluster
    float* y;
    int32_t* isum;          // debug: per-block dots [T][N][K/32] instead of y
    int* err;
};

__device__ __forceinline__ void tma2d(void* dst, const CUtensorMap* map, int x, int y,
                                      uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Physical byte offset of 16-byte chunk c of row r in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return uint32_t(r * 128 + ((c ^ (r & 7)) << 4));
}

// The 32 int8 values of one block row (two 16-byte chunks of a 128-byte-
// swizzled TMA tile) as f16, stored as row r of a K-major no-swizzle operand
// tile at `dst`.
__device__ __forceinline__ void store_row_f16(uint32_t dst, int r, const int4 a, const int4 b) {
    const uint32_t w[8] = {uint32_t(a.x), uint32_t(a.y), uint32_t(a.z), uint32_t(a.w),
                           uint32_t(b.x), uint32_t(b.y), uint32_t(b.z), uint32_t(b.w)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {   // 8 values (one core-matrix row) per c
        uint32_t h[4];
        i8x4_to_f16x4(w[2 * c], h[0], h[1]);
        i8x4_to_f16x4(w[2 * c + 1], h[2], h[3]);
        sts128(dst + tile_offset(r, 8 * c), h[0], h[1], h[2], h[3]);
    }
}

// ------------------------------------------------ packed f32 pairs (sm_100+)

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    return uint64_t(__float_as_uint(lo)) | (uint64_t(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float f2_lo(uint64_t a) { return __uint_as_float(uint32_t(a)); }
__device__ __forceinline__ float f2_hi(uint64_t a) { return __uint_as_float(uint32_t(a >> 32)); }

// ------------------------------------------------------ thread-block clusters

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// 16 consecutive TMEM columns of the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <int MODE, int TT, bool DEBUG>
__global__ void __launch_bounds__(CkCfg<MODE, TT>::kThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_xh,
                 const __grid_constant__ CUtensorMap tm_xl, const __grid_constant__ CUtensorMap tm_s,
                 const __grid_constant__ CUtensorMap tm_xd, const CkParams p) {
    using C = CkCfg<MODE, TT>;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled TMA tiles
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* stages = smem;
    unsigned char* sgroups = stages + size_t(C::kStages) * C::kStage;
    unsigned char* ops = sgroups + size_t(C::kSGroups) * C::kSGroup;
    unsigned char* scl = ops + size_t(kCkPairs) * C::kOpPair;
    uint64_t* bars = reinterpret_cast<uint64_t*>(scl + size_t(C::kSlots) * C::kScl);
    uint64_t* st_full = bars;
    uint64_t* st_empty = st_full + C::kStages;
    uint64_t* sg_full = st_empty + C::kStages;
    uint64_t* sg_empty = sg_full + C::kSGroups;
    uint64_t* op_full = sg_empty + C::kSGroups;
    uint64_t* op_empty = op_full + kCkPairs;
    uint64_t* tm_full = op_empty + kCkPairs;
    uint64_t* tm_empty = tm_full + C::kSlots;
    uint64_t* sc_full = tm_empty + C::kSlots;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sc_full + C::kSlots);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t t0 = int64_t(blockIdx.x) * TT;
    const int64_t m0 = int64_t(blockIdx.y) * kCkM;
    // this CTA's range of K, in 8-block groups
    const int total_groups = int(p.K / (Q8_QK * kCkGroup));
    const int g_begin = int(blockIdx.z) * p.groups_per_split;
    const int g_end = min(total_groups, g_begin + p.groups_per_split);
    const int nblk = g_end > g_begin ? (g_end - g_begin) * kCkGroup : 0;
    const int nst = nblk / 4;
    const int npairs = nblk / 2;
    const int st0 = g_begin * (kCkGroup / 4);   // first TMA stage (global)
    const int64_t trows = p.T - t0 < TT ? p.T - t0 : TT;
    const int np = int((trows + 15) / 16) * 16;   // MMA N

    if (tid == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&st_full[i], 1);
            mbar_init(&st_empty[i], 8);    // each converter warp, once per pair (2 a stage)
        }
        for (int i = 0; i < C::kSGroups; ++i) {
            mbar_init(&sg_full[i], 1);
            mbar_init(&sg_empty[i], 16);   // each converter warp, once per pair (4 a group)
        }
        for (int i = 0; i < kCkPairs; ++i) {
            mbar_init(&op_full[i], 4);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(&tm_full[i], 1);
            mbar_init(&tm_empty[i], kCkEpiWarps);
            mbar_init(&sc_full[i], 4);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    const uint32_t stages_a = smem_u32(stages), sgroups_a = smem_u32(sgroups);
    const uint32_t ops_a = smem_u32(ops), scl_a = smem_u32(scl);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            pdl_wait();
            int issued = 0, sissued = 0;
            for (int s = 0; s < nst; ++s) {
                const int slot = s % C::kStages;
                if (s >= C::kStages &&
                    !mbar_wait(&st_empty[slot], uint32_t(s / C::kStages - 1) & 1u, p.err))
                    break;
                unsigned char* st = stages + size_t(slot) * C::kStage;
                const int kx = (st0 + s) * kCkStageK;   // byte (= element) of K
                mbar_arrive_expect_tx(&st_full[slot], uint32_t(C::kW + C::kX + (DEBUG ? 0 : C::kXD)));
                tma2d(st, &tm_w, kx, int(m0), &st_full[slot]);
                tma2d(st + C::kW, &tm_xh, kx, int(t0), &st_full[slot]);
                if constexpr (MODE == 2)
                    tma2d(st + C::kW + C::kXPlane, &tm_xl, kx, int(t0), &st_full[slot]);
                if constexpr (!DEBUG)
                    tma2d(st + C::kW + C::kX, &tm_xd, kx / Q8_QK, int(t0), &st_full[slot]);
                ++issued;
                if (!DEBUG && (s & 1) == 0) {
                    const int g = s >> 1, gs = g % C::kSGroups;
                    if (g >= C::kSGroups &&
                        !mbar_wait(&sg_empty[gs], uint32_t(g / C::kSGroups - 1) & 1u, p.err))
                        break;
                    mbar_arrive_expect_tx(&sg_full[gs], uint32_t(C::kSGroup));
                    tma2d(sgroups + size_t(gs) * C::kSGroup, &tm_s, kx / Q8_QK, int(m0), &sg_full[gs]);
                    ++sissued;
                }
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int s = issued > C::kStages ? issued - C::kStages : 0; s < issued; ++s)
                mbar_wait(&st_full[s % C::kStages], uint32_t(s / C::kStages) & 1u, p.err);
            for (int g = sissued > C::kSGroups ? sissued - C::kSGroups : 0; g < sissued; ++g)
                mbar_wait(&sg_full[g % C::kSGroups], uint32_t(g / C::kSGroups) & 1u, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(kCkM, np);
            int issued = 0;
            bool ok = true;
            for (int pr = 0; pr < npairs && ok; ++pr) {
                const int ps = pr % kCkPairs;
                if (!mbar_wait(&op_full[ps], uint32_t(pr / kCkPairs) & 1u, p.err)) break;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int b = 2 * pr + h, ts = b % C::kSlots;
                    if (b >= C::kSlots &&
                        !mbar_wait(&tm_empty[ts], uint32_t(b / C::kSlots - 1) & 1u, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = tmem + uint32_t(kCkAccCols + 32 * ps + 16 * h);
                    const uint32_t bb = ops_a + uint32_t(ps * C::kOpPair + h * C::kBBlock);
                    const uint32_t d = tmem + uint32_t(ts * C::kSlotCols);
#pragma unroll
                    for (int pl = 0; pl < C::kPlanes; ++pl)
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2)
                            mma_f16_ts(d + uint32_t(pl * TT), a + uint32_t(8 * s2),
                                       smem_desc_kmajor(bb + uint32_t(pl * C::kBPlane + 256 * s2), 128, 512),
                                       idesc, s2 > 0);
                    mma_commit(smem_u32(&tm_full[ts]));
                    ++issued;
                }
                mma_commit(smem_u32(&op_empty[ps]));
            }
            // nothing may be left in flight when TMEM is released (the epilogue
            // normally drains every block; this covers an early exit)
            if (issued > 0)
                mbar_wait(&tm_full[(issued - 1) % C::kSlots], uint32_t((issued - 1) / C::kSlots) & 1u,
                          p.err);
        }
    } else if (warp < C::kEpiWarp0) {
        // ------------------------------------------------------------ converters
        // group cg converts the pairs pr = cg (mod kConvGroups)
        const int cg = (warp - 2) >> 2;
        const int rw = (warp & 3) * 32 + lane;        // weight row = TMEM lane; activation row
        const uint32_t a_lane = uint32_t((warp & 3) * 32) << 16;
        const bool act = rw < np;                     // the MMA reads activation rows < np only
        bool ok = true;
        for (int pr = cg; pr < npairs; pr += C::kConvGroups) {
            const int s = pr >> 1, half = pr & 1, slot = s % C::kStages;
            const int g = pr >> 2, gs = g % C::kSGroups, ps = pr % kCkPairs;
            const int b0 = 2 * pr, j0 = 2 * half;
            if (ok) ok = mbar_wait(&st_full[slot], uint32_t(s / C::kStages) & 1u, p.err);
            if (!DEBUG && ok) ok = mbar_wait(&sg_full[gs], uint32_t(g / C::kSGroups) & 1u, p.err);
            if (ok && pr >= kCkPairs)
                ok = mbar_wait(&op_empty[ps], uint32_t(pr / kCkPairs - 1) & 1u, p.err);
            // the scale-ring entries of both blocks are free once the epilogue
            // has released the later one's previous user (it releases in order)
            if (!DEBUG && ok && b0 + 1 >= C::kSlots)
                ok = mbar_wait(&tm_empty[(b0 + 1) % C::kSlots], uint32_t((b0 + 1) / C::kSlots - 1) & 1u,
                               p.err);
            // leave together: the warp-wide TMEM store and __syncwarp below need every lane
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t st = stages_a + uint32_t(slot * C::kStage);
            // every shared-memory read first, then convert and store
            int4 w[4], x[4], l[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) w[c] = lds128(st + sw128(rw, 2 * j0 + c));
            if (act) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    x[c] = lds128(st + C::kW + sw128(rw, 2 * j0 + c));
                    if constexpr (MODE == 2) l[c] = lds128(st + C::kW + C::kXPlane + sw128(rw, 2 * j0 + c));
                }
            }
            uint32_t sw2 = 0, xd0 = 0, xd1 = 0;
            if constexpr (!DEBUG) {
                sw2 = lds32(sgroups_a + uint32_t(gs * C::kSGroup + rw * kCkGroup * 2 + (b0 & 7) * 2));
                if (act) {
                    xd0 = lds32(st + uint32_t(C::kW + C::kX + rw * 16 + j0 * 4));
                    xd1 = lds32(st + uint32_t(C::kW + C::kX + rw * 16 + j0 * 4 + 4));
                }
            }
            // weights of both blocks -> 32 TMEM columns of A pair `ps`
            {
                uint32_t hw[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t v[4] = {uint32_t(w[c].x), uint32_t(w[c].y), uint32_t(w[c].z),
                                           uint32_t(w[c].w)};
#pragma unroll
                    for (int i = 0; i < 4; ++i) i8x4_to_f16x4(v[i], hw[8 * c + 2 * i], hw[8 * c + 2 * i + 1]);
                }
                tmem_st32(tmem + a_lane + uint32_t(kCkAccCols + 32 * ps), hw);
            }
            if (act) {
                const uint32_t bb = ops_a + uint32_t(ps * C::kOpPair);
                store_row_f16(bb, rw, x[0], x[1]);
                store_row_f16(bb + C::kBBlock, rw, x[2], x[3]);
                if constexpr (MODE == 2) {
                    store_row_f16(bb + C::kBPlane, rw, l[0], l[1]);
                    store_row_f16(bb + C::kBBlock + C::kBPlane, rw, l[2], l[3]);
                }
            }
            if constexpr (!DEBUG) {
                const uint32_t e0 = scl_a + uint32_t((b0 % C::kSlots) * C::kScl);
                const uint32_t e1 = scl_a + uint32_t(((b0 + 1) % C::kSlots) * C::kScl);
                sts16(e0 + uint32_t(2 * rw), uint16_t(sw2 & 0xFFFFu));
                sts16(e1 + uint32_t(2 * rw), uint16_t(sw2 >> 16));
                if (act) {
                    sts32(e0 + uint32_t(kCkM * 2 + 4 * rw), xd0);
                    sts32(e1 + uint32_t(kCkM * 2 + 4 * rw), xd1);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&op_full[ps]);
                if constexpr (!DEBUG) {
                    mbar_arrive(&sc_full[b0 % C::kSlots]);
                    mbar_arrive(&sc_full[(b0 + 1) % C::kSlots]);
                }
                mbar_arrive(&st_empty[slot]);
                if constexpr (!DEBUG) mbar_arrive(&sg_empty[gs]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // accumulators: pairs of activation rows for one weight row
        uint64_t acc[C::kCW / 2];
#pragma unroll
        for (int i = 0; i < C::kCW / 2; ++i) acc[i] = 0;
        const int ew = warp - C::kEpiWarp0;   // 0..7
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int h = ew >> 2;            // column half
        const int n = q * 32 + lane;      // weight row within the tile
        const int c0 = C::kCW * h;
        bool ok = true;
        for (int b = 0; b < nblk; ++b) {
            const int ts = b % C::kSlots;
            const uint32_t par = uint32_t(b / C::kSlots) & 1u;
            if (!DEBUG && ok) ok = mbar_wait(&sc_full[ts], par, p.err);
            if (ok) ok = mbar_wait(&tm_full[ts], par, p.err);
            ok = __all_sync(0xffffffffu, ok);   // the TMEM loads below are warp-wide
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t(q * 32) << 16) + uint32_t(ts * C::kSlotCols + c0);
            if constexpr (DEBUG) {
                // the plane sums are exact integers below 2^24
                const int64_t row = m0 + n;
#pragma unroll
                for (int cc = 0; cc < C::kCW / 16; ++cc) {
                    if (c0 + 16 * cc >= np) break;
                    float v[16], vl[16];
                    tmem_ld16(d + uint32_t(16 * cc), v);
                    if constexpr (MODE == 2) tmem_ld16(d + TT + uint32_t(16 * cc), vl);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int64_t t = t0 + c0 + 16 * cc + i;
                        if (t < p.T && row < p.N) {
                            int iv = __float2int_rn(v[i]);
                            if constexpr (MODE == 2) iv = 128 * iv + __float2int_rn(vl[i]);
                            p.isum[(t * p.N + row) * (p.K / Q8_QK) + g_begin * kCkGroup + b] = iv;
                        }
                    }
                }
            } else {
                const uint32_t e = scl_a + uint32_t(ts * C::kScl);
                const float sw = half_bits_to_float(lds16(e + uint32_t(2 * n)));
                const uint64_t sw2 = f2_pack(sw, sw);
                const uint32_t xdv = e + uint32_t(kCkM * 2 + c0 * 4);
                // waves of up to 32 columns: all TMEM loads of a wave, one wait
                // registers: two planes or 64 accumulated columns take half-width waves
                constexpr int kWaveMax = (MODE == 2 || C::kCW > 32) ? 16 : 32;
                constexpr int kWave = C::kCW < kWaveMax ? C::kCW : kWaveMax;
#pragma unroll
                for (int w = 0; w < C::kCW / kWave; ++w) {
                    if (c0 + kWave * w >= np) break;   // warp-uniform
                    float v[kWave];
                    float vl[MODE == 2 ? kWave : 1];
#pragma unroll
                    for (int c = 0; c < kWave / 16; ++c) {
                        tmem_ld16(d + uint32_t(kWave * w + 16 * c), *reinterpret_cast<float(*)[16]>(v + 16 * c));
                        if constexpr (MODE == 2)
                            tmem_ld16(d + TT + uint32_t(kWave * w + 16 * c),
                                      *reinterpret_cast<float(*)[16]>(vl + 16 * c));
                    }
                    tmem_wait_ld();
                    if constexpr (MODE == 2) {
                        // 128*hi + lo rounds once: exactly float(isum)
                        const uint64_t k128 = f2_pack(128.0f, 128.0f);
#pragma unroll
                        for (int i = 0; i < kWave / 2; ++i) {
                            const uint64_t r = f2_fma(k128, f2_pack(v[2 * i], v[2 * i + 1]),
                                                      f2_pack(vl[2 * i], vl[2 * i + 1]));
                            v[2 * i] = f2_lo(r);
                            v[2 * i + 1] = f2_hi(r);
                        }
                    }
#pragma unroll
                    for (int i4 = 0; i4 < kWave / 4; ++i4) {
                        const int4 x4 = lds128(xdv + uint32_t(4 * kWave * w + 16 * i4));
                        const uint64_t c01 = f2_mul(sw2, uint64_t(uint32_t(x4.x)) | (uint64_t(uint32_t(x4.y)) << 32));
                        const uint64_t c23 = f2_mul(sw2, uint64_t(uint32_t(x4.z)) | (uint64_t(uint32_t(x4.w)) << 32));
                        const int a = (kWave * w) / 2 + 2 * i4;
                        acc[a] = f2_fma(f2_pack(v[4 * i4], v[4 * i4 + 1]), c01, acc[a]);
                        acc[a + 1] = f2_fma(f2_pack(v[4 * i4 + 2], v[4 * i4 + 3]), c23, acc[a + 1]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tm_empty[ts]);
        }
        if constexpr (!DEBUG) {
            if (gridDim.z == 1) {
                const int64_t row = m0 + n;
                if (row < p.N) {
#pragma unroll
                    for (int i = 0; i < C::kCW; ++i) {
                        const int64_t t = t0 + c0 + i;
                        const float v = (i & 1) ? f2_hi(acc[i >> 1]) : f2_lo(acc[i >> 1]);
                        if (t < p.T) p.y[t * p.N + row] = v;
                    }
                }
            } else {
                // partial tile [TT][128] f32 in the stage buffers: every stage has
                // been consumed once this warp has rescaled the last block
#pragma unroll
                for (int i = 0; i < C::kCW; ++i)
                    sts32(stages_a + uint32_t(((c0 + i) * kCkM + n) * 4),
                          (i & 1) ? uint32_t(acc[i >> 1] >> 32) : uint32_t(acc[i >> 1]));
            }
        }
    }


    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if (!DEBUG && gridDim.z > 1) {
        cluster_sync();
        const uint32_t ks = gridDim.z, rank = blockIdx.z;
        const int n4 = TT * kCkM / 4;
        const int per = (n4 + int(ks) - 1) / int(ks);
        const int i_end = min(n4, int(rank + 1) * per);
        const uint32_t base = stages_a;
        for (int i = int(rank) * per + tid; i < i_end; i += C::kThreads) {
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (uint32_t r = 0; r < ks; ++r) {
                const float4 v = ld_cluster_v4(cluster_map(base + uint32_t(i) * 16u, r));
                s.x += v.x;
                s.y += v.y;
                s.z += v.z;
                s.w += v.w;
            }
            const int e = 4 * i, t = e / kCkM, nn = e % kCkM;
            if (t0 + t < p.T) {
                float* yr = p.y + (t0 + t) * p.N + m0 + nn;
                const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (m0 + nn + u < p.N) yr[u] = sv[u];
            }
        }
        // no CTA may leave while another still reads its shared memory
        cluster_sync();
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                     uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                     CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of `ks` CTAs of this kernel that fit on the device at once.
template <int MODE, int TT, bool DEBUG>
static int active_clusters(int ks, const LaunchCtx& ctx) {
    using C = CkCfg<MODE, TT>;
    // per device and split; threads that race here store the same value
    static std::atomic<int> cache[kMaxDevices][kCkMaxSplit + 1];
    std::atomic<int>& slot = cache[ctx.dev][ks];
    if (const int v = slot.load(std::memory_order_relaxed); v > 0) return v;
    int n = ctx.num_sms / ks;
    if (ks > 1) {
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = unsigned(ks);
        cfg.gridDim = dim3(1, 1, unsigned(ks));
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, chunk_kernel<MODE, TT, DEBUG>, &cfg) == cudaSuccess &&
            c > 0)
            n = c;
        else
            cudaGetLastError();
    }
    n = n > 0 ? n : 1;
    slot.store(n, std::memory_order_relaxed);
    return n;
}

// Split of K over a cluster: the count with the fewest 8-block groups on
// the busiest SM, counting whole waves of clusters.
template <int MODE, int TT, bool DEBUG>
static int choose_split(int64_t tiles, int groups, const LaunchCtx& ctx) {
    int best = 1;
    int64_t best_cost = -1;
    for (int ks = 1; ks <= kCkMaxSplit && ks <= groups; ++ks) {
        const int64_t waves = (tiles + active_clusters<MODE, TT, DEBUG>(ks, ctx) - 1) /
                              active_clusters<MODE, TT, DEBUG>(ks, ctx);
        const int64_t cost = waves * ((groups + ks - 1) / ks);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = ks;
        }
    }
    return best;
}

template <int MODE, int TT, bool DEBUG>
static cudaError_t launch_chunk_t(const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                                  const void* xq, const float* xd, int64_t T, float* y,
                                  int32_t* isum, const LaunchCtx& ctx) {
    using C = CkCfg<MODE, TT>;
    auto kern = chunk_kernel<MODE, TT, DEBUG>;
    static std::atomic<bool> configured[kMaxDevices];
    if (const cudaError_t e = set_smem_once(kern, size_t(C::kSmem), ctx.dev, configured); e != cudaSuccess)
        return e;
    alignas(64) CUtensorMap tw, txh, txl, ts, txd;
    const int64_t nb = K / Q8_QK;
    const int8_t* xh = reinterpret_cast<const int8_t*>(xq);
    bool ok = make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, K, N, K, kCkStageK, kCkM,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&txh, CU_TENSOR_MAP_DATA_TYPE_UINT8, xh, K, T, K, kCkStageK, TT,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&txl, CU_TENSOR_MAP_DATA_TYPE_UINT8, MODE == 2 ? xh + T * K : xh, K, T, K,
                       kCkStageK, TT, CU_TENSOR_MAP_SWIZZLE_128B) &&
              // (the debug variant reads neither scale array: any valid base will do)
              make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, DEBUG ? static_cast<const void*>(q) : s,
                       nb, N, nb * 2, kCkGroup, kCkM, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&txd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, DEBUG ? static_cast<const void*>(q) : xd,
                       DEBUG ? nb / 2 : nb, DEBUG ? N : T, nb * 4, 4, TT, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return cudaErrorInvalidValue;
    const int64_t t_tiles = (T + TT - 1) / TT, n_tiles = (N + kCkM - 1) / kCkM;
    const int groups = int(K / (Q8_QK * kCkGroup));
    const int ks = DEBUG ? 1 : choose_split<MODE, TT, DEBUG>(t_tiles * n_tiles, groups, ctx);
    const int per = (groups + ks - 1) / ks;
    CkParams p{N, K, T, per, y, isum, ctx.dev_err};
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[2];
    cfg.gridDim = dim3(unsigned(t_tiles), unsigned(n_tiles), unsigned((groups + per - 1) / per));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = ctx.stream;
    int na = pdl_attrs(ctx, attrs);
    if (cfg.gridDim.z > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = 1;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = cfg.gridDim.z;
        ++na;
    }
    cfg.numAttrs = na;
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kern, tw, txh, txl, ts, txd, p);
}

bool chunk_supported(int mode, int64_t N, int64_t K, int64_t T) {
    return (mode == 1 || mode == 2) && K % (Q8_QK * kCkGroup) == 0 && T >= 1 && N >= 1 &&
           encode_fn() != nullptr;
}

template <bool DEBUG>
static cudaError_t launch_chunk_any(int mode, const int8_t* q, const uint16_t* s, int64_t N,
                                    int64_t K, const void* xq, const float* xd, int64_t T, float* y,
                                    int32_t* isum, const LaunchCtx& ctx) {
    if (mode == 1) {
        if (T <= 32) return launch_chunk_t<1, 32, DEBUG>(q, s, N, K, xq, xd, T, y, isum, ctx);
        if (T <= 64) return launch_chunk_t<1, 64, DEBUG>(q, s, N, K, xq, xd, T, y, isum, ctx);
        return launch_chunk_t<1, 128, DEBUG>(q, s, N, K, xq, xd, T, y, isum, ctx);
    }
    if (T <= 32) return launch_chunk_t<2, 32, DEBUG>(q, s, N, K, xq, xd, T, y, isum, ctx);
    return launch_chunk_t<2, 64, DEBUG>(q, s, N, K, xq, xd, T, y, isum, ctx);
}

cudaError_t launch_chunk(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                         const void* xq, const float* xd, int64_t T, float* y,
                         const LaunchCtx& ctx) {
    return launch_chunk_any<false>(mode, q, s, N, K, xq, xd, T, y, nullptr, ctx);
}

cudaError_t launch_chunk_debug(int mode, const int8_t* q, int64_t N, int64_t K, const void* xq,
                               int64_t T, int32_t* isum, const LaunchCtx& ctx) {
    return launch_chunk_any<true>(mode, q, nullptr, N, K, xq, nullptr, T, nullptr, isum, ctx);
}

}  // namespace q8

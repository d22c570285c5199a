// chunk.cu -- the prefill-chunk / batched projection on the 5th-generation
// tensor cores (tcgen05, sm_103a): T activation rows at once, every weight
// byte read from HBM once per launch; optionally fused with the LM head's
// arg-max.
//
// Per Q8_0 block b the block dots of a 128-weight-row by TT-activation-row
// tile are one exact tensor-core product: int8 values are exact in f16, and
// 32 products of |q| <= 127 codes sum to < 2^24, so an f32 accumulator holds
// the integer isum exactly (two-word mode: the hi and lo planes stacked along
// the MMA's N, then 128*hi + lo rounds once, exactly like float(isum)).  The
// scales do not fold into the product (they differ per block on both sides),
// so each block's product is read back and rescaled:
//   y[t][n] += isum * (s[n][b] * d[t][b]).
// (tcgen05.mma kind::i8 does not exist for sm_103a; ptxas rejects it.)
//
// One tcgen05.mma (M = 128, K = 16) costs about the same for every N up to
// 128 on this part, so a block costs two MMAs whatever the tile's row count,
// and the per-block work around it decides the speed: the accumulator read
// back from tensor memory (a long-latency load) and the rescale.
//
// CTA tile: 128 weight rows (MMA M) x TT activation rows (MMA N = TT * planes)
// over a range of K.  Warp roles, connected by mbarriers whose waits are
// bounded:
//   warp 0      producer: 2-D TMA tiles of a stage (4 blocks of K): weights
//               (int8, 128-byte swizzle) -- issued before the wait on the
//               previous kernel, since weights never depend on it --, then
//               activation codes (one or two planes) and activation scales;
//               every 8 blocks the weight scales;
//   warp 1      owns TMEM; one thread issues two K = 16 MMAs per block into
//               one of kSlots accumulator slots, and commits once per group
//               of kGS blocks (one barrier a group of slots);
//   next 6-10   converters, a whole stage at a time: 4 or 8 warps (one or
//               two per TMEM lane quadrant) the weights int8 -> f16 into TMEM
//               (the MMA's A operand) and their scales; two warps the
//               activation codes int8 -> f16 into the K-major operand tiles in
//               shared memory (B) and their scales;
//   last 8/16   epilogue: kEG groups take the blocks in turn (so one group's
//               wait on its tensor-memory load overlaps the others' work),
//               kEC warps a lane quadrant split the columns; TMEM ->
//               registers, rescale with packed f32x2 FMAs, accumulate; the
//               groups' partial sums are added in group order at the end.
// A converted stage is freed by its MMAs' own completion (commit); an
// accumulator slot, and a block's entry in the ring of 8 scale entries, by the
// epilogue as soon as it holds them in registers.  TMEM holds the
// accumulator slots, then two or three converted stages (64 columns each).
//
// Split K: when there are too few 128 x TT tiles to fill the GPU, KS CTAs (a
// thread-block cluster along z) share a tile, each over a contiguous range
// of 8-block groups; their partial sums meet in shared memory and each CTA
// adds up a slice of the tile over the cluster (distributed shared memory),
// in rank order, so results do not depend on timing.
//
// Arg-max (the LM head): each tile's best (value, lowest row) per activation
// row goes into a 64-bit key, value-ordered bits above the complemented row,
// merged by one atomicMax per row and tile; the last CTA to take a ticket
// writes the tokens and clears the keys and the ticket.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "gemv.cuh"
#include "launch.h"
#include "tc.cuh"

namespace q8 {

constexpr int kCkM = 128;          // weight rows per tile
constexpr int kCkStageK = 128;     // bytes of K per TMA stage (4 blocks)
constexpr int kCkGroup = 8;        // blocks per weight-scale group (16 bytes of f16)
constexpr int kCkSGroups = 4;      // weight-scale groups in flight
constexpr int kCkACols = 64;       // TMEM columns of one converted stage (4 blocks x 16)
constexpr int kCkAConvWarps = 2;   // activation converters
constexpr int kCkMaxSplit = 8;
constexpr int kCkSmemBudget = 227 * 1024;

// what a launch writes
constexpr int kCkPlain = 0;    // y
constexpr int kCkDebug = 1;    // the per-block integer dots
constexpr int kCkArgmax = 2;   // the arg-max of every row (and y when given)

template <int MODE, int TT>
struct CkCfg {
    // activation planes along the MMA's N: one-word 1, two-word 2 (hi, lo),
    // f32 4 (the byte planes of each block's 31-bit fixed point)
    static constexpr int kPlanes = (MODE == 2) ? 2 : (MODE == 0 ? 4 : 1);
    static constexpr int kN = TT * kPlanes;                            // MMA N
    // converted stages in flight (A in TMEM, B in shared memory): three where
    // the accumulator slots leave room, so the converters run two stages ahead
    static constexpr int kQuads = kN <= 64 ? 3 : 2;
    static constexpr int kAccCols = 512 - kQuads * kCkACols;           // accumulator slots
    static constexpr int kSlotsRaw = (kAccCols / kN) < 8 ? (kAccCols / kN) : 8;
    // epilogue: kEC warps per lane quadrant split the columns, kEG groups
    // take the blocks in turn
    // small tiles: light epilogue work per block, so 8 epilogue warps, and
    // the weight conversion (the same per block whatever the tile) over 8
    // warps, two per TMEM lane quadrant, each half of a stage's blocks;
    // larger tiles: 16 epilogue warps and 4 weight converters
    static constexpr int kWConv = kN <= 32 ? 8 : 4;
    static constexpr int kConv = kWConv + kCkAConvWarps;
    static constexpr int kEpiWarps = kN <= 32 ? 8 : 16;
    // (f32: 8 columns a thread, each four plane sums and an f32-pair sum)
    static constexpr int kEC = MODE == 0 ? TT / 8 : (kN >= 128 ? 4 : (kN >= 64 ? 2 : 1));
    static constexpr int kEG = kEpiWarps / (4 * kEC);
    static constexpr int kSlots = kSlotsRaw / kEG * kEG;               // a multiple of the groups
    // accumulator slots are released in groups of kGS blocks (one barrier a
    // group), so that the MMA issuer waits once per group, not per block
    static constexpr int kGS = kSlots >= 8 ? 4 : (kSlots % 2 == 0 ? kSlots / 2 : 1);
    static constexpr int kSG = kSlots / kGS;
    static constexpr int kCW = TT / kEC;                               // columns per thread
    static constexpr int kW = kCkM * kCkStageK;                        // 16 KB
    static constexpr int kXPlane = TT * kCkStageK;
    // f32: the stage's f32 activation rows, converted in shared memory
    static constexpr int kX = MODE == 0 ? TT * kCkStageK * 4 : kXPlane * kPlanes;
    static constexpr int kXD = MODE == 0 ? 0 : TT * 4 * 4;             // [TT][4 blocks] f32
    static constexpr int kStage = (kW + kX + kXD + 1023) / 1024 * 1024;
    static constexpr int kSGroup = kCkM * kCkGroup * 2;                // [128][8 blocks] f16
    static constexpr int kBBlock = kN * 64;                            // [kN][32] f16
    static constexpr int kBQuad = 4 * kBBlock;
    static constexpr int kScl = kCkM * 2 + TT * 4;                     // sw[128] f16, xd[TT] f32
    static constexpr int kSE = 8;                                      // scale entries: two stages
    static constexpr int kEpiWarp0 = 2 + kConv;
    static constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
    static constexpr int kBarBytes = 1024;
    static constexpr int kFixed = kCkSGroups * kSGroup + kQuads * kBQuad +
                                  (kSE * kScl + 127) / 128 * 128 + kBarBytes + 1024 /*alignment*/;
    static constexpr int kStages = (kCkSmemBudget - kFixed) / kStage < 8
                                       ? (kCkSmemBudget - kFixed) / kStage
                                       : 8;
    static constexpr size_t kSmem = size_t(kStages) * kStage + kFixed;
    // the end-of-tile scratch in the stage area: the groups' partial sums
    // (or the CTA's split-K partial), then the arg-max candidates
    static constexpr int kPartial = kCkM * TT * (MODE == 0 ? 8 : 4);   // f32 mode: f32 pairs
    static constexpr int kBinOff = (kEG > 1 ? kEG - 1 : 1) * kPartial;   // f32: the groups' binades
    static constexpr int kCandOff = kBinOff + (MODE == 0 ? 4 * TT * 4 : 0);
    static_assert(kStages >= 3, "TMA pipeline depth");
    static_assert(kStage % 1024 == 0, "swizzled TMA tiles need 1024-byte alignment");
    static_assert(kCandOff + 4 * TT * 16 <= kStages * kStage, "end-of-tile scratch must fit the stages");
    static_assert(kSmem <= size_t(kCkSmemBudget), "shared memory");
    static_assert(MODE == 0 ? kCW == 8 : (kCW % 16 == 0 && kCW <= 32), "epilogue columns");
    static_assert(kSlots >= 3 && kSlots % kEG == 0, "accumulator slots: each served by one group");
    static_assert(kSE == 8 && kSE % kEG == 0, "scale entries: two stages, each served by one group");
    static_assert(kSlots % kGS == 0 && kSG >= 2 && kGS % kEG == 0 || kGS == 1, "slot groups");
    static_assert(kN <= 256 && kN % 16 == 0, "MMA N");
    static_assert(4 * kEC * kEG == kEpiWarps, "epilogue warps");
};

struct CkParams {
    int64_t N, K, T;
    int groups_per_split;   // 8-block groups of K per CTA of a cluster
    float* y;               // [T][N], may be NULL for the arg-max
    int32_t* isum;          // debug: per-block dots [T][N][K/32] instead of y
    int* err;
    unsigned int* ticket;   // arg-max: CTAs done
    unsigned long long* keys;   // arg-max: one key per activation row
    // f32 mode: y as f64 (instead of y), and the arg-max's (value, row) per
    // tile and activation row [tiles][T]
    double* y64;
    ArgmaxCand* cands;
    int32_t* tok;
    double* maxval;
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

// Four unsigned bytes of w -> two f16x2 words, exact: each byte b maps to the
// f16 1024 + b, then 1024 is subtracted.
__device__ __forceinline__ void u8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(a) : "r"(w), "r"(0x64646464u));   // bytes 0,1
    asm("prmt.b32 %0, %1, %2, 0x7372;" : "=r"(b) : "r"(w), "r"(0x64646464u));   // bytes 2,3
    const __half2 bias = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// The 32 8-bit values of one block row (two 16-byte chunks; signed, or
// unsigned bytes with SIGNED false) as f16, stored as row r of a K-major
// no-swizzle operand tile at `dst`.
template <bool SIGNED = true>
__device__ __forceinline__ void store_row_f16(uint32_t dst, int r, const int4 a, const int4 b) {
    const uint32_t w[8] = {uint32_t(a.x), uint32_t(a.y), uint32_t(a.z), uint32_t(a.w),
                           uint32_t(b.x), uint32_t(b.y), uint32_t(b.z), uint32_t(b.w)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {   // 8 values (one core-matrix row) per c
        uint32_t h[4];
        if constexpr (SIGNED) {
            i8x4_to_f16x4(w[2 * c], h[0], h[1]);
            i8x4_to_f16x4(w[2 * c + 1], h[2], h[3]);
        } else {
            u8x4_to_f16x4(w[2 * c], h[0], h[1]);
            u8x4_to_f16x4(w[2 * c + 1], h[2], h[3]);
        }
        sts128(dst + tile_offset(r, 8 * c), h[0], h[1], h[2], h[3]);
    }
}

// Four 16-byte chunks of int8 weights -> 32 f16x2 words (8 per chunk, the
// lower K index in the low half).
__device__ __forceinline__ void weights_f16(const int4 (&w)[4], uint32_t (&hw)[32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t v[4] = {uint32_t(w[c].x), uint32_t(w[c].y), uint32_t(w[c].z), uint32_t(w[c].w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) i8x4_to_f16x4(v[i], hw[8 * c + 2 * i], hw[8 * c + 2 * i + 1]);
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
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float f2_lo(uint64_t a) { return __uint_as_float(uint32_t(a)); }
__device__ __forceinline__ float f2_hi(uint64_t a) { return __uint_as_float(uint32_t(a >> 32)); }

// The block rescale of four accumulator columns: (a01, a23) += (v01, v23) *
// (sw * x0..x3), two packed products and two packed FMAs (the scale pairs
// formed from the consecutive registers of one shared-memory load).
__device__ __forceinline__ void rescale4(uint64_t& a01, uint64_t& a23, uint64_t v01, uint64_t v23,
                                         const int4& x, uint64_t sw2) {
    asm("{\n\t.reg .b64 x01, x23;\n\t"
        "mov.b64 x01, {%4, %5};\n\t"
        "mov.b64 x23, {%6, %7};\n\t"
        "mul.rn.f32x2 x01, x01, %8;\n\t"
        "mul.rn.f32x2 x23, x23, %8;\n\t"
        "fma.rn.f32x2 %0, %2, x01, %0;\n\t"
        "fma.rn.f32x2 %1, %3, x23, %1;\n\t}"
        : "+l"(a01), "+l"(a23)
        : "l"(v01), "l"(v23), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w), "l"(sw2));
}

__device__ __forceinline__ void sts64(uint32_t a, uint64_t v) {
    asm volatile("st.shared.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t lds64(uint32_t a) {
    uint64_t v;
    asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}

// ------------------------------------------------------ thread-block clusters

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The arriving half of named barrier `id`: counts this warp's threads towards
// `count` without waiting (the other side waits with named_bar).
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
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

// TMEM -> registers as f32 pairs, waited for inside the same PTX (the pairs
// are the load's own consecutive destination registers, so forming them
// costs no moves): 16 or 32 consecutive columns of the warp's 32 lanes, or 16
// columns at each of two addresses (the two-word mode's planes).
__device__ __forceinline__ void tmem_ld16_pairs(uint32_t taddr, uint64_t (&p)[8]) {
    asm volatile(
        "{\n\t.reg .b32 t<16>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "}"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]), "=l"(p[7])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32_pairs(uint32_t taddr, uint64_t (&p)[16]) {
    asm volatile(
        "{\n\t.reg .b32 t<32>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15, t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "}"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]), "=l"(p[7]), "=l"(p[8]), "=l"(p[9]), "=l"(p[10]), "=l"(p[11]), "=l"(p[12]), "=l"(p[13]), "=l"(p[14]), "=l"(p[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld16x2_pairs(uint32_t taddr, uint32_t taddr2, uint64_t (&p)[16]) {
    asm volatile(
        "{\n\t.reg .b32 t<32>;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t0, t1, t2, t3, t4, t5, t6, t7, t8, t9, t10, t11, t12, t13, t14, t15}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {t16, t17, t18, t19, t20, t21, t22, t23, t24, t25, t26, t27, t28, t29, t30, t31}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t"
        "mov.b64 %0, {t0, t1};\n\t"
        "mov.b64 %1, {t2, t3};\n\t"
        "mov.b64 %2, {t4, t5};\n\t"
        "mov.b64 %3, {t6, t7};\n\t"
        "mov.b64 %4, {t8, t9};\n\t"
        "mov.b64 %5, {t10, t11};\n\t"
        "mov.b64 %6, {t12, t13};\n\t"
        "mov.b64 %7, {t14, t15};\n\t"
        "mov.b64 %8, {t16, t17};\n\t"
        "mov.b64 %9, {t18, t19};\n\t"
        "mov.b64 %10, {t20, t21};\n\t"
        "mov.b64 %11, {t22, t23};\n\t"
        "mov.b64 %12, {t24, t25};\n\t"
        "mov.b64 %13, {t26, t27};\n\t"
        "mov.b64 %14, {t28, t29};\n\t"
        "mov.b64 %15, {t30, t31};\n\t"
        "}"
        : "=l"(p[0]), "=l"(p[1]), "=l"(p[2]), "=l"(p[3]), "=l"(p[4]), "=l"(p[5]), "=l"(p[6]), "=l"(p[7]), "=l"(p[8]), "=l"(p[9]), "=l"(p[10]), "=l"(p[11]), "=l"(p[12]), "=l"(p[13]), "=l"(p[14]), "=l"(p[15])
        : "r"(taddr), "r"(taddr2)
        : "memory");
}

// The f32 mode's four plane sums of 8 columns: 8 consecutive TMEM columns at
// taddr + pl * stride for pl = 0..3, waited for.
__device__ __forceinline__ void tmem_ld8x4(uint32_t taddr, uint32_t stride, float (&P)[4][8]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%33];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16, %17, %18, %19, %20, %21, %22, %23}, [%34];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24, %25, %26, %27, %28, %29, %30, %31}, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr), "r"(taddr + stride), "r"(taddr + 2 * stride), "r"(taddr + 3 * stride)
        : "memory");
#pragma unroll
    for (int pl = 0; pl < 4; ++pl)
#pragma unroll
        for (int i = 0; i < 8; ++i) P[pl][i] = __uint_as_float(r[8 * pl + i]);
}

// ------------------------------------------------------------- arg-max keys

// The 64-bit arg-max key of logit v at row n: the value's bits in an order
// that sorts like the value (-0 taken as +0), above the complemented row, so
// the largest key is the largest value at its lowest row.  0 is no key (every
// real key has a non-zero upper word).
__device__ __forceinline__ unsigned long long argmax_key(float v, unsigned n) {
    const unsigned b = __float_as_uint(v == 0.0f ? 0.0f : v);
    const unsigned ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | (0xffffffffu - n);
}

__device__ __forceinline__ void argmax_unkey(unsigned long long key, int32_t& tok, double& val) {
    if (key == 0ull) {   // no candidate: every logit of the row was NaN
        tok = 0;
        val = __longlong_as_double(0x7ff8000000000000ll);
        return;
    }
    const unsigned ord = unsigned(key >> 32);
    const unsigned b = (ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord;
    tok = int32_t(0xffffffffu - unsigned(key & 0xffffffffull));
    val = double(__uint_as_float(b));
}

// The f32 mode's epilogue warps.  Each block's four plane sums per (weight
// row, activation row) are exact integers below 2^20; they combine as in the
// CUDA-core f32 path into the block dot V = P3*2^24 + P2*2^16 + P1*2^8 + P0,
// scaled by the weight scale and the block's binade E as an exact f32 pair and
// added to the column's f32-pair sum.  A column's sum is kept in units of 2^(ecur
// - 30), ecur the largest binade seen so far, and rescaled when a larger one
// comes (exact powers of two; a part more than 2^252 below is dropped).
template <int TT, int KIND, class C>
__device__ __forceinline__ void chunk_epilogue_f32(const CkParams& p, uint32_t tmem, uint32_t scl_a,
                                                   uint32_t stages_a, uint64_t* sc_full, uint64_t* sc_empty,
                                                   uint64_t* tm_full, uint64_t* tm_empty, int warp, int lane,
                                                   int nblk, int64_t m0, int64_t t0, int* s_last) {
    constexpr bool ARGMAX = KIND == kCkArgmax;
    static_assert(KIND != kCkDebug, "the f32 mode has no block-dot debug path");
    constexpr int CW = C::kCW;   // 8
    const int ew = warp - C::kEpiWarp0;
    const int qd = warp & 3;                      // TMEM lane quadrant of this warp
    const int ec = (ew >> 2) % C::kEC;            // column slice
    const int eg = (ew >> 2) / C::kEC;            // block group
    const int n = qd * 32 + lane;                 // weight row within the tile
    const int c0 = ec * CW;
    DF acc[CW];
    int ecur[CW];
#pragma unroll
    for (int i = 0; i < CW; ++i) {
        acc[i] = DF{0.0f, 0.0f};
        ecur[i] = -1000;   // below every binade (the first block sets it)
    }
    bool ok = true;
    for (int b = eg; b < nblk; b += C::kEG) {
        const int ts = b % C::kSlots, se = b % C::kSE;
        const uint32_t par = uint32_t(b / C::kSlots) & 1u;
        if (ok) ok = mbar_wait_fast(&sc_full[(b >> 2) & 1], uint32_t(b >> 3) & 1u, p.err);
        if (ok) ok = mbar_wait_fast(&tm_full[(b / C::kGS) % C::kSG], par, p.err);
        ok = __all_sync(0xffffffffu, ok);   // the TMEM loads below are warp-wide
        if (!ok) break;
        tc_fence_after();
        const uint32_t e = scl_a + uint32_t(se * C::kScl);
        const float sw = half_bits_to_float(lds16(e + uint32_t(2 * n)));
        const int4 e0 = lds128(e + uint32_t(kCkM * 2 + c0 * 4));
        const int4 e1 = lds128(e + uint32_t(kCkM * 2 + c0 * 4 + 16));
        const int eb[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        float P[4][8];
        tmem_ld8x4(tmem + (uint32_t(qd * 32) << 16) + uint32_t(ts * C::kN + c0), uint32_t(TT), P);
        // the data is in registers: the slot and the scale entry go back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&tm_empty[(b / C::kGS) % C::kSG]);
            mbar_arrive(&sc_empty[(b >> 2) & 1]);
        }
        // columns past the last activation row are left out (warp-uniform)
        const int live = int(min64(int64_t(CW), p.T - (t0 + c0)));
#pragma unroll
        for (int i = 0; i < CW; ++i) {
            if (i >= live) break;
            if (eb[i] > ecur[i]) {
                const int dd = ecur[i] - eb[i];
                acc[i] = DF{mul_pow2_neg(acc[i].hi, dd), mul_pow2_neg(acc[i].lo, dd)};
                ecur[i] = eb[i];
            }
            // the column's factor 2^(E - ecur) <= 1: f = sw * g is exact while
            // normal; a block more than 2^100 below the column's largest
            // (below 2^-70 of it after the weight scale) is dropped
            const int dg = eb[i] - ecur[i];
            const float g = dg < -100 ? 0.0f : pow2i(dg < -126 ? -126 : dg);
            const float f = __fmul_rn(sw, g);
            // the plane sums as integers: exact floats below 2^20 read through
            // 1.5 * 2^23 (the offsets cancel below, modulo 2^32)
            const uint32_t b0 = __float_as_uint(__fadd_rn(P[0][i], 12582912.0f));
            const uint32_t b1 = __float_as_uint(__fadd_rn(P[1][i], 12582912.0f));
            const uint32_t b2 = __float_as_uint(__fadd_rn(P[2][i], 12582912.0f));
            const uint32_t b3 = __float_as_uint(__fadd_rn(P[3][i], 12582912.0f));
            const int L = int(b1 * 256u + b0 - 257u * 0x4B400000u);   // P1*2^8 + P0
            const int H = int(b3 * 256u + b2 - 257u * 0x4B400000u);   // P3*2^8 + P2
            const int2 v = make_int2((H >> 5) + (L >> 21) + 1, (H & 31) * 65536 + (L & 0x1fffff) - 2097152);
            acc[i] = df_add(acc[i], scaled_pair_split(f, v));
        }
    }
    constexpr int kEpiThreads = 32 * C::kEpiWarps;
    if constexpr (C::kEG > 1) {
        // group 1 hands its sums and binades to group 0 (the stage area is free:
        // a group's last block lies in the last stage, and its MMAs are done)
        static_assert(C::kEG == 2, "one partial-sum exchange");
        if (eg > 0) {
#pragma unroll
            for (int i = 0; i < CW; ++i) {
                const uint32_t a = stages_a + uint32_t(((c0 + i) * kCkM + n) * 8);
                sts32(a, __float_as_uint(acc[i].hi));
                sts32(a + 4u, __float_as_uint(acc[i].lo));
            }
            if (n == 0) {
#pragma unroll
                for (int i = 0; i < CW; ++i) sts32(stages_a + uint32_t(C::kBinOff + (c0 + i) * 4), uint32_t(ecur[i]));
            }
            named_bar_arrive(1, kEpiThreads);
        } else {
            named_bar(1, kEpiThreads);
#pragma unroll
            for (int i = 0; i < CW; ++i) {
                const uint32_t a = stages_a + uint32_t(((c0 + i) * kCkM + n) * 8);
                const DF o{__uint_as_float(lds32(a)), __uint_as_float(lds32(a + 4u))};
                const int eo = int(lds32(stages_a + uint32_t(C::kBinOff + (c0 + i) * 4)));
                const int em = max(ecur[i], eo);
                const DF x{mul_pow2_neg(acc[i].hi, ecur[i] - em), mul_pow2_neg(acc[i].lo, ecur[i] - em)};
                const DF y{mul_pow2_neg(o.hi, eo - em), mul_pow2_neg(o.lo, eo - em)};
                acc[i] = df_add(x, y);
                ecur[i] = em;
            }
        }
    }
    if (eg != 0) return;
    const int64_t row = m0 + n;
    if (gridDim.z > 1) {
        // split K: the CTA's partial sums and binades for the cluster's sum
        // (after the groups' exchange, in their own words)
#pragma unroll
        for (int i = 0; i < CW; ++i) {
            const uint32_t a = stages_a + uint32_t(((c0 + i) * kCkM + n) * 8);
            sts32(a, __float_as_uint(acc[i].hi));
            sts32(a + 4u, __float_as_uint(acc[i].lo));
        }
        if (n == 0) {
#pragma unroll
            for (int i = 0; i < CW; ++i)
                sts32(stages_a + uint32_t(C::kBinOff + TT * 4 + (c0 + i) * 4), uint32_t(ecur[i]));
        }
        return;
    }
    // outputs: f32 (the pair rounded once, then scaled by 2^(ecur - 30)) or f64
#pragma unroll
    for (int i = 0; i < CW; ++i) {
        const int64_t t = t0 + c0 + i;
        if (t < p.T && row < p.N) {
            const int sc = ecur[i] - 30;   // in [-156, 97]
            if (p.y64)
                p.y64[t * p.N + row] = ldexp(double(acc[i].hi) + double(acc[i].lo), sc);
            else if (p.y)
                p.y[t * p.N + row] = __fmul_rn(__fmul_rn(__fadd_rn(acc[i].hi, acc[i].lo), pow2i(sc >> 1)),
                                               pow2i(sc - (sc >> 1)));
        }
    }
    if constexpr (ARGMAX) {
        // per activation row: the best (value, lowest row) of each quadrant's 32
        // rows, then of the tile, then (the last CTA) of every tile
        constexpr int kG0 = 32 * 4 * C::kEC;   // threads of group 0
        const uint32_t cand = stages_a + uint32_t(C::kCandOff);   // [4][TT] {f64 value, row}
#pragma unroll
        for (int i = 0; i < CW; ++i) {
            double bv = -INFINITY;
            long long bi = 0x7fffffffffffffffll;
            if (row < p.N) argmax_keep(bv, bi, ldexp(double(acc[i].hi) + double(acc[i].lo), ecur[i] - 30), row);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const long long oi = __shfl_xor_sync(0xffffffffu, bi, o);
                argmax_keep(bv, bi, ov, oi);
            }
            if (lane == 0) {
                const uint32_t a = cand + uint32_t((qd * TT + c0 + i) * 16);
                sts64(a, uint64_t(__double_as_longlong(bv)));
                sts64(a + 8u, uint64_t(bi));
            }
        }
        named_bar(2, kG0);
        const int j = (ec * 4 + qd) * 32 + lane;   // 0..kG0-1
        for (int col = j; col < TT; col += kG0) {
            double bv = -INFINITY;
            long long bi = 0x7fffffffffffffffll;
            for (int q2 = 0; q2 < 4; ++q2) {
                const uint32_t a = cand + uint32_t((q2 * TT + col) * 16);
                argmax_keep(bv, bi, __longlong_as_double((long long)lds64(a)), (long long)lds64(a + 8u));
            }
            const int64_t t = t0 + col;
            if (t < p.T) p.cands[int64_t(blockIdx.y) * p.T + t] = ArgmaxCand{bv, bi};
        }
        __threadfence();
        named_bar(2, kG0);
        if (j == 0) *s_last = atomicAdd(p.ticket, 1u) == gridDim.x * gridDim.y - 1u;
        named_bar(2, kG0);
        if (*s_last) {
            __threadfence();
            const uint32_t rs = cand + uint32_t(4 * TT * 16);      // [kG0 / 32] candidates
            const int G = int(gridDim.y);
            for (int64_t t = 0; t < p.T; ++t) {
                double bv = -INFINITY;
                long long bi = 0x7fffffffffffffffll;
                for (int c2 = j; c2 < G; c2 += kG0) {
                    const ArgmaxCand* src = p.cands + int64_t(c2) * p.T + t;
                    argmax_keep(bv, bi, __ldcg(&src->v), __ldcg(&src->i));
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const double ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const long long oi = __shfl_xor_sync(0xffffffffu, bi, o);
                    argmax_keep(bv, bi, ov, oi);
                }
                if (lane == 0) {
                    sts64(rs + uint32_t((j >> 5) * 16), uint64_t(__double_as_longlong(bv)));
                    sts64(rs + uint32_t((j >> 5) * 16 + 8), uint64_t(bi));
                }
                named_bar(2, kG0);
                if (j == 0) {
                    for (int w = 1; w < kG0 / 32; ++w)
                        argmax_keep(bv, bi, __longlong_as_double((long long)lds64(rs + uint32_t(w * 16))),
                                    (long long)lds64(rs + uint32_t(w * 16 + 8)));
                    argmax_store(ArgmaxCand{bv, bi}, p.tok, p.maxval, int(t));
                }
                named_bar(2, kG0);
            }
            if (j == 0) *p.ticket = 0u;
        }
    }
}

template <int MODE, int TT, int KIND>
__global__ void __launch_bounds__(CkCfg<MODE, TT>::kThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_xh,
                 const __grid_constant__ CUtensorMap tm_xl, const __grid_constant__ CUtensorMap tm_s,
                 const __grid_constant__ CUtensorMap tm_xd, const CkParams p) {
    using C = CkCfg<MODE, TT>;
    constexpr bool DEBUG = KIND == kCkDebug;
    constexpr bool ARGMAX = KIND == kCkArgmax;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled TMA tiles
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* stages = smem;
    unsigned char* sgroups = stages + size_t(C::kStages) * C::kStage;
    unsigned char* bquads = sgroups + size_t(kCkSGroups) * C::kSGroup;
    unsigned char* scl = bquads + size_t(C::kQuads) * C::kBQuad;
    uint64_t* bars = reinterpret_cast<uint64_t*>(scl + (C::kSE * C::kScl + 127) / 128 * 128);
    uint64_t* st_full = bars;
    uint64_t* st_empty = st_full + C::kStages;
    uint64_t* sg_full = st_empty + C::kStages;
    uint64_t* sg_empty = sg_full + kCkSGroups;
    uint64_t* a_full = sg_empty + kCkSGroups;
    uint64_t* a_empty = a_full + C::kQuads;
    uint64_t* tm_full = a_empty + C::kQuads;           // per slot group
    uint64_t* tm_empty = tm_full + C::kSG;             // per slot group
    uint64_t* sc_full = tm_empty + C::kSG;             // per stage of scale entries
    uint64_t* sc_empty = sc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sc_empty + 2);
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t t0 = int64_t(blockIdx.x) * TT;
    const int64_t m0 = int64_t(blockIdx.y) * kCkM;
    // this CTA's range of K, in 8-block groups
    const int total_groups = int(p.K / (Q8_QK * kCkGroup));
    const int g_begin = int(blockIdx.z) * p.groups_per_split;
    const int g_end = min(total_groups, g_begin + p.groups_per_split);
    const int nblk = g_end > g_begin ? (g_end - g_begin) * kCkGroup : 0;
    const int nst = nblk / 4;
    const int st0 = g_begin * (kCkGroup / 4);   // first TMA stage (global)

    if (tid == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&st_full[i], 1);
            mbar_init(&st_empty[i], C::kConv);
        }
        for (int i = 0; i < kCkSGroups; ++i) {
            mbar_init(&sg_full[i], 1);
            mbar_init(&sg_empty[i], C::kWConv);
        }
        for (int i = 0; i < C::kQuads; ++i) {
            mbar_init(&a_full[i], C::kConv);
            mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < C::kSG; ++i) mbar_init(&tm_full[i], 1);
        // each block of a group is released by the 4 * kEC warps that read it
        for (int i = 0; i < C::kSG; ++i) mbar_init(&tm_empty[i], C::kGS * 4 * C::kEC);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sc_full[i], C::kConv);
            mbar_init(&sc_empty[i], 4 * 4 * C::kEC);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    const uint32_t stages_a = smem_u32(stages), sgroups_a = smem_u32(sgroups);
    const uint32_t bquads_a = smem_u32(bquads), scl_a = smem_u32(scl);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t stage_tx = uint32_t(C::kW + C::kX + (DEBUG ? 0 : C::kXD));
            const int npre = nst < C::kStages ? nst : C::kStages;
            const int ngroups = nst / 2;
            const int gpre = DEBUG ? 0 : (ngroups < kCkSGroups ? ngroups : kCkSGroups);
            auto weights = [&](int s) {
                const int slot = s % C::kStages;
                mbar_arrive_expect_tx(&st_full[slot], stage_tx);
                tma2d(stages + size_t(slot) * C::kStage, &tm_w, (st0 + s) * kCkStageK, int(m0), &st_full[slot]);
            };
            auto acts = [&](int s) {
                unsigned char* st = stages + size_t(s % C::kStages) * C::kStage;
                const int kx = (st0 + s) * kCkStageK;   // byte (= element) of K
                uint64_t* bar = &st_full[s % C::kStages];
                tma2d(st + C::kW, &tm_xh, kx, int(t0), bar);   // f32 mode: the f32 rows
                if constexpr (MODE == 2) tma2d(st + C::kW + C::kXPlane, &tm_xl, kx, int(t0), bar);
                if constexpr (!DEBUG && MODE != 0) tma2d(st + C::kW + C::kX, &tm_xd, kx / Q8_QK, int(t0), bar);
            };
            auto scales = [&](int g) {
                const int gs = g % kCkSGroups;
                mbar_arrive_expect_tx(&sg_full[gs], uint32_t(C::kSGroup));
                tma2d(sgroups + size_t(gs) * C::kSGroup, &tm_s, (st0 + 2 * g) * kCkStageK / Q8_QK, int(m0),
                      &sg_full[gs]);
            };
            // weights and their scales first: they never depend on the
            // previous kernel on the stream
            for (int s = 0; s < npre; ++s) weights(s);
            for (int g = 0; g < gpre; ++g) scales(g);
            pdl_wait();
            for (int s = 0; s < npre; ++s) acts(s);
            int issued = npre, sissued = gpre;
            for (int s = npre; s < nst; ++s) {
                const int slot = s % C::kStages;
                if (!mbar_wait_fast(&st_empty[slot], uint32_t(s / C::kStages - 1) & 1u, p.err)) break;
                weights(s);
                acts(s);
                ++issued;
                if (!DEBUG && (s & 1) == 0 && s / 2 >= gpre) {
                    const int g = s >> 1;
                    if (!mbar_wait_fast(&sg_empty[g % kCkSGroups], uint32_t(g / kCkSGroups - 1) & 1u, p.err)) break;
                    scales(g);
                    ++sissued;
                }
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int s = issued > C::kStages ? issued - C::kStages : 0; s < issued; ++s)
                mbar_wait_fast(&st_full[s % C::kStages], uint32_t(s / C::kStages) & 1u, p.err);
            for (int g = sissued > kCkSGroups ? sissued - kCkSGroups : 0; g < sissued; ++g)
                mbar_wait_fast(&sg_full[g % kCkSGroups], uint32_t(g / kCkSGroups) & 1u, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(kCkM, C::kN);
            int issued = 0;
            bool ok = true;
            for (int s = 0; s < nst && ok; ++s) {
                const int qs = s % C::kQuads;
                if (!mbar_wait_fast(&a_full[qs], uint32_t(s / C::kQuads) & 1u, p.err)) break;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int b = 4 * s + j, ts = b % C::kSlots;
                    if (b >= C::kSlots && b % C::kGS == 0 &&
                        !mbar_wait_fast(&tm_empty[(b / C::kGS) % C::kSG], uint32_t(b / C::kSlots - 1) & 1u, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = tmem + uint32_t(C::kAccCols + kCkACols * qs + 16 * j);
                    const uint32_t bb = bquads_a + uint32_t(qs * C::kBQuad + j * C::kBBlock);
                    const uint32_t d = tmem + uint32_t(ts * C::kN);
                    mma_f16_ts(d, a, smem_desc_kmajor(bb, 128, 512), idesc, false);
                    mma_f16_ts(d, a + 8u, smem_desc_kmajor(bb + 256u, 128, 512), idesc, true);
                    // one commit a slot group: its accumulators are ready together
                    if ((b + 1) % C::kGS == 0) mma_commit(smem_u32(&tm_full[(b / C::kGS) % C::kSG]));
                    ++issued;
                }
                if (ok) mma_commit(smem_u32(&a_empty[qs]));
            }
            // nothing may be left in flight when TMEM is released (the epilogue
            // normally drains every block; this covers an early exit, whose
            // last group may still want its commit)
            if (issued > 0) {
                const int bl = issued - 1;
                if (issued % C::kGS != 0) mma_commit(smem_u32(&tm_full[(bl / C::kGS) % C::kSG]));
                mbar_wait_fast(&tm_full[(bl / C::kGS) % C::kSG], uint32_t(bl / C::kSlots) & 1u, p.err);
            }
        }
    } else if (warp < C::kEpiWarp0) {
        // ------------------------------------------------------------ converters
        // warps 2 .. 2+kWConv-1: the weights of one TMEM lane quadrant each
        // (all four blocks of a stage, or with two warps a quadrant, half of
        // them) and their scales; the next two warps the activation codes and
        // their scales, one (row, block) pair a lane and pass, rows first
        // (consecutive lanes take consecutive rows of one block, so the
        // swizzled loads and the operand stores stay free of bank
        // conflicts).  Both sets follow the same stages in step.
        const bool wconv = warp < 2 + C::kWConv;
        const int qd = warp & 3;                      // TMEM lane quadrant
        const int rw = qd * 32 + lane;                // weight row = TMEM lane
        const uint32_t a_lane = uint32_t(qd * 32) << 16;
        constexpr int kHalves = C::kWConv == 8 ? 1 : 2;   // 32-column halves a weight warp converts
        const int h0 = C::kWConv == 8 ? (warp - 2) / 4 : 0;
        const int aw = warp - 2 - C::kWConv;               // activation warp 0 or 1
        constexpr int kAPasses = (TT * 4 + 63) / 64;      // (row, block) pairs a lane (TT <= 32)
        bool ok = true;
        for (int s = 0; s < nst; ++s) {
            const int slot = s % C::kStages, qs = s % C::kQuads;
            const int g = s >> 1, gs = g % kCkSGroups;
            if (ok) ok = mbar_wait_fast(&st_full[slot], uint32_t(s / C::kStages) & 1u, p.err);
            if (!DEBUG && wconv && ok && (s & 1) == 0)
                ok = mbar_wait_fast(&sg_full[gs], uint32_t(g / kCkSGroups) & 1u, p.err);
            if (ok && s >= C::kQuads) ok = mbar_wait_fast(&a_empty[qs], uint32_t(s / C::kQuads - 1) & 1u, p.err);
            // the stage's scale entries are free once the epilogue has read
            // the scales of the stage two back
            if (!DEBUG && ok && s >= 2) ok = mbar_wait_fast(&sc_empty[s & 1], uint32_t(s / 2 - 1) & 1u, p.err);
            // leave together: the warp-wide TMEM stores below need every lane
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const uint32_t st = stages_a + uint32_t(slot * C::kStage);
            if (wconv) {
                tc_fence_after();
                // weights of two blocks (32 TMEM columns) a half
#pragma unroll
                for (int hh = 0; hh < kHalves; ++hh) {
                    const int h = h0 + hh;
                    int4 w[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) w[c] = lds128(st + sw128(rw, 4 * h + c));
                    uint32_t hw[32];
                    weights_f16(w, hw);
                    tmem_st32(tmem + a_lane + uint32_t(C::kAccCols + kCkACols * qs + 32 * h), hw);
                }
                if constexpr (!DEBUG) {
                    // this row's weight scales of those blocks (its 16-byte group row)
                    const uint32_t sgr = sgroups_a + uint32_t(gs * C::kSGroup + rw * kCkGroup * 2 + (s & 1) * 8);
#pragma unroll
                    for (int hh = 0; hh < kHalves; ++hh) {
                        const int h = h0 + hh;
                        const uint32_t sw2 = lds32(sgr + uint32_t(4 * h));
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
                            sts16(scl_a + uint32_t(((4 * s + 2 * h + jj) % C::kSE) * C::kScl + 2 * rw),
                                  uint16_t(jj ? (sw2 >> 16) : (sw2 & 0xFFFFu)));
                    }
                }
                tmem_wait_st();
                tc_fence_before();
            } else {
                if constexpr (MODE == 0) {
                    // f32 rows: each (row, block) pair of the stage gives its
                    // binade E and the four byte planes of X = rint(x *
                    // 2^(30-E)) (planes 0-2 unsigned, plane 3 signed), stored
                    // as the block's B rows pl * TT + row; E goes to the
                    // block's scale entry in place of a scale
                    static_assert(TT * 4 == kAPasses * 64, "activation pairs");
#pragma unroll 1
                    for (int pass = 0; pass < kAPasses; ++pass) {
                        const int item = (2 * pass + aw) * 32 + lane;   // j * TT + ra
                        const int ra = item % TT, j = item / TT;
                        const uint32_t xs = st + uint32_t(C::kW + ra * (kCkStageK * 4) + j * (Q8_QK * 4));
                        float v[32];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int4 x4 = lds128(xs + uint32_t(16 * u));
                            v[4 * u + 0] = __int_as_float(x4.x);
                            v[4 * u + 1] = __int_as_float(x4.y);
                            v[4 * u + 2] = __int_as_float(x4.z);
                            v[4 * u + 3] = __int_as_float(x4.w);
                        }
                        const FixChunk32 f = fix_chunk32(v);
                        const uint32_t bq = bquads_a + uint32_t(qs * C::kBQuad + j * C::kBBlock);
#pragma unroll
                        for (int pl = 0; pl < 4; ++pl) {
                            const int4 lo4 = make_int4(f.p[pl][0], f.p[pl][1], f.p[pl][2], f.p[pl][3]);
                            const int4 hi4 = make_int4(f.p[pl][4], f.p[pl][5], f.p[pl][6], f.p[pl][7]);
                            if (pl == 3)
                                store_row_f16<true>(bq, pl * TT + ra, lo4, hi4);
                            else
                                store_row_f16<false>(bq, pl * TT + ra, lo4, hi4);
                        }
                        if constexpr (!DEBUG)
                            sts32(scl_a + uint32_t(((4 * s + j) % C::kSE) * C::kScl + kCkM * 2 + 4 * ra),
                                  uint32_t(f.e));
                    }
                } else if constexpr (TT <= 32) {
                    // exactly 4 * TT (row, block) pairs: two warps of 32 lanes,
                    // kAPasses passes, rows first within a block
                    static_assert(TT * 4 == kAPasses * 64, "activation pairs");
#pragma unroll
                    for (int pass = 0; pass < kAPasses; ++pass) {
                        const int item = (2 * pass + aw) * 32 + lane;   // j * TT + ra
                        const int ra = item % TT, j = item / TT;
                        const uint32_t bq = bquads_a + uint32_t(qs * C::kBQuad + j * C::kBBlock);
#pragma unroll
                        for (int pl = 0; pl < C::kPlanes; ++pl) {
                            const uint32_t xs = st + uint32_t(C::kW + pl * C::kXPlane);
                            const int4 x0 = lds128(xs + sw128(ra, 2 * j));
                            const int4 x1 = lds128(xs + sw128(ra, 2 * j + 1));
                            store_row_f16(bq, pl * TT + ra, x0, x1);
                        }
                        if constexpr (!DEBUG)
                            sts32(scl_a + uint32_t(((4 * s + j) % C::kSE) * C::kScl + kCkM * 2 + 4 * ra),
                                  lds32(st + uint32_t(C::kW + C::kX + ra * 16 + j * 4)));
                    }
                } else {
                    // one row a lane, its four blocks (the row's 128 bytes
                    // loaded at once), rows in groups of 8 consecutive rows,
                    // group g to warp g % 2, 64 rows a pass
#pragma unroll
                    for (int pass = 0; pass < TT / 64; ++pass) {
                        const int ra = 8 * (2 * (4 * pass + (lane >> 3)) + aw) + (lane & 7);
                        const uint32_t bq = bquads_a + uint32_t(qs * C::kBQuad);
#pragma unroll
                        for (int pl = 0; pl < C::kPlanes; ++pl) {
                            const uint32_t xs = st + uint32_t(C::kW + pl * C::kXPlane);
                            int4 x[8];
#pragma unroll
                            for (int c = 0; c < 8; ++c) x[c] = lds128(xs + sw128(ra, c));
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                store_row_f16(bq + uint32_t(j * C::kBBlock), pl * TT + ra, x[2 * j], x[2 * j + 1]);
                        }
                        if constexpr (!DEBUG) {
                            const int4 xd4 = lds128(st + uint32_t(C::kW + C::kX + ra * 16));
                            const uint32_t xdv[4] = {uint32_t(xd4.x), uint32_t(xd4.y), uint32_t(xd4.z),
                                                     uint32_t(xd4.w)};
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                sts32(scl_a + uint32_t(((4 * s + j) % C::kSE) * C::kScl + kCkM * 2 + 4 * ra),
                                      xdv[j]);
                        }
                    }
                }
                fence_proxy_async_smem();   // the B operand is read by the tensor core
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&a_full[qs]);
                if constexpr (!DEBUG) {
                    mbar_arrive(&sc_full[s & 1]);
                    if (wconv && (s & 1)) mbar_arrive(&sg_empty[gs]);
                }
                mbar_arrive(&st_empty[slot]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        pdl_wait();   // outputs and arg-max keys belong to the previous kernel until here
        if constexpr (MODE == 0) {
            chunk_epilogue_f32<TT, KIND, C>(p, tmem, scl_a, stages_a, sc_full, sc_empty, tm_full, tm_empty,
                                           warp, lane, nblk, m0, t0, &s_last);
        } else {
        constexpr int CW = C::kCW;
        const int ew = warp - C::kEpiWarp0;           // 0..15
        const int qd = warp & 3;                      // TMEM lane quadrant of this warp
        const int ec = (ew >> 2) % C::kEC;            // column slice
        const int eg = (ew >> 2) / C::kEC;            // block group
        const int n = qd * 32 + lane;                 // weight row within the tile
        const int c0 = ec * CW;
        uint64_t acc[CW / 2];
#pragma unroll
        for (int i = 0; i < CW / 2; ++i) acc[i] = 0;
        bool ok = true;
        for (int b = eg; b < nblk; b += C::kEG) {
            const int ts = b % C::kSlots, se = b % C::kSE;
            const uint32_t par = uint32_t(b / C::kSlots) & 1u;
            if (!DEBUG && ok) ok = mbar_wait_fast(&sc_full[(b >> 2) & 1], uint32_t(b >> 3) & 1u, p.err);
            if (ok) ok = mbar_wait_fast(&tm_full[(b / C::kGS) % C::kSG], par, p.err);
            ok = __all_sync(0xffffffffu, ok);   // the TMEM loads below are warp-wide
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t(qd * 32) << 16) + uint32_t(ts * C::kN + c0);
            if constexpr (DEBUG) {
                float v[CW];
                float vl[MODE == 2 ? CW : 1];
#pragma unroll
                for (int c = 0; c < CW / 16; ++c) {
                    tmem_ld16(d + uint32_t(16 * c), v + 16 * c);
                    if constexpr (MODE == 2) tmem_ld16(d + uint32_t(TT + 16 * c), vl + 16 * c);
                }
                tmem_wait_ld();
                // the data is in registers: the slot goes back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tm_empty[(b / C::kGS) % C::kSG]);
                // the plane sums are exact integers below 2^24
                const int64_t row = m0 + n;
#pragma unroll
                for (int i = 0; i < CW; ++i) {
                    const int64_t t = t0 + c0 + i;
                    if (t < p.T && row < p.N) {
                        int iv = __float2int_rn(v[i]);
                        if constexpr (MODE == 2) iv = 128 * iv + __float2int_rn(vl[i]);
                        p.isum[(t * p.N + row) * (p.K / Q8_QK) + g_begin * kCkGroup + b] = iv;
                    }
                }
            } else {
                // the block's weight scale, then its accumulator columns as
                // f32 pairs (the load waited for inside the same PTX)
                const uint32_t e = scl_a + uint32_t(se * C::kScl);
                const float sw = half_bits_to_float(lds16(e + uint32_t(2 * n)));
                uint64_t vp[CW / 2];
                if constexpr (MODE == 2) {
                    static_assert(CW == 16, "two-word tiles: 16 columns a thread");
                    uint64_t hl[16];
                    tmem_ld16x2_pairs(d, d + uint32_t(TT), hl);
                    // 128*hi + lo rounds once: exactly float(isum)
                    const uint64_t k128 = f2_pack(128.0f, 128.0f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) vp[i] = f2_fma(hl[i], k128, hl[8 + i]);
                } else if constexpr (CW == 32) {
                    tmem_ld32_pairs(d, vp);
                } else {
                    static_assert(CW == 16, "16 or 32 columns a thread");
                    tmem_ld16_pairs(d, vp);
                }
                // the data is in registers: the slot goes back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tm_empty[(b / C::kGS) % C::kSG]);
                const uint64_t sw2 = f2_pack(sw, sw);
#pragma unroll
                for (int i4 = 0; i4 < CW / 4; ++i4) {
                    const int4 x4 = lds128(e + uint32_t(kCkM * 2 + c0 * 4 + 16 * i4));
                    rescale4(acc[2 * i4], acc[2 * i4 + 1], vp[2 * i4], vp[2 * i4 + 1], x4, sw2);
                }
                // the block's scales are read: its scale entry goes back
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc_empty[(b >> 2) & 1]);
            }
        }
        if constexpr (!DEBUG) {
            constexpr int kEpiThreads = 32 * C::kEpiWarps;
            // The stage area is free for the end-of-tile scratch once a warp
            // has its last block: that block's MMAs have completed, so the
            // converters have read every stage.  Group 1 (its last block is
            // the tile's last) writes its partial sums there and group 0 waits
            // only for that.
            if constexpr (C::kEG > 1) {
                static_assert(C::kEG == 2, "one partial-sum exchange");
                if (eg > 0) {
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        sts32(stages_a + uint32_t(((eg - 1) * C::kPartial) + ((c0 + i) * kCkM + n) * 4),
                              (i & 1) ? uint32_t(acc[i >> 1] >> 32) : uint32_t(acc[i >> 1]));
                    named_bar_arrive(1, kEpiThreads);
                } else {
                    named_bar(1, kEpiThreads);
                }
                if (eg == 0) {
                    // the groups' partial sums in group order
                    for (int g2 = 1; g2 < C::kEG; ++g2) {
#pragma unroll
                        for (int i = 0; i < CW / 2; ++i) {
                            const uint32_t a0 = stages_a + uint32_t((g2 - 1) * C::kPartial + ((c0 + 2 * i) * kCkM + n) * 4);
                            const uint64_t o = uint64_t(lds32(a0)) | (uint64_t(lds32(a0 + kCkM * 4)) << 32);
                            acc[i] = f2_add(acc[i], o);
                        }
                    }
                }
            }
            if (eg == 0) {
                const int64_t row = m0 + n;
                if (gridDim.z == 1) {
                    if (p.y && row < p.N) {
#pragma unroll
                        for (int i = 0; i < CW; ++i) {
                            const int64_t t = t0 + c0 + i;
                            const float v = (i & 1) ? f2_hi(acc[i >> 1]) : f2_lo(acc[i >> 1]);
                            if (t < p.T) p.y[t * p.N + row] = v;
                        }
                    }
                } else {
                    // the CTA's partial tile [TT][128] f32 for the cluster sum
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        sts32(stages_a + uint32_t(((c0 + i) * kCkM + n) * 4),
                              (i & 1) ? uint32_t(acc[i >> 1] >> 32) : uint32_t(acc[i >> 1]));
                }
                if constexpr (ARGMAX) {
                    // per activation row: the best (value, lowest row) of this
                    // warp's 32 weight rows, then of the four quadrants
                    const uint32_t cand = stages_a + uint32_t(C::kCandOff);
#pragma unroll
                    for (int i = 0; i < CW; ++i) {
                        float v = (i & 1) ? f2_hi(acc[i >> 1]) : f2_lo(acc[i >> 1]);
                        unsigned ni = unsigned(row);
                        const bool valid = row < p.N && !(v != v);
                        if (!valid) {
                            v = -INFINITY;
                            ni = 0xffffffffu;
                        }
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
                            const unsigned on = __shfl_xor_sync(0xffffffffu, ni, o);
                            if (ov > v || (ov == v && on < ni)) {
                                v = ov;
                                ni = on;
                            }
                        }
                        if (lane == 0) {
                            sts32(cand + uint32_t((qd * TT + c0 + i) * 8), __float_as_uint(v));
                            sts32(cand + uint32_t((qd * TT + c0 + i) * 8 + 4), ni);
                        }
                    }
                }
            }
            if constexpr (ARGMAX) {
                constexpr int kG0 = 32 * 4 * C::kEC;   // threads of group 0
                if (eg == 0) {
                    named_bar(2, kG0);
                    const int j = (ec * 4 + ((warp - C::kEpiWarp0) & 3)) * 32 + lane;   // 0..kG0-1
                    const uint32_t cand = stages_a + uint32_t(C::kCandOff);
                    for (int col = j; col < TT; col += kG0) {
                        float bv = -INFINITY;
                        unsigned bn = 0xffffffffu;
                        for (int q2 = 0; q2 < 4; ++q2) {   // quadrants in row order
                            const float ov = __uint_as_float(lds32(cand + uint32_t((q2 * TT + col) * 8)));
                            const unsigned on = lds32(cand + uint32_t((q2 * TT + col) * 8 + 4));
                            if (ov > bv || (ov == bv && on < bn)) {
                                bv = ov;
                                bn = on;
                            }
                        }
                        const int64_t t = t0 + col;
                        if (t < p.T && bn != 0xffffffffu) atomicMax(p.keys + t, argmax_key(bv, bn));
                    }
                    __threadfence();
                    named_bar(2, kG0);
                    if (j == 0) s_last = atomicAdd(p.ticket, 1u) == gridDim.x * gridDim.y - 1u;
                    named_bar(2, kG0);
                    if (s_last) {
                        // the last CTA: every row's token, and the keys and the
                        // ticket cleared for the next call
                        __threadfence();
                        for (int64_t t = j; t < p.T; t += kG0) {
                            const unsigned long long key = atomicExch(p.keys + t, 0ull);
                            int32_t tk;
                            double val;
                            argmax_unkey(key, tk, val);
                            p.tok[t] = tk;
                            if (p.maxval) p.maxval[t] = val;
                        }
                        if (j == 0) *p.ticket = 0u;
                    }
                }
            }
        }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (MODE == 0 && gridDim.z > 1) {
        // f32 mode, split K: each CTA adds up a slice of the tile over the
        // cluster in rank order, each partial first brought to the column's
        // largest binade (exact powers of two)
        cluster_sync();
        const uint32_t ks = gridDim.z, rank = blockIdx.z;
        const int ne = TT * kCkM;
        const int per = (ne + int(ks) - 1) / int(ks);
        const int i_end = min(ne, int(rank + 1) * per);
        for (int i = int(rank) * per + tid; i < i_end; i += C::kThreads) {
            const int t = i / kCkM, nn = i % kCkM;
            const uint32_t pa = stages_a + uint32_t(i) * 8u;
            const uint32_t ba = stages_a + uint32_t(C::kBinOff + TT * 4 + t * 4);
            int em = -1000;
            for (uint32_t r = 0; r < ks; ++r) em = max(em, int(ld_cluster_u32(cluster_map(ba, r))));
            DF sum{0.0f, 0.0f};
            for (uint32_t r = 0; r < ks; ++r) {
                const uint32_t pr = cluster_map(pa, r);
                const int d = int(ld_cluster_u32(cluster_map(ba, r))) - em;
                const DF v{mul_pow2_neg(__uint_as_float(ld_cluster_u32(pr)), d),
                           mul_pow2_neg(__uint_as_float(ld_cluster_u32(pr + 4u)), d)};
                sum = df_add(sum, v);
            }
            const int64_t tg = t0 + t, row = m0 + nn;
            if (tg < p.T && row < p.N) {
                const int sc = em - 30;
                if (p.y64)
                    p.y64[tg * p.N + row] = ldexp(double(sum.hi) + double(sum.lo), sc);
                else if (p.y)
                    p.y[tg * p.N + row] = __fmul_rn(__fmul_rn(__fadd_rn(sum.hi, sum.lo), pow2i(sc >> 1)),
                                                    pow2i(sc - (sc >> 1)));
            }
        }
        // no CTA may leave while another still reads its shared memory
        cluster_sync();
    } else if (!DEBUG && gridDim.z > 1) {
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
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(p);
            fn.store(f, std::memory_order_release);
        }
    }
    return f;
}

// A 2-D tiled tensor map (also used by the batched kernel of gemv_rpl.cuh).
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
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

// A 3-D tiled tensor map for the batched kernel of gemv_rpl.cuh: dims[0] is
// contiguous, strides[] are the byte strides of dims 1 and 2 (in any order in
// memory, so one box can gather the 128-byte chunks of a tile of rows).
bool make_map3(CUtensorMap* m, CUtensorMapDataType dt, const void* base, const uint64_t dims[3],
               const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of `ks` CTAs of this kernel that fit on the device at once.
template <int MODE, int TT, int KIND>
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
        if (cudaOccupancyMaxActiveClusters(&c, chunk_kernel<MODE, TT, KIND>, &cfg) == cudaSuccess &&
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
// the busiest SM, counting whole waves of clusters.  Powers of two only:
// clusters of 3 (48 of them, where the occupancy query allows 50) ran a
// 6144 x 4096 projection at 1.6x the time of clusters of 2 in back-to-back
// launches, although this count favours them.
template <int MODE, int TT, int KIND>
static int choose_split(int64_t tiles, int groups, const LaunchCtx& ctx) {
    int best = 1;
    int64_t best_cost = -1;
    for (int ks = 1; ks <= kCkMaxSplit && ks <= groups; ks *= 2) {
        const int ac = active_clusters<MODE, TT, KIND>(ks, ctx);
        const int64_t waves = (tiles + ac - 1) / ac;
        const int64_t cost = waves * ((groups + ks - 1) / ks);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = ks;
        }
    }
    return best;
}

struct ChunkOut {
    float* y = nullptr;
    double* y64 = nullptr;   // f32 mode: f64 outputs instead of y
    int32_t* isum = nullptr;
    // arg-max
    unsigned char* ws = nullptr;
    int32_t* tok = nullptr;
    double* maxval = nullptr;
};

template <int MODE, int TT, int KIND>
static cudaError_t launch_chunk_t(const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                                  const void* xq, const float* xd, int64_t T, const ChunkOut& out,
                                  const LaunchCtx& ctx) {
    using C = CkCfg<MODE, TT>;
    constexpr bool DEBUG = KIND == kCkDebug;
    auto kern = chunk_kernel<MODE, TT, KIND>;
    static std::atomic<bool> configured[kMaxDevices];
    if (const cudaError_t e = set_smem_once(kern, size_t(C::kSmem), ctx.dev, configured); e != cudaSuccess)
        return e;
    alignas(64) CUtensorMap tw, txh, txl, ts, txd;
    const int64_t nb = K / Q8_QK;
    const int8_t* xh = reinterpret_cast<const int8_t*>(xq);
    bool ok = make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, K, N, K, kCkStageK, kCkM,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              // f32 mode: the f32 rows, a stage's 128 values of TT rows, unswizzled
              (MODE == 0 ? make_map(&txh, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xq, K, T, K * 4, kCkStageK, TT,
                                    CU_TENSOR_MAP_SWIZZLE_NONE)
                         : make_map(&txh, CU_TENSOR_MAP_DATA_TYPE_UINT8, xh, K, T, K, kCkStageK, TT,
                                    CU_TENSOR_MAP_SWIZZLE_128B)) &&
              make_map(&txl, CU_TENSOR_MAP_DATA_TYPE_UINT8, MODE == 2 ? xh + T * K : xh, K, T, K,
                       kCkStageK, TT, CU_TENSOR_MAP_SWIZZLE_128B) &&
              // (the debug variant reads neither scale array: any valid base will do)
              make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, DEBUG ? static_cast<const void*>(q) : s,
                       nb, N, nb * 2, kCkGroup, kCkM, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              // (the f32 mode reads no activation scales: any valid map will do)
              make_map(&txd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                       (DEBUG || MODE == 0) ? static_cast<const void*>(q) : xd,
                       (DEBUG || MODE == 0) ? nb / 2 : nb, (DEBUG || MODE == 0) ? N : T, nb * 4, 4, TT,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return cudaErrorInvalidValue;
    const int64_t t_tiles = (T + TT - 1) / TT, n_tiles = (N + kCkM - 1) / kCkM;
    if (t_tiles > 65535 || n_tiles > 65535) return cudaErrorInvalidValue;
    const int groups = int(K / (Q8_QK * kCkGroup));
    const int ks = KIND != kCkPlain ? 1 : choose_split<MODE, TT, KIND>(t_tiles * n_tiles, groups, ctx);
    const int per = (groups + ks - 1) / ks;
    CkParams p{};
    p.N = N;
    p.K = K;
    p.T = T;
    p.groups_per_split = per;
    p.y = out.y;
    p.y64 = out.y64;
    p.isum = out.isum;
    p.err = ctx.dev_err;
    if (KIND == kCkArgmax) {
        if (MODE == 0) {
            // the CUDA-core arg-max's layout: its ticket, then one (value,
            // row) per n tile and activation row
            if (n_tiles > kMaxGrid || T > kArgmaxGroupRows) return cudaErrorInvalidValue;
            p.ticket = reinterpret_cast<unsigned int*>(out.ws + kArgmaxGemvOff);
            p.cands = reinterpret_cast<ArgmaxCand*>(out.ws + kArgmaxGemvOff + kArgmaxHeader);
        } else {
            p.ticket = reinterpret_cast<unsigned int*>(out.ws);
            p.keys = reinterpret_cast<unsigned long long*>(out.ws + kArgmaxHeader);
        }
        p.tok = out.tok;
        p.maxval = out.maxval;
    }
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

template <int MODE, int TT, int KIND>
static void plan_of(int64_t N, int64_t K, const int64_t T, const LaunchCtx& ctx, int64_t* out) {
    const int64_t tiles = ((T + TT - 1) / TT) * ((N + kCkM - 1) / kCkM);
    const int groups = int(K / (Q8_QK * kCkGroup));
    const int kc = KIND != kCkPlain ? 1 : choose_split<MODE, TT, KIND>(tiles, groups, ctx);
    const int per = (groups + kc - 1) / kc, ks = (groups + per - 1) / per;
    const int64_t ac = active_clusters<MODE, TT, KIND>(ks, ctx);
    out[0] = TT;
    out[1] = ks;
    out[2] = tiles;
    out[3] = ac;
    out[4] = (tiles + ac - 1) / ac;
    out[5] = CkCfg<MODE, TT>::kStages;
}

template <int KIND>
static void plan_any(int mode, int64_t N, int64_t K, int64_t T, const LaunchCtx& ctx, int64_t* out) {
    if (mode == 0) {
        if (T <= 16) return plan_of<0, 16, KIND>(N, K, T, ctx, out);
        return plan_of<0, 32, KIND>(N, K, T, ctx, out);
    }
    if (mode == 1) {
        if (T <= 16) return plan_of<1, 16, KIND>(N, K, T, ctx, out);
        if (T <= 32) return plan_of<1, 32, KIND>(N, K, T, ctx, out);
        if (T <= 64) return plan_of<1, 64, KIND>(N, K, T, ctx, out);
        return plan_of<1, 128, KIND>(N, K, T, ctx, out);
    }
    if (T <= 16) return plan_of<2, 16, KIND>(N, K, T, ctx, out);
    if (T <= 32) return plan_of<2, 32, KIND>(N, K, T, ctx, out);
    return plan_of<2, 64, KIND>(N, K, T, ctx, out);
}

bool chunk_plan(int mode, int64_t N, int64_t K, int64_t T, bool argmax, const LaunchCtx& ctx,
                int64_t* out) {
    if (!chunk_supported(mode, N, K, T)) return false;
    if (argmax)
        plan_any<kCkArgmax>(mode, N, K, T, ctx, out);
    else
        plan_any<kCkPlain>(mode, N, K, T, ctx, out);
    return true;
}

bool chunk_supported(int mode, int64_t N, int64_t K, int64_t T) {
    return (mode == 0 || mode == 1 || mode == 2) && K % (Q8_QK * kCkGroup) == 0 && T >= 1 && N >= 1 &&
           encode_fn() != nullptr;
}

template <int KIND>
static cudaError_t launch_chunk_any(int mode, const int8_t* q, const uint16_t* s, int64_t N,
                                    int64_t K, const void* xq, const float* xd, int64_t T,
                                    const ChunkOut& out, const LaunchCtx& ctx) {
    if (mode == 0) {
        if constexpr (KIND == kCkDebug) return cudaErrorInvalidValue;   // no f32 block dots
        else {
            if (T <= 16) return launch_chunk_t<0, 16, KIND>(q, s, N, K, xq, xd, T, out, ctx);
            return launch_chunk_t<0, 32, KIND>(q, s, N, K, xq, xd, T, out, ctx);
        }
    }
    if (mode == 1) {
        if (T <= 16) return launch_chunk_t<1, 16, KIND>(q, s, N, K, xq, xd, T, out, ctx);
        if (T <= 32) return launch_chunk_t<1, 32, KIND>(q, s, N, K, xq, xd, T, out, ctx);
        if (T <= 64) return launch_chunk_t<1, 64, KIND>(q, s, N, K, xq, xd, T, out, ctx);
        return launch_chunk_t<1, 128, KIND>(q, s, N, K, xq, xd, T, out, ctx);
    }
    if (T <= 16) return launch_chunk_t<2, 16, KIND>(q, s, N, K, xq, xd, T, out, ctx);
    if (T <= 32) return launch_chunk_t<2, 32, KIND>(q, s, N, K, xq, xd, T, out, ctx);
    return launch_chunk_t<2, 64, KIND>(q, s, N, K, xq, xd, T, out, ctx);
}

cudaError_t launch_chunk(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                         const void* xq, const float* xd, int64_t T, void* y, bool out_f64,
                         const LaunchCtx& ctx) {
    ChunkOut out;
    if (out_f64)
        out.y64 = static_cast<double*>(y);
    else
        out.y = static_cast<float*>(y);
    return launch_chunk_any<kCkPlain>(mode, q, s, N, K, xq, xd, T, out, ctx);
}

cudaError_t launch_chunk_debug(int mode, const int8_t* q, int64_t N, int64_t K, const void* xq,
                               int64_t T, int32_t* isum, const LaunchCtx& ctx) {
    ChunkOut out;
    out.isum = isum;
    return launch_chunk_any<kCkDebug>(mode, q, nullptr, N, K, xq, nullptr, T, out, ctx);
}

cudaError_t launch_chunk_argmax(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                                const void* xq, const float* xd, int64_t T, void* logits,
                                int32_t* tok, double* maxval, void* ws, const LaunchCtx& ctx) {
    ChunkOut out;
    if (mode == 0)
        out.y64 = static_cast<double*>(logits);   // f32 mode: f64 logits
    else
        out.y = static_cast<float*>(logits);
    out.ws = static_cast<unsigned char*>(ws);
    out.tok = tok;
    out.maxval = maxval;
    return launch_chunk_any<kCkArgmax>(mode, q, s, N, K, xq, xd, T, out, ctx);
}

}  // namespace q8

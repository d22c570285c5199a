// chunk.cu -- the prefill-chunk / batched projection on the 5th-generation
// tensor cores (tcgen05, sm_103a): T activation rows at once, every weight
// byte read once per 128-row activation tile.
//
// Per Q8_0 block b the block dots of a 128-weight-row by Tt-activation-row
// tile are one exact tensor-core product: int8 values are exact in f16, and
// 32 products of |q| <= 127 codes sum to < 2^24, so an f32 accumulator holds
// the integer isum exactly (two-word mode: one product per plane, then
// 128*hi + lo rounds once, exactly like float(isum)).  The scales do not fold
// into the product (they differ per block on both sides), so each block's
// accumulator is read back and rescaled:  y[t][n] += isum * (s[n][b] * d[t][b]).
//
// CTA tile: 128 weight rows (MMA M) x up to 128 activation rows (MMA N).
// Warp roles, all connected by mbarriers with bounded waits:
//   warp 0      producer: 2-D TMA tiles of weights (int8, 128-byte swizzle),
//               activation codes (one or two planes), activation scales and,
//               every 8 blocks, weight scales;
//   warp 1      owns TMEM; one thread issues the MMAs (kind::f16, K = 16,
//               two per block per activation plane) and commits them;
//   warps 2-5   converters: int8 tiles -> f16 operand tiles in the K-major
//               no-swizzle canonical layout, plus the block's scales;
//   warps 6-13  epilogue: TMEM -> registers, rescale, accumulate in f32.
// TMEM holds two accumulator buffers (MMA of block b+1 overlaps the epilogue
// of block b).
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace q8 {

constexpr int kCkM = 128;        // weight rows per tile
constexpr int kCkTT = 128;       // activation rows per tile
constexpr int kCkStageK = 128;   // bytes of K per TMA stage (4 blocks)
constexpr int kCkOpSlots = 3;
constexpr int kCkThreads = 14 * 32;

template <int MODE>
struct CkCfg {
    static constexpr int kPlanes = (MODE == 2) ? 2 : 1;
    static constexpr int kStages = (MODE == 2) ? 2 : 3;
    static constexpr int kW = kCkM * kCkStageK;                  // 16 KB
    static constexpr int kX = kCkTT * kCkStageK * kPlanes;       // 16 / 32 KB
    static constexpr int kXD = kCkTT * 4 * 4;                    // [Tt][4 blocks] f32
    static constexpr int kStage = kW + kX + kXD;                 // multiple of 1024
    static constexpr int kSGroup = kCkM * 8 * 2;                 // [128][8 blocks] f16
    static constexpr int kA = kCkM * 64;                         // [128][32] f16
    static constexpr int kB = kCkTT * 64 * kPlanes;              // [Tt][32] f16 per plane
    static constexpr int kOp = ((kA + kB + kCkM * 2 + kCkTT * 4) + 1023) / 1024 * 1024;
    static constexpr int kTmemCols = (MODE == 2) ? 512 : 256;
    static constexpr int kDStride = 128 * kPlanes;               // TMEM columns per buffer
    static constexpr size_t kSmem = size_t(kStages) * kStage + 2 * kSGroup +
                                    size_t(kCkOpSlots) * kOp + 1024 /*barriers*/ + 1024 /*align*/;
};

struct CkParams {
    int64_t N, K, T;
    float* y;
    int32_t* isum;   // debug: per-block dots [T][N][K/32] instead of y
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

// Converts one 32-byte int8 row segment (two swizzled 16-byte chunks) to the
// f16 operand tile row r (K-major, no swizzle).
__device__ __forceinline__ void convert_row(const unsigned char* src_tile, int r, int j,
                                            unsigned char* dst_tile) {
    const int4 a = *reinterpret_cast<const int4*>(src_tile + sw128(r, 2 * j));
    const int4 b = *reinterpret_cast<const int4*>(src_tile + sw128(r, 2 * j + 1));
    const uint32_t w[8] = {uint32_t(a.x), uint32_t(a.y), uint32_t(a.z), uint32_t(a.w),
                           uint32_t(b.x), uint32_t(b.y), uint32_t(b.z), uint32_t(b.w)};
#pragma unroll
    for (int c = 0; c < 4; ++c) {   // 8 values (one core-matrix row) per c
        uint32_t h[4];
        i8x4_to_f16x4(w[2 * c], h[0], h[1]);
        i8x4_to_f16x4(w[2 * c + 1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst_tile + tile_offset(r, 8 * c)) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

template <int MODE, bool DEBUG>
__global__ void __launch_bounds__(kCkThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_xh,
                 const __grid_constant__ CUtensorMap tm_xl, const __grid_constant__ CUtensorMap tm_s,
                 const __grid_constant__ CUtensorMap tm_xd, const CkParams p) {
    using C = CkCfg<MODE>;
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled TMA tiles
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* stages = smem;
    unsigned char* sgroups = stages + size_t(C::kStages) * C::kStage;
    unsigned char* ops = sgroups + 2 * C::kSGroup;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ops + size_t(kCkOpSlots) * C::kOp);
    uint64_t* st_full = bars;
    uint64_t* st_empty = st_full + C::kStages;
    uint64_t* s_full = st_empty + C::kStages;
    uint64_t* s_empty = s_full + 2;
    uint64_t* op_full = s_empty + 2;
    uint64_t* op_empty = op_full + kCkOpSlots;
    uint64_t* d_full = op_empty + kCkOpSlots;
    uint64_t* d_empty = d_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(d_empty + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t m0 = int64_t(blockIdx.y) * kCkM;
    const int64_t t0 = int64_t(blockIdx.x) * kCkTT;
    const int nblk = int(p.K / Q8_QK);
    const int nst = int(p.K / kCkStageK);
    const int64_t trows = p.T - t0 < kCkTT ? p.T - t0 : kCkTT;
    const int np = int((trows + 15) / 16) * 16;   // MMA N

    if (tid == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&st_full[i], 1);
            mbar_init(&st_empty[i], 4);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], 8);
        }
        for (int i = 0; i < kCkOpSlots; ++i) {
            mbar_init(&op_full[i], 4);
            mbar_init(&op_empty[i], 8);
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

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            pdl_wait();
            int issued = 0, sissued = 0;
            for (int s = 0; s < nst; ++s) {
                const int slot = s % C::kStages;
                const uint32_t ph = uint32_t(s / C::kStages) & 1u;
                if (s >= C::kStages && !mbar_wait(&st_empty[slot], ph ^ 1u, p.err)) break;
                unsigned char* st = stages + size_t(slot) * C::kStage;
                mbar_arrive_expect_tx(&st_full[slot], uint32_t(C::kW + C::kX + (DEBUG ? 0 : C::kXD)));
                tma2d(st, &tm_w, s * kCkStageK, int(m0), &st_full[slot]);
                tma2d(st + C::kW, &tm_xh, s * kCkStageK, int(t0), &st_full[slot]);
                if constexpr (MODE == 2)
                    tma2d(st + C::kW + kCkTT * kCkStageK, &tm_xl, s * kCkStageK, int(t0), &st_full[slot]);
                if constexpr (!DEBUG) tma2d(st + C::kW + C::kX, &tm_xd, s * 4, int(t0), &st_full[slot]);
                ++issued;
                if (!DEBUG && (s & 1) == 0) {
                    const int g = s >> 1, gs = g & 1;
                    if (g >= 2 && !mbar_wait(&s_empty[gs], uint32_t((g >> 1) - 1) & 1u, p.err)) break;
                    mbar_arrive_expect_tx(&s_full[gs], uint32_t(C::kSGroup));
                    tma2d(sgroups + size_t(gs) * C::kSGroup, &tm_s, g * 8, int(m0), &s_full[gs]);
                    ++sissued;
                }
            }
            // never leave with copies in flight into this CTA's shared memory
            for (int s = issued > C::kStages ? issued - C::kStages : 0; s < issued; ++s)
                mbar_wait(&st_full[s % C::kStages], uint32_t(s / C::kStages) & 1u, p.err);
            for (int g = sissued > 2 ? sissued - 2 : 0; g < sissued; ++g)
                mbar_wait(&s_full[g & 1], uint32_t(g >> 1) & 1u, p.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(kCkM, np);
            bool ok = true;
            int issued = 0;
            for (int b = 0; b < nblk && ok; ++b) {
                const int os = b % kCkOpSlots, db = b & 1;
                ok = mbar_wait(&op_full[os], uint32_t(b / kCkOpSlots) & 1u, p.err);
                if (ok && b >= 2) ok = mbar_wait(&d_empty[db], uint32_t((b >> 1) - 1) & 1u, p.err);
                if (!ok) break;
                tc_fence_after();
                const unsigned char* op = ops + size_t(os) * C::kOp;
                const uint32_t a_addr = smem_u32(op);
                const uint32_t d = tmem + uint32_t(db * C::kDStride);
#pragma unroll
                for (int pl = 0; pl < C::kPlanes; ++pl) {
                    const uint32_t b_addr = smem_u32(op + C::kA + pl * (kCkTT * 64));
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2)
                        mma_f16(d + uint32_t(pl * 128), smem_desc_kmajor(a_addr + 256 * s2, 128, 512),
                                smem_desc_kmajor(b_addr + 256 * s2, 128, 512), idesc, s2 > 0);
                }
                mma_commit(smem_u32(&d_full[db]));
                ++issued;
            }
            // nothing may be left in flight when TMEM is released (the epilogue
            // normally drains every block; this covers an early exit)
            if (issued > 0)
                mbar_wait(&d_full[(issued - 1) & 1], uint32_t((issued - 1) >> 1) & 1u, p.err);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ converters
        const int ct = tid - 64;   // 0..127: weight row / activation row
        bool ok = true;
        for (int b = 0; b < nblk; ++b) {
            const int s = b >> 2, j = b & 3, slot = s % C::kStages;
            const int g = b >> 3, gs = g & 1, os = b % kCkOpSlots;
            if (ok && j == 0) ok = mbar_wait(&st_full[slot], uint32_t(s / C::kStages) & 1u, p.err);
            if (!DEBUG && ok && (b & 7) == 0) ok = mbar_wait(&s_full[gs], uint32_t(g >> 1) & 1u, p.err);
            if (ok && b >= kCkOpSlots)
                ok = mbar_wait(&op_empty[os], uint32_t(b / kCkOpSlots - 1) & 1u, p.err);
            if (!ok) break;
            const unsigned char* st = stages + size_t(slot) * C::kStage;
            unsigned char* op = ops + size_t(os) * C::kOp;
            convert_row(st, ct, j, op);                                   // weights -> A
            convert_row(st + C::kW, ct, j, op + C::kA);                   // codes -> B
            if constexpr (MODE == 2)
                convert_row(st + C::kW + kCkTT * kCkStageK, ct, j, op + C::kA + kCkTT * 64);
            if constexpr (!DEBUG) {
                const uint16_t* sg = reinterpret_cast<const uint16_t*>(sgroups + size_t(gs) * C::kSGroup);
                reinterpret_cast<uint16_t*>(op + C::kA + C::kB)[ct] = sg[ct * 8 + (b & 7)];
                const float* xd = reinterpret_cast<const float*>(st + C::kW + C::kX);
                reinterpret_cast<float*>(op + C::kA + C::kB + kCkM * 2)[ct] = xd[ct * 4 + j];
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&op_full[os]);
                if (j == 3) mbar_arrive(&st_empty[slot]);
                if (!DEBUG && (b & 7) == 7) mbar_arrive(&s_empty[gs]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 6;          // 0..7
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int h = ew >> 2;            // column half
        const int n = q * 32 + lane;      // weight row within the tile
        const int c0 = 64 * h;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
        bool ok = true;
        for (int b = 0; b < nblk; ++b) {
            const int db = b & 1, os = b % kCkOpSlots;
            if (ok) ok = mbar_wait(&d_full[db], uint32_t(b >> 1) & 1u, p.err);
            if (!ok) break;
            tc_fence_after();
            const unsigned char* op = ops + size_t(os) * C::kOp;
            const float sw = half_bits_to_float(reinterpret_cast<const uint16_t*>(op + C::kA + C::kB)[n]);
            const float* xdv = reinterpret_cast<const float*>(op + C::kA + C::kB + kCkM * 2);
            if (c0 < np) {
                const uint32_t d = tmem + (uint32_t(q * 32) << 16) + uint32_t(db * C::kDStride + c0);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    float v[32];
                    float vl[32];
                    tmem_ld32(d + uint32_t(32 * cc), v);
                    if constexpr (MODE == 2) tmem_ld32(d + 128 + uint32_t(32 * cc), vl);
                    tmem_wait_ld();
                    if constexpr (DEBUG) {
                        // the plane sums are exact integers below 2^24
                        const int64_t row = m0 + n;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int64_t t = t0 + c0 + 32 * cc + i;
                            if (t < p.T && row < p.N) {
                                int iv = __float2int_rn(v[i]);
                                if constexpr (MODE == 2) iv = 128 * iv + __float2int_rn(vl[i]);
                                p.isum[(t * p.N + row) * nblk + b] = iv;
                            }
                        }
                    } else {
                        if constexpr (MODE == 2) {
                            // 128*hi + lo rounds once: exactly float(isum)
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __fmaf_rn(128.0f, v[i], vl[i]);
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            acc[32 * cc + i] = __fmaf_rn(v[i], __fmul_rn(sw, xdv[c0 + 32 * cc + i]),
                                                         acc[32 * cc + i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&d_empty[db]);
                mbar_arrive(&op_empty[os]);
            }
        }
        if constexpr (!DEBUG) {
            const int64_t row = m0 + n;
            if (row < p.N) {
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int64_t t = t0 + c0 + i;
                    if (t < p.T) p.y[t * p.N + row] = acc[i];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
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

template <int MODE, bool DEBUG>
static cudaError_t launch_chunk_t(const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                                  const void* xq, const float* xd, int64_t T, float* y,
                                  int32_t* isum, const LaunchCtx& ctx) {
    using C = CkCfg<MODE>;
    auto kern = chunk_kernel<MODE, DEBUG>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(C::kSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    alignas(64) CUtensorMap tw, txh, txl, ts, txd;
    const int64_t nb = K / Q8_QK;
    const int8_t* xh = reinterpret_cast<const int8_t*>(xq);
    bool ok = make_map(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, K, N, K, kCkStageK, kCkM,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&txh, CU_TENSOR_MAP_DATA_TYPE_UINT8, xh, K, T, K, kCkStageK, kCkTT,
                       CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&txl, CU_TENSOR_MAP_DATA_TYPE_UINT8, MODE == 2 ? xh + T * K : xh, K, T, K,
                       kCkStageK, kCkTT, CU_TENSOR_MAP_SWIZZLE_128B) &&
              // (the debug variant reads neither scale array: any valid base will do)
              make_map(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, DEBUG ? static_cast<const void*>(q) : s,
                       nb, N, nb * 2, 8, kCkM, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&txd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, DEBUG ? static_cast<const void*>(q) : xd,
                       DEBUG ? nb / 2 : nb, DEBUG ? N : T, nb * 4, 4, kCkTT, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return cudaErrorInvalidValue;
    CkParams p{N, K, T, y, isum, ctx.dev_err};
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[1];
    cfg.gridDim = dim3(unsigned((T + kCkTT - 1) / kCkTT), unsigned((N + kCkM - 1) / kCkM));
    cfg.blockDim = dim3(kCkThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = ctx.stream;
    cfg.numAttrs = pdl_attrs(ctx, attrs);
    cfg.attrs = attrs;
    return cudaLaunchKernelEx(&cfg, kern, tw, txh, txl, ts, txd, p);
}

bool chunk_supported(int mode, int64_t N, int64_t K, int64_t T) {
    return (mode == 1 || mode == 2) && K % 256 == 0 && T >= 1 && N >= 1 && encode_fn() != nullptr;
}

cudaError_t launch_chunk(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                         const void* xq, const float* xd, int64_t T, float* y,
                         const LaunchCtx& ctx) {
    if (mode == 1) return launch_chunk_t<1, false>(q, s, N, K, xq, xd, T, y, nullptr, ctx);
    return launch_chunk_t<2, false>(q, s, N, K, xq, xd, T, y, nullptr, ctx);
}

cudaError_t launch_chunk_debug(int mode, const int8_t* q, int64_t N, int64_t K, const void* xq,
                               int64_t T, int32_t* isum, const LaunchCtx& ctx) {
    if (mode == 1) return launch_chunk_t<1, true>(q, nullptr, N, K, xq, nullptr, T, nullptr, isum, ctx);
    return launch_chunk_t<2, true>(q, nullptr, N, K, xq, nullptr, T, nullptr, isum, ctx);
}

}  // namespace q8

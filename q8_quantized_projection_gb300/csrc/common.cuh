// common.cuh -- device helpers shared by the kernels of libq8proj (sm_103a).
//
// Inline PTX for the pieces CUDA C++ does not spell directly: mbarriers, the
// bulk-copy (TMA) engine, programmatic dependent launch and the global timer
// used to bound every wait.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define Q8_QK 32

// Device error codes written to the library's error word.
#define Q8_DEVERR_TIMEOUT 1
#define Q8_DEVERR_POSITION 2   // a KV-cache position outside the cache

// A bounded wait gives up after this many nanoseconds of global time.
#define Q8_WAIT_LIMIT_NS 2000000000ull

namespace q8 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}



// Waits for the phase with the given parity to complete.  Gives up after
// Q8_WAIT_LIMIT_NS, records Q8_DEVERR_TIMEOUT in *err and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > Q8_WAIT_LIMIT_NS) {
            atomicExch(err, Q8_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// The polling loop of mbar_wait_fast, out of line.
static __device__ __noinline__ bool mbar_wait_poll(uint64_t* bar, uint32_t parity, int* err) {
    const uint64_t t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > Q8_WAIT_LIMIT_NS) {
            atomicExch(err, Q8_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// mbar_wait whose common case (a phase that has already completed) costs one
// try_wait, without the polling loop's reconvergence around it (measured:
// about 50 cycles against 170), for fine-grained pipelines where most waits
// find the phase complete.  The out-of-line loop costs registers at the call
// site, so register-bound kernels keep mbar_wait.
__device__ __forceinline__ bool mbar_wait_fast(uint64_t* bar, uint32_t parity, int* err) {
    return mbar_try_wait(bar, parity) || mbar_wait_poll(bar, parity, err);
}

// ----------------------------------------------------------- bulk copy (TMA)

// Contiguous global -> shared copy on the bulk-copy engine; completion is
// counted in bytes on `bar`.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (weights are streamed once).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier `id` (1..15) over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------- programmatic dependent launch

// Blocks until every grid this one depends on has completed and its memory
// operations are visible.  Returns at once when launched without PDL.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next grid on the stream be scheduled before this one finishes.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------- global loads

// 16-byte read-only load through the non-coherent path.
__device__ __forceinline__ int4 ldg_nc_v4(const void* p) {
    int4 v;
    asm volatile("ld.global.nc.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int4 lds_v4(const void* p) {
    return *reinterpret_cast<const int4*>(p);
}

// Explicit shared-space loads on 32-bit shared addresses (data written by the
// bulk-copy engine and published through an mbarrier wait).
__device__ __forceinline__ int4 lds128(uint32_t addr) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ float half_bits_to_float(uint16_t bits) {
    return __half2float(__ushort_as_half(bits));
}

// ------------------------------------------------------------ block dots

// float(v) for |v| < 2^22 without a conversion instruction: v added to the
// bit pattern of 1.5*2^23 is that float plus v, exactly.
__device__ __forceinline__ float small_int_to_float(int v) {
    return __fsub_rn(__int_as_float(0x4B400000 + v), 12582912.0f);
}

// Exact int32 dot of 16 int8 weights with 16 int8 activation codes.
__device__ __forceinline__ int dot16_i8(const int4 w, const int4 a) {
    int acc = __dp4a(w.x, a.x, 0);
    acc = __dp4a(w.y, a.y, acc);
    acc = __dp4a(w.z, a.z, acc);
    acc = __dp4a(w.w, a.w, acc);
    return acc;
}

// Exact int32 dot of 16 weights with the 14-bit code 128*hi + lo.
// |result| <= 16 * 127 * 8191 < 2^24, so it also converts to float exactly.
__device__ __forceinline__ int dot16_i8x2(const int4 w, const int4 hi, const int4 lo) {
    return 128 * dot16_i8(w, hi) + dot16_i8(w, lo);
}

// Signed byte j (0..3) of a packed word, as float.
__device__ __forceinline__ float byte_as_float(int word, int j) {
    return static_cast<float>(static_cast<int>(word << (24 - 8 * j)) >> 24);
}

// Round-half-away-from-zero quotient of x by d, clamped to [-lim, lim]
// (0 when d == 0).  IEEE division, as the quantisers are defined.
__device__ __forceinline__ int quantize_code(float x, float d, float lim) {
    if (d == 0.0f) return 0;
    float v = roundf(__fdiv_rn(x, d));
    v = fminf(fmaxf(v, -lim), lim);
    return static_cast<int>(v);
}

}  // namespace q8

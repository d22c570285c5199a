// noalloc.cu -- head_argmax for callers that cannot allocate device memory.
//
// The arg-max epilogues need a little scratch (ticket counters, one key per
// activation row, and one candidate per CTA and row).  head_argmax takes it from the caller; this
// entry point keeps it instead in a file-scope device array of fixed size,
// which every GPU that loads the library holds until the process exits.
//
// Host code must not hand the array's name to a kernel: on the host it is a
// stand-in symbol, not a device address.  The first call on each device,
// with that device current, looks the real address up with
// cudaGetSymbolAddress and caches it; that first call should therefore come
// before any stream capture.  All calls share the one array and it keeps the
// last call's contents, so each call clears the counters and keys it relies on
// (an asynchronous memset on the caller's stream) and calls that overlap on
// the GPU race on the array.  Nothing here allocates.
#include <mutex>

#include "launch.h"
#include "q8proj.h"

namespace {

constexpr size_t kNoAllocScratch = q8::kArgmaxGemvOff + q8::kArgmaxHeader +
                                   size_t(q8::kMaxGrid) * q8::kArgmaxGroupRows * sizeof(q8::ArgmaxCand);

__device__ __align__(256) unsigned char g_q8_head_scratch[kNoAllocScratch];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev];
std::mutex g_scratch_mu;

}  // namespace

extern "C" {

size_t head_argmax_noalloc_scratch_bytes(void) { return kNoAllocScratch; }

q8_status head_argmax_noalloc(int mode, const int8_t* q, const uint16_t* s, int64_t N,
                              int64_t K, const void* xq, const float* xd, int64_t rows,
                              int32_t* tok, double* maxval, void* logits, void* stream) {
    if (rows < 1 || rows > Q8_MAX_ROWS) return Q8_ERR_SHAPE;
    if (head_argmax_workspace(rows) > kNoAllocScratch) return Q8_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q8_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return Q8_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_q8_head_scratch) != cudaSuccess || !p)
                return Q8_ERR_CUDA;
            g_scratch_ptr[dev] = p;
        }
        ptr = g_scratch_ptr[dev];
    }
    // the ticket counters and the keys must read zero when the kernel starts
    if (cudaMemsetAsync(ptr, 0, q8::kArgmaxGemvOff + q8::kArgmaxHeader,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return Q8_ERR_CUDA;
    return head_argmax(mode, q, s, N, K, xq, xd, rows, tok, maxval, logits, ptr, kNoAllocScratch,
                       stream);
}

}  // extern "C"

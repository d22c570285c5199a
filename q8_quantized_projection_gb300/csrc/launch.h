// launch.h -- host-side launch interface between the C ABI (api.cu) and the
// kernel translation units.  Internal to libq8proj.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace q8 {

constexpr int kMaxDevices = 64;   // devices one process may use

// Raises a kernel's dynamic shared-memory limit once per device: the attribute
// belongs to that device's context.  `done` is the kernel's own flag array;
// two threads that race here both set the same value.
template <typename F>
inline cudaError_t set_smem_once(F kern, size_t smem, int dev, std::atomic<bool>* done) {
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
    return e;
}

struct LaunchCtx {
    int dev;         // current device, 0 <= dev < kMaxDevices
    cudaStream_t stream;
    bool pdl;        // programmatic dependent launch
    int num_sms;     // SMs of the current device
    int* dev_err;    // device error word of the current device
};

// Fills `attrs` with the PDL attribute when enabled; returns the count.
int pdl_attrs(const LaunchCtx& ctx, cudaLaunchAttribute* attrs);

cudaError_t launch_pack(const float* w, int64_t N, int64_t K, int8_t* q, uint16_t* s,
                        int32_t* overflow, const LaunchCtx& ctx);

// prod: 0 plain (h, norm as given), 1 residual (h + res, normalised), 2 SwiGLU
// (h the fused gate+up output, rows of 2K values; no norm)
cudaError_t launch_act_quant(int mode, int prod, const float* h, const float* res, float* s_out,
                             int64_t rows, int64_t K, int norm, const float* gain, float eps, void* xq,
                             float* xd, const LaunchCtx& ctx);

// One CUDA-core GEMV launch over a group of at most `gemv_max_rows(mode)`
// activation rows.
struct GemvArgs {
    int mode;
    const int8_t* q;
    const uint16_t* s;
    int64_t N, K;
    const void* act;    // activation of the group's first row (mode layout)
    const float* xd;    // block scales of the group's first row
    int64_t plane;      // elements between the hi and lo planes (two-word mode)
    int rows;           // rows in the group
    void* y;            // output of the group's first row (row stride N), may be NULL
    int out_f64;
    // arg-max epilogue (head): all NULL for a plain projection
    int32_t* tok;
    double* maxval;
    void* ws;
    // producer fused into the projection (decode step, one row): when h is
    // set, act/xd are ignored and the kernel runs RMSNorm -> quant itself
    const float* h;
    int prod;            // producer input: 0 h, 1 h + res, 2 SwiGLU of h (gate+up row)
    const float* res;    // residual added before the norm, or NULL
    float* s_out;        // h + res written back, or NULL
    const float* gain;
    float eps;
    // KV-row epilogue (see GemvParams); k_cache NULL: none
    const int32_t* pos;
    int64_t kv_col, kv_dim, n_pos;
    float* k_cache;
    float* v_cache;
};

// Largest K the decode kernel quantises in its own shared memory.
constexpr int64_t kFusedMaxK = 16384;

// Rows per CUDA-core launch: the decode kernel's widest row count per mode
// (more rows run as groups, each reading the weights once); f32 runs a row
// per launch: it is issue-bound, and a two-row pass cost 1.5x two one-row
// passes (LM head, 16 rows: 3.19 ms in pairs, 2.07 ms row by row).
constexpr int gemv_max_rows(int mode) { return mode == 0 ? 1 : mode == 1 ? 8 : 4; }
// The rows one such launch takes for a projection with K values: f32 pairs
// where the row-per-lane kernel holds both rows in shared memory (K % 1024 ==
// 0, K <= 8192; plain or with the arg-max), else gemv_max_rows(mode).
constexpr int gemv_group_rows(int mode, int64_t K) {
    return (mode == 0 && K % 1024 == 0 && K <= 8192) ? 2 : gemv_max_rows(mode);
}

// tensor-core chunk path (chunk.cu): modes 1 and 2, K % 256 == 0
bool chunk_supported(int mode, int64_t N, int64_t K, int64_t T);
// (f32 mode: xq is the f32 activation, xd unused; y is double [T][N] with
// out_f64, float else)
cudaError_t launch_chunk(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                         const void* xq, const float* xd, int64_t T, void* y, bool out_f64,
                         const LaunchCtx& ctx);
cudaError_t launch_chunk_debug(int mode, const int8_t* q, int64_t N, int64_t K, const void* xq,
                               int64_t T, int32_t* isum, const LaunchCtx& ctx);
// The chunk projection fused with the arg-max of every activation row (the LM
// head): ws is the arg-max workspace (int8 modes: ticket and keys; f32 mode:
// the CUDA-core layout from kArgmaxGemvOff, at most kMaxGrid tiles of 128
// rows and kArgmaxGroupRows activation rows); logits (float [T][N], f32 mode
// double) may be NULL.
cudaError_t launch_chunk_argmax(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                                const void* xq, const float* xd, int64_t T, void* logits,
                                int32_t* tok, double* maxval, void* ws, const LaunchCtx& ctx);
// The launch plan the chunk path would use (host side; occupancy queries
// only): out[6] = TT, ks (CTAs splitting K), tiles, clusters that fit at once,
// waves, pipeline stages.  False where the path does not apply (mode, K).
bool chunk_plan(int mode, int64_t N, int64_t K, int64_t T, bool argmax, const LaunchCtx& ctx,
                int64_t* out);
// Activation rows from which projections run on the tensor cores: where one
// chunk launch beats the decode kernel's groups of rows (one-word: groups of
// 8, so 9 rows and more; two-word: groups of 4, so 5 and more; f32: a row a
// pass, measured on the d = 4096 layer: even at 3 rows, 199 against 239 us
// at 4).  The f32 LM head (a launch per row) breaks even at 6 rows.
inline int64_t chunk_min_rows(int mode) { return mode == 2 ? 5 : mode == 0 ? 4 : 9; }
inline int64_t chunk_min_head_rows(int mode) { return mode == 0 ? 6 : chunk_min_rows(mode); }

// K/V slices of y [rows][N] into cache row pos[m] of each row's cache
cudaError_t launch_kv_scatter(const float* y, int64_t rows, int64_t N, const int32_t* pos, int64_t kv_col,
                              int64_t kv_dim, int64_t n_pos, float* k_cache, float* v_cache,
                              const LaunchCtx& ctx);

cudaError_t launch_debug_dots(int mode, const int8_t* q, const void* xq, int64_t N, int64_t K,
                              int64_t rows, int32_t* isum, const LaunchCtx& ctx);

// Workspace layout of the arg-max epilogues, all at fixed offsets so that one
// workspace serves calls of any row count:
//   [0, 256)                      the tensor-core path's ticket counter
//   [256, 256 + kArgmaxKeyBytes)  its 64-bit key per activation row
//   [kArgmaxGemvOff, ...)         the CUDA-core path: a ticket counter, then
//                                 from kArgmaxHeader on one (value, index)
//                                 candidate per CTA and row of a group.
// Counters and keys must be zero before the first call; every completed call
// leaves them zero.
constexpr size_t kArgmaxHeader = 256;
constexpr size_t kArgmaxKeyBytes = 8 * 256;   // one key per row, up to the largest row count
constexpr size_t kArgmaxGemvOff = kArgmaxHeader + kArgmaxKeyBytes;
constexpr int kMaxGrid = 1024;
struct ArgmaxCand {
    double v;
    long long i;
};
// Rows of one arg-max launch the workspace is sized for (every mode's group).
constexpr int kArgmaxGroupRows = 16;
static_assert(gemv_max_rows(0) <= kArgmaxGroupRows && gemv_max_rows(1) <= kArgmaxGroupRows &&
                  gemv_max_rows(2) <= kArgmaxGroupRows,
              "the arg-max workspace holds one candidate per CTA and row of a group");

}  // namespace q8

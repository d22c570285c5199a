// api.cu -- the C ABI of libq8proj (declared in include/q8proj.h): argument
// validation on the host, then launches of the kernels on the caller's stream.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "q8proj.h"

namespace q8 {
cudaError_t launch_gemv_mode0(const GemvArgs& a, const LaunchCtx& ctx);
cudaError_t launch_gemv_mode1(const GemvArgs& a, const LaunchCtx& ctx);
cudaError_t launch_gemv_mode2(const GemvArgs& a, const LaunchCtx& ctx);
cudaError_t launch_gemv_fused_mode0(const GemvArgs& a, const LaunchCtx& ctx);
cudaError_t launch_gemv_fused_mode1(const GemvArgs& a, const LaunchCtx& ctx);
cudaError_t launch_gemv_fused_mode2(const GemvArgs& a, const LaunchCtx& ctx);
}  // namespace q8

using namespace q8;

// Device error word: bounded waits that run out record a code here.
__device__ int g_q8_dev_err;

namespace {

thread_local int t_last_cuda = 0;
std::atomic<int> g_pdl{1};   // q8_set_pdl may race with launches on other threads

struct DevInfo {
    bool ready = false;
    int num_sms = 0;
    int* dev_err = nullptr;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

q8_status cuda_fail(cudaError_t e) {
    t_last_cuda = int(e);
    return Q8_ERR_CUDA;
}

q8_status make_ctx(void* stream, LaunchCtx& ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return Q8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevInfo& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_q8_dev_err);
        if (e != cudaSuccess) return cuda_fail(e);
        d.dev_err = static_cast<int*>(p);
        d.ready = true;
    }
    ctx.dev = dev;
    ctx.stream = static_cast<cudaStream_t>(stream);
    ctx.pdl = g_pdl.load(std::memory_order_relaxed) != 0;
    ctx.num_sms = d.num_sms;
    ctx.dev_err = d.dev_err;
    return Q8_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

q8_status launched(cudaError_t e) { return e == cudaSuccess ? Q8_OK : cuda_fail(e); }

bool valid_mode(int mode) { return mode >= Q8_ACT_F32 && mode <= Q8_ACT_I8X2; }

q8_status check_shape(int64_t N, int64_t K) {
    if (N < 1 || K < Q8_QK || K % Q8_QK != 0) return Q8_ERR_SHAPE;
    if (N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 24)) return Q8_ERR_SHAPE;
    return Q8_OK;
}

size_t act_bytes(int mode, int64_t rows, int64_t K) {
    if (mode == Q8_ACT_F32) return size_t(rows) * K * 4;
    if (mode == Q8_ACT_I8) return size_t(rows) * K;
    return size_t(2) * rows * K;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

cudaError_t gemv_dispatch(const GemvArgs& a, const LaunchCtx& ctx) {
    if (a.mode == Q8_ACT_F32) return launch_gemv_mode0(a, ctx);
    if (a.mode == Q8_ACT_I8) return launch_gemv_mode1(a, ctx);
    return launch_gemv_mode2(a, ctx);
}

// The KV-row epilogue's arguments (k_cache NULL: none).
struct KvArgs {
    const int32_t* pos = nullptr;
    int64_t kv_col = 0, kv_dim = 0, n_pos = 0;
    float* k_cache = nullptr;
    float* v_cache = nullptr;
};

// Runs the CUDA-core projection over groups of gemv_group_rows(mode, K)
// activation rows (each group one launch reading the weights once).
q8_status run_projection(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                         const void* xq, const float* xd, int64_t rows, void* y, int out_f64,
                         int32_t* tok, double* maxval, void* ws, const LaunchCtx& ctx) {
    const int64_t nb = K / Q8_QK;
    const int group = gemv_group_rows(mode, K);
    const size_t elem = (mode == Q8_ACT_F32) ? 4 : 1;
    const size_t ysz = (mode == Q8_ACT_F32 && out_f64) ? 8 : 4;
    for (int64_t g0 = 0; g0 < rows; g0 += group) {
        GemvArgs a{};
        a.mode = mode;
        a.q = q;
        a.s = s;
        a.N = N;
        a.K = K;
        a.act = static_cast<const unsigned char*>(xq) + size_t(g0) * K * elem;
        a.xd = xd ? xd + g0 * nb : nullptr;
        a.plane = rows * K;
        a.rows = int(rows - g0 < group ? rows - g0 : group);
        a.y = y ? static_cast<unsigned char*>(y) + size_t(g0) * N * ysz : nullptr;
        a.out_f64 = out_f64;
        a.tok = tok ? tok + g0 : nullptr;
        a.maxval = maxval ? maxval + g0 : nullptr;
        a.ws = ws;
        cudaError_t e = gemv_dispatch(a, ctx);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return Q8_OK;
}

// Plain projection of an activation: the tensor-core chunk kernel from
// chunk_min_rows(mode) rows on (K % 256 == 0), the CUDA-core kernels else.
q8_status project_dispatch(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                           const void* xq, const float* xd, int64_t rows, void* y, int out_f64,
                           const LaunchCtx& ctx) {
    // (f32 at 4 rows runs as two row pairs where the row-per-lane kernel holds
    // a pair: 2 x 87 against 197 us for the d = 4096 layer)
    const bool f32_pairs = mode == Q8_ACT_F32 && rows == 4 && gemv_group_rows(mode, K) == 2;
    if (!f32_pairs && (!out_f64 || mode == Q8_ACT_F32) && rows >= chunk_min_rows(mode) &&
        chunk_supported(mode, N, K, rows))
        return launched(launch_chunk(mode, q, s, N, K, xq, xd, rows, y, out_f64 != 0, ctx));
    return run_projection(mode, q, s, N, K, xq, xd, rows, y, out_f64, nullptr, nullptr, nullptr,
                          ctx);
}

q8_status check_proj_args(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                          const void* xq, const float* xd, int64_t rows, const void* y) {
    if (!valid_mode(mode)) return Q8_ERR_MODE;
    if (!q || !s || !xq || !y || (mode != Q8_ACT_F32 && !xd)) return Q8_ERR_ARG;
    q8_status st = check_shape(N, K);
    if (st != Q8_OK) return st;
    if (rows < 1 || rows > Q8_MAX_ROWS) return Q8_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(s) || !aligned16(xq) || !aligned16(y) ||
        (xd && !aligned16(xd)))
        return Q8_ERR_ALIGN;
    return Q8_OK;
}

}  // namespace

extern "C" {

const char* q8_status_str(int status) {
    switch (status) {
        case Q8_OK: return "Q8_OK";
        case Q8_ERR_ARG: return "Q8_ERR_ARG";
        case Q8_ERR_SHAPE: return "Q8_ERR_SHAPE";
        case Q8_ERR_ALIGN: return "Q8_ERR_ALIGN";
        case Q8_ERR_MODE: return "Q8_ERR_MODE";
        case Q8_ERR_CUDA: return "Q8_ERR_CUDA";
        case Q8_ERR_UNSUPPORTED: return "Q8_ERR_UNSUPPORTED";
        case Q8_ERR_WORKSPACE: return "Q8_ERR_WORKSPACE";
        default: return "Q8_ERR_UNKNOWN";
    }
}

int q8_version(void) { return 106; }

int q8_last_cuda_error(void) { return t_last_cuda; }

void q8_set_pdl(int enable) { g_pdl.store(enable ? 1 : 0, std::memory_order_relaxed); }

q8_status q8_device_error(int32_t* code, void* stream) {
    if (!code) return Q8_ERR_ARG;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_q8_dev_err, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_q8_dev_err, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    *code = v;
    return Q8_OK;
}

q8_status q8_pack(const float* w, int64_t N, int64_t K, int8_t* q, uint16_t* s,
                  int32_t* overflow, void* stream) {
    if (!w || !q || !s) return Q8_ERR_ARG;
    q8_status st = check_shape(N, K);
    if (st != Q8_OK) return st;
    if (!aligned16(w) || !aligned16(q) || !aligned16(s) || (overflow && !aligned16(overflow)))
        return Q8_ERR_ALIGN;
    LaunchCtx ctx;
    if ((st = make_ctx(stream, ctx)) != Q8_OK) return st;
    return launched(launch_pack(w, N, K, q, s, overflow, ctx));
}

// [a, a + n) and [b, b + n) overlap (either NULL: no)
static bool overlaps(const void* a, const void* b, size_t n) {
    if (!a || !b) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + n && y < x + n;
}

// The residual's arguments: r required; s_out optional, 16-byte aligned and
// disjoint from h and r (every CTA of a fused call reads all of h and r).
static q8_status check_residual(const float* h, const float* r, const float* s_out, int64_t rows,
                                int64_t K) {
    if (!r) return Q8_ERR_ARG;
    if (!aligned16(r) || (s_out && !aligned16(s_out))) return Q8_ERR_ALIGN;
    const size_t n = size_t(rows) * size_t(K) * sizeof(float);
    if (overlaps(s_out, h, n) || overlaps(s_out, r, n)) return Q8_ERR_ARG;
    return Q8_OK;
}

// prod: 0 plain, 1 residual, 2 SwiGLU (h: the gate+up output, rows of 2K)
static q8_status act_quant_impl(int mode, int prod, const float* h, const float* res, float* s_out,
                                int64_t rows, int64_t K, int norm, const float* gain, float eps,
                                void* xq, float* xd, void* stream) {
    if (!valid_mode(mode)) return Q8_ERR_MODE;
    if (!h || !xq || (mode != Q8_ACT_F32 && !xd)) return Q8_ERR_ARG;
    if (norm != 0 && norm != 1) return Q8_ERR_ARG;
    if (!(eps >= 0.0f)) return Q8_ERR_ARG;
    q8_status st = check_shape(1, K);
    if (st != Q8_OK) return st;
    if (rows < 1 || rows > Q8_MAX_ROWS) return Q8_ERR_SHAPE;
    if (!aligned16(h) || !aligned16(xq) || (xd && !aligned16(xd)) || (gain && !aligned16(gain)))
        return Q8_ERR_ALIGN;
    LaunchCtx ctx;
    if ((st = make_ctx(stream, ctx)) != Q8_OK) return st;
    return launched(launch_act_quant(mode, prod, h, res, s_out, rows, K, norm, gain, eps, xq, xd, ctx));
}

q8_status act_quant(int mode, const float* h, int64_t rows, int64_t K, int norm,
                    const float* gain, float eps, void* xq, float* xd, void* stream) {
    return act_quant_impl(mode, 0, h, nullptr, nullptr, rows, K, norm, gain, eps, xq, xd, stream);
}

q8_status act_quant_residual(int mode, const float* h, const float* r, float* s_out, int64_t rows,
                             int64_t K, const float* gain, float eps, void* xq, float* xd,
                             void* stream) {
    if (!h) return Q8_ERR_ARG;
    const q8_status st = check_residual(h, r, s_out, rows, K);
    if (st != Q8_OK) return st;
    return act_quant_impl(mode, 1, h, r, s_out, rows, K, 1, gain, eps, xq, xd, stream);
}

q8_status act_quant_swiglu(int mode, const float* gu, int64_t rows, int64_t K, void* xq, float* xd,
                           void* stream) {
    return act_quant_impl(mode, 2, gu, nullptr, nullptr, rows, K, 0, nullptr, 0.0f, xq, xd, stream);
}

q8_status q8_proj(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                  const void* xq, const float* xd, int64_t rows, void* y, int out_f64,
                  void* stream) {
    q8_status st = check_proj_args(mode, q, s, N, K, xq, xd, rows, y);
    if (st != Q8_OK) return st;
    if (out_f64 && mode != Q8_ACT_F32) return Q8_ERR_MODE;
    LaunchCtx ctx;
    if ((st = make_ctx(stream, ctx)) != Q8_OK) return st;
    return project_dispatch(mode, q, s, N, K, xq, xd, rows, y, out_f64 ? 1 : 0, ctx);
}

q8_status q8_proj_chunk(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                        const void* xq, const float* xd, int64_t T, float* y, void* stream) {
    q8_status st = check_proj_args(mode, q, s, N, K, xq, xd, T, y);
    if (st != Q8_OK) return st;
    LaunchCtx ctx;
    if ((st = make_ctx(stream, ctx)) != Q8_OK) return st;
    return project_dispatch(mode, q, s, N, K, xq, xd, T, y, 0, ctx);
}

q8_status q8_debug_chunk_plan(int mode, int64_t N, int64_t K, int64_t T, int argmax, int64_t* out) {
    if (!out) return Q8_ERR_ARG;
    if (!valid_mode(mode)) return Q8_ERR_MODE;
    if (N < 1 || N > (int64_t(1) << 31) || T < 1 || T > Q8_MAX_ROWS || K < 256 || K % 256 != 0 ||
        K > (int64_t(1) << 24))
        return Q8_ERR_SHAPE;
    LaunchCtx ctx;
    q8_status st = make_ctx(nullptr, ctx);
    if (st != Q8_OK) return st;
    return chunk_plan(mode, N, K, T, argmax != 0, ctx, out) ? Q8_OK : Q8_ERR_UNSUPPORTED;
}

size_t q8_proj_fused_workspace(int mode, int64_t rows, int64_t K) {
    if (!valid_mode(mode) || rows < 1 || K < Q8_QK) return 0;
    return round_up(act_bytes(mode, rows, K), 256) + round_up(size_t(rows) * (K / Q8_QK) * 4, 256);
}

static q8_status proj_fused_impl(int mode, int prod, const int8_t* q, const uint16_t* s, int64_t N,
                                 int64_t K, const float* h, const float* res, float* s_out, int64_t rows,
                                 const float* gain, float eps, void* y, int out_f64, void* workspace,
                                 size_t ws_bytes, void* stream, const KvArgs& kv = KvArgs{}) {
    if (!workspace) return Q8_ERR_WORKSPACE;
    // (h stands in for the scales argument: the fused call has none)
    q8_status st = check_proj_args(mode, q, s, N, K, h, h, rows, y);
    if (st != Q8_OK) return st;
    if (out_f64 && mode != Q8_ACT_F32) return Q8_ERR_MODE;
    if (gain && !aligned16(gain)) return Q8_ERR_ALIGN;
    if (!(eps >= 0.0f)) return Q8_ERR_ARG;
    if (!aligned16(workspace)) return Q8_ERR_ALIGN;
    if (ws_bytes < q8_proj_fused_workspace(mode, rows, K)) return Q8_ERR_WORKSPACE;
    LaunchCtx ctx;
    if ((st = make_ctx(stream, ctx)) != Q8_OK) return st;
    if (rows == 1 && K <= kFusedMaxK) {
        // decode step: one launch, the producer runs inside the projection
        GemvArgs a{};
        a.mode = mode;
        a.q = q;
        a.s = s;
        a.N = N;
        a.K = K;
        a.rows = 1;
        a.plane = K;
        a.y = y;
        a.out_f64 = out_f64 ? 1 : 0;
        a.h = h;
        a.prod = prod;
        a.res = res;
        a.s_out = s_out;
        a.gain = gain;
        a.eps = eps;
        a.pos = kv.pos;
        a.kv_col = kv.kv_col;
        a.kv_dim = kv.kv_dim;
        a.n_pos = kv.n_pos;
        a.k_cache = kv.k_cache;
        a.v_cache = kv.v_cache;
        return launched(mode == Q8_ACT_F32 ? launch_gemv_fused_mode0(a, ctx)
                        : mode == Q8_ACT_I8 ? launch_gemv_fused_mode1(a, ctx)
                                            : launch_gemv_fused_mode2(a, ctx));
    }
    unsigned char* act = static_cast<unsigned char*>(workspace);
    float* xd = reinterpret_cast<float*>(act + round_up(act_bytes(mode, rows, K), 256));
    cudaError_t e = launch_act_quant(mode, prod, h, res, s_out, rows, K, prod == 2 ? 0 : 1, gain, eps,
                                     act, xd, ctx);
    if (e != cudaSuccess) return cuda_fail(e);
    if (kv.k_cache) {
        // batches: the projection, then the K/V slices copied into the caches
        const q8_status st2 = project_dispatch(mode, q, s, N, K, act, mode == Q8_ACT_F32 ? nullptr : xd,
                                               rows, y, 0, ctx);
        if (st2 != Q8_OK) return st2;
        return launched(launch_kv_scatter(static_cast<const float*>(y), rows, N, kv.pos, kv.kv_col,
                                          kv.kv_dim, kv.n_pos, kv.k_cache, kv.v_cache, ctx));
    }
    return project_dispatch(mode, q, s, N, K, act, mode == Q8_ACT_F32 ? nullptr : xd, rows, y,
                            out_f64 ? 1 : 0, ctx);
}

q8_status q8_proj_fused(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                        const float* h, int64_t rows, const float* gain, float eps, void* y,
                        int out_f64, void* workspace, size_t ws_bytes, void* stream) {
    return proj_fused_impl(mode, 0, q, s, N, K, h, nullptr, nullptr, rows, gain, eps, y, out_f64,
                           workspace, ws_bytes, stream);
}

q8_status q8_proj_fused_residual(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                                 const float* h, const float* r, float* s_out, int64_t rows,
                                 const float* gain, float eps, void* y, int out_f64,
                                 void* workspace, size_t ws_bytes, void* stream) {
    if (!h) return Q8_ERR_ARG;
    if (rows < 1 || rows > Q8_MAX_ROWS) return Q8_ERR_SHAPE;
    const q8_status st = check_residual(h, r, s_out, rows, K);
    if (st != Q8_OK) return st;
    return proj_fused_impl(mode, 1, q, s, N, K, h, r, s_out, rows, gain, eps, y, out_f64, workspace,
                           ws_bytes, stream);
}

q8_status q8_proj_fused_kv(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                           const float* h, int64_t rows, const float* gain, float eps, void* y,
                           const int32_t* pos, int64_t kv_col, int64_t kv_dim, float* k_cache,
                           float* v_cache, int64_t n_pos, void* workspace, size_t ws_bytes,
                           void* stream) {
    if (!pos || !k_cache || !v_cache) return Q8_ERR_ARG;
    if (rows < 1 || rows > Q8_MAX_ROWS) return Q8_ERR_SHAPE;
    if (kv_dim < 1 || kv_col < 0 || kv_dim > N / 2 || kv_col > N - 2 * kv_dim) return Q8_ERR_SHAPE;
    // positions are int32; a cache of more than 2^40 bytes exceeds any device
    if (n_pos < 1 || n_pos > INT32_MAX || kv_dim > (int64_t(1) << 38) / (rows * n_pos))
        return Q8_ERR_SHAPE;
    if (K > kFusedMaxK) return Q8_ERR_UNSUPPORTED;   // the decode kernel's K
    if (!aligned16(pos) || !aligned16(k_cache) || !aligned16(v_cache)) return Q8_ERR_ALIGN;
    const size_t cache = size_t(rows) * size_t(n_pos) * size_t(kv_dim) * sizeof(float);
    if (overlaps(k_cache, v_cache, cache)) return Q8_ERR_ARG;
    KvArgs kv;
    kv.pos = pos;
    kv.kv_col = kv_col;
    kv.kv_dim = kv_dim;
    kv.n_pos = n_pos;
    kv.k_cache = k_cache;
    kv.v_cache = v_cache;
    return proj_fused_impl(mode, 0, q, s, N, K, h, nullptr, nullptr, rows, gain, eps, y, 0, workspace,
                           ws_bytes, stream, kv);
}

q8_status q8_proj_fused_swiglu(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                               const float* gu, int64_t rows, void* y, int out_f64, void* workspace,
                               size_t ws_bytes, void* stream) {
    return proj_fused_impl(mode, 2, q, s, N, K, gu, nullptr, nullptr, rows, nullptr, 0.0f, y, out_f64,
                           workspace, ws_bytes, stream);
}

size_t head_argmax_workspace(int64_t rows) {
    if (rows < 1) return 0;
    const int64_t g = rows < kArgmaxGroupRows ? rows : kArgmaxGroupRows;
    return kArgmaxGemvOff + kArgmaxHeader + size_t(kMaxGrid) * size_t(g) * sizeof(ArgmaxCand);
}

q8_status head_argmax(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                      const void* xq, const float* xd, int64_t rows, int32_t* tok,
                      double* maxval, void* logits, void* workspace, size_t ws_bytes,
                      void* stream) {
    if (!valid_mode(mode)) return Q8_ERR_MODE;
    if (!q || !s || !xq || !tok || (mode != Q8_ACT_F32 && !xd)) return Q8_ERR_ARG;
    q8_status st = check_shape(N, K);
    if (st != Q8_OK) return st;
    if (rows < 1 || rows > Q8_MAX_ROWS) return Q8_ERR_SHAPE;
    if (!workspace || ws_bytes < head_argmax_workspace(rows)) return Q8_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(s) || !aligned16(xq) || (xd && !aligned16(xd)) ||
        !aligned16(workspace) || (logits && !aligned16(logits)) ||
        (reinterpret_cast<uintptr_t>(tok) & 3u) || (reinterpret_cast<uintptr_t>(maxval) & 7u))
        return Q8_ERR_ALIGN;
    LaunchCtx ctx;
    if ((st = make_ctx(stream, ctx)) != Q8_OK) return st;
    static_assert(kArgmaxKeyBytes >= 8 * Q8_MAX_ROWS, "one arg-max key per row");
    // the tensor-core path from chunk_min_head_rows(mode) rows; in f32 mode up to
    // kArgmaxGroupRows rows and kMaxGrid tiles (its candidates use the
    // CUDA-core layout of the workspace)
    const bool f32_fits = mode != Q8_ACT_F32 || (rows <= kArgmaxGroupRows && (N + 127) / 128 <= kMaxGrid);
    // (f32 row pairs, where they fit, beat the tensor cores up to 7 rows)
    const int64_t min_rows =
        (mode == Q8_ACT_F32 && gemv_group_rows(mode, K) == 2) ? 8 : chunk_min_head_rows(mode);
    if (f32_fits && rows >= min_rows && chunk_supported(mode, N, K, rows))
        return launched(launch_chunk_argmax(mode, q, s, N, K, xq, xd, rows, logits, tok, maxval, workspace,
                                            ctx));
    return run_projection(mode, q, s, N, K, xq, xd, rows, logits, mode == Q8_ACT_F32 ? 1 : 0, tok,
                          maxval, static_cast<unsigned char*>(workspace) + kArgmaxGemvOff, ctx);
}

q8_status q8_debug_block_dots(int mode, const int8_t* q, const void* xq, int64_t N, int64_t K,
                              int64_t rows, int32_t* isum, int path, void* stream) {
    if (mode != Q8_ACT_I8 && mode != Q8_ACT_I8X2) return Q8_ERR_MODE;
    if (!q || !xq || !isum) return Q8_ERR_ARG;
    q8_status st = check_shape(N, K);
    if (st != Q8_OK) return st;
    if (rows < 1 || rows > Q8_MAX_ROWS) return Q8_ERR_SHAPE;
    if (rows * N * (K / Q8_QK) > (int64_t(1) << 26)) return Q8_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(xq) || !aligned16(isum)) return Q8_ERR_ALIGN;
    if (path != 0 && path != 1) return Q8_ERR_ARG;
    LaunchCtx ctx;
    if ((st = make_ctx(stream, ctx)) != Q8_OK) return st;
    if (path == 1) {
        if (!chunk_supported(mode, N, K, rows)) return Q8_ERR_UNSUPPORTED;
        return launched(launch_chunk_debug(mode, q, N, K, xq, rows, isum, ctx));
    }
    return launched(launch_debug_dots(mode, q, xq, N, K, rows, isum, ctx));
}

}  // extern "C"

/*
 * q8proj.h -- C ABI of the Q8_0 quantized-projection library (libq8proj.so),
 * written for one NVIDIA GB300 (sm_103a).
 *
 * What it computes.  The compiled generation lane of logicaffeine_compile
 * (codegen_cuda::lane, module description) reads every quantized projection
 * "as rows read in place from the checkpoint", stored as a Q8_0 pair of files
 * <var>.q / <var>.s (model::author, module description: "Q8_0 quants and
 * block scales").  Its CudaKnobs pick the projection numerics: f32
 * activations with f64 sums, a two-word ~14-bit int8 activation (the
 * default), or llama.cpp's one int8 word; fuse_quant quantizes the
 * activation in its producer.  A step has rows = 1 (decode), rows = B (a
 * batch, every weight read once for all sequences) or T rows (a prefill
 * chunk, every projection reading its weights once for the block), and ends
 * with the arg-max of the logits (model::author, decode_step / decode_head).
 *
 * Layouts (all row-major, planar, dense pitch):
 *   Q   int8   [N][K]      weight quants, the ".q" file
 *   S   uint16 [N][K/32]   binary16 bit patterns of the block scales, ".s"
 *   activations, by mode:
 *     Q8_ACT_F32   float  [rows][K]                    (xd unused, may be NULL)
 *     Q8_ACT_I8    int8   [rows][K]  + xd float [rows][K/32]
 *     Q8_ACT_I8X2  int8   [2][rows][K] (hi plane, then lo plane)
 *                                     + xd float [rows][K/32]
 *   outputs: float [rows][N], or double [rows][N] for Q8_ACT_F32 with out_f64.
 *
 * Numerics (the pages name these modes but give no formulas; the readings):
 *   block of 32 values along K; weight scale s = binary16(amax/127) and
 *   q = round_half_away(w / s) in [-127, 127];
 *   one-word activation: d = amax/127 (f32), q = round_half_away(x/d);
 *   two-word activation: d = amax/8191 (f32), Q = round_half_away(x/d) in
 *   [-8191, 8191], lo = ((Q + 64) mod 128) - 64, hi = (Q - lo) / 128;
 *   projection (one/two-word): y = sum_b float(isum_b) * (s_b * d_b), where
 *   isum_b is the exact int32 dot of block b (two-word: 128*dot(hi)+dot(lo));
 *   projection (f32): y = sum_k (s_b * q_k) * x_k, summed to f64 accuracy;
 *   RMSNorm producer: r = 1/sqrt(sum h^2 / K + eps) with the sum in f64,
 *   x = (h * float(r)) * g.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller unless stated.  The
 *     library allocates no device memory; scratch comes from caller-sized
 *     workspaces.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Argument errors are found on the host and returned
 *     before anything is launched.
 *   - Every pointer must be 16-byte aligned; K must be a multiple of 32;
 *     N, rows >= 1.  Violations return Q8_ERR_ALIGN / Q8_ERR_SHAPE.
 *   - A failed launch returns Q8_ERR_CUDA; q8_last_cuda_error() gives the
 *     CUDA error number.  The library never exits, aborts or traps.
 *   - Each call runs on the calling thread's current device (cudaSetDevice).
 *     One process may use several devices (up to 64) and call from several
 *     threads: the per-device state (SM count, device error word, kernel
 *     attributes) is set up once per device under a lock or atomically.
 *   - Device-side waits are bounded.  A wait that runs out records a code
 *     that q8_device_error() reports; the kernel then returns early and its
 *     outputs are undefined.
 *   - By default consecutive launches use programmatic dependent launch: a
 *     projection may start streaming its WEIGHTS before the preceding kernel
 *     on the stream has finished (activations, outputs and workspaces are
 *     only touched after it has).  So the kernel launched just before a
 *     projection must not write that projection's Q or S; synchronise the
 *     stream (or q8_set_pdl(0)) after writing weights.
 */
#ifndef Q8PROJ_H
#define Q8PROJ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    Q8_OK = 0,
    Q8_ERR_ARG = 1,          /* null pointer, bad flag or bad value */
    Q8_ERR_SHAPE = 2,        /* K % 32 != 0, N or rows out of range */
    Q8_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned */
    Q8_ERR_MODE = 4,         /* activation mode not valid for this call */
    Q8_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed */
    Q8_ERR_UNSUPPORTED = 6,  /* valid request this build does not serve */
    Q8_ERR_WORKSPACE = 7     /* workspace missing or too small */
} q8_status;

typedef enum {
    Q8_ACT_F32 = 0,   /* f32 activations, f64 sums */
    Q8_ACT_I8 = 1,    /* one int8 word per value (llama.cpp style) */
    Q8_ACT_I8X2 = 2   /* two-word ~14-bit int8 code (the lane's default) */
} q8_act_mode;

/* Largest activation row count one call accepts (decode batch or prefill chunk). */
#define Q8_MAX_ROWS 256

/* Name of a status code; never NULL. */
const char* q8_status_str(int status);

/* Library ABI version (major * 100 + minor). */
int q8_version(void);

/* The CUDA error number behind the last Q8_ERR_CUDA returned on this thread. */
int q8_last_cuda_error(void);

/*
 * Synchronises `stream`, then reads and clears the device error word of the
 * current device: 0 = none, 1 = a bounded wait ran out, 2 = a KV-cache
 * position outside its cache (q8_proj_fused_kv).  *code receives it.
 */
q8_status q8_device_error(int32_t* code /* host */, void* stream);

/* Programmatic dependent launch on (1, default) or off (0) for this process. */
void q8_set_pdl(int enable);

/*
 * Q8_0 pack (model::author, module description: <var>.q / <var>.s).
 *   w  float [N][K] -> q int8 [N][K], s uint16 [N][K/32] (binary16 bits).
 * Per 32-value block: s = binary16(amax/127), q = round_half_away(w/s)
 * clamped to [-127, 127] (q = 0 where s == 0).  overflow (device int32,
 * nullable) is incremented by the number of blocks whose scale overflowed
 * binary16 (their q are 0); the caller zeroes it.
 */
q8_status q8_pack(const float* w, int64_t N, int64_t K, int8_t* q, uint16_t* s,
                  int32_t* overflow, void* stream);

/*
 * Activation producer (codegen_cuda::lane, CudaKnobs fuse_quant; "Modules:
 * kernels", an activation quantized in a producer's epilogue, a norm).
 *   h     float [rows][K] hidden state
 *   norm  0: quantize h as given; 1: RMSNorm first, x = (h * r) * gain
 *   gain  float [K] or NULL (gain of one); eps the RMSNorm epsilon
 *   xq    output in the mode's activation layout (see top of file)
 *   xd    float [rows][K/32] block scales (ignored for Q8_ACT_F32)
 * rows <= Q8_MAX_ROWS.
 */
q8_status act_quant(int mode, const float* h, int64_t rows, int64_t K, int norm,
                    const float* gain, float eps, void* xq, float* xd, void* stream);

/*
 * The producer with a residual added before the norm (codegen_cuda::lane,
 * "Modules: kernels": a residual added before a norm).
 *   s = h + r per value (one f32 rounding) is the producer's input: RMSNorm
 *   of s, x = (s * rs) * gain, then the mode's quantisation, exactly as
 *   act_quant with norm = 1 applied to s.
 *   r      float [rows][K], required
 *   s_out  float [rows][K] or NULL: receives s (the updated residual stream);
 *          it must not overlap h or r (Q8_ERR_ARG)
 */
q8_status act_quant_residual(int mode, const float* h, const float* r, float* s_out, int64_t rows,
                             int64_t K, const float* gain, float eps, void* xq, float* xd,
                             void* stream);

/*
 * The SwiGLU producer of the down projection (codegen_cuda::lane, "Modules:
 * kernels": an activation quantized in its producer's epilogue; the FFN's gate
 * and up projections run as one fused matrix).
 *   gu  float [rows][2K]: each row the fused gate+up output, gate first
 *       (gu[m][0..K)), then up (gu[m][K..2K))
 *   x = silu(gate) * up, silu(g) = g / (1 + e^-g), every step one binary32
 *   rounding with e^x computed by a fixed method (Cody-Waite reduction, the
 *   degree-7 Taylor series), then the mode's quantisation (no norm); the
 *   rest as act_quant.
 */
q8_status act_quant_swiglu(int mode, const float* gu, int64_t rows, int64_t K, void* xq, float* xd,
                           void* stream);

/*
 * Quantized projection of a stacked activation (codegen_cuda::lane: the
 * decode step, rows = 1, and a batch's step, rows = B, with each weight read
 * once for a group of rows: up to 8 rows (one-word) or 4 (two-word) a pass,
 * with a weight row per lane when K % 1024 == 0 (f32: one row up to 16384
 * values, or two up to 8192); from 9 (one-word), 5 (two-word) or 4 (f32) rows
 * with K % 256 == 0 one pass on the tensor cores, except f32 at 4 rows where
 * two row pairs fit; f32 below 4 rows otherwise runs one row a pass, its
 * arithmetic being the bound).
 *   y[m][n] for m < rows, n < N; y is float, or double when mode is
 *   Q8_ACT_F32 and out_f64 != 0.  1 <= rows <= Q8_MAX_ROWS.
 */
q8_status q8_proj(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                  const void* xq, const float* xd, int64_t rows, void* y, int out_f64,
                  void* stream);

/*
 * Prefill-chunk projection (codegen_cuda::lane: author::prefill's chunks of
 * 2, 4, ... rows, every projection reading its weights once for the block).
 * Same contract as q8_proj with rows = T (1 <= T <= Q8_MAX_ROWS) and a float
 * output; large chunks run on the tensor cores.
 */
q8_status q8_proj_chunk(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                        const void* xq, const float* xd, int64_t T, float* y, void* stream);

/*
 * Producer fused with the projection (CudaKnobs fuse_quant): RMSNorm of h
 * (gain nullable) quantized in the producer's epilogue, then the projection.
 * workspace holds the quantized activation; its size is
 * q8_proj_fused_workspace(mode, rows, K) bytes, 16-byte aligned.
 */
q8_status q8_proj_fused(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                        const float* h, int64_t rows, const float* gain, float eps, void* y,
                        int out_f64, void* workspace, size_t ws_bytes, void* stream);
size_t q8_proj_fused_workspace(int mode, int64_t rows, int64_t K);

/*
 * q8_proj_fused with the K/V slices of a fused QKV projection also written
 * into the row of a cache that a position names (codegen_cuda::lane, "Modules:
 * kernels": a result written into the row of a cache a position names).
 *   y        float [rows][N]: the whole projection output, as q8_proj_fused
 *   pos      int32 [rows], device memory: row m's position (read by the
 *            launch, so one captured graph serves every step)
 *   kv_col   first column of the K slice: K = columns [kv_col, kv_col + kv_dim),
 *            V = [kv_col + kv_dim, kv_col + 2 kv_dim); kv_col + 2 kv_dim <= N
 *   k_cache, v_cache  float [rows][n_pos][kv_dim], one cache per row's
 *            sequence, disjoint; row m's slices go to cache row pos[m];
 *            1 <= n_pos <= 2^31 - 1 and each cache at most 2^40 bytes
 *            (Q8_ERR_SHAPE otherwise)
 * K <= 16384.  A position outside [0, n_pos) writes no cache entry of its row
 * and sets device error 2 (q8_device_error); y is written either way.
 */
q8_status q8_proj_fused_kv(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                           const float* h, int64_t rows, const float* gain, float eps, void* y,
                           const int32_t* pos, int64_t kv_col, int64_t kv_dim, float* k_cache,
                           float* v_cache, int64_t n_pos, void* workspace, size_t ws_bytes,
                           void* stream);

/*
 * q8_proj_fused with the residual added before the norm: the producer's
 * input is s = h + r (see act_quant_residual), written to s_out when it is
 * not NULL (s_out must not overlap h or r: every block of the decode launch
 * reads all of h and r).  Same workspace as q8_proj_fused.
 */
q8_status q8_proj_fused_residual(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                                 const float* h, const float* r, float* s_out, int64_t rows,
                                 const float* gain, float eps, void* y, int out_f64,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * The down projection with its SwiGLU producer fused (act_quant_swiglu, then
 * the projection; one launch at rows = 1): q [N][K], gu [rows][2K].  Same
 * workspace as q8_proj_fused.
 */
q8_status q8_proj_fused_swiglu(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                               const float* gu, int64_t rows, void* y, int out_f64, void* workspace,
                               size_t ws_bytes, void* stream);

/*
 * LM head fused with its arg-max (model::author, decode_head: "the final
 * norm, the LM head and the arg-max"; decode_batch_head: one token per
 * sequence).  Modes Q8_ACT_F32 (logits to f64 accuracy) and Q8_ACT_I8 /
 * Q8_ACT_I8X2 (f32 logits).  From 9 (one-word), 5 (two-word) or 6 (f32, up
 * to 16 rows and N <= 131072; 8 where f32 row pairs fit, K % 1024 == 0 and
 * K <= 8192) rows on, with K % 256 == 0, the head is read
 * once for all rows on the tensor cores; below that, once per group of up to
 * 8 (one-word) or 4 (two-word) rows (with a weight row per lane when
 * K % 1024 == 0), and f32 once per row pair (K % 1024 == 0, K <= 8192) or row.
 *   tok     int32 [rows]: the smallest n holding the row's maximum logit; NaN
 *           logits are never the maximum, and a row of NaN gives 0
 *   maxval  double [rows] or NULL: that maximum (NaN for a row of NaN)
 *   logits  float [rows][N] (double for Q8_ACT_F32) or NULL
 *   workspace: head_argmax_workspace(rows) bytes, zeroed whole before the
 *   first call on it; every completed call leaves the counters and keys it
 *   uses zero again.  Calls sharing a workspace must not overlap.
 */
q8_status head_argmax(int mode, const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                      const void* xq, const float* xd, int64_t rows, int32_t* tok,
                      double* maxval, void* logits, void* workspace, size_t ws_bytes,
                      void* stream);
size_t head_argmax_workspace(int64_t rows);

/*
 * head_argmax without a workspace, for callers that cannot allocate device
 * memory: code that runs where a framework's allocator owns all device memory
 * (raw cudaMalloc is forbidden or would fragment its pool), or a serving loop
 * that must not allocate once it is running.  The pages describing the method
 * have no counterpart to this call; it exists only for those callers.
 *   Same arguments and results as head_argmax, minus the workspace.  The
 *   scratch is a fixed device array inside the library,
 *   head_argmax_noalloc_scratch_bytes() bytes (about 256 KB), which every GPU
 *   that loads the library keeps until the process exits; it covers every
 *   rows <= Q8_MAX_ROWS, and larger rows return Q8_ERR_SHAPE.
 *   The first call on a device (with that device current) looks up the
 *   array's device address, so make that first call before any stream
 *   capture.  Each call clears the array's counter on `stream` first.  All
 *   calls share the one array: calls that overlap on the GPU race and give
 *   undefined results.  No allocation happens in any call.
 */
q8_status head_argmax_noalloc(int mode, const int8_t* q, const uint16_t* s, int64_t N,
                              int64_t K, const void* xq, const float* xd, int64_t rows,
                              int32_t* tok, double* maxval, void* logits, void* stream);
size_t head_argmax_noalloc_scratch_bytes(void);

/*
 * Debug: the per-block int32 dot products the projections fold with their
 * scales (modes Q8_ACT_I8 / Q8_ACT_I8X2), isum int32 [rows][N][K/32].
 * path 0 runs the CUDA-core inner product the GEMV kernels use, path 1 the
 * tensor-core chunk kernel's per-block accumulators.  Small shapes only:
 * rows * N * K/32 <= 2^26.
 */
q8_status q8_debug_block_dots(int mode, const int8_t* q, const void* xq, int64_t N, int64_t K,
                              int64_t rows, int32_t* isum, int path, void* stream);

/*
 * Debug, host only (no device work, no CUDA call): the stage geometry the
 * decode kernel (rows <= 8 one-word, <= 4 two-word, 1 f32) uses for CTA `cta`
 * of a grid of `grid` CTAs (the library launches min(SM count, N) of them).
 * That kernel serves the LM head's arg-max and the projections whose K is not
 * a multiple of 1024 (f32: or above 16384); the others of those row counts
 * run the row-per-lane kernel, whose geometry is fixed (a lane per weight
 * row, 32-row groups, whole groups per CTA, stages of 1024 values).
 * out (host, 21 int64) receives: R (activation rows the kernel is built for),
 * KS (bytes of K a slice), nks (slices a row), PB (bytes a part), npr (parts a
 * slice, a power of two), nprr (parts holding data), RS (rows a stage), rpw
 * (rows a warp serves per stage), items (RS*npr/rpw), stride (warp groups,
 * 16/items), stage_bytes, nstages, r0, r1 (the CTA's rows [r0, r1)), sbrows
 * (rows a super-block), ep_off, ring bytes, part-sum bytes, part-sum bytes a
 * row-part, CPL (16-byte chunks a lane), consumer warps.  Returns
 * Q8_ERR_UNSUPPORTED when the projection would use its slice-major kernel.
 */
q8_status q8_debug_row_geometry(int mode, int64_t rows, int64_t N, int64_t K, int grid, int cta,
                                int64_t* out);

/*
 * Debug, host only: the same 21 fields for the decode launch of a fused call
 * at rows = 1 and K <= 16384 values, by its producer: prod 0 q8_proj_fused
 * (and its KV-row form), 1 q8_proj_fused_residual, 2 q8_proj_fused_swiglu.
 * (Fused calls whose K is a multiple of 1024 run the row-per-lane kernel
 * instead, as the plain projections do.)
 * The int8 modes and the plain producer run the rows = 1 geometry above.  In
 * f32 mode the residual and SwiGLU producers above 4096 values shorten the
 * ring (field 16): the converted activation (128 bytes a 32-value block, 4K
 * bytes rounded up to 1 KB) stays in shared memory after it for the whole
 * launch.  Errors as q8_debug_row_geometry (prod outside 0..2: Q8_ERR_ARG);
 * Q8_ERR_UNSUPPORTED above 16384 values.
 */
q8_status q8_debug_row_geometry_fused(int mode, int prod, int64_t N, int64_t K, int grid,
                                      int cta, int64_t* out);

/*
 * Debug, host side (the current device's occupancy is queried; nothing is
 * launched): the plan of the tensor-core path for a projection of T rows
 * (argmax = 0: q8_proj_chunk and q8_proj from 9 one-word / 5 two-word / 4
 * f32 rows; argmax = 1: head_argmax).  out (host, 6 int64) receives: TT
 * (activation rows a tile), ks (CTAs of a cluster, each over 1/ks of K),
 * tiles (128 x TT, one cluster each), clusters that fit on the device at
 * once, waves, pipeline stages.  Any activation mode, K % 256 == 0,
 * 1 <= T <= Q8_MAX_ROWS; otherwise Q8_ERR_MODE / Q8_ERR_SHAPE.
 */
q8_status q8_debug_chunk_plan(int mode, int64_t N, int64_t K, int64_t T, int argmax, int64_t* out);

#ifdef __cplusplus
}
#endif

#endif /* Q8PROJ_H */

/*
 * qk.h -- C ABI of libqk: quantize-once activation images for GB300 (sm_103a).
 *
 * An F32 activation is quantised once into a 32-element-block Q8 "image" by
 * the kernel that produces it (an RMSNorm or a GLU), and that one image is
 * then read by every quantised-weight projection that consumes the
 * activation: q/k/v or gate/up, ordinary (MUL_MAT) or routed per expert
 * (MUL_MAT_ID).
 *
 * Sources (page titles and sections):
 *   llama.cpp PR #117 "activation image emission" -- Overview and Coverage:
 *     the shared Q8_1 image, RMS/GLU producers that emit it beside their
 *     original F32 output, ordinary and routed MMVQ readers.
 *   minfer doc 52 "r49 A-quantize prepass shared-A dedup" -- sections 1-3:
 *     the prefill Q8_0 prepass read by the MMQ GEMMs, once per distinct A;
 *     out-of-pool scratch; errors surfaced at entry, before any launch.
 *   TensorFold PR #1047 "padding rows no longer go through routed experts"
 *     -- "The fix": a device-side live-row count read by every kernel at
 *     each graph replay, launches sized for the bucket, stable grouped plan.
 *
 * Conventions (every call):
 *   - Pointers named x, w, img, y, ids ... are DEVICE pointers owned by the
 *     caller; the library never frees or keeps them after the call.
 *   - The library allocates no memory and never synchronises; each call
 *     validates its arguments on the host, then enqueues its kernel(s) on
 *     `stream` (NULL = the legacy default stream) and returns.
 *   - Kernels are launched with programmatic stream serialization: a kernel
 *     of this library may start while the library kernel before it on the
 *     stream is finishing, and waits for it before reading anything it may
 *     have written. The projection kernels may begin streaming their packed
 *     weights early, so packed weights must not be written by the library
 *     kernel enqueued immediately before a projection that reads them
 *     (qk_weight_pack itself always completes first).
 *   - On an invalid argument nothing is launched and a status other than
 *     QK_OK is returned; qk_last_error() gives a one-line reason (per host
 *     thread).
 *   - d_live_rows: optional DEVICE pointer to one int32, the number of live
 *     rows. Kernels read it on the device at every launch or graph replay;
 *     rows at or past it (clamped to [0, rows]) are not read for work and
 *     their outputs are not written. NULL means every row is live. Grids are
 *     always sized for `rows`, so a captured CUDA graph stays valid while the
 *     count changes between replays.
 *   - A row count of 0, where a call accepts it (the producers' T, the
 *     routing calls' rows), enqueues nothing and writes nothing, except
 *     qk_moe_plan and qk_route_plan, which write the zero counts and offsets
 *     of an empty plan. The projections take T (rows) >= 1.
 *   - Results depend only on the input bytes and shape arguments (no state
 *     kept between calls, no cross-call caching; an image is rebuilt on every
 *     call and replay).
 *   - Strides are in elements of the pointed-to type unless named *_blocks.
 */
#ifndef QK_H
#define QK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QK_API __attribute__((visibility("default")))
#else
#define QK_API
#endif

struct CUstream_st;
typedef struct CUstream_st *qk_stream; /* a cudaStream_t */

typedef enum qk_status {
    QK_OK = 0,
    QK_ERR_ARG = 1,         /* null pointer, negative size or bad enum */
    QK_ERR_SHAPE = 2,       /* a width that must be whole 32-blocks is not, or a stride too small */
    QK_ERR_ALIAS = 3,       /* an output overlaps an input or another output */
    QK_ERR_WORKSPACE = 4,   /* a packed buffer or workspace is too small */
    QK_ERR_UNSUPPORTED = 5, /* a size outside what the kernel supports (e.g. T > 8) */
    QK_ERR_CUDA = 6         /* a CUDA launch failed; see qk_last_error() */
} qk_status;

typedef enum qk_norm_kind {
    QK_NORM_PLAIN = 0,   /* y = x * r               */
    QK_NORM_MUL = 1,     /* y = (x * r) * w          */
    QK_NORM_MUL_ADD = 2, /* y = (x * r) * w + b      */
    QK_NORM_SCALE = 3    /* y = (x * r) * scale      */
} qk_norm_kind;

typedef enum qk_glu_kind {
    QK_GLU_SWIGLU = 0,     /* out = g * sigmoid(g) * u */
    QK_GLU_GEGLU_TANH = 1, /* out = 0.5 g (1 + tanh(sqrt(2/pi)(g + 0.044715 g^3))) * u */
    QK_GLU_REGLU = 2,      /* out = max(g, 0) * u */
    QK_GLU_GEGLU_ERF = 3,  /* out = 0.5 g (1 + erf(g / sqrt 2)) * u   (exact GELU) */
    QK_GLU_GEGLU_QUICK = 4,/* out = g * sigmoid(1.702 g) * u          (sigmoid GELU) */
    QK_GLU_SWIGLU_OAI = 5, /* x = min(g, limit), v = clamp(u, -limit, limit):
                              out = x * sigmoid(alpha x) * (v + 1)     */
    QK_GLU_SWIGLU_CLAMP = 6/* x = min(g, limit), v = clamp(u, -limit, limit):
                              out = x * sigmoid(x) * v  (a reading: the
                              pages give no formula)                   */
} qk_glu_kind;

typedef enum qk_glu_layout {
    QK_GLU_SEPARATE = 0,      /* g rows at a (a_stride), u rows at b (b_stride) */
    QK_GLU_PACKED = 1,        /* row of a = [g (N) | u (N)]; b unused          */
    QK_GLU_PACKED_SWAPPED = 2 /* row of a = [u (N) | g (N)]; b unused          */
} qk_glu_layout;

typedef enum qk_wtype {
    QK_W_Q4_0 = 0, /* 18-byte blocks: half d, 16 nibble bytes; value (nibble - 8) * d */
    QK_W_Q8_0 = 1  /* 34-byte blocks: half d, 32 int8; value q * d                    */
} qk_wtype;

/* ------------------------------------------------------------------ misc */

/* Short name of a status code (static string). */
QK_API const char *qk_status_string(qk_status s);

/* One-line reason for the last non-QK_OK status returned on this host thread. */
QK_API const char *qk_last_error(void);

/* The same string as qk_last_error (the name used by the boundary's first sketch). */
QK_API const char *qk_last_error_string(void);

/* Number of kernels this library has launched in this process (all threads). */
QK_API uint64_t qk_launch_count(void);

/*
 * Device-side fault word of the current device, then cleared. Bit 0: a
 * kernel's bounded wait on a shared-memory barrier gave up (the kernel then
 * stopped early and its outputs are not valid). Covers qk_mmvq, qk_mmvq_id
 * and qk_mmq. Bit 1: a routed projection's counts held more passes than any
 * plan of its bucket can (not the output of qk_moe_plan); it did no work.
 * Synchronises the device.
 */
QK_API qk_status qk_device_faults(uint32_t *faults);

/*
 * Failure-path self-test: launches one CTA whose bounded wait on a
 * shared-memory barrier that nothing completes runs out (about a second at
 * most), sets bit 0 of the fault word and returns. The device stays usable;
 * read the word with qk_device_faults. For tests of the timeout path.
 */
QK_API qk_status qk_selftest_wait_timeout(qk_stream stream);

/* ------------------------------------------------------------ the image */

/*
 * Q8_1 activation image (llama.cpp PR #117, Coverage: the "standard Q8_1
 * activation image" read by every MMVQ weight format).
 *
 * Layout: img[t] is a row of img_row_blocks blocks of 36 bytes, rows back to
 * back (row stride 36 * img_row_blocks bytes). Block b of row t covers
 * activation columns 32b .. 32b+31:
 *   bytes 0-1  d  = half(amax / 127), amax = max |x| over the block, binary32
 *   bytes 2-3  s  = half(d * sum(q)), product in binary32
 *   bytes 4-35 q_i = rint(x_i / d) in binary32, ties to even, int8 in [-127, 127]
 * An all-zero block has d = s = 0 and q = 0. Columns past K inside the last
 * block are taken as 0; blocks ceil(K/32) .. img_row_blocks-1 are written as
 * 36 zero bytes. Halves are IEEE binary16, round to nearest even, little
 * endian.
 */
#define QK_Q8_1_BLOCK_BYTES 36

/*
 * qk_quantize_q8_1 -- standalone quantiser (the separate launch that producer
 * emission replaces; kept for unfused use and as the fused kernels' control).
 *   x        [T][x_stride] F32, columns 0..K-1 read
 *   img      [T][img_row_blocks] Q8_1 blocks, img_row_blocks >= ceil(K/32)
 * Errors: QK_ERR_ARG (null, T < 0, K < 1 or K > 2^25, img_row_blocks > 2^20),
 * QK_ERR_SHAPE (x_stride < K, img_row_blocks < ceil(K/32)), QK_ERR_ALIAS (img
 * overlaps x).
 */
QK_API qk_status qk_quantize_q8_1(const float *x, int64_t T, int64_t K, int64_t x_stride,
                           void *img, int64_t img_row_blocks,
                           const int32_t *d_live_rows, qk_stream stream);

/*
 * qk_quantize_q8_0 -- the prefill prepass (minfer doc 52, section 1: per
 * 32-block amax, rintf scaling, zero pad). Same d and codes as the Q8_1
 * image, no s, stored as two planes so tensor-core tiles load rows directly:
 *   qs  [T][row_blocks * 32] int8 codes
 *   d   [T][row_blocks]      binary16 bits (uint16)
 * Blocks ceil(K/32) .. row_blocks-1 are zero. Errors as qk_quantize_q8_1.
 */
QK_API qk_status qk_quantize_q8_0(const float *x, int64_t T, int64_t K, int64_t x_stride,
                           int8_t *qs, uint16_t *d, int64_t row_blocks,
                           const int32_t *d_live_rows, qk_stream stream);

/* ------------------------------------------------------- the producers */

/*
 * qk_rmsnorm_q8_1 -- RMS producer that emits the image (llama.cpp PR #117,
 * Coverage: RMS-alone, RMS+MUL, RMS+MUL+ADD and RMS+SCALE producers emit
 * images while keeping their original F32 output).
 *   r = 1 / sqrt(sum(x^2)/K + eps) per row (binary32 arithmetic)
 *   y = x*r, (x*r)*w, (x*r)*w + b, or (x*r)*scale  by `kind`
 *   y   [T][y_stride] F32, written for live rows, columns 0..K-1
 *   img the Q8_1 image of exactly the stored y values (bit-identical to
 *       qk_quantize_q8_1 applied to y)
 *   w, b: [K] F32, required by MUL / MUL_ADD (b only by MUL_ADD), else ignored
 * Errors: QK_ERR_ARG, QK_ERR_SHAPE (K % 32 != 0: the producer's width must be
 * whole Q8_1 blocks; strides too small), QK_ERR_UNSUPPORTED (K > 32768),
 * QK_ERR_ALIAS (y or img overlapping x, w, b or each other).
 */
QK_API qk_status qk_rmsnorm_q8_1(const float *x, int64_t T, int64_t K, int64_t x_stride,
                          qk_norm_kind kind, const float *w, const float *b,
                          float scale, float eps,
                          float *y, int64_t y_stride, void *img, int64_t img_row_blocks,
                          const int32_t *d_live_rows, qk_stream stream);

/*
 * qk_rmsnorm_q8_0 -- the same RMS producer emitting the prefill Q8_0 planes
 * that qk_mmq reads (minfer doc 52, "r51" fused RMSNorm -> Q8_0 producer: the
 * separate quantize pass and its re-read of y go away).
 *   y   as qk_rmsnorm_q8_1
 *   qs  [T][row_blocks*32] int8 codes, 16-byte aligned; d [T][row_blocks] half
 *       scales: bit-identical to qk_quantize_q8_0 applied to the stored y
 *       (blocks from K/32 up to row_blocks are zero)
 * Errors: as qk_rmsnorm_q8_1.
 */
QK_API qk_status qk_rmsnorm_q8_0(const float *x, int64_t T, int64_t K, int64_t x_stride,
                                 qk_norm_kind kind, const float *w, const float *b,
                                 float scale, float eps, float *y, int64_t y_stride,
                                 int8_t *qs, uint16_t *d, int64_t row_blocks,
                                 const int32_t *d_live_rows, qk_stream stream);

/*
 * qk_glu_q8_1 -- GLU producer that emits the image (llama.cpp PR #117,
 * Coverage: F32 ReGLU, GeGLU, SwiGLU, GeGLU-erf, GeGLU-quick, SwiGLU-OAI and
 * SwiGLU-clamp with separate, packed and packed-swapped inputs and independent
 * source row strides; output width whole Q8_1 blocks).
 *   out [T][out_stride] F32 = act(g) * u for live rows, columns 0..N-1
 *   img the Q8_1 image of exactly the stored out values
 *   SEPARATE: g = a + t*a_stride, u = b + t*b_stride
 *   PACKED: g = a + t*a_stride, u = g + N;  PACKED_SWAPPED: u = a + t*a_stride, g = u + N
 * Errors: QK_ERR_ARG (N > 2^25), QK_ERR_SHAPE (N % 32 != 0, strides too small),
 * QK_ERR_ALIAS (out or img overlapping the inputs or each other).
 */
QK_API qk_status qk_glu_q8_1(qk_glu_kind kind, qk_glu_layout layout,
                      const float *a, int64_t a_stride, const float *b, int64_t b_stride,
                      int64_t T, int64_t N,
                      float *out, int64_t out_stride, void *img, int64_t img_row_blocks,
                      const int32_t *d_live_rows, qk_stream stream);

/*
 * qk_glu_q8_1_ex -- qk_glu_q8_1 with the SwiGLU-OAI parameters (llama.cpp PR
 * #117, Coverage: the GLU producers keep their alpha/limit parameters).
 * alpha is read by QK_GLU_SWIGLU_OAI, limit by it and QK_GLU_SWIGLU_CLAMP;
 * qk_glu_q8_1 passes alpha = 1.702, limit = 7.0. Errors: as qk_glu_q8_1, and QK_ERR_ARG for a
 * non-finite alpha or a limit that is not a positive finite number.
 */
QK_API qk_status qk_glu_q8_1_ex(qk_glu_kind kind, qk_glu_layout layout,
                                const float *a, int64_t a_stride, const float *b, int64_t b_stride,
                                int64_t T, int64_t N,
                                float *out, int64_t out_stride, void *img, int64_t img_row_blocks,
                                float alpha, float limit, const int32_t *d_live_rows, qk_stream stream);

/* ------------------------------------------------------------- weights */

/*
 * Weights arrive as canonical row-major blocks ([N][K/32] blocks of
 * QK_W_Q4_0 or QK_W_Q8_0 bytes; Q4_0 element j < 16 is the low nibble of byte
 * j, element j+16 its high nibble). qk_weight_pack rearranges them once into
 * the device layout the projection kernels stream with 128-bit loads. The
 * packed layout is private to this library and may change between versions;
 * its size is qk_weight_packed_bytes(). K must be a multiple of 32.
 */
QK_API size_t qk_weight_packed_bytes(qk_wtype wtype, int64_t N, int64_t K);

QK_API qk_status qk_weight_pack(qk_wtype wtype, const void *blocks, int64_t N, int64_t K,
                         void *packed, size_t packed_bytes, qk_stream stream);

/* ---------------------------------------------------------- projections */

/* One projection read from a shared image: y[t][n] = sum_k W[n][k] x_t[k]. */
typedef struct qk_proj {
    int32_t wtype;     /* qk_wtype */
    int32_t reserved;  /* 0 */
    const void *w;     /* packed weights (qk_weight_pack) */
    int64_t N;         /* output features */
    int64_t K;         /* input features, multiple of 32 */
    float *y;          /* [T][y_stride] F32 output */
    int64_t y_stride;  /* >= N */
} qk_proj;

/*
 * qk_mmvq -- ordinary MUL_MAT on one shared Q8_1 image, several projections
 * in ONE launch (llama.cpp PR #117, Overview/Coverage: q/k/v or gate/up read
 * the same image; the page's "Ordinary, K8192 / T8" component).
 * Per 32-block b, from the stored halves (exact integer block dot D):
 *   Q4_0: y += d_w * (d_a * D - 8 * s_a),  D = sum nibble_i * q_i
 *   Q8_0: y += d_w * d_a * D,              D = sum w_i * q_i
 *   img  [T][img_row_blocks] Q8_1; every projection's K <= 32*img_row_blocks
 *   T    1..8 image rows (tokens); rows >= *d_live_rows are not written
 *   projs host array of n_proj (1..8) descriptors; outputs must not share a
 *        byte. Outputs with one y_stride may be disjoint column windows of
 *        one buffer (q, k and v as columns of a fused [T][Nq+Nk+Nv] output).
 *   ws   device workspace of at least qk_mmvq_workspace_bytes(n_proj, projs)
 *        bytes, 16-byte aligned, ZEROED ONCE before its first use (e.g. by
 *        cudaMemset). It holds completion counters, which every call returns
 *        to zero before its kernels finish, and scratch partial sums; so it
 *        can be reused by later calls (and graph replays) on the same stream
 *        without zeroing again. Calls that may run concurrently need
 *        separate workspaces.
 * The work is split by bytes over the device's SMs; partial sums of a row
 * tile shared by several CTAs go through ws and are added in a fixed order,
 * so outputs are deterministic on a given device.
 * Errors: QK_ERR_ARG, QK_ERR_UNSUPPORTED (T > 8 or n_proj > 8),
 * QK_ERR_SHAPE (K % 32, K beyond the image, y_stride < N), QK_ERR_ALIAS,
 * QK_ERR_WORKSPACE (ws null or too small).
 */
QK_API size_t qk_mmvq_workspace_bytes(int32_t n_proj, const qk_proj *projs);

QK_API qk_status qk_mmvq(const void *img, int64_t img_row_blocks, int64_t T,
                         int32_t n_proj, const qk_proj *projs,
                         const int32_t *d_live_rows, void *ws, size_t ws_bytes,
                         qk_stream stream);

/*
 * qk_mmvq_static_ws -- qk_mmvq for callers that cannot allocate device memory.
 * (The pages this library follows have no counterpart for this call.)
 *
 * Some callers cannot call cudaMalloc at all or at the point where they
 * project: a plugin or kernel-library shim that is handed only the tensors it
 * reads and writes (it owns no allocator and may not keep memory between
 * calls), or a latency-critical path that must not touch the allocator
 * (cudaMalloc can synchronise the device and take milliseconds). This entry point takes the same
 * arguments as qk_mmvq minus the workspace, and uses instead a fixed scratch
 * array of QK_MMVQ_STATIC_WS_BYTES bytes that lives in the library's own
 * device memory (every GPU that loads the library holds it until the process
 * exits). Inputs and outputs are still passed by the caller.
 *   - The first call on a device looks up the array's device address once,
 *     with that device current; later calls on the device reuse it.
 *   - Every argument is checked as in qk_mmvq before anything is enqueued.
 *   - Calls whose workspace need (qk_mmvq_workspace_bytes) exceeds
 *     QK_MMVQ_STATIC_WS_BYTES are refused with QK_ERR_UNSUPPORTED.
 *   - Each call clears the array's completion counters (only those) on its
 *     stream before its kernels run; it allocates nothing.
 *   - All calls on a device share the one array, so calls that may overlap on
 *     the GPU (for instance on different streams) race and give wrong
 *     results; order them on one stream.
 */
#define QK_MMVQ_STATIC_WS_BYTES (2u << 20)

QK_API qk_status qk_mmvq_static_ws(const void *img, int64_t img_row_blocks, int64_t T,
                                   int32_t n_proj, const qk_proj *projs,
                                   const int32_t *d_live_rows, qk_stream stream);

/* ---------------------------------------------------------- routing */

/*
 * qk_topk_route -- router probabilities and top-k experts for the live rows
 * (TensorFold PR #1047, "The fix": tf_moe_router and tf_moe_topk skip rows
 * from the live count up).
 *   logits [rows][E] F32; ids [rows][k] int32; wts [rows][k] F32
 *   experts ranked by logit, larger first, equal logits to the lower index;
 *   ids in rank order; wts = softmax(logits)[id] (not renormalised).
 * Rows >= *d_live_rows keep their previous ids/wts bytes. rows = 0 launches nothing.
 * Errors: QK_ERR_ARG, QK_ERR_UNSUPPORTED (E > 256, k > 32, k > E).
 */
QK_API qk_status qk_topk_route(const float *logits, int64_t rows, int32_t E, int32_t k,
                        int32_t *ids, float *wts,
                        const int32_t *d_live_rows, qk_stream stream);

/*
 * qk_moe_plan -- stable grouped plan of the live pairs (TensorFold PR #1047,
 * "The fix": counts and ranks, exclusive-scan offsets, scatter, over the
 * first live*k pairs only).
 *   pairs p = row*k + slot for rows < live; expert ids[p]
 *   counts [E]   pairs per expert
 *   offsets[E+1] exclusive scan of counts, offsets[E] = live*k
 *   items  [rows*k] positions 0..live*k-1 hold the pairs grouped by expert,
 *          ascending p within each expert; positions past live*k untouched
 * One launch for any width, also for rows = 0 or a live count of 0 (zero
 * counts and offsets). Errors: QK_ERR_ARG, QK_ERR_UNSUPPORTED (E > 1024),
 * QK_ERR_ALIAS.
 */
QK_API qk_status qk_moe_plan(const int32_t *ids, int64_t rows, int32_t k, int32_t E,
                      int32_t *counts, int32_t *offsets, int32_t *items,
                      const int32_t *d_live_rows, qk_stream stream);

/*
 * qk_route_plan -- qk_topk_route then qk_moe_plan, in one launch when the
 * bucket has at most 32 rows (one CTA: a warp per row, then the plan), else
 * as the two launches. Outputs (ids, wts, counts, offsets, items) are the
 * same bytes as the two calls'; arguments and limits as theirs (E <= 256).
 * Errors: QK_ERR_ARG, QK_ERR_UNSUPPORTED, QK_ERR_ALIAS.
 */
QK_API qk_status qk_route_plan(const float *logits, int64_t rows, int32_t E, int32_t k, int32_t *ids,
                               float *wts, int32_t *counts, int32_t *offsets, int32_t *items,
                               const int32_t *d_live_rows, qk_stream stream);

/* One routed projection: E experts' packed weights back to back. */
typedef struct qk_proj_id {
    int32_t wtype;          /* qk_wtype */
    int32_t n_experts;      /* E */
    const void *w;          /* expert e at w + e * qk_weight_packed_bytes(wtype, N, K) */
    int64_t N;              /* output features per expert */
    int64_t K;              /* input features, multiple of 32 */
    float *y;               /* [rows*k][N] F32, pair p at row p */
} qk_proj_id;

/*
 * qk_mmvq_id -- routed MUL_MAT_ID reading the one shared image (llama.cpp
 * PR #117, Coverage: the image is independent of route ids; TensorFold PR
 * #1047: padding rows get no plan items and no expert work).
 * For every expert e and every planned item p in items[offsets[e] ..
 * offsets[e+1]): y[p][:] = W_e * image row (p / k), with the per-block
 * arithmetic of qk_mmvq. Experts with no items read no weights; pairs not in
 * the plan are not written. The plan (counts/offsets/items, device) is the
 * output of qk_moe_plan; ids is not needed. A plan from anywhere else gives
 * unspecified outputs but no read outside counts, offsets and items: counts
 * are clamped to [0, rows * k] and an item position outside items, or a pair
 * outside the bucket, is skipped.
 *   rows: bucket rows (image rows >= rows never read); n_proj 1..8
 * Errors: QK_ERR_ARG, QK_ERR_UNSUPPORTED (n_experts > 1024), QK_ERR_SHAPE,
 * QK_ERR_ALIAS (also an output over counts, offsets or items).
 */
QK_API qk_status qk_mmvq_id(const void *img, int64_t img_row_blocks, int64_t rows, int32_t k,
                     int32_t n_proj, const qk_proj_id *projs,
                     const int32_t *counts, const int32_t *offsets, const int32_t *items,
                     qk_stream stream);

/*
 * qk_mmvq_id_slots -- qk_mmvq_id with one image row per pair: y[p][:] =
 * W_e * image row p (the per-slot down projection of a routed FFN, whose
 * input is each pair's own GLU output; llama.cpp PR #117, "GLU producer
 * evidence" table, the per-slot routed components "K8192 / 32 slots / T8" and
 * "K2560 / 128 slots / T8"). img has rows * k rows.
 * In a routed FFN the per-pair image comes from qk_glu_q8_1 over the rows * k
 * gate/up output rows; passing offsets + E (the plan's count of planned pairs,
 * live * k) as that call's d_live_rows leaves the padding pairs untouched.
 * Errors: as qk_mmvq_id.
 */
QK_API qk_status qk_mmvq_id_slots(const void *img, int64_t img_row_blocks, int64_t rows, int32_t k,
                                  int32_t n_proj, const qk_proj_id *projs, const int32_t *counts,
                                  const int32_t *offsets, const int32_t *items, qk_stream stream);

/*
 * qk_moe_combine -- weighted combine of the routed experts' outputs (the
 * closing step of the routed FFN; TensorFold PR #1047: live-row aware).
 *   y[r][n] = sum over s = 0..k-1 (in that order, one binary32 fma each) of
 *             wts[r*k + s] * expert_out[r*k + s][n],   for rows r < live
 *   expert_out [rows*k][out_stride] F32, wts [rows][k] F32 (qk_topk_route's),
 *   y [rows][y_stride] F32; rows >= *d_live_rows are not read or written.
 *   expert_out and y 16-byte aligned; strides and N multiples of 4; N <= 2^25.
 * Errors: QK_ERR_ARG, QK_ERR_SHAPE, QK_ERR_ALIAS.
 */
QK_API qk_status qk_moe_combine(const float *expert_out, int64_t out_stride, const float *wts, int64_t rows,
                                int32_t k, int64_t N, float *y, int64_t y_stride, const int32_t *d_live_rows,
                                qk_stream stream);

/* ---------------------------------------------------------- prefill */

/*
 * qk_mmq -- prefill dense contraction on a Q8_0 image (minfer doc 52,
 * sections 1 and 5: the q/k/v and gate/up GEMMs that share one quantised A).
 *   qs [T][row_blocks*32] int8 and d [T][row_blocks] half: qk_quantize_q8_0
 *   C[t][n] = sum_b d_w[n][b] * d_a[t][b] * sum_{i in b} w_i * q_i
 *   (Q4_0: w_i = nibble - 8) written to projs[j].y ([T][y_stride] F32);
 *   outputs must not share a byte (disjoint column windows of one buffer
 *   with one y_stride are allowed, as for qk_mmvq)
 * Runs on the tensor cores with binary16 operands (nibble - 8) * d_w and
 * q * d_a, each rounded once, accumulated in binary32: within about 2^-11
 * relative per product of the exact block form (NMSE ~1e-7).
 *   ws: caller workspace of qk_mmq_workspace_bytes bytes, 128-byte aligned;
 *   it holds the dequantised image for this call (scratch, no state kept).
 *   Two launches on the stream (the dequantisation, then the GEMM).
 * Errors: QK_ERR_ARG, QK_ERR_SHAPE, QK_ERR_UNSUPPORTED, QK_ERR_ALIAS,
 * QK_ERR_WORKSPACE.
 */
/*
 * qk_image_memo -- the consecutive-window memo of minfer doc 52 ("r49 A-quantize
 * prepass shared-A dedup", sections 2 and 3.1): which activation the caller's
 * image buffers hold, so that the GEMMs that read one activation (q/k/v,
 * gate/up) quantise it once. Caller-owned plain data; all zeros is empty.
 *   key: image format (QK_MEMO_Q8_0 planes or QK_MEMO_Q8_1 image), the source
 *   pointer x, T, K, x_stride, row_blocks, the stream, and the buffers the image
 *   was written to (qs and d, or img and NULL): a hit needs every field equal,
 *   the destination pointers included (the page's physical-pointer check).
 *   The quantisers are pure functions of these, so a hit equals a recompute byte
 *   for byte -- provided x was not written since. The memo cannot see writes, so
 *   it is valid only while that holds, which the page guarantees with two rules
 *   that the CALLER applies by calling qk_image_memo_clear:
 *     1. any node that is not a quantised-weight GEMM reading this image clears it
 *        (the window is consecutive GEMMs; a buffer can only be rewritten by some
 *        other node, and that node has cleared the memo first);
 *     2. every synchronisation or graph execution boundary clears it (the next
 *        execution can hand the same addresses to new data).
 *   The image buffers must not be any node's output (they live outside the
 *   caller's activation pool), or another node could overwrite them.
 *   Live-row counts are not supported (a device-side value cannot be a key).
 * qk_image_memo_quantize_q8_0 / _q8_1: on a hit nothing is enqueued and *hit = 1;
 * otherwise as qk_quantize_q8_0 / qk_quantize_q8_1 (no live count), *hit = 0,
 * and on success the memo records the call's key. Any error clears the memo.
 * qk_image_memo_match: 1 if a call with these arguments would be a hit, else 0
 * (host only; enqueues nothing).
 * Errors: those of the quantisers; QK_ERR_ARG for a null memo or hit pointer.
 */
typedef enum qk_memo_format { QK_MEMO_EMPTY = 0, QK_MEMO_Q8_0 = 1, QK_MEMO_Q8_1 = 2 } qk_memo_format;
typedef struct qk_image_memo {
    int32_t format; /* qk_memo_format; QK_MEMO_EMPTY: nothing recorded */
    int32_t reserved;
    const void *x;
    int64_t T, K, x_stride, row_blocks;
    const void *dst0, *dst1; /* qs and d, or img and NULL */
    qk_stream stream;
} qk_image_memo;
QK_API void qk_image_memo_clear(qk_image_memo *memo);
QK_API int32_t qk_image_memo_match(const qk_image_memo *memo, int32_t format, const float *x, int64_t T,
                                   int64_t K, int64_t x_stride, const void *dst0, const void *dst1,
                                   int64_t row_blocks, qk_stream stream);
QK_API qk_status qk_image_memo_quantize_q8_0(qk_image_memo *memo, const float *x, int64_t T, int64_t K,
                                             int64_t x_stride, int8_t *qs, uint16_t *d, int64_t row_blocks,
                                             int32_t *hit, qk_stream stream);
QK_API qk_status qk_image_memo_quantize_q8_1(qk_image_memo *memo, const float *x, int64_t T, int64_t K,
                                             int64_t x_stride, void *img, int64_t img_row_blocks,
                                             int32_t *hit, qk_stream stream);

QK_API size_t qk_mmq_workspace_bytes(int64_t T, int32_t n_proj, const qk_proj *projs);
QK_API qk_status qk_mmq(const int8_t *qs, const uint16_t *d, int64_t row_blocks, int64_t T,
                 int32_t n_proj, const qk_proj *projs, void *ws, size_t ws_bytes,
                 qk_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* QK_H */

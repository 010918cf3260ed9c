// Internal declarations shared by libqk's translation units (not installed).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qk.h"

namespace qk {

// ---------------------------------------------------------------- host side
qk_status fail(qk_status s, const char *fmt, ...);  // records qk_last_error(), returns s
qk_status check_launch(const char *what);           // cudaGetLastError -> QK_ERR_CUDA
void count_launch(unsigned n = 1);                   // feeds qk_launch_count()

// Half-open byte range of a device buffer, for overlap checks.
struct Span {
    uintptr_t lo, hi;
};
inline Span span(const void *p, size_t bytes) {
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + bytes};
}
inline bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Bytes spanned by `rows` rows of `row_bytes` with a row pitch of `pitch_bytes`.
inline size_t rows_span(int64_t rows, int64_t pitch_bytes, int64_t row_bytes) {
    return rows <= 0 ? 0 : (size_t)((rows - 1) * pitch_bytes + row_bytes);
}

// Whether two row sets (`rows` rows of la / lb bytes at pitches pa / pb) share a byte. Row sets
// with one pitch whose column windows are disjoint within the pitch (the q, k and v outputs as
// column ranges of one fused [T][N_q + N_k + N_v] buffer) do not overlap; any other pair whose
// byte ranges meet counts as overlapping.
inline bool rows_overlap(const void *a, int64_t pa, int64_t la, const void *b, int64_t pb, int64_t lb, int64_t rows) {
    if (!overlap(span(a, rows_span(rows, pa, la)), span(b, rows_span(rows, pb, lb)))) return false;
    if (rows <= 1 || pa != pb || la > pa || lb > pb) return true;
    const int64_t diff = (int64_t)(reinterpret_cast<uintptr_t>(b) - reinterpret_cast<uintptr_t>(a));
    const int64_t d = ((diff % pa) + pa) % pa;   // b's column offset within a's row period
    return !(d >= la && d + lb <= pa);
}

// ------------------------------------------------------------- device side
constexpr int QB = 32;           // elements per quant block
constexpr int Q8_1_BYTES = 36;   // half d, half s, 32 codes
constexpr int Q4_0_BYTES = 18;
constexpr int Q8_0_BYTES = 34;

// Programmatic dependent launch. Every compute kernel of the library lets the
// next kernel on the stream start launching as soon as all of its own CTAs are
// resident (trigger), and waits for the previous kernel's completion and
// memory before it reads anything that kernel may have written (wait). Both
// are no-ops when the launch has no programmatic dependency.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Live rows: min(rows, max(0, *live)), or rows when no pointer is given.
__device__ __forceinline__ int live_rows(const int32_t *live, int rows) {
    if (!live) return rows;
    int n = __ldg(live);
    return n < 0 ? 0 : (n > rows ? rows : n);
}

// Packed weights: units of 128 rows x 128 columns (8 row groups of 16 rows x
// 4 quant blocks), ordered (row tile, column chunk) and block-major inside a
// unit, so one warp reads everything it needs for one 32-column block of all
// 8 row groups with conflict-free 128-bit loads. Lane l = 4g + t; "word t" of
// a row's block = its bytes 4t..4t+3 (Q4_0: nibble bytes; Q8_0: codes 4t..4t+3
// "lo" and codes 16+4t..16+4t+3 "hi").
//   Q4_0 unit, 9216 B: block jb at jb*2048, four 512-B regions; region k,
//     lane l: 16 B = word t of rows 32k+g, 32k+g+8, 32k+16+g, 32k+24+g.
//     Scales at 8192 + jb*256 + g*32: eight half2 (row 16r+g, row 16r+g+8),
//     r = 0..7.
//   Q8_0 unit, 17408 B: block jb at jb*4096, eight 512-B regions; region k,
//     lane l: 16 B = [row 16k+g lo, hi][row 16k+g+8 lo, hi]. Scales at
//     16384 + jb*256 as for Q4_0.
constexpr int UNIT_ROWS = 128;
constexpr int UNIT_GROUPS = 8;
constexpr int UNIT_COLS = 128;
constexpr int Q4_UNIT_BYTES = 9216;
constexpr int Q8_UNIT_BYTES = 17408;
constexpr int Q4_BLOCK_STRIDE = 2048;
constexpr int Q8_BLOCK_STRIDE = 4096;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t unit_bytes(int wtype) { return wtype == QK_W_Q4_0 ? Q4_UNIT_BYTES : Q8_UNIT_BYTES; }
inline int64_t packed_bytes(int wtype, int64_t N, int64_t K) {
    return ceil_div(N, UNIT_ROWS) * ceil_div(K, UNIT_COLS) * unit_bytes(wtype);
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Reads and clears the device-side fault word (bit 0: a bounded mbarrier
// wait gave up). Synchronous.
qk_status read_device_faults(uint32_t *faults);
// One CTA whose bounded wait runs out and sets bit 0 of the fault word.
qk_status launch_wait_selftest(cudaStream_t s);

// Launch with programmatic stream serialization (see pdl_trigger/pdl_wait).
template <typename... KArgs, typename... Args>
qk_status launch_pdl(const char *name, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    count_launch();
    if (e != cudaSuccess) return fail(QK_ERR_CUDA, "%s: %s", name, cudaGetErrorString(e));
    return check_launch(name);
}

// ------------------------------------------------------- kernel launchers
// Defined in the kernel translation units; arguments already validated.
qk_status launch_quantize_q8_1(const float *x, int T, int K, int64_t x_stride, uint8_t *img,
                               int64_t row_blocks, const int32_t *live, cudaStream_t s);
qk_status launch_quantize_q8_0(const float *x, int T, int K, int64_t x_stride, int8_t *qs,
                               uint16_t *d, int64_t row_blocks, const int32_t *live, cudaStream_t s);
qk_status launch_rmsnorm_q8_1(const float *x, int T, int K, int64_t x_stride, int kind,
                              const float *w, const float *b, float scale, float eps, float *y,
                              int64_t y_stride, uint8_t *img, int64_t row_blocks,
                              const int32_t *live, cudaStream_t s);
qk_status launch_rmsnorm_q8_0(const float *x, int T, int K, int64_t x_stride, int kind, const float *w,
                              const float *b, float scale, float eps, float *y, int64_t y_stride, int8_t *qs,
                              uint16_t *dh, int64_t row_blocks, const int32_t *live, cudaStream_t s);
qk_status launch_glu_q8_1(int kind, int layout, const float *a, int64_t a_stride, const float *b,
                          int64_t b_stride, int T, int N, float *out, int64_t out_stride,
                          uint8_t *img, int64_t row_blocks, float alpha, float limit, const int32_t *live,
                          cudaStream_t s);
qk_status launch_weight_pack(int wtype, const uint8_t *blocks, int64_t N, int64_t K,
                             uint8_t *packed, cudaStream_t s);
int64_t mmvq_workspace_bytes(int n_proj, const qk_proj *projs);
// Every argument check of qk_mmvq except those of the workspace (nothing is enqueued).
qk_status mmvq_validate(const void *img, int64_t img_row_blocks, int64_t T, int32_t n_proj, const qk_proj *projs);
// Byte range of the ordinary path's completion counters inside its workspace, for the
// projections of one weight type (they start at zero and every launch leaves them at zero).
void mmvq_counter_range(int n_proj, const qk_proj *projs, int64_t *offset, int64_t *bytes);
qk_status launch_mmvq(const uint8_t *img, int64_t row_blocks, int T, int n_proj,
                      const qk_proj *projs, const int32_t *live, void *ws, size_t ws_bytes,
                      cudaStream_t s);
qk_status launch_mmvq_id(const uint8_t *img, int64_t row_blocks, int rows, int k, int n_proj,
                         const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                         const int32_t *items, bool per_pair, cudaStream_t s);
qk_status launch_moe_combine(const float *expert_out, int64_t out_stride, const float *wts, int rows, int k, int N,
                             float *y, int64_t y_stride, const int32_t *live, cudaStream_t s);
qk_status launch_topk_route(const float *logits, int rows, int E, int k, int32_t *ids,
                            float *wts, const int32_t *live, cudaStream_t s);
qk_status launch_moe_plan(const int32_t *ids, int rows, int k, int E, int32_t *counts,
                          int32_t *offsets, int32_t *items, const int32_t *live, cudaStream_t s);
// Top-k then plan in one launch (buckets of up to 32 rows; larger ones take the two launches).
qk_status launch_route_plan(const float *logits, int rows, int E, int k, int32_t *ids, float *wts, int32_t *counts,
                            int32_t *offsets, int32_t *items, const int32_t *live, cudaStream_t s);
qk_status launch_mmq(const int8_t *qs, const uint16_t *d, int64_t row_blocks, int T, int n_proj,
                     const qk_proj *projs, void *ws, size_t ws_bytes, cudaStream_t s);
int64_t mmq_workspace_bytes(int64_t T, int64_t kmax);
qk_status read_mmq_faults(uint32_t *faults);

}  // namespace qk

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

// ------------------------------------------------------------- device side
constexpr int QB = 32;           // elements per quant block
constexpr int Q8_1_BYTES = 36;   // half d, half s, 32 codes
constexpr int Q4_0_BYTES = 18;
constexpr int Q8_0_BYTES = 34;

// Live rows: min(rows, max(0, *live)), or rows when no pointer is given.
__device__ __forceinline__ int live_rows(const int32_t *live, int rows) {
    if (!live) return rows;
    int n = __ldg(live);
    return n < 0 ? 0 : (n > rows ? rows : n);
}

// Packed Q4_0 weights: 16-row groups x 128-column chunks, 1152-byte tiles.
//   bytes    0..511 : lane l = 4g+t holds 16 B = for blocks j=0..3 of the chunk,
//                     nibble bytes 4t..4t+3 of row g of the group
//   bytes  512..1023: the same for row g+8
//   bytes 1024..1151: scales, row r (0..15) at 1024 + 8r, block j half at +2j
// Packed Q8_0 weights: same tiling, 2176-byte tiles.
//   bytes    0..1023: lane l holds 32 B = for blocks j=0..3: codes 4t..4t+3 and
//                     16+4t..16+4t+3 of row g (8 B per block)
//   bytes 1024..2047: the same for row g+8
//   bytes 2048..2175: scales as for Q4_0
constexpr int TILE_ROWS = 16;
constexpr int TILE_COLS = 128;
constexpr int Q4_TILE_BYTES = 1152;
constexpr int Q8_TILE_BYTES = 2176;

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t tile_bytes(int wtype) { return wtype == QK_W_Q4_0 ? Q4_TILE_BYTES : Q8_TILE_BYTES; }
inline int64_t packed_bytes(int wtype, int64_t N, int64_t K) {
    return ceil_div(N, TILE_ROWS) * ceil_div(K, TILE_COLS) * tile_bytes(wtype);
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
qk_status launch_glu_q8_1(int kind, int layout, const float *a, int64_t a_stride, const float *b,
                          int64_t b_stride, int T, int N, float *out, int64_t out_stride,
                          uint8_t *img, int64_t row_blocks, const int32_t *live, cudaStream_t s);
qk_status launch_weight_pack(int wtype, const uint8_t *blocks, int64_t N, int64_t K,
                             uint8_t *packed, cudaStream_t s);
qk_status launch_mmvq(const uint8_t *img, int64_t row_blocks, int T, int n_proj,
                      const qk_proj *projs, const int32_t *live, cudaStream_t s);
qk_status launch_mmvq_id(const uint8_t *img, int64_t row_blocks, int rows, int k, int n_proj,
                         const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                         const int32_t *items, cudaStream_t s);
qk_status launch_topk_route(const float *logits, int rows, int E, int k, int32_t *ids,
                            float *wts, const int32_t *live, cudaStream_t s);
qk_status launch_moe_plan(const int32_t *ids, int rows, int k, int E, int32_t *counts,
                          int32_t *offsets, int32_t *items, const int32_t *live, cudaStream_t s);
qk_status launch_mmq(const int8_t *qs, const uint16_t *d, int64_t row_blocks, int T, int n_proj,
                     const qk_proj *projs, cudaStream_t s);

}  // namespace qk

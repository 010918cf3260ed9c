// libqk C ABI: argument checks on the host, then the kernel launchers.
//
// Every check happens before anything is enqueued, so a bad call leaves the
// stream untouched (minfer doc 52 "r49 A-quantize prepass shared-A dedup",
// section 3.1: errors surface at entry, not as a fault in a later launch).
// Aliasing outputs are refused (llama.cpp PR #117 "activation image
// emission", Coverage: unsafe input/output aliases keep the original path).

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "qk_internal.cuh"

namespace qk {

static thread_local char g_err[512] = "";
static std::atomic<uint64_t> g_launches{0};

qk_status fail(qk_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

qk_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(QK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return QK_OK;
}

void count_launch(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace qk

using namespace qk;

#define REQUIRE(cond, status, ...) \
    do {                           \
        if (!(cond)) return fail(status, __VA_ARGS__); \
    } while (0)

static bool aligned(const void *p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static qk_status check_proj_common(int32_t wtype, const void *w, int64_t N, int64_t K, int64_t img_row_blocks) {
    REQUIRE(wtype == QK_W_Q4_0 || wtype == QK_W_Q8_0, QK_ERR_ARG, "bad wtype %d", (int)wtype);
    REQUIRE(w, QK_ERR_ARG, "null weight pointer");
    REQUIRE(aligned(w, 16), QK_ERR_ARG, "packed weights must be 16-byte aligned");
    REQUIRE(N >= 1 && N <= INT32_MAX && K >= 32 && K <= INT32_MAX, QK_ERR_ARG, "N or K out of range");
    REQUIRE(K % QB == 0, QK_ERR_SHAPE, "K=%lld is not a multiple of 32", (long long)K);
    REQUIRE(K / QB <= img_row_blocks, QK_ERR_SHAPE, "K=%lld reaches past the image row (%lld blocks)",
            (long long)K, (long long)img_row_blocks);
    return QK_OK;
}

namespace qk {
// Every check of qk_mmvq except those of the workspace: the image, T, the
// projections, their outputs and aliasing between them.
qk_status mmvq_validate(const void *img, int64_t img_row_blocks, int64_t T, int32_t n_proj, const qk_proj *projs) {
    REQUIRE(img && projs, QK_ERR_ARG, "null pointer");
    REQUIRE(aligned(img, 4), QK_ERR_ARG, "img not 4-byte aligned");
    REQUIRE(T >= 1 && img_row_blocks >= 1, QK_ERR_ARG, "T or img_row_blocks < 1");
    REQUIRE(T <= 8, QK_ERR_UNSUPPORTED, "T=%lld > 8 (use qk_mmq for larger batches)", (long long)T);
    REQUIRE(n_proj >= 1 && n_proj <= 8, QK_ERR_UNSUPPORTED, "n_proj=%d not in 1..8", (int)n_proj);
    Span si = span(img, (size_t)(T * img_row_blocks * Q8_1_BYTES));
    for (int j = 0; j < n_proj; j++) {
        const qk_proj &p = projs[j];
        qk_status st = check_proj_common(p.wtype, p.w, p.N, p.K, img_row_blocks);
        if (st != QK_OK) return st;
        REQUIRE(p.y, QK_ERR_ARG, "projection %d: y is null", j);
        REQUIRE(p.y_stride >= p.N, QK_ERR_SHAPE, "projection %d: y_stride < N", j);
        Span sy = span(p.y, rows_span(T, p.y_stride * 4, p.N * 4));
        Span sw = span(p.w, (size_t)packed_bytes(p.wtype, p.N, p.K));
        REQUIRE(!overlap(sy, si) && !overlap(sy, sw), QK_ERR_ALIAS, "projection %d: y overlaps img or w", j);
        for (int i = 0; i < j; i++) {
            REQUIRE(!rows_overlap(projs[i].y, projs[i].y_stride * 4, projs[i].N * 4, p.y, p.y_stride * 4, p.N * 4, T),
                    QK_ERR_ALIAS, "outputs of projections %d and %d overlap", i, j);
        }
    }
    return QK_OK;
}
}  // namespace qk

extern "C" {

const char *qk_status_string(qk_status s) {
    switch (s) {
        case QK_OK: return "QK_OK";
        case QK_ERR_ARG: return "QK_ERR_ARG";
        case QK_ERR_SHAPE: return "QK_ERR_SHAPE";
        case QK_ERR_ALIAS: return "QK_ERR_ALIAS";
        case QK_ERR_WORKSPACE: return "QK_ERR_WORKSPACE";
        case QK_ERR_UNSUPPORTED: return "QK_ERR_UNSUPPORTED";
        case QK_ERR_CUDA: return "QK_ERR_CUDA";
    }
    return "QK_ERR_UNKNOWN";
}

const char *qk_last_error(void) { return g_err; }
const char *qk_last_error_string(void) { return g_err; }

uint64_t qk_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// ------------------------------------------------------------------ image
static qk_status check_quant_in(const float *x, int64_t T, int64_t K, int64_t x_stride) {
    REQUIRE(T >= 0 && T <= INT32_MAX, QK_ERR_ARG, "T=%lld out of range", (long long)T);
    REQUIRE(K >= 1 && K <= (1LL << 25), QK_ERR_ARG, "K=%lld out of range", (long long)K);
    REQUIRE(x || T == 0, QK_ERR_ARG, "x is null");
    REQUIRE(x_stride >= K, QK_ERR_SHAPE, "x_stride=%lld < K=%lld", (long long)x_stride, (long long)K);
    REQUIRE(aligned(x, 4), QK_ERR_ARG, "x not 4-byte aligned");
    return QK_OK;
}

qk_status qk_quantize_q8_1(const float *x, int64_t T, int64_t K, int64_t x_stride, void *img,
                           int64_t img_row_blocks, const int32_t *d_live_rows, qk_stream stream) {
    qk_status st = check_quant_in(x, T, K, x_stride);
    if (st != QK_OK) return st;
    REQUIRE(img || T == 0, QK_ERR_ARG, "img is null");
    REQUIRE(aligned(img, 4), QK_ERR_ARG, "img not 4-byte aligned");
    REQUIRE(img_row_blocks >= ceil_div(K, QB), QK_ERR_SHAPE, "img_row_blocks=%lld < ceil(K/32)=%lld",
            (long long)img_row_blocks, (long long)ceil_div(K, QB));
    REQUIRE(img_row_blocks <= (1 << 20), QK_ERR_ARG, "img_row_blocks > 2^20");
    Span sx = span(x, rows_span(T, x_stride * 4, K * 4));
    Span si = span(img, (size_t)(T * img_row_blocks * Q8_1_BYTES));
    REQUIRE(!overlap(sx, si), QK_ERR_ALIAS, "img overlaps x");
    return launch_quantize_q8_1(x, (int)T, (int)K, x_stride, static_cast<uint8_t *>(img), img_row_blocks,
                                d_live_rows, (cudaStream_t)stream);
}

qk_status qk_quantize_q8_0(const float *x, int64_t T, int64_t K, int64_t x_stride, int8_t *qs,
                           uint16_t *d, int64_t row_blocks, const int32_t *d_live_rows, qk_stream stream) {
    qk_status st = check_quant_in(x, T, K, x_stride);
    if (st != QK_OK) return st;
    REQUIRE((qs && d) || T == 0, QK_ERR_ARG, "qs or d is null");
    REQUIRE(aligned(qs, 4) && aligned(d, 2), QK_ERR_ARG, "qs must be 4-byte and d 2-byte aligned");
    REQUIRE(row_blocks >= ceil_div(K, QB), QK_ERR_SHAPE, "row_blocks=%lld < ceil(K/32)", (long long)row_blocks);
    REQUIRE(row_blocks <= (1 << 20), QK_ERR_ARG, "row_blocks > 2^20");
    Span sx = span(x, rows_span(T, x_stride * 4, K * 4));
    Span sq = span(qs, (size_t)(T * row_blocks * QB));
    Span sd = span(d, (size_t)(T * row_blocks * 2));
    REQUIRE(!overlap(sx, sq) && !overlap(sx, sd) && !overlap(sq, sd), QK_ERR_ALIAS, "qs/d overlap x or each other");
    return launch_quantize_q8_0(x, (int)T, (int)K, x_stride, qs, d, row_blocks, d_live_rows, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ image memo
void qk_image_memo_clear(qk_image_memo *memo) {
    if (memo) *memo = qk_image_memo{};
}

int32_t qk_image_memo_match(const qk_image_memo *m, int32_t format, const float *x, int64_t T, int64_t K,
                            int64_t x_stride, const void *dst0, const void *dst1, int64_t row_blocks,
                            qk_stream stream) {
    return m && m->format != QK_MEMO_EMPTY && m->format == format && m->x == x && m->T == T && m->K == K &&
           m->x_stride == x_stride && m->row_blocks == row_blocks && m->dst0 == dst0 && m->dst1 == dst1 &&
           m->stream == stream;
}

static qk_status memo_record(qk_image_memo *m, qk_status st, int32_t format, const float *x, int64_t T,
                             int64_t K, int64_t x_stride, const void *dst0, const void *dst1, int64_t row_blocks,
                             qk_stream stream) {
    qk_image_memo_clear(m);
    if (st == QK_OK) {
        m->format = format;
        m->x = x;
        m->T = T;
        m->K = K;
        m->x_stride = x_stride;
        m->row_blocks = row_blocks;
        m->dst0 = dst0;
        m->dst1 = dst1;
        m->stream = stream;
    }
    return st;
}

qk_status qk_image_memo_quantize_q8_0(qk_image_memo *memo, const float *x, int64_t T, int64_t K, int64_t x_stride,
                                      int8_t *qs, uint16_t *d, int64_t row_blocks, int32_t *hit, qk_stream stream) {
    REQUIRE(memo, QK_ERR_ARG, "memo is null");
    if (!hit) {
        qk_image_memo_clear(memo);
        return fail(QK_ERR_ARG, "hit is null");
    }
    *hit = qk_image_memo_match(memo, QK_MEMO_Q8_0, x, T, K, x_stride, qs, d, row_blocks, stream);
    if (*hit) return QK_OK;
    const qk_status st = qk_quantize_q8_0(x, T, K, x_stride, qs, d, row_blocks, nullptr, stream);
    return memo_record(memo, st, QK_MEMO_Q8_0, x, T, K, x_stride, qs, d, row_blocks, stream);
}

qk_status qk_image_memo_quantize_q8_1(qk_image_memo *memo, const float *x, int64_t T, int64_t K, int64_t x_stride,
                                      void *img, int64_t img_row_blocks, int32_t *hit, qk_stream stream) {
    REQUIRE(memo, QK_ERR_ARG, "memo is null");
    if (!hit) {
        qk_image_memo_clear(memo);
        return fail(QK_ERR_ARG, "hit is null");
    }
    *hit = qk_image_memo_match(memo, QK_MEMO_Q8_1, x, T, K, x_stride, img, nullptr, img_row_blocks, stream);
    if (*hit) return QK_OK;
    const qk_status st = qk_quantize_q8_1(x, T, K, x_stride, img, img_row_blocks, nullptr, stream);
    return memo_record(memo, st, QK_MEMO_Q8_1, x, T, K, x_stride, img, nullptr, img_row_blocks, stream);
}

// ------------------------------------------------------------------ producers
qk_status qk_rmsnorm_q8_1(const float *x, int64_t T, int64_t K, int64_t x_stride, qk_norm_kind kind,
                          const float *w, const float *b, float scale, float eps, float *y,
                          int64_t y_stride, void *img, int64_t img_row_blocks,
                          const int32_t *d_live_rows, qk_stream stream) {
    qk_status st = check_quant_in(x, T, K, x_stride);
    if (st != QK_OK) return st;
    REQUIRE(kind >= QK_NORM_PLAIN && kind <= QK_NORM_SCALE, QK_ERR_ARG, "bad norm kind %d", (int)kind);
    REQUIRE(K % QB == 0, QK_ERR_SHAPE, "K=%lld is not a whole number of 32-blocks", (long long)K);
    REQUIRE(K <= 32768, QK_ERR_UNSUPPORTED, "K=%lld > 32768 (a row is kept in registers)", (long long)K);
    REQUIRE((y && img) || T == 0, QK_ERR_ARG, "y or img is null");
    const bool need_w = kind == QK_NORM_MUL || kind == QK_NORM_MUL_ADD;
    REQUIRE(!need_w || w, QK_ERR_ARG, "w is null for a MUL kind");
    REQUIRE(kind != QK_NORM_MUL_ADD || b, QK_ERR_ARG, "b is null for MUL_ADD");
    REQUIRE(y_stride >= K, QK_ERR_SHAPE, "y_stride < K");
    REQUIRE(img_row_blocks >= K / QB, QK_ERR_SHAPE, "img_row_blocks < K/32");
    REQUIRE(aligned(y, 4) && aligned(img, 4) && aligned(w, 4) && aligned(b, 4), QK_ERR_ARG, "misaligned pointer");
    Span sx = span(x, rows_span(T, x_stride * 4, K * 4));
    Span sy = span(y, rows_span(T, y_stride * 4, K * 4));
    Span si = span(img, (size_t)(T * img_row_blocks * Q8_1_BYTES));
    Span sw = span(need_w ? w : nullptr, need_w ? (size_t)K * 4 : 0);
    Span sb = span(kind == QK_NORM_MUL_ADD ? b : nullptr, kind == QK_NORM_MUL_ADD ? (size_t)K * 4 : 0);
    REQUIRE(!overlap(sy, sx) && !overlap(sy, si) && !overlap(si, sx) && !overlap(sy, sw) && !overlap(sy, sb) &&
                !overlap(si, sw) && !overlap(si, sb),
            QK_ERR_ALIAS, "y or img overlaps an input or each other");
    return launch_rmsnorm_q8_1(x, (int)T, (int)K, x_stride, (int)kind, w, b, scale, eps, y, y_stride,
                               static_cast<uint8_t *>(img), img_row_blocks, d_live_rows, (cudaStream_t)stream);
}

qk_status qk_rmsnorm_q8_0(const float *x, int64_t T, int64_t K, int64_t x_stride, qk_norm_kind kind,
                          const float *w, const float *b, float scale, float eps, float *y, int64_t y_stride,
                          int8_t *qs, uint16_t *d, int64_t row_blocks, const int32_t *d_live_rows,
                          qk_stream stream) {
    qk_status st = check_quant_in(x, T, K, x_stride);
    if (st != QK_OK) return st;
    REQUIRE(kind >= QK_NORM_PLAIN && kind <= QK_NORM_SCALE, QK_ERR_ARG, "bad norm kind %d", (int)kind);
    REQUIRE(K % QB == 0, QK_ERR_SHAPE, "K=%lld is not a whole number of 32-blocks", (long long)K);
    REQUIRE(K <= 32768, QK_ERR_UNSUPPORTED, "K=%lld > 32768 (a row is kept in registers)", (long long)K);
    REQUIRE((y && qs && d) || T == 0, QK_ERR_ARG, "y, qs or d is null");
    const bool need_w = kind == QK_NORM_MUL || kind == QK_NORM_MUL_ADD;
    REQUIRE(!need_w || w, QK_ERR_ARG, "w is null for a MUL kind");
    REQUIRE(kind != QK_NORM_MUL_ADD || b, QK_ERR_ARG, "b is null for MUL_ADD");
    REQUIRE(y_stride >= K, QK_ERR_SHAPE, "y_stride < K");
    REQUIRE(row_blocks >= K / QB, QK_ERR_SHAPE, "row_blocks < K/32");
    REQUIRE(aligned(y, 4) && aligned(qs, 16) && aligned(d, 4) && aligned(w, 4) && aligned(b, 4), QK_ERR_ARG,
            "misaligned pointer (qs must be 16-byte aligned)");
    Span sx = span(x, rows_span(T, x_stride * 4, K * 4));
    Span sy = span(y, rows_span(T, y_stride * 4, K * 4));
    Span sq = span(qs, (size_t)(T * row_blocks * QB)), sd = span(d, (size_t)(T * row_blocks * 2));
    Span sw = span(need_w ? w : nullptr, need_w ? (size_t)K * 4 : 0);
    Span sb = span(kind == QK_NORM_MUL_ADD ? b : nullptr, kind == QK_NORM_MUL_ADD ? (size_t)K * 4 : 0);
    const Span outs[3] = {sy, sq, sd}, ins[3] = {sx, sw, sb};
    for (int o = 0; o < 3; o++) {
        for (int i = 0; i < 3; i++) REQUIRE(!overlap(outs[o], ins[i]), QK_ERR_ALIAS, "an output overlaps an input");
        for (int q = 0; q < o; q++) REQUIRE(!overlap(outs[o], outs[q]), QK_ERR_ALIAS, "outputs overlap each other");
    }
    return launch_rmsnorm_q8_0(x, (int)T, (int)K, x_stride, (int)kind, w, b, scale, eps, y, y_stride, qs, d,
                               row_blocks, d_live_rows, (cudaStream_t)stream);
}

qk_status qk_glu_q8_1(qk_glu_kind kind, qk_glu_layout layout, const float *a, int64_t a_stride,
                      const float *b, int64_t b_stride, int64_t T, int64_t N, float *out,
                      int64_t out_stride, void *img, int64_t img_row_blocks, const int32_t *d_live_rows,
                      qk_stream stream) {
    return qk_glu_q8_1_ex(kind, layout, a, a_stride, b, b_stride, T, N, out, out_stride, img, img_row_blocks,
                          1.702f, 7.0f, d_live_rows, stream);
}

qk_status qk_glu_q8_1_ex(qk_glu_kind kind, qk_glu_layout layout, const float *a, int64_t a_stride,
                         const float *b, int64_t b_stride, int64_t T, int64_t N, float *out,
                         int64_t out_stride, void *img, int64_t img_row_blocks, float alpha, float limit,
                         const int32_t *d_live_rows, qk_stream stream) {
    REQUIRE(kind >= QK_GLU_SWIGLU && kind <= QK_GLU_SWIGLU_CLAMP, QK_ERR_ARG, "bad glu kind %d", (int)kind);
    REQUIRE(std::isfinite(alpha) && std::isfinite(limit) && limit > 0.0f, QK_ERR_ARG,
            "alpha must be finite and limit positive and finite");
    REQUIRE(layout >= QK_GLU_SEPARATE && layout <= QK_GLU_PACKED_SWAPPED, QK_ERR_ARG, "bad glu layout %d", (int)layout);
    REQUIRE(T >= 0 && T <= INT32_MAX && N >= 1 && N <= (1LL << 25), QK_ERR_ARG, "T or N out of range");
    REQUIRE(N % QB == 0, QK_ERR_SHAPE, "N=%lld is not a whole number of 32-blocks", (long long)N);
    REQUIRE((a && out && img && (layout != QK_GLU_SEPARATE || b)) || T == 0, QK_ERR_ARG, "null pointer");
    const int64_t a_row = layout == QK_GLU_SEPARATE ? N : 2 * N;
    REQUIRE(a_stride >= a_row, QK_ERR_SHAPE, "a_stride too small");
    REQUIRE(layout != QK_GLU_SEPARATE || b_stride >= N, QK_ERR_SHAPE, "b_stride < N");
    REQUIRE(out_stride >= N && img_row_blocks >= N / QB, QK_ERR_SHAPE, "out_stride or img_row_blocks too small");
    REQUIRE(aligned(a, 4) && aligned(b, 4) && aligned(out, 4) && aligned(img, 4), QK_ERR_ARG, "misaligned pointer");
    Span sa = span(a, rows_span(T, a_stride * 4, a_row * 4));
    Span sb = span(layout == QK_GLU_SEPARATE ? b : nullptr,
                   layout == QK_GLU_SEPARATE ? rows_span(T, b_stride * 4, N * 4) : 0);
    Span so = span(out, rows_span(T, out_stride * 4, N * 4));
    Span si = span(img, (size_t)(T * img_row_blocks * Q8_1_BYTES));
    REQUIRE(!overlap(so, sa) && !overlap(so, sb) && !overlap(so, si) && !overlap(si, sa) && !overlap(si, sb),
            QK_ERR_ALIAS, "out or img overlaps an input or each other");
    return launch_glu_q8_1((int)kind, (int)layout, a, a_stride, b, b_stride, (int)T, (int)N, out, out_stride,
                           static_cast<uint8_t *>(img), img_row_blocks, alpha, limit, d_live_rows,
                           (cudaStream_t)stream);
}

// ------------------------------------------------------------------ weights
size_t qk_weight_packed_bytes(qk_wtype wtype, int64_t N, int64_t K) {
    if ((wtype != QK_W_Q4_0 && wtype != QK_W_Q8_0) || N < 0 || K < 0) return 0;
    return (size_t)packed_bytes(wtype, N, K);
}

qk_status qk_weight_pack(qk_wtype wtype, const void *blocks, int64_t N, int64_t K, void *packed,
                         size_t packed_bytes_, qk_stream stream) {
    REQUIRE(wtype == QK_W_Q4_0 || wtype == QK_W_Q8_0, QK_ERR_ARG, "bad wtype %d", (int)wtype);
    REQUIRE(N >= 1 && K >= 32 && N <= INT32_MAX && K <= INT32_MAX, QK_ERR_ARG, "N or K out of range");
    REQUIRE(K % QB == 0, QK_ERR_SHAPE, "K=%lld is not a multiple of 32", (long long)K);
    REQUIRE(blocks && packed, QK_ERR_ARG, "null pointer");
    REQUIRE(aligned(packed, 16), QK_ERR_ARG, "packed must be 16-byte aligned");
    const size_t need = (size_t)packed_bytes(wtype, N, K);
    REQUIRE(packed_bytes_ >= need, QK_ERR_WORKSPACE, "packed_bytes=%zu < %zu", packed_bytes_, need);
    const size_t src = (size_t)(N * (K / QB) * (wtype == QK_W_Q4_0 ? Q4_0_BYTES : Q8_0_BYTES));
    REQUIRE(!overlap(span(blocks, src), span(packed, need)), QK_ERR_ALIAS, "packed overlaps blocks");
    return launch_weight_pack(wtype, static_cast<const uint8_t *>(blocks), N, K, static_cast<uint8_t *>(packed),
                              (cudaStream_t)stream);
}

// ------------------------------------------------------------------ projections

size_t qk_mmvq_workspace_bytes(int32_t n_proj, const qk_proj *projs) {
    if (n_proj < 1 || n_proj > 8 || !projs) return 0;
    size_t need = 0;
    for (int wt = QK_W_Q4_0; wt <= QK_W_Q8_0; wt++) {
        qk_proj group[8];
        int n = 0;
        for (int j = 0; j < n_proj; j++)
            if (projs[j].wtype == wt) group[n++] = projs[j];
        if (n == 0) continue;
        const size_t g = (size_t)mmvq_workspace_bytes(n, group);
        need = g > need ? g : need;
    }
    return need;
}

qk_status qk_device_faults(uint32_t *faults) {
    REQUIRE(faults, QK_ERR_ARG, "faults is null");
    uint32_t a = 0, b = 0;
    qk_status st = read_device_faults(&a);
    if (st == QK_OK) st = read_mmq_faults(&b);
    *faults = a | b;
    return st;
}

qk_status qk_selftest_wait_timeout(qk_stream stream) { return launch_wait_selftest((cudaStream_t)stream); }

qk_status qk_mmvq(const void *img, int64_t img_row_blocks, int64_t T, int32_t n_proj, const qk_proj *projs,
                  const int32_t *d_live_rows, void *ws, size_t ws_bytes, qk_stream stream) {
    qk_status vs = mmvq_validate(img, img_row_blocks, T, n_proj, projs);
    if (vs != QK_OK) return vs;
    Span si = span(img, (size_t)(T * img_row_blocks * Q8_1_BYTES));
    REQUIRE(ws && aligned(ws, 16), QK_ERR_WORKSPACE, "workspace null or not 16-byte aligned");
    // one launch per weight type present, in order on the stream; they share ws
    for (int wt = QK_W_Q4_0; wt <= QK_W_Q8_0; wt++) {
        qk_proj group[8];
        int n = 0;
        for (int j = 0; j < n_proj; j++)
            if (projs[j].wtype == wt) group[n++] = projs[j];
        if (n == 0) continue;
        const size_t need = (size_t)mmvq_workspace_bytes(n, group);
        REQUIRE(ws_bytes >= need, QK_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
        Span sws = span(ws, need);
        REQUIRE(!overlap(sws, si), QK_ERR_ALIAS, "workspace overlaps img");
        for (int j = 0; j < n_proj; j++)
            REQUIRE(!overlap(sws, span(projs[j].y, rows_span(T, projs[j].y_stride * 4, projs[j].N * 4))) &&
                        !overlap(sws, span(projs[j].w, (size_t)packed_bytes(projs[j].wtype, projs[j].N, projs[j].K))),
                    QK_ERR_ALIAS, "workspace overlaps projection %d", j);
    }
    for (int wt = QK_W_Q4_0; wt <= QK_W_Q8_0; wt++) {
        qk_proj group[8];
        int n = 0;
        for (int j = 0; j < n_proj; j++)
            if (projs[j].wtype == wt) group[n++] = projs[j];
        if (n == 0) continue;
        qk_status st = launch_mmvq(static_cast<const uint8_t *>(img), img_row_blocks, (int)T, n, group,
                                   d_live_rows, ws, ws_bytes, (cudaStream_t)stream);
        if (st != QK_OK) return st;
    }
    return QK_OK;
}

static qk_status mmvq_id_common(const void *img, int64_t img_row_blocks, int64_t rows, int32_t k, int32_t n_proj,
                                const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                                const int32_t *items, bool per_pair, qk_stream stream) {
    REQUIRE(img && projs && counts && offsets && items, QK_ERR_ARG, "null pointer");
    REQUIRE(aligned(img, 4), QK_ERR_ARG, "img not 4-byte aligned");
    REQUIRE(rows >= 1 && rows <= (1 << 24) && k >= 1 && k <= 64 && img_row_blocks >= 1, QK_ERR_ARG,
            "rows, k or img_row_blocks out of range");
    REQUIRE(n_proj >= 1 && n_proj <= 8, QK_ERR_UNSUPPORTED, "n_proj=%d not in 1..8", (int)n_proj);
    Span si = span(img, (size_t)((per_pair ? rows * k : rows) * img_row_blocks * Q8_1_BYTES));
    // the plan is read while outputs are written: no output may overlap it
    const int64_t E = projs[0].n_experts;
    const Span plan[3] = {span(counts, (size_t)(E > 0 ? E : 0) * 4), span(offsets, (size_t)(E > 0 ? E + 1 : 0) * 4),
                          span(items, (size_t)(rows * k * 4))};
    for (int j = 0; j < n_proj; j++) {
        const qk_proj_id &p = projs[j];
        qk_status st = check_proj_common(p.wtype, p.w, p.N, p.K, img_row_blocks);
        if (st != QK_OK) return st;
        REQUIRE(p.n_experts >= 1 && p.n_experts <= 1024, QK_ERR_UNSUPPORTED, "n_experts=%d", (int)p.n_experts);
        REQUIRE(p.y, QK_ERR_ARG, "projection %d: y is null", j);
        REQUIRE(projs[0].n_experts == p.n_experts, QK_ERR_ARG, "projections disagree on n_experts");
        Span sy = span(p.y, (size_t)(rows * k * p.N * 4));
        Span sw = span(p.w, (size_t)packed_bytes(p.wtype, p.N, p.K) * p.n_experts);
        REQUIRE(!overlap(sy, si) && !overlap(sy, sw), QK_ERR_ALIAS, "projection %d: y overlaps img or w", j);
        REQUIRE(!overlap(sy, plan[0]) && !overlap(sy, plan[1]) && !overlap(sy, plan[2]), QK_ERR_ALIAS,
                "projection %d: y overlaps counts, offsets or items", j);
        for (int i = 0; i < j; i++)
            REQUIRE(!overlap(sy, span(projs[i].y, (size_t)(rows * k * projs[i].N * 4))), QK_ERR_ALIAS,
                    "outputs of projections %d and %d overlap", i, j);
    }
    // the routed kernel counts its work items in int: (passes of any plan) x (row tiles) < 2^31
    int64_t tiles = 0;
    for (int j = 0; j < n_proj; j++) tiles += ceil_div(projs[j].N, UNIT_ROWS);
    REQUIRE(((rows * k + 7) / 8 + E) * tiles < (1LL << 31), QK_ERR_UNSUPPORTED,
            "rows * k * row tiles too large for one routed launch");
    for (int wt = QK_W_Q4_0; wt <= QK_W_Q8_0; wt++) {
        qk_proj_id group[8];
        int n = 0;
        for (int j = 0; j < n_proj; j++)
            if (projs[j].wtype == wt) group[n++] = projs[j];
        if (n == 0) continue;
        qk_status st = launch_mmvq_id(static_cast<const uint8_t *>(img), img_row_blocks, (int)rows, k, n, group,
                                      counts, offsets, items, per_pair, (cudaStream_t)stream);
        if (st != QK_OK) return st;
    }
    return QK_OK;
}

qk_status qk_mmvq_id(const void *img, int64_t img_row_blocks, int64_t rows, int32_t k, int32_t n_proj,
                     const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                     const int32_t *items, qk_stream stream) {
    return mmvq_id_common(img, img_row_blocks, rows, k, n_proj, projs, counts, offsets, items, false, stream);
}

qk_status qk_mmvq_id_slots(const void *img, int64_t img_row_blocks, int64_t rows, int32_t k, int32_t n_proj,
                           const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                           const int32_t *items, qk_stream stream) {
    return mmvq_id_common(img, img_row_blocks, rows, k, n_proj, projs, counts, offsets, items, true, stream);
}

qk_status qk_moe_combine(const float *expert_out, int64_t out_stride, const float *wts, int64_t rows, int32_t k,
                         int64_t N, float *y, int64_t y_stride, const int32_t *d_live_rows, qk_stream stream) {
    REQUIRE(expert_out && wts && y, QK_ERR_ARG, "null pointer");
    REQUIRE(rows >= 0 && rows <= (1 << 24) && k >= 1 && k <= 64 && N >= 1 && N <= (1LL << 25), QK_ERR_ARG,
            "rows, k or N out of range");
    REQUIRE(out_stride >= N && y_stride >= N, QK_ERR_SHAPE, "out_stride or y_stride < N");
    REQUIRE(aligned(expert_out, 16) && aligned(y, 16) && out_stride % 4 == 0 && y_stride % 4 == 0 && N % 4 == 0,
            QK_ERR_ARG, "expert_out and y must be 16-byte aligned with strides and N multiples of 4");
    Span se = span(expert_out, rows_span(rows * k, out_stride * 4, N * 4));
    Span sw = span(wts, (size_t)(rows * k * 4));
    Span sy = span(y, rows_span(rows, y_stride * 4, N * 4));
    REQUIRE(!overlap(sy, se) && !overlap(sy, sw), QK_ERR_ALIAS, "y overlaps expert_out or wts");
    if (rows == 0) return QK_OK;
    return launch_moe_combine(expert_out, out_stride, wts, (int)rows, k, (int)N, y, y_stride, d_live_rows,
                              (cudaStream_t)stream);
}

// ------------------------------------------------------------------ routing
qk_status qk_topk_route(const float *logits, int64_t rows, int32_t E, int32_t k, int32_t *ids, float *wts,
                        const int32_t *d_live_rows, qk_stream stream) {
    REQUIRE(logits && ids && wts, QK_ERR_ARG, "null pointer");
    REQUIRE(rows >= 0 && rows <= (1 << 24) && E >= 1 && k >= 1, QK_ERR_ARG, "rows, E or k out of range");
    REQUIRE(E <= 256 && k <= 32 && k <= E, QK_ERR_UNSUPPORTED, "E=%d k=%d (need E <= 256, k <= min(32, E))", E, k);
    Span sl = span(logits, (size_t)(rows * E * 4));
    Span si = span(ids, (size_t)(rows * k * 4));
    Span sw = span(wts, (size_t)(rows * k * 4));
    REQUIRE(!overlap(si, sl) && !overlap(sw, sl) && !overlap(si, sw), QK_ERR_ALIAS, "ids/wts overlap logits or each other");
    return launch_topk_route(logits, (int)rows, E, k, ids, wts, d_live_rows, (cudaStream_t)stream);
}

qk_status qk_moe_plan(const int32_t *ids, int64_t rows, int32_t k, int32_t E, int32_t *counts, int32_t *offsets,
                      int32_t *items, const int32_t *d_live_rows, qk_stream stream) {
    REQUIRE(ids && counts && offsets && items, QK_ERR_ARG, "null pointer");
    REQUIRE(rows >= 0 && rows <= (1 << 24) && k >= 1 && k <= 64 && E >= 1, QK_ERR_ARG, "rows, k or E out of range");
    REQUIRE(E <= 1024, QK_ERR_UNSUPPORTED, "E=%d > 1024", E);
    Span s_ids = span(ids, (size_t)(rows * k * 4));
    Span sc = span(counts, (size_t)E * 4), so = span(offsets, (size_t)(E + 1) * 4);
    Span sit = span(items, (size_t)(rows * k * 4));
    REQUIRE(!overlap(sc, s_ids) && !overlap(so, s_ids) && !overlap(sit, s_ids) && !overlap(sc, so) &&
                !overlap(sc, sit) && !overlap(so, sit),
            QK_ERR_ALIAS, "plan outputs overlap ids or each other");
    return launch_moe_plan(ids, (int)rows, k, E, counts, offsets, items, d_live_rows, (cudaStream_t)stream);
}

qk_status qk_route_plan(const float *logits, int64_t rows, int32_t E, int32_t k, int32_t *ids, float *wts,
                        int32_t *counts, int32_t *offsets, int32_t *items, const int32_t *d_live_rows,
                        qk_stream stream) {
    REQUIRE(logits && ids && wts && counts && offsets && items, QK_ERR_ARG, "null pointer");
    REQUIRE(rows >= 0 && rows <= (1 << 24) && E >= 1 && k >= 1, QK_ERR_ARG, "rows, E or k out of range");
    REQUIRE(E <= 256 && k <= 32 && k <= E, QK_ERR_UNSUPPORTED, "E=%d k=%d (need E <= 256, k <= min(32, E))", E, k);
    Span sl = span(logits, (size_t)(rows * E * 4));
    Span si = span(ids, (size_t)(rows * k * 4));
    Span sw = span(wts, (size_t)(rows * k * 4));
    Span sc = span(counts, (size_t)E * 4), so = span(offsets, (size_t)(E + 1) * 4);
    Span sit = span(items, (size_t)(rows * k * 4));
    const Span outs[5] = {si, sw, sc, so, sit};
    for (int a = 0; a < 5; a++) {
        REQUIRE(!overlap(outs[a], sl), QK_ERR_ALIAS, "an output overlaps logits");
        for (int b = 0; b < a; b++) REQUIRE(!overlap(outs[a], outs[b]), QK_ERR_ALIAS, "outputs overlap each other");
    }
    // rows == 0 still launches: like qk_moe_plan, the plan of no pairs writes zero counts and offsets
    return launch_route_plan(logits, (int)rows, E, k, ids, wts, counts, offsets, items, d_live_rows,
                             (cudaStream_t)stream);
}

// ------------------------------------------------------------------ prefill
size_t qk_mmq_workspace_bytes(int64_t T, int32_t n_proj, const qk_proj *projs) {
    if (T < 1 || n_proj < 1 || n_proj > 8 || !projs) return 0;
    int64_t kmax = 0;
    for (int j = 0; j < n_proj; j++) kmax = projs[j].K > kmax ? projs[j].K : kmax;
    return (size_t)mmq_workspace_bytes(T, kmax);
}

qk_status qk_mmq(const int8_t *qs, const uint16_t *d, int64_t row_blocks, int64_t T, int32_t n_proj,
                 const qk_proj *projs, void *ws, size_t ws_bytes, qk_stream stream) {
    REQUIRE(qs && d && projs, QK_ERR_ARG, "null pointer");
    REQUIRE(T >= 1 && T <= INT32_MAX && row_blocks >= 1, QK_ERR_ARG, "T or row_blocks out of range");
    REQUIRE(n_proj >= 1 && n_proj <= 8, QK_ERR_UNSUPPORTED, "n_proj=%d not in 1..8", (int)n_proj);
    REQUIRE(aligned(qs, 16) && aligned(d, 4), QK_ERR_ARG, "qs must be 16-byte and d 4-byte aligned");
    Span sq = span(qs, (size_t)(T * row_blocks * QB)), sd = span(d, (size_t)(T * row_blocks * 2));
    for (int j = 0; j < n_proj; j++) {
        const qk_proj &p = projs[j];
        qk_status st = check_proj_common(p.wtype, p.w, p.N, p.K, row_blocks);
        if (st != QK_OK) return st;
        REQUIRE(p.wtype == QK_W_Q4_0, QK_ERR_UNSUPPORTED, "qk_mmq takes Q4_0 weights");
        REQUIRE(p.y && p.y_stride >= p.N, QK_ERR_SHAPE, "projection %d: y null or y_stride < N", j);
        Span sy = span(p.y, rows_span(T, p.y_stride * 4, p.N * 4));
        REQUIRE(!overlap(sy, sq) && !overlap(sy, sd) && !overlap(sy, span(p.w, (size_t)packed_bytes(p.wtype, p.N, p.K))),
                QK_ERR_ALIAS, "projection %d: y overlaps an input", j);
        for (int i = 0; i < j; i++)
            REQUIRE(!rows_overlap(projs[i].y, projs[i].y_stride * 4, projs[i].N * 4, p.y, p.y_stride * 4, p.N * 4, T),
                    QK_ERR_ALIAS, "outputs of projections %d and %d overlap", i, j);
    }
    const size_t need = qk_mmq_workspace_bytes(T, n_proj, projs);
    REQUIRE(ws && aligned(ws, 128), QK_ERR_WORKSPACE, "workspace null or not 128-byte aligned");
    REQUIRE(ws_bytes >= need, QK_ERR_WORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
    Span sws = span(ws, need);
    REQUIRE(!overlap(sws, sq) && !overlap(sws, sd), QK_ERR_ALIAS, "workspace overlaps the image");
    for (int j = 0; j < n_proj; j++)
        REQUIRE(!overlap(sws, span(projs[j].y, rows_span(T, projs[j].y_stride * 4, projs[j].N * 4))) &&
                    !overlap(sws, span(projs[j].w, (size_t)packed_bytes(projs[j].wtype, projs[j].N, projs[j].K))),
                QK_ERR_ALIAS, "workspace overlaps projection %d", j);
    return launch_mmq(qs, d, row_blocks, (int)T, n_proj, projs, ws, ws_bytes, (cudaStream_t)stream);
}

}  // extern "C"

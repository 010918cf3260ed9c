// Router top-k, the stable expert plan and the weighted combine, all live-row
// aware (TensorFold PR #1047 "padding rows no longer go through routed experts",
// "The fix": router, top-k, plan and combine read the live-row count on the
// device and skip rows from it up; launches stay sized for the bucket).

#include "qk_internal.cuh"

namespace qk {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int MAX_E_PER_LANE = 8;   // E <= 256
constexpr int ROUTE_PLAN_MAX_ROWS = 32;   // fused top-k + plan: one row per warp of one CTA

// ---------------------------------------------------------------- top-k
// One warp per row; lane l holds experts l, l+32, ... Ranking by logit,
// larger first, equal logits to the lower expert index (exact f32 compares,
// so ids are reproducible bit for bit). Weights are the softmax probabilities
// of the chosen experts.
//
// Each pick is two warp reductions: the largest key, then the lowest expert
// index holding it. A logit's key is its bit pattern mapped so that unsigned
// order is float order (negative: all bits flipped; positive: sign bit set),
// after adding +0 so that -0 and +0 share a key, as they compare equal.
__device__ __forceinline__ unsigned order_key(float v) {
    const unsigned u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of row r (one warp): the logits are already in v (lane l: experts l, l+32, ...).
__device__ __forceinline__ void topk_row(const float v[MAX_E_PER_LANE], int r, int E, int k, int lane,
                                         int32_t *__restrict__ ids, float *__restrict__ wts) {
    unsigned key[MAX_E_PER_LANE];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < MAX_E_PER_LANE; i++) {
        const int e = lane + 32 * i;
        key[i] = e < E ? order_key(v[i]) : 0u;   // 0: below every logit, never picked
        if (e < E) mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < MAX_E_PER_LANE; i++)
        if (lane + 32 * i < E) z += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(FULL, z, o);

    for (int s = 0; s < k; s++) {
        unsigned bk = 0u;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < MAX_E_PER_LANE; i++)   // ascending expert index: strict > keeps the lowest on ties
            if (key[i] > bk) {
                bk = key[i];
                bi = lane + 32 * i;
            }
        const unsigned mk = __reduce_max_sync(FULL, bk);
        const int idx = (int)__reduce_min_sync(FULL, bk == mk && bk != 0u ? (unsigned)bi : 0x7fffffffu);
        if ((idx & 31) == lane) {
#pragma unroll
            for (int i = 0; i < MAX_E_PER_LANE; i++)
                if (i == (idx >> 5)) key[i] = 0u;   // taken
        }
        if (lane == 0) {
            ids[(int64_t)r * k + s] = idx;
            wts[(int64_t)r * k + s] = expf(key_value(mk) - mx) / z;
        }
    }
}

__device__ __forceinline__ void load_logits(const float *__restrict__ logits, int r, int E, int lane,
                                            float v[MAX_E_PER_LANE]) {
    const float *l = logits + (int64_t)r * E;
#pragma unroll
    for (int i = 0; i < MAX_E_PER_LANE; i++) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(l + e) : -INFINITY;
    }
}

__global__ void __launch_bounds__(256) topk_kernel(const float *__restrict__ logits, int rows, int E,
                                                   int k, int32_t *__restrict__ ids,
                                                   float *__restrict__ wts, const int32_t *live) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;   // warp-uniform
    // the row's logits are loaded together with the live count (row r < rows is in the
    // caller's buffer even when it is padding), so the two global reads overlap
    float v[MAX_E_PER_LANE];
    load_logits(logits, r, E, lane, v);
    if (r >= live_rows(live, rows)) return;   // warp-uniform
    topk_row(v, r, E, k, lane, ids, wts);
}

// ---------------------------------------------------------------- plan
// One CTA of 1024 threads (32 warps) for any width. Warp w owns a contiguous
// segment of the live pairs. Pass 1 counts each segment per expert (warp
// match, no atomics); then each expert's segment counts are prefix-summed
// over warps and the totals scanned over experts; pass 2 re-walks every
// segment in order and scatters, so each expert's items come out in
// ascending pair order (a stable counting sort). Pairs naming an expert
// outside [0, E) are left out of the plan.
// The plan of the first npairs pairs of ids, by one CTA of 1024 threads (ids read with plain
// loads: in the fused launch this CTA wrote them). sm: 32 * E + E + 1 ints of dynamic shared memory.
__device__ __forceinline__ void plan_body(const int32_t *ids, int npairs, int E, int32_t *__restrict__ counts,
                                          int32_t *__restrict__ offsets, int32_t *__restrict__ items,
                                          int32_t *sm, int32_t *wsum) {
    int32_t *seg = sm;                 // [32][E] per-warp counts, then per-warp bases
    int32_t *off = sm + 32 * E;        // [E + 1]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (npairs + 31) / 32;
    const int p_begin = warp * per, p_end = min(npairs, p_begin + per);
    const unsigned lt = (1u << lane) - 1u;

    for (int i = tid; i < 32 * E; i += 1024) seg[i] = 0;
    __syncthreads();

    for (int p0 = p_begin; p0 < p_end; p0 += 32) {
        const int p = p0 + lane;
        const int e = p < p_end ? ids[p] : -1;
        const bool ok = e >= 0 && e < E;
        const unsigned m = __match_any_sync(FULL, ok ? e : -1);
        if (ok && (m & lt) == 0) seg[warp * E + e] += __popc(m);
        __syncwarp();
    }
    __syncthreads();

    // per expert: prefix over warps (seg becomes the warp's base), total count
    for (int e = tid; e < E; e += 1024) {
        int s = 0;
        for (int w = 0; w < 32; w++) {
            const int c = seg[w * E + e];
            seg[w * E + e] = s;
            s += c;
        }
        counts[e] = s;
        off[e] = s;
    }
    __syncthreads();
    // exclusive scan of off[0..E) (E <= 1024: one value per thread)
    int v = tid < E ? off[tid] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int ws = wsum[lane];
        int wi = ws;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(FULL, wi, o);
            if (lane >= o) wi += n;
        }
        wsum[lane] = wi - ws;   // exclusive warp offsets
    }
    __syncthreads();
    const int excl = wsum[warp] + incl - v;
    __syncthreads();
    if (tid < E) off[tid] = excl;
    if (tid == E - 1) off[E] = excl + v;
    __syncthreads();
    for (int e = tid; e <= E; e += 1024) offsets[e] = off[e];

    for (int p0 = p_begin; p0 < p_end; p0 += 32) {
        const int p = p0 + lane;
        const int e = p < p_end ? ids[p] : -1;
        const bool ok = e >= 0 && e < E;
        const unsigned m = __match_any_sync(FULL, ok ? e : -1);
        if (ok) {
            const int rank = __popc(m & lt);
            items[off[e] + seg[warp * E + e] + rank] = p;
        }
        __syncwarp();
        if (ok && (m & lt) == 0) seg[warp * E + e] += __popc(m);
        __syncwarp();
    }
}


__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *__restrict__ ids, int rows, int k,
                                                    int E, int32_t *__restrict__ counts,
                                                    int32_t *__restrict__ offsets,
                                                    int32_t *__restrict__ items, const int32_t *live) {
    extern __shared__ int32_t sm[];
    __shared__ int32_t wsum[32];
    pdl_trigger();
    pdl_wait();
    plan_body(ids, live_rows(live, rows) * k, E, counts, offsets, items, sm, wsum);
}

// Top-k and plan in one CTA of 1024 threads for buckets of up to 32 rows (one row per warp):
// the same ids, weights and plan as the two launches, one launch boundary fewer on the path.
__global__ void __launch_bounds__(1024) route_plan_kernel(const float *__restrict__ logits, int rows, int E, int k,
                                                          int32_t *ids, float *__restrict__ wts,
                                                          int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                                          int32_t *__restrict__ items, const int32_t *live) {
    extern __shared__ int32_t sm[];
    __shared__ int32_t wsum[32];
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, r = threadIdx.x >> 5;
    float v[MAX_E_PER_LANE];
    if (r < rows) load_logits(logits, r, E, lane, v);
    const int n_live = live_rows(live, rows);
    if (r < n_live) topk_row(v, r, E, k, lane, ids, wts);
    __syncthreads();   // this CTA's ids are visible to all its threads
    plan_body(ids, n_live * k, E, counts, offsets, items, sm, wsum);
}

// ---------------------------------------------------------------- combine
// y[r][n] = sum over slots s (ascending) of wts[r][s] * expert_out[r*k + s][n], one binary32 fma
// per slot, for live rows r. Grid (rows, ceil(N/1024)); thread i of CTA (r, cy) handles columns
// 1024*cy + 4i .. +3 of row r.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ eo, int64_t eo_stride,
                                                      const float *__restrict__ wts, int rows, int k, int N,
                                                      float *__restrict__ y, int64_t y_stride, const int32_t *live) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    if (r >= live_rows(live, rows)) return;
    const int c = (blockIdx.y * 256 + threadIdx.x) * 4;
    if (c >= N) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < k; s++) {
        const float w = wts[(int64_t)r * k + s];
        const float4 e = *reinterpret_cast<const float4 *>(eo + ((int64_t)r * k + s) * eo_stride + c);
        acc.x = fmaf(w, e.x, acc.x);
        acc.y = fmaf(w, e.y, acc.y);
        acc.z = fmaf(w, e.z, acc.z);
        acc.w = fmaf(w, e.w, acc.w);
    }
    *reinterpret_cast<float4 *>(y + (int64_t)r * y_stride + c) = acc;
}

}  // namespace

qk_status launch_topk_route(const float *logits, int rows, int E, int k, int32_t *ids, float *wts,
                            const int32_t *live, cudaStream_t s) {
    if (rows == 0) return QK_OK;
    return launch_pdl("topk_route", topk_kernel, dim3((unsigned)ceil_div(rows, 8)), dim3(256), 0, s, logits, rows,
                      E, k, ids, wts, live);
}

qk_status launch_route_plan(const float *logits, int rows, int E, int k, int32_t *ids, float *wts, int32_t *counts,
                            int32_t *offsets, int32_t *items, const int32_t *live, cudaStream_t s) {
    if (rows > ROUTE_PLAN_MAX_ROWS) {   // one row per warp in one CTA: larger buckets use the two launches
        qk_status st = launch_topk_route(logits, rows, E, k, ids, wts, live, s);
        return st != QK_OK ? st : launch_moe_plan(ids, rows, k, E, counts, offsets, items, live, s);
    }
    const size_t smem = sizeof(int32_t) * (32 * (size_t)E + E + 1);
    static int configured = 0;
    if (smem > 48 * 1024 && configured < (int)smem) {
        cudaFuncSetAttribute(route_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        configured = (int)smem;
    }
    return launch_pdl("route_plan", route_plan_kernel, dim3(1), dim3(1024), smem, s, logits, rows, E, k, ids, wts,
                      counts, offsets, items, live);
}

qk_status launch_moe_plan(const int32_t *ids, int rows, int k, int E, int32_t *counts,
                          int32_t *offsets, int32_t *items, const int32_t *live, cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (32 * (size_t)E + E + 1);
    static int configured = 0;
    if (smem > 48 * 1024 && configured < (int)smem) {
        cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        configured = (int)smem;
    }
    return launch_pdl("moe_plan", plan_kernel, dim3(1), dim3(1024), smem, s, ids, rows, k, E, counts, offsets,
                      items, live);
}

qk_status launch_moe_combine(const float *expert_out, int64_t out_stride, const float *wts, int rows, int k, int N,
                             float *y, int64_t y_stride, const int32_t *live, cudaStream_t s) {
    dim3 grid((unsigned)rows, (unsigned)ceil_div(N, 1024));   // rows on x: up to 2^31-1 blocks
    return launch_pdl("moe_combine", combine_kernel, grid, dim3(256), 0, s, expert_out, out_stride, wts, rows, k, N,
                      y, y_stride, live);
}
}  // namespace qk

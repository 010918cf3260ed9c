// Router top-k and the stable expert plan, both live-row aware
// (TensorFold PR #1047 "padding rows no longer go through routed experts",
// "The fix": router, top-k and plan read the live-row count on the device and
// skip rows from it up; launches stay sized for the bucket).

#include "qk_internal.cuh"

namespace qk {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int MAX_E_PER_LANE = 8;   // E <= 256

// ---------------------------------------------------------------- top-k
// One warp per row; lane l holds experts l, l+32, ... Ranking by logit,
// larger first, equal logits to the lower expert index (exact f32 compares,
// so ids are reproducible bit for bit). Weights are the softmax probabilities
// of the chosen experts.
__global__ void __launch_bounds__(256) topk_kernel(const float *__restrict__ logits, int rows, int E,
                                                   int k, int32_t *__restrict__ ids,
                                                   float *__restrict__ wts, const int32_t *live) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= live_rows(live, rows)) return;   // warp-uniform
    const float *l = logits + (int64_t)r * E;
    float v[MAX_E_PER_LANE];
    int n = 0;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < MAX_E_PER_LANE; i++) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldg(l + e) : -INFINITY;
        if (e < E) { mx = fmaxf(mx, v[i]); n++; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
    float z = 0.0f;
#pragma unroll
    for (int i = 0; i < MAX_E_PER_LANE; i++)
        if (lane + 32 * i < E) z += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(FULL, z, o);

    unsigned taken = 0;   // bit i: expert lane + 32 i already chosen
    for (int s = 0; s < k; s++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < MAX_E_PER_LANE; i++) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi) || bi == 0x7fffffff)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(FULL, bv, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == 0) {
            ids[(int64_t)r * k + s] = bi;
            wts[(int64_t)r * k + s] = expf(bv - mx) / z;
        }
    }
    (void)n;
}

// ---------------------------------------------------------------- plan
// One CTA of 1024 threads (32 warps) for any width. Warp w owns a contiguous
// segment of the live pairs. Pass 1 counts each segment per expert (warp
// match, no atomics); then each expert's segment counts are prefix-summed
// over warps and the totals scanned over experts; pass 2 re-walks every
// segment in order and scatters, so each expert's items come out in
// ascending pair order (a stable counting sort). Pairs naming an expert
// outside [0, E) are left out of the plan.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t *__restrict__ ids, int rows, int k,
                                                    int E, int32_t *__restrict__ counts,
                                                    int32_t *__restrict__ offsets,
                                                    int32_t *__restrict__ items, const int32_t *live) {
    extern __shared__ int32_t sm[];
    int32_t *seg = sm;                 // [32][E] per-warp counts, then per-warp bases
    int32_t *off = sm + 32 * E;        // [E + 1]
    __shared__ int32_t wsum[32];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int npairs = live_rows(live, rows) * k;
    const int per = (npairs + 31) / 32;
    const int p_begin = warp * per, p_end = min(npairs, p_begin + per);
    const unsigned lt = (1u << lane) - 1u;

    for (int i = tid; i < 32 * E; i += 1024) seg[i] = 0;
    __syncthreads();

    for (int p0 = p_begin; p0 < p_end; p0 += 32) {
        const int p = p0 + lane;
        const int e = p < p_end ? __ldg(ids + p) : -1;
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
        const int e = p < p_end ? __ldg(ids + p) : -1;
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

}  // namespace

qk_status launch_topk_route(const float *logits, int rows, int E, int k, int32_t *ids, float *wts,
                            const int32_t *live, cudaStream_t s) {
    if (rows == 0) return QK_OK;
    return launch_pdl("topk_route", topk_kernel, dim3((unsigned)ceil_div(rows, 8)), dim3(256), 0, s, logits, rows,
                      E, k, ids, wts, live);
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

}  // namespace qk

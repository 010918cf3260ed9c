// Q8 activation images and the producers that emit them.
//
//   quantize_q8_1 / quantize_q8_0 : standalone quantisers (llama.cpp PR #117
//       "activation image emission", Coverage: the standard Q8_1 image;
//       minfer doc 52 "r49 A-quantize prepass shared-A dedup", section 1: the
//       Q8_0 prepass with per-32-block amax, rintf scaling and zero pad).
//   rmsnorm_q8_1 / glu_q8_1       : producers that write their original F32
//       output and the Q8_1 image of exactly the stored values (PR #117,
//       Coverage: RMS and F32 GLU producers emit the image).
//
// Work layout: every quant block of 32 elements is handled by 8 consecutive
// lanes, 4 elements each, so a warp quantises 4 blocks at once with 3-step
// xor shuffles for the block max and the code sum. All block arithmetic is
// binary32 with IEEE division (no fast-math in this file), the codes use
// round-to-nearest-even and the halves use __float2half_rn.

#include "qk_internal.cuh"

namespace qk {
namespace {

constexpr unsigned FULL = 0xffffffffu;

// Four consecutive floats from p (16-byte aligned fast path, else scalar with
// a bound: elements at index >= n read as 0).
__device__ __forceinline__ void load4(const float *p, int n, float v[4]) {
    if (n >= 4 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
        float4 t = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) v[i] = i < n ? __ldg(p + i) : 0.0f;
    }
}

__device__ __forceinline__ void store4(float *p, const float v[4]) {
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) p[i] = v[i];
    }
}

// Quantises one 32-element block held by 8 lanes (4 values each; j8 = the
// lane's index in its group). All 32 lanes of the warp must call this.
// Returns the binary32 scale d; codes are packed little-endian into *codes
// and the block's code sum into *sum.
// ZEROS: for inputs where exact zeros are common (ReGLU outputs: half of them), zeros skip the
// division (the same codes; a division of zero measured slower on this GPU).
template <bool ZEROS = false>
__device__ __forceinline__ float q8_block(const float v[4], uint32_t *codes, int *sum) {
    float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 1));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 2));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 4));
    const float d = a / 127.0f;
    int q[4] = {0, 0, 0, 0};
    if (a != 0.0f) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            if (ZEROS) {   // a zero's code is 0: its quotient is taken as 1 / 1 and dropped
                const bool z = v[i] == 0.0f;
                const int qi = __float2int_rn((z ? d : v[i]) / d);
                q[i] = z ? 0 : qi;
            } else {
                q[i] = __float2int_rn(v[i] / d);
            }
        }
    }
    int s = q[0] + q[1] + q[2] + q[3];
    s += __shfl_xor_sync(FULL, s, 1);
    s += __shfl_xor_sync(FULL, s, 2);
    s += __shfl_xor_sync(FULL, s, 4);
    *codes = (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) |
             ((uint32_t)(q[2] & 0xff) << 16) | ((uint32_t)(q[3] & 0xff) << 24);
    *sum = s;
    return d;
}

// Writes lane j8's share of a Q8_1 block: codes at bytes 4+4*j8, and for
// j8 == 0 the header [half d][half d*sum].
__device__ __forceinline__ void put_q8_1(uint8_t *blk, int j8, float d, uint32_t codes, int sum) {
    reinterpret_cast<uint32_t *>(blk + 4)[j8] = codes;
    if (j8 == 0) {
        __half2 h = __halves2half2(__float2half_rn(d), __float2half_rn(d * (float)sum));
        *reinterpret_cast<__half2 *>(blk) = h;
    }
}

// ---------------------------------------------------------------- quantizers
// grid (T, ceil(row_blocks / (G*QPB))), NT threads, G = NT / 8 lane groups: lane group m of
// warp w handles blocks G*QPB*blockIdx.y + G*j + 4*w + m (j < QPB) of row blockIdx.x (rows on
// x: up to 2^31-1). A lane loads its QPB float4s before it quantises, so that large images
// keep several loads per thread in flight, while small ones spread over more CTAs (QPB = 1).
// Large images with rows of at most 128 blocks take a 128-thread CTA per row with QPB =
// ceil(row_blocks / 16) (more rows in flight per SM, few idle lanes), wider rows 256 threads
// with QPB = 4. Every block is quantised on its own, so the bytes do not depend on the shape.
template <bool Q81, int QPB, int NT = 256>
__global__ void __launch_bounds__(NT) quantize_kernel(const float *__restrict__ x, int K,
                                                       int64_t x_stride, uint8_t *__restrict__ out,
                                                       int8_t *__restrict__ qs, uint16_t *__restrict__ dh,
                                                       int64_t row_blocks, int T, const int32_t *live) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, j8 = lane & 7;
    constexpr int G = NT / 8;
    const int64_t b0 = (int64_t)blockIdx.y * G * QPB + (threadIdx.x >> 5) * 4 + (lane >> 3);
    float v[QPB][4];
    // the row's values are loaded together with the live count (row t < T is in the caller's
    // buffer even when it is padding), so the global reads overlap
#pragma unroll
    for (int j = 0; j < QPB; j++) {
        const int64_t b = b0 + G * j, col = b * QB + 4 * j8;
        v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.0f;
        if (b < row_blocks && col < K) load4(x + t * x_stride + col, (int)(K - col < 4 ? K - col : 4), v[j]);
    }
    if (t >= live_rows(live, T)) return;
#pragma unroll
    for (int j = 0; j < QPB; j++) {
        const int64_t b = b0 + G * j;
        uint32_t codes;
        int sum;
        const float d = q8_block(v[j], &codes, &sum);   // all lanes take part in the shuffles
        if (b >= row_blocks) continue;                   // whole 8-lane group agrees
        if (Q81) {
            put_q8_1(out + (t * row_blocks + b) * Q8_1_BYTES, j8, d, codes, sum);
        } else {
            reinterpret_cast<uint32_t *>(qs + (t * row_blocks + b) * QB)[j8] = codes;
            if (j8 == 0) dh[t * row_blocks + b] = __half_as_ushort(__float2half_rn(d));
        }
    }
}

// ---------------------------------------------------------------- RMS producer
// One CTA per row; the row stays in registers between the sum of squares and
// the output. The reference shape is 1024 threads (thread i holds columns
// 4i + 4096*it for it < ITEMS, ITEMS = 1, 2, 4 or 8 by K, so K <= 32768). For
// many rows a smaller CTA takes the row instead (128 threads for K <= 4096,
// eight rows in flight per SM; 256 threads for K <= 8192, four): its thread j
// plays the reference threads j + NT*m (m < 1024 / NT) and reduces their
// partial sums in the same order (one warp tree per m, then the same 32-entry
// tree), so the bits are those of the 1024-thread shape.
// With ITEMS <= 2 the weight and bias are loaded together with the row, before
// the reduction.
constexpr int RMS_THREADS = 1024;
constexpr int RMS_ITEMS = 8;
constexpr int RMS_ROWS_FOR_SMALL = 256;   // rows from which the 256-thread shape is used

// Q81: the image is Q8_1 blocks (img); else Q8_0 split planes (qs codes, dh half scales), the
// prefill layout that qk_mmq reads.
template <int NT, int ITEMS, bool Q81>
__global__ void __launch_bounds__(NT, RMS_THREADS / NT) rmsnorm_q8_1_kernel(
    const float *__restrict__ x, int K, int64_t x_stride, int kind, const float *__restrict__ w,
    const float *__restrict__ bias, float scale, float eps, float *__restrict__ y, int64_t y_stride,
    uint8_t *__restrict__ img, int8_t *__restrict__ qs, uint16_t *__restrict__ dh, int64_t row_blocks, int T,
    const int32_t *live) {
    constexpr bool EARLY = ITEMS <= 2;   // registers for the weight and bias next to the row
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    const float *xr = x + t * x_stride;
    const int tid = threadIdx.x, lane = tid & 31, j8 = lane & 7;
    const bool use_w = kind == QK_NORM_MUL || kind == QK_NORM_MUL_ADD, use_b = kind == QK_NORM_MUL_ADD;

    // the row (and with EARLY its weight and bias) is loaded together with the live count (row
    // t < T is in the caller's buffer even when it is padding), so the global reads overlap
    float v[ITEMS][4], wv[EARLY ? ITEMS : 1][4], bv[EARLY ? ITEMS : 1][4];
#pragma unroll
    for (int it = 0; it < ITEMS; it++) {
        const int c = 4 * tid + 4 * NT * it;
        v[it][0] = v[it][1] = v[it][2] = v[it][3] = 0.0f;
        if (c < K) {
            load4(xr + c, 4, v[it]);
            if (EARLY && use_w) load4(w + c, 4, wv[EARLY ? it : 0]);
            if (EARLY && use_b) load4(bias + c, 4, bv[EARLY ? it : 0]);
        }
    }
    if (t >= live_rows(live, T)) return;
    // reference thread j + NT*m holds items m, m + R, m + 2R, ... of this thread (R = 1024 / NT)
    constexpr int R = RMS_THREADS / NT;
    __shared__ float red[RMS_THREADS / 32];
#pragma unroll
    for (int m = 0; m < R; m++) {
        float ss = 0.0f;
#pragma unroll
        for (int it = m; it < ITEMS; it += R)
            ss += v[it][0] * v[it][0] + v[it][1] * v[it][1] + v[it][2] * v[it][2] + v[it][3] * v[it][3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
        if (lane == 0) red[(tid >> 5) + m * (NT / 32)] = ss;
    }
    __syncthreads();
    if (tid < 32) {
        float tot = red[tid];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
        if (tid == 0) red[0] = 1.0f / sqrtf(tot / (float)K + eps);
    }
    __syncthreads();
    const float r = red[0];

    float *yr = y + t * y_stride;
    uint8_t *ir = Q81 ? img + t * row_blocks * Q8_1_BYTES : nullptr;
    int8_t *qr = Q81 ? nullptr : qs + t * row_blocks * QB;
    uint16_t *dr = Q81 ? nullptr : dh + t * row_blocks;
#pragma unroll
    for (int it = 0; it < ITEMS; it++) {
        if (4 * NT * it >= K) break;                        // uniform: no warp has columns left
        const int c = 4 * tid + 4 * NT * it;
        const bool ok = c < K;                               // K % 32 == 0: whole 8-lane groups agree
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
            float wl[4], bl[4];
            const float *wq = wl, *bq = bl;
            if (EARLY) {
                wq = wv[EARLY ? it : 0];
                bq = bv[EARLY ? it : 0];
            } else {
                if (use_w) load4(w + c, 4, wl);
                if (use_b) load4(bias + c, 4, bl);
            }
#pragma unroll
            for (int i = 0; i < 4; i++) {
                float q = v[it][i] * r;
                if (kind == QK_NORM_MUL) q = q * wq[i];
                else if (kind == QK_NORM_MUL_ADD) q = q * wq[i] + bq[i];
                else if (kind == QK_NORM_SCALE) q = q * scale;
                o[i] = q;
            }
            store4(yr + c, o);
        }
        uint32_t codes;
        int sum;
        const float d = q8_block(o, &codes, &sum);   // all lanes of the warp take part
        if (ok) {
            if (Q81) {
                put_q8_1(ir + (int64_t)(c / QB) * Q8_1_BYTES, j8, d, codes, sum);
            } else {
                reinterpret_cast<uint32_t *>(qr + (int64_t)(c / QB) * QB)[j8] = codes;
                if (j8 == 0) dr[c / QB] = __half_as_ushort(__float2half_rn(d));
            }
        }
    }
    // zero blocks of the row padding
    for (int64_t bb = K / QB + tid; bb < row_blocks; bb += NT) {
        if (Q81) {
            uint32_t *p = reinterpret_cast<uint32_t *>(ir + bb * Q8_1_BYTES);
#pragma unroll
            for (int i = 0; i < 9; i++) p[i] = 0u;
        } else {
            uint32_t *p = reinterpret_cast<uint32_t *>(qr + bb * QB);
#pragma unroll
            for (int i = 0; i < 8; i++) p[i] = 0u;
            dr[bb] = 0;
        }
    }
}

// ---------------------------------------------------------------- GLU producer
// act(g) * u for the GLU kinds; SwiGLU-OAI and SwiGLU-clamp clamp g from above and u both
// ways at limit (SwiGLU-OAI also scales the gate by alpha and multiplies by u + 1).
__device__ __forceinline__ float glu_out(int kind, float g, float u, float alpha, float limit) {
    switch (kind) {
        case QK_GLU_SWIGLU: return g / (1.0f + expf(-g)) * u;
        case QK_GLU_GEGLU_TANH: {
            const float c = 0.7978845608028654f;  // sqrt(2/pi)
            return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g))) * u;
        }
        case QK_GLU_GEGLU_ERF: return 0.5f * g * (1.0f + erff(g * 0.7071067811865476f)) * u;
        case QK_GLU_GEGLU_QUICK: return g / (1.0f + expf(-1.702f * g)) * u;
        case QK_GLU_SWIGLU_OAI: {
            const float x = fminf(g, limit), v = fminf(fmaxf(u, -limit), limit);
            return x / (1.0f + expf(-alpha * x)) * (v + 1.0f);
        }
        case QK_GLU_SWIGLU_CLAMP: {
            const float x = fminf(g, limit), v = fminf(fmaxf(u, -limit), limit);
            return x / (1.0f + expf(-x)) * v;
        }
        default: return fmaxf(g, 0.0f) * u;
    }
}

// grid (T, ceil(N/1024)), 256 threads; thread i of CTA (t, cy) handles columns 1024*cy + 4i of row t.
__global__ void __launch_bounds__(256) glu_q8_1_kernel(
    int kind, int layout, const float *__restrict__ a, int64_t a_stride, const float *__restrict__ b,
    int64_t b_stride, int N, float *__restrict__ out, int64_t out_stride, uint8_t *__restrict__ img,
    int64_t row_blocks, int T, float alpha, float limit, const int32_t *live) {
    pdl_trigger();
    pdl_wait();
    const int t = blockIdx.x;
    const int tid = threadIdx.x, j8 = tid & 7;
    const int c = blockIdx.y * 1024 + 4 * tid;
    const float *g, *u;
    if (layout == QK_GLU_SEPARATE) {
        g = a + t * a_stride;
        u = b + t * b_stride;
    } else if (layout == QK_GLU_PACKED) {
        g = a + t * a_stride;
        u = g + N;
    } else {
        u = a + t * a_stride;
        g = u + N;
    }
    const bool ok = c < N;
    // the inputs are loaded together with the live count (row t < T is in the caller's
    // buffers even when it is padding), so the global reads overlap
    float gv[4] = {0.f, 0.f, 0.f, 0.f}, uv[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
        load4(g + c, 4, gv);
        load4(u + c, 4, uv);
    }
    if (t >= live_rows(live, T)) return;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
#pragma unroll
        for (int i = 0; i < 4; i++) v[i] = glu_out(kind, gv[i], uv[i], alpha, limit);
        store4(out + t * out_stride + c, v);
    }
    uint32_t codes;
    int sum;
    const float d = kind == QK_GLU_REGLU ? q8_block<true>(v, &codes, &sum) : q8_block(v, &codes, &sum);
    uint8_t *ir = img + t * row_blocks * Q8_1_BYTES;
    if (ok) put_q8_1(ir + (int64_t)(c / QB) * Q8_1_BYTES, j8, d, codes, sum);
    if (blockIdx.y == 0) {  // zero blocks of the row padding
        for (int64_t bb = N / QB + tid; bb < row_blocks; bb += 256) {
            uint32_t *p = reinterpret_cast<uint32_t *>(ir + bb * Q8_1_BYTES);
#pragma unroll
            for (int i = 0; i < 9; i++) p[i] = 0u;
        }
    }
}

constexpr int64_t QUANT_BIG_BLOCKS = 1 << 17;   // blocks per call from which QPB = 4 is used

}  // namespace

// Large images with rows of at most 128 blocks: one 128-thread CTA per row (QPB = ceil(rb / 16)).
template <bool Q81>
static qk_status launch_quantize_rows128(const char *name, const float *x, int T, int K, int64_t x_stride,
                                         uint8_t *img, int8_t *qs, uint16_t *d, int64_t row_blocks,
                                         const int32_t *live, cudaStream_t s) {
    const int qpb = (int)ceil_div(row_blocks, 16);
    auto kernel = qpb <= 5   ? quantize_kernel<Q81, 5, 128>
                  : qpb == 6 ? quantize_kernel<Q81, 6, 128>
                  : qpb == 7 ? quantize_kernel<Q81, 7, 128>
                             : quantize_kernel<Q81, 8, 128>;
    return launch_pdl(name, kernel, dim3((unsigned)T, 1u), dim3(128), 0, s, x, K, x_stride, img, qs, d, row_blocks,
                      T, live);
}

qk_status launch_quantize_q8_1(const float *x, int T, int K, int64_t x_stride, uint8_t *img,
                               int64_t row_blocks, const int32_t *live, cudaStream_t s) {
    if (T == 0) return QK_OK;
    const bool big = (int64_t)T * row_blocks >= QUANT_BIG_BLOCKS;
    if (big && row_blocks > 64 && row_blocks <= 128)
        return launch_quantize_rows128<true>("quantize_q8_1", x, T, K, x_stride, img, nullptr, nullptr, row_blocks,
                                             live, s);
    dim3 grid((unsigned)T, (unsigned)ceil_div(row_blocks, big ? 128 : 32));
    return launch_pdl("quantize_q8_1", big ? quantize_kernel<true, 4> : quantize_kernel<true, 1>, grid, dim3(256),
                      0, s, x, K, x_stride, img, (int8_t *)nullptr, (uint16_t *)nullptr, row_blocks, T, live);
}

qk_status launch_quantize_q8_0(const float *x, int T, int K, int64_t x_stride, int8_t *qs,
                               uint16_t *d, int64_t row_blocks, const int32_t *live, cudaStream_t s) {
    if (T == 0) return QK_OK;
    const bool big = (int64_t)T * row_blocks >= QUANT_BIG_BLOCKS;
    if (big && row_blocks > 64 && row_blocks <= 128)
        return launch_quantize_rows128<false>("quantize_q8_0", x, T, K, x_stride, nullptr, qs, d, row_blocks, live,
                                              s);
    dim3 grid((unsigned)T, (unsigned)ceil_div(row_blocks, big ? 128 : 32));
    return launch_pdl("quantize_q8_0", big ? quantize_kernel<false, 4> : quantize_kernel<false, 1>, grid,
                      dim3(256), 0, s, x, K, x_stride, (uint8_t *)nullptr, qs, d, row_blocks, T, live);
}

template <bool Q81>
static qk_status launch_rmsnorm(const float *x, int T, int K, int64_t x_stride, int kind, const float *w,
                                const float *b, float scale, float eps, float *y, int64_t y_stride, uint8_t *img,
                                int8_t *qs, uint16_t *dh, int64_t row_blocks, const int32_t *live, cudaStream_t s) {
    if (T == 0) return QK_OK;
    const int per = 4 * RMS_THREADS;   // columns per item of the reference shape
    if (T >= RMS_ROWS_FOR_SMALL && K <= 2 * per) {   // 256 threads, four times the items
        if (K <= per)   // 128 threads: eight rows in flight per SM
            return launch_pdl(Q81 ? "rmsnorm_q8_1" : "rmsnorm_q8_0", rmsnorm_q8_1_kernel<128, 8, Q81>,
                              dim3((unsigned)T), dim3(128), 0, s, x, K, x_stride, kind, w, b, scale, eps, y, y_stride,
                              img, qs, dh, row_blocks, T, live);
        return launch_pdl(Q81 ? "rmsnorm_q8_1" : "rmsnorm_q8_0", rmsnorm_q8_1_kernel<256, 8, Q81>, dim3((unsigned)T),
                          dim3(256), 0, s, x, K, x_stride, kind, w, b, scale, eps, y, y_stride, img, qs, dh,
                          row_blocks, T, live);
    }
    auto kernel = K <= per ? rmsnorm_q8_1_kernel<RMS_THREADS, 1, Q81>
                  : K <= 2 * per ? rmsnorm_q8_1_kernel<RMS_THREADS, 2, Q81>
                  : K <= 4 * per ? rmsnorm_q8_1_kernel<RMS_THREADS, 4, Q81>
                                 : rmsnorm_q8_1_kernel<RMS_THREADS, RMS_ITEMS, Q81>;
    return launch_pdl(Q81 ? "rmsnorm_q8_1" : "rmsnorm_q8_0", kernel, dim3((unsigned)T), dim3(RMS_THREADS), 0, s, x,
                      K, x_stride, kind, w, b, scale, eps, y, y_stride, img, qs, dh, row_blocks, T, live);
}

qk_status launch_rmsnorm_q8_1(const float *x, int T, int K, int64_t x_stride, int kind,
                              const float *w, const float *b, float scale, float eps, float *y,
                              int64_t y_stride, uint8_t *img, int64_t row_blocks,
                              const int32_t *live, cudaStream_t s) {
    return launch_rmsnorm<true>(x, T, K, x_stride, kind, w, b, scale, eps, y, y_stride, img, nullptr, nullptr,
                                row_blocks, live, s);
}

qk_status launch_rmsnorm_q8_0(const float *x, int T, int K, int64_t x_stride, int kind, const float *w,
                              const float *b, float scale, float eps, float *y, int64_t y_stride, int8_t *qs,
                              uint16_t *dh, int64_t row_blocks, const int32_t *live, cudaStream_t s) {
    return launch_rmsnorm<false>(x, T, K, x_stride, kind, w, b, scale, eps, y, y_stride, nullptr, qs, dh,
                                 row_blocks, live, s);
}

qk_status launch_glu_q8_1(int kind, int layout, const float *a, int64_t a_stride, const float *b,
                          int64_t b_stride, int T, int N, float *out, int64_t out_stride,
                          uint8_t *img, int64_t row_blocks, float alpha, float limit, const int32_t *live,
                          cudaStream_t s) {
    if (T == 0) return QK_OK;
    dim3 grid((unsigned)T, (unsigned)ceil_div(N, 1024));
    return launch_pdl("glu_q8_1", glu_q8_1_kernel, grid, dim3(256), 0, s, kind, layout, a, a_stride, b, b_stride,
                      N, out, out_stride, img, row_blocks, T, alpha, limit, live);
}

}  // namespace qk

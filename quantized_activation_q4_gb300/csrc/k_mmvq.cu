// Quantised-weight projections that read one shared Q8_1 activation image.
//
//   mmvq    : ordinary MUL_MAT, several projections (q/k/v, gate/up) in one
//             launch (llama.cpp PR #117 "activation image emission",
//             Overview/Coverage; its "Ordinary, K8192 / T8" component).
//   mmvq_id : routed MUL_MAT_ID over a stable expert plan; experts with no
//             planned pair read no weights (TensorFold PR #1047, "The fix").
//
// Per 32-block b of weight row n and image row t, from the stored halves:
//   Q4_0: y += d_w * (d_a * D - 8 * s_a),   D = sum nibble_i * q_i
//   Q8_0: y += d_w * (d_a * D),             D = sum w_i * q_i
//
// GB300 design. The exact integer block dot D runs on the f16 tensor path:
// nibbles, int8 weights and int8 codes are all exact in binary16, products
// are exact and every partial sum stays below 2^22, so the f32 accumulator
// holds D exactly. (Blackwell Ultra's int8 MMA and dp4a rates are a quarter
// of its f16 rate, too low to keep up with HBM at 8 tokens.) A nibble becomes
// a half in one logic op by OR-ing it under a binary16 exponent (1024 + lo for
// low nibbles, 64 + hi for high nibbles); the resulting bias sum_i bias * q_i
// depends only on the token, so one pair of MMAs with a constant -bias A
// operand per block yields it, and it seeds the accumulator of every row
// group. Weights stream once from HBM with 128-bit no-L1-allocate loads in a
// tile order written by qk_weight_pack; the small image is read through L1.
//
// CTA: NW warps share RG 16-row groups and split their K chunks (128 columns
// each); partial sums are reduced across warps in shared memory and across
// the CTAs of a thread-block cluster (split K) through distributed shared
// memory, always in the same order, so results are deterministic.

#include <cooperative_groups.h>

#include "qk_internal.cuh"

namespace cg = cooperative_groups;

namespace qk {
namespace {

constexpr int MAX_PROJ = 8;
constexpr int NW = 8;   // warps per CTA
constexpr int RG = 2;   // 16-row groups per CTA

struct ProjDesc {
    const uint8_t *w;        // packed tiles (expert 0 for routed)
    float *y;
    int64_t y_stride;        // elements between output rows of consecutive tokens / pairs
    int64_t expert_bytes;    // routed: bytes per expert's packed matrix
    int N, K;
    int n_groups;            // ceil(N/16)
    int chunks;              // ceil(K/128)
    int row_tiles;           // ceil(n_groups / RG)
    int experts;             // routed: E; ordinary: 1
    int tiles_begin;         // first tile index of this projection
};

struct Args {
    const uint8_t *img;
    int64_t img_row_bytes;
    int T;                   // image rows (tokens or bucket rows)
    const int32_t *live;     // ordinary only
    int n_proj;
    int ksplit;              // cluster size along K
    const int32_t *counts, *offsets, *items;  // routed plan
    int k;                   // routed: slots per row
    ProjDesc p[MAX_PROJ];
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream8(const void *p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_img4(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}

// D = A * B + C for one m16n8k16 f16 MMA with f32 accumulators.
__device__ __forceinline__ void mma_f16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four int8 codes (bytes c0..c3 of w) -> two exact half2: (c0, c2) and (c1, c3).
// XOR 0x80 makes u = c + 128 in 1..255; under the exponent of 1024 the half
// 0x64uu is 1024 + u; subtracting 1152 leaves c exactly.
__device__ __forceinline__ void codes_to_half2(uint32_t w, uint32_t &h02, uint32_t &h13) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4240);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4341);
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    h02 = *reinterpret_cast<uint32_t *>(&ha);
    h13 = *reinterpret_cast<uint32_t *>(&hb);
}

// Four Q4_0 nibble bytes (B0..B3) -> biased halves for the two MMAs of a block:
//   lo02 = (1024+lo(B0), 1024+lo(B2)), lo13 = (1024+lo(B1), 1024+lo(B3))
//   hi02 = (  64+hi(B0),   64+hi(B2)), hi13 = (  64+hi(B1),   64+hi(B3))
__device__ __forceinline__ void nibbles_to_half2(uint32_t w, uint32_t &lo02, uint32_t &lo13,
                                                 uint32_t &hi02, uint32_t &hi13) {
    const uint32_t w8 = w >> 8;
    lo02 = (w & 0x000F000Fu) | 0x64006400u;
    hi02 = (w & 0x00F000F0u) | 0x54005400u;
    lo13 = (w8 & 0x000F000Fu) | 0x64006400u;
    hi13 = (w8 & 0x00F000F0u) | 0x54005400u;
}

// Q8_0 weight codes keep the +1152 bias (removed by the correction MMAs).
__device__ __forceinline__ void wcodes_to_half2(uint32_t w, uint32_t &h02, uint32_t &h13) {
    const uint32_t u = w ^ 0x80808080u;
    h02 = __byte_perm(u, 0x64646464u, 0x4240);
    h13 = __byte_perm(u, 0x64646464u, 0x4341);
}

__device__ __forceinline__ float half_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xffffu))); }
__device__ __forceinline__ float half_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

// ---------------------------------------------------------------- the kernel
//
// Fragment map (m16n8k16, lane = 4g + t): A rows g and g+8, B column (token) g,
// C rows g, g+8 and columns (tokens) 2t, 2t+1. Within a 32-block, MMA 0 takes
// the elements 4t..4t+3 and MMA 1 the elements 16+4t..16+4t+3, in the order
// (4t, 4t+2 | 4t+1, 4t+3) on both the A and the B side.
template <int WT, bool ROUTED>
__global__ void __launch_bounds__(NW * 32) mmvq_kernel(const __grid_constant__ Args args) {
    constexpr int TILE = WT == QK_W_Q4_0 ? Q4_TILE_BYTES : Q8_TILE_BYTES;
    constexpr int SCALE_OFF = WT == QK_W_Q4_0 ? 1024 : 2048;
    constexpr int HALF_OFF = WT == QK_W_Q4_0 ? 512 : 1024;   // rows g+8
    // constant A operand of the correction MMAs (-bias of each half)
    constexpr uint32_t NEG_BIAS_LO = WT == QK_W_Q4_0 ? 0xE400E400u : 0xE480E480u;  // -1024 | -1152
    constexpr uint32_t NEG_BIAS_HI = WT == QK_W_Q4_0 ? 0xD400D400u : 0xE480E480u;  //   -64 | -1152

    __shared__ float red[NW][RG * 4][32];
    __shared__ int tok_img[8], tok_out[8];

    const int C = args.ksplit;
    const int rank = (int)(blockIdx.x % (unsigned)C);
    const int tile = (int)(blockIdx.x / (unsigned)C);
    int j = 0;
#pragma unroll 1
    while (j + 1 < args.n_proj && tile >= args.p[j + 1].tiles_begin) j++;
    const ProjDesc &P = args.p[j];
    const int local = tile - P.tiles_begin;
    const int e = ROUTED ? local / P.row_tiles : 0;
    const int rt = ROUTED ? local % P.row_tiles : local;
    const int g0 = rt * RG;

    int n_items = 0, item0 = 0;
    if (ROUTED) {
        n_items = __ldg(args.counts + e);
        if (n_items <= 0) return;          // uniform over the cluster: no weights read
        item0 = __ldg(args.offsets + e);
    }
    const uint8_t *wbase = P.w + (ROUTED ? (int64_t)e * P.expert_bytes : 0);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int Kb = P.K / QB;
    const int per = (P.chunks + C - 1) / C;
    const int c_begin = rank * per;
    const int c_end = min(P.chunks, c_begin + per);
    const int n_passes = ROUTED ? (n_items + 7) / 8 : 1;

    for (int pass = 0; pass < n_passes; pass++) {
        if (threadIdx.x < 8) {
            const int s = threadIdx.x;
            if (ROUTED) {
                const int idx = pass * 8 + s;
                int p = idx < n_items ? __ldg(args.items + item0 + idx) : -1;
                if (p < 0 || p / args.k >= args.T) p = -1;     // not a pair of this bucket: skip
                tok_img[s] = p >= 0 ? p / args.k : -1;
                tok_out[s] = p;
            } else {
                const int tl = live_rows(args.live, args.T);
                tok_img[s] = s < tl ? s : -1;
                tok_out[s] = s < tl ? s : -1;
            }
        }
        __syncthreads();
        const int rowB = tok_img[g];
        const int rowS0 = tok_img[2 * t4], rowS1 = tok_img[2 * t4 + 1];
        const uint8_t *imgB = rowB >= 0 ? args.img + (int64_t)rowB * args.img_row_bytes : nullptr;
        const uint8_t *imgS0 = rowS0 >= 0 ? args.img + (int64_t)rowS0 * args.img_row_bytes : nullptr;
        const uint8_t *imgS1 = rowS1 >= 0 ? args.img + (int64_t)rowS1 * args.img_row_bytes : nullptr;

        float acc[RG][4];
#pragma unroll
        for (int r = 0; r < RG; r++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[r][i] = 0.0f;

        for (int c = c_begin + warp; c < c_end; c += NW) {
            // weights of this chunk for every row group (issued first: HBM latency)
            uint4 wv[RG][WT == QK_W_Q4_0 ? 2 : 4];
            uint2 sv[RG][2];
#pragma unroll
            for (int r = 0; r < RG; r++) {
                if (g0 + r < P.n_groups) {
                    const uint8_t *tp = wbase + ((int64_t)(g0 + r) * P.chunks + c) * TILE;
                    if (WT == QK_W_Q4_0) {
                        wv[r][0] = ld_stream16(tp + lane * 16);
                        wv[r][1] = ld_stream16(tp + HALF_OFF + lane * 16);
                    } else {
                        wv[r][0] = ld_stream16(tp + lane * 32);
                        wv[r][1] = ld_stream16(tp + lane * 32 + 16);
                        wv[r][2] = ld_stream16(tp + HALF_OFF + lane * 32);
                        wv[r][3] = ld_stream16(tp + HALF_OFF + lane * 32 + 16);
                    }
                    sv[r][0] = ld_stream8(tp + SCALE_OFF + g * 8);
                    sv[r][1] = ld_stream8(tp + SCALE_OFF + (g + 8) * 8);
                } else {
#pragma unroll
                    for (int i = 0; i < (WT == QK_W_Q4_0 ? 2 : 4); i++) wv[r][i] = make_uint4(0, 0, 0, 0);
                    sv[r][0] = sv[r][1] = make_uint2(0, 0);
                }
            }
#pragma unroll
            for (int jb = 0; jb < 4; jb++) {
                const int b = 4 * c + jb;
                if (b >= Kb) break;
                // B side: this lane's token g, elements 4t..4t+3 and 16+4t..16+4t+3
                uint32_t blo02 = 0, blo13 = 0, bhi02 = 0, bhi13 = 0;
                if (imgB) {
                    const uint8_t *blk = imgB + (int64_t)b * Q8_1_BYTES;
                    codes_to_half2(ld_img4(blk + 4 + 4 * t4), blo02, blo13);
                    codes_to_half2(ld_img4(blk + 20 + 4 * t4), bhi02, bhi13);
                }
                // activation scales of tokens 2t and 2t+1
                float da0 = 0.f, da1 = 0.f, ns0 = 0.f, ns1 = 0.f;
                if (imgS0) {
                    const uint32_t ds = ld_img4(imgS0 + (int64_t)b * Q8_1_BYTES);
                    da0 = half_lo(ds);
                    if (WT == QK_W_Q4_0) ns0 = -8.0f * half_hi(ds);
                }
                if (imgS1) {
                    const uint32_t ds = ld_img4(imgS1 + (int64_t)b * Q8_1_BYTES);
                    da1 = half_lo(ds);
                    if (WT == QK_W_Q4_0) ns1 = -8.0f * half_hi(ds);
                }
                // bias correction: -sum(bias_i * q_i) per token, same for every row
                float corr[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16(corr, NEG_BIAS_LO, NEG_BIAS_LO, NEG_BIAS_LO, NEG_BIAS_LO, blo02, blo13);
                mma_f16(corr, NEG_BIAS_HI, NEG_BIAS_HI, NEG_BIAS_HI, NEG_BIAS_HI, bhi02, bhi13);
#pragma unroll
                for (int r = 0; r < RG; r++) {
                    uint32_t a_lo[4], a_hi[4];  // {row g k0, row g+8 k0, row g k8, row g+8 k8}
                    if (WT == QK_W_Q4_0) {
                        const uint32_t wg = (&wv[r][0].x)[jb];
                        const uint32_t wg8 = (&wv[r][1].x)[jb];
                        nibbles_to_half2(wg, a_lo[0], a_lo[2], a_hi[0], a_hi[2]);
                        nibbles_to_half2(wg8, a_lo[1], a_lo[3], a_hi[1], a_hi[3]);
                    } else {
                        const uint32_t *vg = &wv[r][jb >> 1].x + 2 * (jb & 1);
                        const uint32_t *vg8 = &wv[r][2 + (jb >> 1)].x + 2 * (jb & 1);
                        wcodes_to_half2(vg[0], a_lo[0], a_lo[2]);
                        wcodes_to_half2(vg[1], a_hi[0], a_hi[2]);
                        wcodes_to_half2(vg8[0], a_lo[1], a_lo[3]);
                        wcodes_to_half2(vg8[1], a_hi[1], a_hi[3]);
                    }
                    float dv[4] = {corr[0], corr[1], corr[2], corr[3]};
                    mma_f16(dv, a_lo[0], a_lo[1], a_lo[2], a_lo[3], blo02, blo13);
                    mma_f16(dv, a_hi[0], a_hi[1], a_hi[2], a_hi[3], bhi02, bhi13);
                    const uint32_t sg = (jb < 2) ? sv[r][0].x : sv[r][0].y;
                    const uint32_t sg8 = (jb < 2) ? sv[r][1].x : sv[r][1].y;
                    const float dwg = (jb & 1) ? half_hi(sg) : half_lo(sg);
                    const float dwg8 = (jb & 1) ? half_hi(sg8) : half_lo(sg8);
                    acc[r][0] = fmaf(dwg, fmaf(da0, dv[0], ns0), acc[r][0]);
                    acc[r][1] = fmaf(dwg, fmaf(da1, dv[1], ns1), acc[r][1]);
                    acc[r][2] = fmaf(dwg8, fmaf(da0, dv[2], ns0), acc[r][2]);
                    acc[r][3] = fmaf(dwg8, fmaf(da1, dv[3], ns1), acc[r][3]);
                }
            }
        }

        // reduce: warps (fixed order), then cluster ranks (fixed order)
#pragma unroll
        for (int r = 0; r < RG; r++)
#pragma unroll
            for (int i = 0; i < 4; i++) red[warp][r * 4 + i][lane] = acc[r][i];
        __syncthreads();
        float *part = &red[0][0][0];
        for (int v = threadIdx.x; v < RG * 4 * 32; v += NW * 32) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < NW; w++) s += (&red[w][0][0])[v];
            part[v] = s;   // each v is read and written by one thread only
        }
        if (C > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();
            if (rank == 0) {
                for (int v = threadIdx.x; v < RG * 4 * 32; v += NW * 32) {
                    float s = part[v];
                    for (int q = 1; q < C; q++) s += cluster.map_shared_rank(part, q)[v];
                    part[v] = s;
                }
            }
            cluster.sync();
        } else {
            __syncthreads();
        }
        if (rank == 0) {
            for (int v = threadIdx.x; v < RG * 4 * 32; v += NW * 32) {
                const int l = v & 31, ri = v >> 5, r = ri >> 2, i = ri & 3;
                const int row = (g0 + r) * 16 + (l >> 2) + ((i & 2) ? 8 : 0);
                const int slot = 2 * (l & 3) + (i & 1);
                const int orow = tok_out[slot];
                if (row < P.N && orow >= 0) P.y[(int64_t)orow * P.y_stride + row] = part[v];
            }
        }
        __syncthreads();   // tok_* and red reused by the next pass
    }
}

// ---------------------------------------------------------------- weight pack
// One CTA of 128 threads per 16x128 tile. Canonical source blocks are read
// byte by byte (18- and 34-byte blocks are only 2-byte aligned).
template <int WT>
__global__ void __launch_bounds__(128) pack_kernel(const uint8_t *__restrict__ src, int N, int K,
                                                   int chunks, uint8_t *__restrict__ dst) {
    constexpr int TILE = WT == QK_W_Q4_0 ? Q4_TILE_BYTES : Q8_TILE_BYTES;
    constexpr int SB = WT == QK_W_Q4_0 ? Q4_0_BYTES : Q8_0_BYTES;
    constexpr int SCALE_OFF = WT == QK_W_Q4_0 ? 1024 : 2048;
    const int64_t tile = blockIdx.x;
    const int grp = (int)(tile / chunks), c = (int)(tile % chunks);
    const int Kb = K / QB;
    uint8_t *out = dst + tile * TILE;
    const int tid = threadIdx.x;
    auto byte_at = [&](int n, int b, int off) -> uint32_t {
        if (n >= N || b >= Kb) return 0u;
        return src[((int64_t)n * Kb + b) * SB + off];
    };
    if (tid < 64) {
        const int half = tid >> 5, l = tid & 31, gg = l >> 2, t = l & 3;
        const int n = grp * 16 + gg + 8 * half;
        if (WT == QK_W_Q4_0) {
            uint32_t v[4];
            for (int jb = 0; jb < 4; jb++) {
                const int b = 4 * c + jb;
                v[jb] = byte_at(n, b, 2 + 4 * t) | (byte_at(n, b, 3 + 4 * t) << 8) |
                        (byte_at(n, b, 4 + 4 * t) << 16) | (byte_at(n, b, 5 + 4 * t) << 24);
            }
            *reinterpret_cast<uint4 *>(out + half * 512 + l * 16) = make_uint4(v[0], v[1], v[2], v[3]);
        } else {
            uint32_t v[8];
            for (int jb = 0; jb < 4; jb++) {
                const int b = 4 * c + jb;
                for (int h = 0; h < 2; h++) {
                    const int o = 2 + 16 * h + 4 * t;
                    v[2 * jb + h] = byte_at(n, b, o) | (byte_at(n, b, o + 1) << 8) |
                                    (byte_at(n, b, o + 2) << 16) | (byte_at(n, b, o + 3) << 24);
                }
            }
            uint4 *o4 = reinterpret_cast<uint4 *>(out + half * 1024 + l * 32);
            o4[0] = make_uint4(v[0], v[1], v[2], v[3]);
            o4[1] = make_uint4(v[4], v[5], v[6], v[7]);
        }
    } else if (tid < 80) {
        const int r = tid - 64, n = grp * 16 + r;
        uint16_t h[4];
        for (int jb = 0; jb < 4; jb++) {
            const int b = 4 * c + jb;
            h[jb] = (uint16_t)(byte_at(n, b, 0) | (byte_at(n, b, 1) << 8));
        }
        *reinterpret_cast<uint2 *>(out + SCALE_OFF + r * 8) =
            make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
    }
}

// Split K over a cluster so that the grid holds at least ~4 CTAs per SM.
int pick_ksplit(int64_t tiles, int chunks, int n_sm) {
    int C = 1;
    while (C < 8 && tiles * C < 4LL * n_sm && chunks >= 2 * C * NW) C *= 2;
    return C;
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

template <int WT, bool ROUTED>
qk_status launch(const Args &a, int64_t tiles, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)(tiles * a.ksplit));
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.numAttrs = 0;
    if (a.ksplit > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)a.ksplit;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t err = cudaLaunchKernelEx(&cfg, mmvq_kernel<WT, ROUTED>, a);
    count_launch();
    if (err != cudaSuccess) return fail(QK_ERR_CUDA, "%s: %s", ROUTED ? "mmvq_id" : "mmvq", cudaGetErrorString(err));
    return check_launch(ROUTED ? "mmvq_id" : "mmvq");
}

}  // namespace

qk_status launch_weight_pack(int wtype, const uint8_t *blocks, int64_t N, int64_t K,
                             uint8_t *packed, cudaStream_t s) {
    const int64_t chunks = ceil_div(K, TILE_COLS);
    const int64_t tiles = ceil_div(N, TILE_ROWS) * chunks;
    if (tiles == 0) return QK_OK;
    if (wtype == QK_W_Q4_0)
        pack_kernel<QK_W_Q4_0><<<(unsigned)tiles, 128, 0, s>>>(blocks, (int)N, (int)K, (int)chunks, packed);
    else
        pack_kernel<QK_W_Q8_0><<<(unsigned)tiles, 128, 0, s>>>(blocks, (int)N, (int)K, (int)chunks, packed);
    count_launch();
    return check_launch("weight_pack");
}

static void fill_desc(ProjDesc &d, int wtype, const void *w, float *y, int64_t y_stride, int64_t N,
                      int64_t K, int experts, int tiles_begin) {
    d.w = static_cast<const uint8_t *>(w);
    d.y = y;
    d.y_stride = y_stride;
    d.expert_bytes = packed_bytes(wtype, N, K);
    d.N = (int)N;
    d.K = (int)K;
    d.n_groups = (int)ceil_div(N, TILE_ROWS);
    d.chunks = (int)ceil_div(K, TILE_COLS);
    d.row_tiles = (int)ceil_div(d.n_groups, RG);
    d.experts = experts;
    d.tiles_begin = tiles_begin;
}

qk_status launch_mmvq(const uint8_t *img, int64_t row_blocks, int T, int n_proj,
                      const qk_proj *projs, const int32_t *live, cudaStream_t s) {
    Args a = {};
    a.img = img;
    a.img_row_bytes = row_blocks * Q8_1_BYTES;
    a.T = T;
    a.live = live;
    a.n_proj = n_proj;
    a.k = 1;
    int64_t tiles = 0;
    int min_chunks = 1 << 30;
    for (int j = 0; j < n_proj; j++) {
        fill_desc(a.p[j], projs[j].wtype, projs[j].w, projs[j].y, projs[j].y_stride, projs[j].N,
                  projs[j].K, 1, (int)tiles);
        tiles += a.p[j].row_tiles;
        min_chunks = min(min_chunks, a.p[j].chunks);
    }
    a.ksplit = pick_ksplit(tiles, min_chunks, sm_count());
    // one weight type per launch: mixed groups are split by the caller side below
    const int wt = projs[0].wtype;
    return wt == QK_W_Q4_0 ? launch<QK_W_Q4_0, false>(a, tiles, s) : launch<QK_W_Q8_0, false>(a, tiles, s);
}

qk_status launch_mmvq_id(const uint8_t *img, int64_t row_blocks, int rows, int k, int n_proj,
                         const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                         const int32_t *items, cudaStream_t s) {
    Args a = {};
    a.img = img;
    a.img_row_bytes = row_blocks * Q8_1_BYTES;
    a.T = rows;
    a.n_proj = n_proj;
    a.counts = counts;
    a.offsets = offsets;
    a.items = items;
    a.k = k;
    int64_t tiles = 0;
    int min_chunks = 1 << 30;
    for (int j = 0; j < n_proj; j++) {
        fill_desc(a.p[j], projs[j].wtype, projs[j].w, projs[j].y, projs[j].N, projs[j].N, projs[j].K,
                  projs[j].n_experts, (int)tiles);
        tiles += (int64_t)a.p[j].row_tiles * projs[j].n_experts;
        min_chunks = min(min_chunks, a.p[j].chunks);
    }
    a.ksplit = pick_ksplit(tiles, min_chunks, sm_count());
    const int wt = projs[0].wtype;
    return wt == QK_W_Q4_0 ? launch<QK_W_Q4_0, true>(a, tiles, s) : launch<QK_W_Q8_0, true>(a, tiles, s);
}

}  // namespace qk

// Prefill dense contraction on a Q8_0 activation image (minfer doc 52 "r49
// A-quantize prepass shared-A dedup", sections 1 and 5: the q/k/v and
// gate/up GEMMs that read one quantised A).
//
//   C[t][n] = sum_b d_w[n][b] * d_a[t][b] * D,   D = sum_{i in b} (nibble_i - 8) * q_i
//
// Like the MMVQ kernels, the exact integer block dot D runs on the f16 tensor
// path (mma.sync m16n8k16): nibbles and codes are exact halves and every
// partial sum stays below 2^22. Nibbles are turned into halves by OR-ing them
// under an exponent (1024 + lo, 64 + hi); the per-token correction
// -(1032 * sum of the low-half codes + 72 * sum of the high-half codes)
// removes both that bias and the "- 8" of Q4_0 at once, so it seeds the
// accumulator and D comes out exact. The block scales d_w * d_a are applied
// per block in f32 (two FP operations per output per block), which makes this
// contraction bound by FP32 issue rather than by the tensor pipe.
//
// CTA: 8 warps, a 128-row weight tile (one packed unit row, warp w = row
// group w) by 64 tokens (8 token groups). Per 128-column chunk the CTA stages
// the unit (cp.async, 9216 B) and the 64 tokens' codes and scales, converts
// the codes once into f16 B fragments with their corrections, then every warp
// runs 8 token groups x 4 blocks of MMAs. Two stages double-buffer the
// copies.

#include "qk_internal.cuh"

namespace qk {
namespace {

constexpr int MW = 8;        // warps = row groups of the 128-row tile
constexpr int TT = 64;       // tokens per CTA
constexpr int TG = TT / 8;   // token groups
constexpr int MAX_PROJ = 8;

struct MmqProj {
    const uint8_t *w;
    float *y;
    int64_t y_stride;
    int N, K, chunks, row_tiles, tiles_begin;
};
struct MmqArgs {
    const int8_t *qs;
    const uint16_t *d;
    int64_t row_blocks;
    int T, n_proj;
    MmqProj p[MAX_PROJ];
};

// shared memory per stage
struct Stage {
    uint8_t unit[Q4_UNIT_BYTES];       // packed weights of the chunk
    int8_t codes[TT][128];             // the chunk's codes of 64 tokens
    uint16_t dh[TT][4];                // their block scales (half bits)
};
struct Frags {
    uint4 b[4][TG][32];                // [block][token group][lane]: (lo02, lo13, hi02, hi13)
    float corr[4][TT];                 // -(1032 S_lo + 72 S_hi) per block and token
    float da[4][TT];                   // d_a per block and token
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;   // 0 source bytes: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                        const float c[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Four int8 codes -> exact half2 (c0, c2) and (c1, c3) (XOR 0x80, exponent of
// 1024, minus 1152).
__device__ __forceinline__ void codes_to_half2(uint32_t w, uint32_t &h02, uint32_t &h13) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4240);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4341);
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    h02 = *reinterpret_cast<uint32_t *>(&ha);
    h13 = *reinterpret_cast<uint32_t *>(&hb);
}

__device__ __forceinline__ void nibbles_to_half2(uint32_t w, uint32_t &lo02, uint32_t &lo13, uint32_t &hi02,
                                                 uint32_t &hi13) {
    const uint32_t w8 = w >> 8;
    lo02 = (w & 0x000F000Fu) | 0x64006400u;
    hi02 = (w & 0x00F000F0u) | 0x54005400u;
    lo13 = (w8 & 0x000F000Fu) | 0x64006400u;
    hi13 = (w8 & 0x00F000F0u) | 0x54005400u;
}

// Sum of four signed bytes.
__device__ __forceinline__ int sum4(uint32_t w) {
    return (int)(int8_t)(w & 0xff) + (int)(int8_t)((w >> 8) & 0xff) + (int)(int8_t)((w >> 16) & 0xff) +
           (int)(int8_t)(w >> 24);
}

__global__ void __launch_bounds__(MW * 32) mmq_kernel(const __grid_constant__ MmqArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    Stage *st = reinterpret_cast<Stage *>(smem);                       // [2]
    Frags *fr = reinterpret_cast<Frags *>(smem + 2 * sizeof(Stage));
    pdl_trigger();
    pdl_wait();

    const int tile = blockIdx.x;
    int j = 0;
    while (j + 1 < a.n_proj && tile >= a.p[j + 1].tiles_begin) j++;
    const MmqProj &P = a.p[j];
    const int rt = tile - P.tiles_begin;
    const int tok0 = blockIdx.y * TT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
    const int Kb = P.K / QB;
    const uint8_t *wtile = P.w + (int64_t)rt * P.chunks * Q4_UNIT_BYTES;

    auto issue = [&](int c, int s) {
        Stage &S = st[s];
        const uint8_t *src = wtile + (int64_t)c * Q4_UNIT_BYTES;
        for (int i = tid; i < Q4_UNIT_BYTES / 16; i += MW * 32) cp_async16(S.unit + i * 16, src + i * 16, true);
        // codes: 64 tokens x 8 x 16 bytes; blocks past K and tokens past T read as zero
        for (int i = tid; i < TT * 8; i += MW * 32) {
            const int tk = i >> 3, part = i & 7, b = 4 * c + (part >> 1);
            const bool ok = tok0 + tk < a.T && b < Kb;
            const int8_t *s8 = ok ? a.qs + (int64_t)(tok0 + tk) * a.row_blocks * QB + (int64_t)4 * c * QB + part * 16
                                  : a.qs;
            cp_async16(&S.codes[tk][part * 16], s8, ok);
        }
        // scales (4 halves per token; plain loads: the scale rows are only 2-byte aligned)
        for (int i = tid; i < TT; i += MW * 32) {
            const bool ok = tok0 + i < a.T;
            const uint16_t *s16 = a.d + (int64_t)(tok0 + i) * a.row_blocks + 4 * c;
#pragma unroll
            for (int q = 0; q < 4; q++) S.dh[i][q] = ok && 4 * c + q < Kb ? __ldg(s16 + q) : (uint16_t)0;
        }
        cp_commit();
    };

    float acc[TG][4];
#pragma unroll
    for (int q = 0; q < TG; q++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[q][i] = 0.0f;

    issue(0, 0);
    for (int c = 0; c < P.chunks; c++) {
        const int s = c & 1;
        if (c + 1 < P.chunks) {
            issue(c + 1, s ^ 1);
            cp_wait<1>();
        } else {
            cp_wait<0>();
        }
        __syncthreads();   // stage s landed; fr free (previous chunk's MMAs done)
        // convert codes -> f16 fragments, corrections and scales (one item per thread per block)
        Stage &S = st[s];
#pragma unroll
        for (int jb = 0; jb < 4; jb++) {
            const int qg = tid >> 5, l = tid & 31, tg_ = l >> 2, tt = l & 3;   // tid = tg*32 + lane
            const int tk = qg * 8 + tg_;
            const uint32_t lo = *reinterpret_cast<const uint32_t *>(&S.codes[tk][jb * 32 + 4 * tt]);
            const uint32_t hi = *reinterpret_cast<const uint32_t *>(&S.codes[tk][jb * 32 + 16 + 4 * tt]);
            uint4 f;
            codes_to_half2(lo, f.x, f.y);
            codes_to_half2(hi, f.z, f.w);
            fr->b[jb][qg][l] = f;
            if (tid < TT) {
                int slo = 0, shi = 0;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    slo += sum4(*reinterpret_cast<const uint32_t *>(&S.codes[tid][jb * 32 + 4 * q]));
                    shi += sum4(*reinterpret_cast<const uint32_t *>(&S.codes[tid][jb * 32 + 16 + 4 * q]));
                }
                fr->corr[jb][tid] = -(1032.0f * (float)slo + 72.0f * (float)shi);
                const bool ok = 4 * c + jb < Kb;
                fr->da[jb][tid] = ok ? __half2float(__ushort_as_half(S.dh[tid][jb])) : 0.0f;
            }
        }
        __syncthreads();
        // MMAs: warp = row group, all token groups, 4 blocks
#pragma unroll
        for (int jb = 0; jb < 4; jb++) {
            if (4 * c + jb >= Kb) break;
            const uint8_t *blk = S.unit + jb * Q4_BLOCK_STRIDE;
            const uint4 v = *reinterpret_cast<const uint4 *>(blk + (warp >> 1) * 512 + lane * 16);
            const uint32_t wg = (warp & 1) ? v.z : v.x, wg8 = (warp & 1) ? v.w : v.y;
            uint32_t a_lo[4], a_hi[4];
            nibbles_to_half2(wg, a_lo[0], a_lo[2], a_hi[0], a_hi[2]);
            nibbles_to_half2(wg8, a_lo[1], a_lo[3], a_hi[1], a_hi[3]);
            const uint32_t dw2 = *reinterpret_cast<const uint32_t *>(S.unit + 8192 + jb * 256 + g * 32 + warp * 4);
            const float2 dw = __half22float2(*reinterpret_cast<const __half2 *>(&dw2));
#pragma unroll
            for (int q = 0; q < TG; q++) {
                const uint4 bf = fr->b[jb][q][lane];
                const float2 cr = *reinterpret_cast<const float2 *>(&fr->corr[jb][q * 8 + 2 * t4]);
                const float2 da = *reinterpret_cast<const float2 *>(&fr->da[jb][q * 8 + 2 * t4]);
                const float c4[4] = {cr.x, cr.y, cr.x, cr.y};
                float d1[4], dv[4];
                mma_f16(d1, a_lo, bf.x, bf.y, c4);
                mma_f16(dv, a_hi, bf.z, bf.w, d1);
                acc[q][0] = fmaf(dw.x, da.x * dv[0], acc[q][0]);
                acc[q][1] = fmaf(dw.x, da.y * dv[1], acc[q][1]);
                acc[q][2] = fmaf(dw.y, da.x * dv[2], acc[q][2]);
                acc[q][3] = fmaf(dw.y, da.y * dv[3], acc[q][3]);
            }
        }
        __syncthreads();   // stage s and fr are rewritten next
    }

    // outputs: row = 16*warp + g (+8), token = tok0 + 8q + 2*t4 (+1)
    const int row0 = rt * UNIT_ROWS + 16 * warp + g;
#pragma unroll
    for (int q = 0; q < TG; q++) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int row = row0 + ((i & 2) ? 8 : 0);
            const int tok = tok0 + 8 * q + 2 * t4 + (i & 1);
            if (row < P.N && tok < a.T) P.y[(int64_t)tok * P.y_stride + row] = acc[q][i];
        }
    }
}

}  // namespace

qk_status launch_mmq(const int8_t *qs, const uint16_t *d, int64_t row_blocks, int T, int n_proj,
                     const qk_proj *projs, cudaStream_t s) {
    MmqArgs a = {};
    a.qs = qs;
    a.d = d;
    a.row_blocks = row_blocks;
    a.T = T;
    a.n_proj = n_proj;
    int tiles = 0;
    for (int j = 0; j < n_proj; j++) {
        MmqProj &p = a.p[j];
        p.w = static_cast<const uint8_t *>(projs[j].w);
        p.y = projs[j].y;
        p.y_stride = projs[j].y_stride;
        p.N = (int)projs[j].N;
        p.K = (int)projs[j].K;
        p.chunks = (int)ceil_div(p.K, UNIT_COLS);
        p.row_tiles = (int)ceil_div(p.N, UNIT_ROWS);
        p.tiles_begin = tiles;
        tiles += p.row_tiles;
    }
    const size_t smem = 2 * sizeof(Stage) + sizeof(Frags);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(mmq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return fail(QK_ERR_CUDA, "mmq: shared memory attribute: %s", cudaGetErrorString(e));
        configured = true;
    }
    dim3 grid((unsigned)tiles, (unsigned)ceil_div(T, TT));
    return launch_pdl("mmq", mmq_kernel, grid, dim3(MW * 32), smem, s, a);
}

}  // namespace qk

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
// Block dot on the f16 tensor path. Nibbles, int8 weights and int8 codes are
// exact in binary16, products are exact and every partial sum stays below
// 2^22, so the f32 accumulator of mma.sync m16n8k16 holds the integer D
// exactly. (Blackwell Ultra's int8 mma and dp4a run at about a quarter of its
// f16 mma rate -- measured 150 vs 590 T/s -- too slow to keep up with HBM at
// 8 tokens.) A nibble becomes a half with one logic op by OR-ing it under a
// binary16 exponent (1024 + lo for low nibbles, 64 + hi for high ones); the
// bias this adds, sum_i bias * q_i, depends only on the token, so a pair of
// MMAs with a constant -bias A operand computes it once per block and it
// seeds the accumulator of all 8 row groups.
//
// Ordinary path: one persistent CTA per SM. A producer warp streams 128x128
// weight units with TMA bulk copies (cp.async.bulk, L2 evict-first) into a
// ring of shared-memory slots guarded by full/empty mbarriers; 15 consumer
// warps take the units' 32-column blocks round-robin (block j of the CTA's
// range goes to warp j mod 15), each computing all 128 rows x 8 tokens of its
// block. Work is split by equal bytes over the CTAs (stream-K): a row tile
// cut between CTAs leaves partial sums in a small caller workspace (written
// when the CTA has finished its whole range, so no consumer waits on global
// memory mid-stream), and the last CTA to publish its part (atomic counter,
// reset after use) adds the parts in CTA order. All sums run in a fixed order, so results do not depend on
// timing or on the live-row count.

#include <mutex>

#include "qk_internal.cuh"

namespace qk {
namespace {

__device__ unsigned int g_qk_faults = 0;

constexpr int MAX_PROJ = 8;
constexpr int CW = 15;                       // consumer warps (ordinary path); with the
constexpr int THREADS = (CW + 1) * 32;       // producer, 16 warps = 4 per SM sub-partition
constexpr int VALS = UNIT_GROUPS * 4 * 32;   // accumulators of one 128-row tile per warp
constexpr int HALF_VALS = VALS / 2;          // reduced in two passes of 4 row groups
constexpr int MAXP = 8;                      // partial sums loaded per batch
constexpr uint32_t SPIN_LIMIT = 1u << 22;

template <int WT> struct Layout;
template <> struct Layout<QK_W_Q4_0> {
    static constexpr int UNIT = Q4_UNIT_BYTES, BLOCK = Q4_BLOCK_STRIDE, SCALES = 8192, SLOTS = 16;
};
template <> struct Layout<QK_W_Q8_0> {
    static constexpr int UNIT = Q8_UNIT_BYTES, BLOCK = Q8_BLOCK_STRIDE, SCALES = 16384, SLOTS = 8;
};

struct SkProj {
    const uint8_t *w;
    float *y;
    int64_t y_stride;
    int64_t unit_base;   // first unit of this projection in the flat unit space
    int N, K, chunks, row_tiles, rt_base;
};

struct SkArgs {
    const uint8_t *img;
    int64_t img_row_bytes;
    int T;
    const int32_t *live;
    int n_proj;
    int64_t U;           // total units
    float *ws_part;      // [G][2][VALS]
    unsigned int *ws_cnt;
    SkProj p[MAX_PROJ];
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_img4(const uint8_t *p) {
    return __ldg(reinterpret_cast<const unsigned int *>(p));
}
__device__ __forceinline__ __half2 as_h2(uint32_t v) { return *reinterpret_cast<__half2 *>(&v); }
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after SPIN_LIMIT tries, records a fault and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity) {
    for (uint32_t i = 0; i < SPIN_LIMIT; i++)
        if (mbar_try_wait(a, parity)) return true;
    atomicOr(&g_qk_faults, 1u);
    return false;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(mbar), "l"(pol)
        : "memory");
}
// Atomic add with acquire-release semantics at GPU scope (returns the old value).
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// A row tile this CTA shares with others (stream-K): where its parts live.
struct SharedTile {
    float *y;
    int64_t y_stride;
    int N, rt, R;            // rows, row tile in its projection, global row-tile index
    int c_first, c_last;     // contributing CTAs
    int first_slot;          // part slot used by c_first (later CTAs use slot 0)
};

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(CW * 32) : "memory");
}

// D = A * B + C (m16n8k16, f16 inputs, f32 accumulate); D and C may differ.
__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                        const float c[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}

// Four int8 codes (bytes c0..c3) -> exact half2 (c0, c2) and (c1, c3):
// XOR 0x80 gives u = c + 128; the half 0x64uu is 1024 + u; minus 1152 is c.
__device__ __forceinline__ void codes_to_half2(uint32_t w, uint32_t &h02, uint32_t &h13) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4240);
    uint32_t b = __byte_perm(u, 0x64646464u, 0x4341);
    __half2 ha = __hsub2(as_h2(a), bias);
    __half2 hb = __hsub2(as_h2(b), bias);
    h02 = *reinterpret_cast<uint32_t *>(&ha);
    h13 = *reinterpret_cast<uint32_t *>(&hb);
}

// Q4_0 word (nibble bytes B0..B3) -> biased halves of one row for the two MMAs:
//   lo02 = (1024+lo B0, 1024+lo B2), lo13 = (1024+lo B1, 1024+lo B3)
//   hi02 = (  64+hi B0,   64+hi B2), hi13 = (  64+hi B1,   64+hi B3)
__device__ __forceinline__ void nibbles_to_half2(uint32_t w, uint32_t &lo02, uint32_t &lo13,
                                                 uint32_t &hi02, uint32_t &hi13) {
    const uint32_t w8 = w >> 8;
    lo02 = (w & 0x000F000Fu) | 0x64006400u;
    hi02 = (w & 0x00F000F0u) | 0x54005400u;
    lo13 = (w8 & 0x000F000Fu) | 0x64006400u;
    hi13 = (w8 & 0x00F000F0u) | 0x54005400u;
}

// Q8_0 weight codes keep their +1152 bias (removed by the correction MMAs).
__device__ __forceinline__ void wcodes_to_half2(uint32_t w, uint32_t &h02, uint32_t &h13) {
    const uint32_t u = w ^ 0x80808080u;
    h02 = __byte_perm(u, 0x64646464u, 0x4240);
    h13 = __byte_perm(u, 0x64646464u, 0x4341);
}

// ---------------------------------------------------------------- one block
// Activation side of block b for this lane: B fragments of token g (elements
// 4t..4t+3 and 16+4t..16+4t+3), scales of tokens 2t and 2t+1, and the bias
// correction shared by every row group. The four image words are loaded one
// block ahead (Raw) so their latency overlaps the previous block's MMAs.
struct Raw {
    uint32_t lo, hi, ds0, ds1;
};
struct BSide {
    uint32_t lo02, lo13, hi02, hi13;
    float da0, da1, ns0, ns1;
    float corr[4];
};

__device__ __forceinline__ Raw load_raw(const uint8_t *imgB, const uint8_t *imgS0, const uint8_t *imgS1, int b,
                                        int t4) {
    Raw r = {0u, 0u, 0u, 0u};
    const int64_t off = (int64_t)b * Q8_1_BYTES;
    if (imgB) {
        r.lo = ld_img4(imgB + off + 4 + 4 * t4);
        r.hi = ld_img4(imgB + off + 20 + 4 * t4);
    }
    if (imgS0) r.ds0 = ld_img4(imgS0 + off);
    if (imgS1) r.ds1 = ld_img4(imgS1 + off);
    return r;
}

template <int WT>
__device__ __forceinline__ void bside(const Raw &r, BSide &s) {
    constexpr uint32_t NEG_LO = WT == QK_W_Q4_0 ? 0xE400E400u : 0xE480E480u;  // -1024 | -1152
    constexpr uint32_t NEG_HI = WT == QK_W_Q4_0 ? 0xD400D400u : 0xE480E480u;  //   -64 | -1152
    codes_to_half2(r.lo, s.lo02, s.lo13);   // an absent token has zero words: exact zeros
    codes_to_half2(r.hi, s.hi02, s.hi13);
    const float2 d0 = __half22float2(as_h2(r.ds0)), d1 = __half22float2(as_h2(r.ds1));
    s.da0 = d0.x;
    s.da1 = d1.x;
    s.ns0 = WT == QK_W_Q4_0 ? -8.0f * d0.y : 0.0f;
    s.ns1 = WT == QK_W_Q4_0 ? -8.0f * d1.y : 0.0f;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t alo[4] = {NEG_LO, NEG_LO, NEG_LO, NEG_LO};
    const uint32_t ahi[4] = {NEG_HI, NEG_HI, NEG_HI, NEG_HI};
    float c1[4];
    mma_f16(c1, alo, s.lo02, s.lo13, zero);
    mma_f16(s.corr, ahi, s.hi02, s.hi13, c1);
}

// Row group: two MMAs seeded with the correction, then the scale epilogue.
__device__ __forceinline__ void row_group(const uint32_t a_lo[4], const uint32_t a_hi[4], uint32_t dw2,
                                          const BSide &s, float acc[4]) {
    float d1[4], dv[4];
    mma_f16(d1, a_lo, s.lo02, s.lo13, s.corr);
    mma_f16(dv, a_hi, s.hi02, s.hi13, d1);
    const float2 dw = __half22float2(as_h2(dw2));   // (row g, row g+8)
    acc[0] = fmaf(dw.x, fmaf(s.da0, dv[0], s.ns0), acc[0]);
    acc[1] = fmaf(dw.x, fmaf(s.da1, dv[1], s.ns1), acc[1]);
    acc[2] = fmaf(dw.y, fmaf(s.da0, dv[2], s.ns0), acc[2]);
    acc[3] = fmaf(dw.y, fmaf(s.da1, dv[3], s.ns1), acc[3]);
}

// All 8 row groups of one block, from shared memory (SMEM, 32-bit shared
// addresses) or with streaming global loads.
template <int WT, bool SMEM>
__device__ __forceinline__ void block_rows(const uint8_t *gblk, uint32_t sblk, const uint8_t *gsc, uint32_t ssc,
                                           int lane, const BSide &s, float acc[UNIT_GROUPS][4]) {
    const int g = lane >> 2;
    uint4 sc0, sc1;
    if (SMEM) {
        sc0 = lds128(ssc + g * 32);
        sc1 = lds128(ssc + g * 32 + 16);
    } else {
        sc0 = ldg_stream16(gsc + g * 32);
        sc1 = ldg_stream16(gsc + g * 32 + 16);
    }
    const uint32_t scw[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
    if (WT == QK_W_Q4_0) {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const uint4 v = SMEM ? lds128(sblk + k * 512 + lane * 16) : ldg_stream16(gblk + k * 512 + lane * 16);
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint32_t wg = h ? v.z : v.x, wg8 = h ? v.w : v.y;
                uint32_t a_lo[4], a_hi[4];
                nibbles_to_half2(wg, a_lo[0], a_lo[2], a_hi[0], a_hi[2]);
                nibbles_to_half2(wg8, a_lo[1], a_lo[3], a_hi[1], a_hi[3]);
                row_group(a_lo, a_hi, scw[2 * k + h], s, acc[2 * k + h]);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const uint4 v = SMEM ? lds128(sblk + k * 512 + lane * 16) : ldg_stream16(gblk + k * 512 + lane * 16);
            uint32_t a_lo[4], a_hi[4];
            wcodes_to_half2(v.x, a_lo[0], a_lo[2]);
            wcodes_to_half2(v.y, a_hi[0], a_hi[2]);
            wcodes_to_half2(v.z, a_lo[1], a_lo[3]);
            wcodes_to_half2(v.w, a_hi[1], a_hi[3]);
            row_group(a_lo, a_hi, scw[k], s, acc[k]);
        }
    }
}

// Output position of accumulator value v (0..VALS-1) of a 128-row tile.
__device__ __forceinline__ void val_pos(int v, int &row, int &slot) {
    const int l = v & 31, i = (v >> 5) & 3, r = v >> 7;
    row = 16 * r + (l >> 2) + ((i & 2) ? 8 : 0);
    slot = 2 * (l & 3) + (i & 1);
}

__device__ __forceinline__ int64_t cta_start(int c, int64_t U, int G) {
    return (int64_t)(((uint64_t)c * (uint64_t)U) / (uint32_t)G);
}
__device__ __forceinline__ int cta_of(int64_t u, int64_t U, int G) {
    int c = (int)((u * G) / U);
    while (c + 1 < G && cta_start(c + 1, U, G) <= u) c++;
    while (c > 0 && cta_start(c, U, G) > u) c--;
    return c;
}

// ---------------------------------------------------------------- ordinary path
template <int WT>
__global__ void __launch_bounds__(THREADS, 1) mmvq_sk_kernel(const __grid_constant__ SkArgs a) {
    using L = Layout<WT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *ring = smem;
    float *red = reinterpret_cast<float *>(smem + L::SLOTS * L::UNIT);
    float *keep = red + CW * HALF_VALS;   // [2][VALS]
    uint64_t *full = reinterpret_cast<uint64_t *>(keep + 2 * VALS);
    uint64_t *empty = full + L::SLOTS;
    __shared__ int s_last[2];
    __shared__ SharedTile s_tile[2];

    pdl_trigger();
    const int G = gridDim.x, cta = blockIdx.x;
    const int64_t u0 = cta_start(cta, a.U, G), u1 = cta_start(cta + 1, a.U, G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::SLOTS; s++) {
            mbar_init(smem_addr(full + s), 1);
            mbar_init(smem_addr(empty + s), 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    auto decode = [&](int64_t u, int &j, int &rt, int &c) {
        j = 0;
        while (j + 1 < a.n_proj && u >= a.p[j + 1].unit_base) j++;
        const int64_t local = u - a.p[j].unit_base;
        rt = (int)(local / a.p[j].chunks);
        c = (int)(local % a.p[j].chunks);
    };

    if (warp == CW) {   // ---------------- producer
        if (lane == 0 && u0 < u1) {
            const uint64_t pol = evict_first_policy();
            int j, rt, c;
            decode(u0, j, rt, c);
            // units of one projection are contiguous in its packed buffer
            const uint8_t *src = a.p[j].w + ((int64_t)rt * a.p[j].chunks + c) * L::UNIT;
            int64_t left_in_proj = a.p[j].unit_base + (int64_t)a.p[j].row_tiles * a.p[j].chunks - u0;
            for (int i = 0; u0 + i < u1; i++) {
                const int slot = i % L::SLOTS;
                const uint32_t n = (uint32_t)i / L::SLOTS;
                if (n > 0 && !mbar_wait(smem_addr(empty + slot), (n - 1) & 1u)) break;
                if (left_in_proj == 0) {   // next projection
                    j++;
                    src = a.p[j].w;
                    left_in_proj = (int64_t)a.p[j].row_tiles * a.p[j].chunks;
                }
                mbar_expect_tx(smem_addr(full + slot), L::UNIT);
                bulk_g2s(smem_addr(ring + (size_t)slot * L::UNIT), src, L::UNIT, smem_addr(full + slot), pol);
                src += L::UNIT;
                left_in_proj--;
            }
        }
        return;
    }

    // ---------------- consumers
    // The producer above streams weights without waiting for the previous
    // kernel (no library kernel that may run just before writes packed
    // weights); the consumers wait before reading the image, the live count or
    // the workspace, or writing outputs.
    pdl_wait();
    const int g = lane >> 2, t4 = lane & 3, tid = threadIdx.x;
    const int tl = live_rows(a.live, a.T);
    const uint8_t *imgB = g < tl ? a.img + (int64_t)g * a.img_row_bytes : nullptr;
    const uint8_t *imgS0 = 2 * t4 < tl ? a.img + (int64_t)(2 * t4) * a.img_row_bytes : nullptr;
    const uint8_t *imgS1 = 2 * t4 + 1 < tl ? a.img + (int64_t)(2 * t4 + 1) * a.img_row_bytes : nullptr;
    bool ok = true;

    // Row tiles this CTA shares (at most its first, slot 0, and its last, slot
    // 1), planned now so that the tail only stores, counts and adds.
    if (tid < 2) {
        SharedTile st = {};
        st.R = -1;
        if (u0 < u1) {
            int jj, rr, cc;
            decode(tid == 0 ? u0 : u1 - 1, jj, rr, cc);
            const SkProj &P = a.p[jj];
            const int64_t rs = P.unit_base + (int64_t)rr * P.chunks, re = rs + P.chunks;
            const bool first_tile_too = tid == 1 && rs <= u0;   // last tile == first tile
            if (!first_tile_too && (rs < u0 || re > u1)) {
                st.y = P.y;
                st.y_stride = P.y_stride;
                st.N = P.N;
                st.rt = rr;
                st.R = P.rt_base + rr;
                st.c_first = cta_of(rs, a.U, G);
                st.c_last = cta_of(re - 1, a.U, G);
                st.first_slot = cta_start(st.c_first, a.U, G) < rs ? 1 : 0;
            }
        }
        s_tile[tid] = st;
    }

    int j = 0, rt = 0, c0 = 0;
    if (u0 < u1) decode(u0, j, rt, c0);
    for (int64_t u = u0; u < u1;) {
        const SkProj &P = a.p[j];
        const int64_t rt_start = P.unit_base + (int64_t)rt * P.chunks, rt_end = rt_start + P.chunks;
        const int64_t s1 = u1 < rt_end ? u1 : rt_end;
        const int nblk = (int)(4 * (s1 - u));
        const int Kb = P.K / QB;
        float acc[UNIT_GROUPS][4];
#pragma unroll
        for (int r = 0; r < UNIT_GROUPS; r++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[r][i] = 0.0f;

        auto blk_of = [&](int jj) { return 4 * (c0 + (jj >> 2)) + (jj & 3); };
        Raw next = {0u, 0u, 0u, 0u};
        if (warp < nblk && blk_of(warp) < Kb) next = load_raw(imgB, imgS0, imgS1, blk_of(warp), t4);
        for (int jj = warp; jj < nblk; jj += CW) {
            const Raw cur = next;
            const int jn = jj + CW;
            if (jn < nblk && blk_of(jn) < Kb) next = load_raw(imgB, imgS0, imgS1, blk_of(jn), t4);
            const int i = (int)(u - u0) + (jj >> 2);
            const int slot = i % L::SLOTS;
            if (ok) ok = mbar_wait(smem_addr(full + slot), ((uint32_t)i / L::SLOTS) & 1u);
            const int jb = jj & 3;
            if (ok && blk_of(jj) < Kb) {
                BSide s;
                bside<WT>(cur, s);
                const uint32_t ub = smem_addr(ring + (size_t)slot * L::UNIT);
                block_rows<WT, true>(nullptr, ub + jb * L::BLOCK, nullptr, ub + L::SCALES + jb * 256, lane, s, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(empty + slot));
        }

        // CTA reduction over the consumer warps in fixed order, in two passes
        // of 4 row groups (value v of pass h is accumulator index h*512 + v)
        const bool whole = u == rt_start && s1 == rt_end;
        const int part_slot = u0 >= rt_start ? 0 : 1;
#pragma unroll
        for (int h = 0; h < 2; h++) {
#pragma unroll
            for (int r = 0; r < UNIT_GROUPS / 2; r++)
#pragma unroll
                for (int i = 0; i < 4; i++) red[warp * HALF_VALS + (r * 4 + i) * 32 + lane] = acc[h * 4 + r][i];
            consumer_sync();
            for (int t = tid; t < HALF_VALS; t += CW * 32) {
                float sum = 0.0f;
#pragma unroll
                for (int w = 0; w < CW; w++) sum += red[w * HALF_VALS + t];
                const int tv = h * HALF_VALS + t;
                if (whole) {
                    int row, slot;
                    val_pos(tv, row, slot);
                    row += rt * UNIT_ROWS;
                    if (row < P.N && slot < tl) P.y[(int64_t)slot * P.y_stride + row] = sum;
                } else {
                    keep[part_slot * VALS + tv] = sum;
                }
            }
            consumer_sync();   // red is rewritten by the next pass / row tile
        }
        u = s1;
        // next segment starts at chunk 0 of the next row tile (or projection)
        c0 = 0;
        if (++rt == P.row_tiles) {
            rt = 0;
            j++;
        }
    }

    // Publish this CTA's parts of shared row tiles; the last contributor of a
    // tile adds every part in CTA order and writes the output. Thread 0/1's
    // acquire-release atomic after the barrier covers the whole CTA's stores.
    const SharedTile t0 = s_tile[0], t1 = s_tile[1];
    if (t0.R < 0 && t1.R < 0) return;
    for (int ps = 0; ps < 2; ps++) {
        if ((ps ? t1.R : t0.R) < 0) continue;
        float *mine = a.ws_part + ((int64_t)cta * 2 + ps) * VALS;
        for (int t = tid; t < VALS; t += CW * 32) mine[t] = keep[ps * VALS + t];
    }
    consumer_sync();
    if (tid < 2) {
        const SharedTile &st = tid ? t1 : t0;
        int last = 0;
        if (st.R >= 0) {
            const unsigned old = atom_add_acq_rel(a.ws_cnt + st.R, 1u);
            last = old == (unsigned)(st.c_last - st.c_first);
        }
        s_last[tid] = last;
    }
    consumer_sync();
    for (int ps = 0; ps < 2; ps++) {
        if (!s_last[ps]) continue;
        const SharedTile &st = ps ? t1 : t0;
        constexpr int PER = (VALS + CW * 32 - 1) / (CW * 32);
        float sums[PER];
#pragma unroll
        for (int k = 0; k < PER; k++) sums[k] = 0.0f;
        for (int cb = st.c_first; cb <= st.c_last; cb += MAXP) {   // MAXP parts in flight at once
            const float *src[MAXP];
#pragma unroll
            for (int q = 0; q < MAXP; q++) {
                const int cc = cb + q <= st.c_last ? cb + q : st.c_last;
                const int pslot = cc == st.c_first ? st.first_slot : 0;
                src[q] = a.ws_part + ((int64_t)cc * 2 + pslot) * VALS;
            }
#pragma unroll
            for (int k = 0; k < PER; k++) {
                const int t = tid + k * CW * 32;
                if (t < VALS) {
                    float part[MAXP];
#pragma unroll
                    for (int q = 0; q < MAXP; q++) part[q] = __ldcg(src[q] + t);
#pragma unroll
                    for (int q = 0; q < MAXP; q++)
                        if (cb + q <= st.c_last) sums[k] += part[q];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < PER; k++) {
            const int t = tid + k * CW * 32;
            if (t < VALS) {
                int row, slot;
                val_pos(t, row, slot);
                row += st.rt * UNIT_ROWS;
                if (row < st.N && slot < tl) st.y[(int64_t)slot * st.y_stride + row] = sums[k];
            }
        }
        if (tid == 0) a.ws_cnt[st.R] = 0u;
    }
}

// ---------------------------------------------------------------- routed path
// One CTA of 8 warps per (projection, expert, 128-row tile). Experts with no
// planned pair return at once. Warps take the K blocks round-robin, reading
// the expert's packed units from global memory, and reduce in shared memory
// in fixed warp order. Up to 8 planned pairs per pass; more pairs re-run the
// pass (the weights then come from L2).
constexpr int RW = 8;

struct IdProj {
    const uint8_t *w;
    float *y;
    int64_t expert_bytes;
    int N, K, chunks, row_tiles, tiles_begin;
};
struct IdArgs {
    const uint8_t *img;
    int64_t img_row_bytes;
    int rows, k, n_proj;
    const int32_t *counts, *offsets, *items;
    IdProj p[MAX_PROJ];
};

template <int WT>
__global__ void __launch_bounds__(RW * 32) mmvq_id_kernel(const __grid_constant__ IdArgs a) {
    using L = Layout<WT>;
    extern __shared__ __align__(16) float red_id[];   // [RW][VALS]
    __shared__ int tok_img[8], tok_out[8];
    pdl_trigger();
    pdl_wait();
    const int tile = blockIdx.x;
    int j = 0;
    while (j + 1 < a.n_proj && tile >= a.p[j + 1].tiles_begin) j++;
    const IdProj &P = a.p[j];
    const int local = tile - P.tiles_begin;
    const int e = local / P.row_tiles, rt = local % P.row_tiles;
    const int n_items = __ldg(a.counts + e);
    if (n_items <= 0) return;   // no planned pair: no weights read
    const int item0 = __ldg(a.offsets + e);
    const uint8_t *wbase = P.w + (int64_t)e * P.expert_bytes + (int64_t)rt * P.chunks * L::UNIT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t4 = lane & 3, g = lane >> 2;
    const int Kb = P.K / QB;

    for (int pass = 0; pass * 8 < n_items; pass++) {
        if (threadIdx.x < 8) {
            const int idx = pass * 8 + threadIdx.x;
            int p = idx < n_items ? __ldg(a.items + item0 + idx) : -1;
            if (p < 0 || p / a.k >= a.rows) p = -1;   // not a pair of this bucket: skip
            tok_img[threadIdx.x] = p >= 0 ? p / a.k : -1;
            tok_out[threadIdx.x] = p;
        }
        __syncthreads();
        const int rB = tok_img[g], rS0 = tok_img[2 * t4], rS1 = tok_img[2 * t4 + 1];
        const uint8_t *imgB = rB >= 0 ? a.img + (int64_t)rB * a.img_row_bytes : nullptr;
        const uint8_t *imgS0 = rS0 >= 0 ? a.img + (int64_t)rS0 * a.img_row_bytes : nullptr;
        const uint8_t *imgS1 = rS1 >= 0 ? a.img + (int64_t)rS1 * a.img_row_bytes : nullptr;
        float acc[UNIT_GROUPS][4];
#pragma unroll
        for (int r = 0; r < UNIT_GROUPS; r++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[r][i] = 0.0f;
        for (int b = warp; b < Kb; b += RW) {
            const uint8_t *unit = wbase + (int64_t)(b >> 2) * L::UNIT;
            BSide s;
            bside<WT>(load_raw(imgB, imgS0, imgS1, b, t4), s);
            block_rows<WT, false>(unit + (b & 3) * L::BLOCK, 0, unit + L::SCALES + (b & 3) * 256, 0, lane, s, acc);
        }
#pragma unroll
        for (int r = 0; r < UNIT_GROUPS; r++)
#pragma unroll
            for (int i = 0; i < 4; i++) red_id[warp * VALS + (r * 4 + i) * 32 + lane] = acc[r][i];
        __syncthreads();
        for (int t = threadIdx.x; t < VALS; t += RW * 32) {
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < RW; w++) sum += red_id[w * VALS + t];
            int row, slot;
            val_pos(t, row, slot);
            row += rt * UNIT_ROWS;
            const int orow = tok_out[slot];
            if (row < P.N && orow >= 0) P.y[(int64_t)orow * P.N + row] = sum;
        }
        __syncthreads();   // tok_* and red_id are reused by the next pass
    }
}

// ---------------------------------------------------------------- weight pack
// One CTA of 256 threads per 128x128 unit. Canonical blocks are only 2-byte
// aligned, so they are read byte by byte.
template <int WT>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ src, int N, int K, int chunks,
                                                   uint8_t *__restrict__ dst) {
    using L = Layout<WT>;
    constexpr int SB = WT == QK_W_Q4_0 ? Q4_0_BYTES : Q8_0_BYTES;
    constexpr int REGIONS = WT == QK_W_Q4_0 ? 4 : 8;
    const int64_t unit = blockIdx.x;
    const int rt = (int)(unit / chunks), c = (int)(unit % chunks);
    const int Kb = K / QB;
    uint8_t *out = dst + unit * L::UNIT;
    auto byte_at = [&](int n, int b, int off) -> uint32_t {
        if (n >= N || b >= Kb) return 0u;
        return src[((int64_t)n * Kb + b) * SB + off];
    };
    auto word_at = [&](int n, int b, int off) -> uint32_t {
        return byte_at(n, b, off) | (byte_at(n, b, off + 1) << 8) | (byte_at(n, b, off + 2) << 16) |
               (byte_at(n, b, off + 3) << 24);
    };
    const int n0 = rt * UNIT_ROWS;
    for (int idx = threadIdx.x; idx < 4 * REGIONS * 32; idx += 256) {
        const int jb = idx / (REGIONS * 32), k = (idx / 32) % REGIONS, l = idx % 32, g = l >> 2, t = l & 3;
        const int b = 4 * c + jb;
        uint4 v;
        if (WT == QK_W_Q4_0) {
            const int off = 2 + 4 * t;
            v.x = word_at(n0 + 32 * k + g, b, off);
            v.y = word_at(n0 + 32 * k + g + 8, b, off);
            v.z = word_at(n0 + 32 * k + 16 + g, b, off);
            v.w = word_at(n0 + 32 * k + 24 + g, b, off);
        } else {
            v.x = word_at(n0 + 16 * k + g, b, 2 + 4 * t);
            v.y = word_at(n0 + 16 * k + g, b, 18 + 4 * t);
            v.z = word_at(n0 + 16 * k + g + 8, b, 2 + 4 * t);
            v.w = word_at(n0 + 16 * k + g + 8, b, 18 + 4 * t);
        }
        *reinterpret_cast<uint4 *>(out + jb * L::BLOCK + k * 512 + l * 16) = v;
    }
    // scales: block jb, lane group g, row group r -> half2 (row 16r+g, row 16r+g+8)
    for (int idx = threadIdx.x; idx < 4 * 8 * 8; idx += 256) {
        const int jb = idx / 64, g = (idx / 8) % 8, r = idx % 8;
        const int b = 4 * c + jb, n = n0 + 16 * r + g;
        const uint32_t lo = byte_at(n, b, 0) | (byte_at(n, b, 1) << 8);
        const uint32_t hi = byte_at(n + 8, b, 0) | (byte_at(n + 8, b, 1) << 8);
        *reinterpret_cast<uint32_t *>(out + L::SCALES + jb * 256 + g * 32 + r * 4) = lo | (hi << 16);
    }
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

template <int WT>
size_t sk_smem() {
    using L = Layout<WT>;
    return (size_t)L::SLOTS * L::UNIT + ((size_t)CW * HALF_VALS + 2 * VALS) * sizeof(float) +
           2 * L::SLOTS * sizeof(uint64_t);
}

}  // namespace

// Workspace of the ordinary path: [G][2][VALS] partial sums, then one counter
// per 128-row tile; G = min(units, SMs) CTAs.
int64_t mmvq_workspace_bytes(int n_proj, const qk_proj *projs) {
    int64_t U = 0, R = 0;
    for (int j = 0; j < n_proj; j++) {
        const int64_t rts = ceil_div(projs[j].N, UNIT_ROWS);
        U += rts * ceil_div(projs[j].K, UNIT_COLS);
        R += rts;
    }
    const int64_t G = U < sm_count() ? U : sm_count();
    return G * 2 * VALS * (int64_t)sizeof(float) + R * (int64_t)sizeof(unsigned int);
}

qk_status read_device_faults(uint32_t *faults) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_qk_faults, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_qk_faults, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(QK_ERR_CUDA, "qk_device_faults: %s", cudaGetErrorString(e));
    *faults = v;
    return QK_OK;
}

qk_status launch_weight_pack(int wtype, const uint8_t *blocks, int64_t N, int64_t K, uint8_t *packed,
                             cudaStream_t s) {
    const int64_t chunks = ceil_div(K, UNIT_COLS);
    const int64_t units = ceil_div(N, UNIT_ROWS) * chunks;
    if (units == 0) return QK_OK;
    if (wtype == QK_W_Q4_0)
        pack_kernel<QK_W_Q4_0><<<(unsigned)units, 256, 0, s>>>(blocks, (int)N, (int)K, (int)chunks, packed);
    else
        pack_kernel<QK_W_Q8_0><<<(unsigned)units, 256, 0, s>>>(blocks, (int)N, (int)K, (int)chunks, packed);
    count_launch();
    return check_launch("weight_pack");
}

template <int WT>
static qk_status launch_sk(const SkArgs &a, int G, cudaStream_t s) {
    static bool configured = false;
    const size_t smem = sk_smem<WT>();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(mmvq_sk_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return fail(QK_ERR_CUDA, "mmvq: shared memory attribute: %s", cudaGetErrorString(e));
        configured = true;
    }
    return launch_pdl("mmvq", mmvq_sk_kernel<WT>, dim3(G), dim3(THREADS), smem, s, a);
}

qk_status launch_mmvq(const uint8_t *img, int64_t row_blocks, int T, int n_proj, const qk_proj *projs,
                      const int32_t *live, void *ws, size_t ws_bytes, cudaStream_t s) {
    SkArgs a = {};
    a.img = img;
    a.img_row_bytes = row_blocks * Q8_1_BYTES;
    a.T = T;
    a.live = live;
    a.n_proj = n_proj;
    int64_t U = 0;
    int R = 0;
    for (int j = 0; j < n_proj; j++) {
        SkProj &d = a.p[j];
        d.w = static_cast<const uint8_t *>(projs[j].w);
        d.y = projs[j].y;
        d.y_stride = projs[j].y_stride;
        d.N = (int)projs[j].N;
        d.K = (int)projs[j].K;
        d.chunks = (int)ceil_div(d.K, UNIT_COLS);
        d.row_tiles = (int)ceil_div(d.N, UNIT_ROWS);
        d.unit_base = U;
        d.rt_base = R;
        U += (int64_t)d.row_tiles * d.chunks;
        R += d.row_tiles;
    }
    a.U = U;
    const int G = (int)(U < sm_count() ? U : sm_count());
    const int64_t need = mmvq_workspace_bytes(n_proj, projs);
    if (!ws || ws_bytes < (size_t)need)
        return fail(QK_ERR_WORKSPACE, "mmvq: workspace %zu < %lld bytes", ws_bytes, (long long)need);
    a.ws_part = static_cast<float *>(ws);
    a.ws_cnt = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(ws) + (int64_t)G * 2 * VALS * sizeof(float));
    return projs[0].wtype == QK_W_Q4_0 ? launch_sk<QK_W_Q4_0>(a, G, s) : launch_sk<QK_W_Q8_0>(a, G, s);
}

qk_status launch_mmvq_id(const uint8_t *img, int64_t row_blocks, int rows, int k, int n_proj,
                         const qk_proj_id *projs, const int32_t *counts, const int32_t *offsets,
                         const int32_t *items, cudaStream_t s) {
    IdArgs a = {};
    a.img = img;
    a.img_row_bytes = row_blocks * Q8_1_BYTES;
    a.rows = rows;
    a.k = k;
    a.n_proj = n_proj;
    a.counts = counts;
    a.offsets = offsets;
    a.items = items;
    int tiles = 0;
    for (int j = 0; j < n_proj; j++) {
        IdProj &d = a.p[j];
        d.w = static_cast<const uint8_t *>(projs[j].w);
        d.y = projs[j].y;
        d.expert_bytes = packed_bytes(projs[j].wtype, projs[j].N, projs[j].K);
        d.N = (int)projs[j].N;
        d.K = (int)projs[j].K;
        d.chunks = (int)ceil_div(d.K, UNIT_COLS);
        d.row_tiles = (int)ceil_div(d.N, UNIT_ROWS);
        d.tiles_begin = tiles;
        tiles += d.row_tiles * projs[j].n_experts;
    }
    const size_t smem = (size_t)RW * VALS * sizeof(float);
    if (projs[0].wtype == QK_W_Q4_0)
        return launch_pdl("mmvq_id", mmvq_id_kernel<QK_W_Q4_0>, dim3(tiles), dim3(RW * 32), smem, s, a);
    return launch_pdl("mmvq_id", mmvq_id_kernel<QK_W_Q8_0>, dim3(tiles), dim3(RW * 32), smem, s, a);
}

}  // namespace qk

// ------------------------------------------------------------------ no-allocation variant
// qk_mmvq_static_ws: the workspace is this file-scope device array instead of
// caller memory. In host code the array's name is only a host-side stand-in,
// so its device address is looked up once per device (with that device
// current) and cached.
static __device__ __align__(256) unsigned char g_mmvq_static_ws[QK_MMVQ_STATIC_WS_BYTES];

namespace {
constexpr int MAX_DEVICES = 64;
std::mutex g_static_ws_mu;
void *g_static_ws_ptr[MAX_DEVICES] = {};
}  // namespace

extern "C" QK_API qk_status qk_mmvq_static_ws(const void *img, int64_t img_row_blocks, int64_t T,
                                              int32_t n_proj, const qk_proj *projs,
                                              const int32_t *d_live_rows, qk_stream stream) {
    if (!projs || n_proj < 1 || n_proj > 8)
        return qk::fail(QK_ERR_ARG, "qk_mmvq_static_ws: projs null or n_proj=%d not in 1..8", (int)n_proj);
    const size_t need = qk_mmvq_workspace_bytes(n_proj, projs);
    if (need > QK_MMVQ_STATIC_WS_BYTES)
        return qk::fail(QK_ERR_UNSUPPORTED, "qk_mmvq_static_ws: needs %zu bytes of scratch, the static array holds %u",
                    need, (unsigned)QK_MMVQ_STATIC_WS_BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return qk::fail(QK_ERR_CUDA, "qk_mmvq_static_ws: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES) return qk::fail(QK_ERR_UNSUPPORTED, "qk_mmvq_static_ws: device %d", dev);
    void *ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_ws_mu);
        if (!g_static_ws_ptr[dev]) {
            e = cudaGetSymbolAddress(&g_static_ws_ptr[dev], g_mmvq_static_ws);
            if (e != cudaSuccess) {
                g_static_ws_ptr[dev] = nullptr;
                return qk::fail(QK_ERR_CUDA, "qk_mmvq_static_ws: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            }
        }
        ws = g_static_ws_ptr[dev];
    }
    // the counters (and, simply, all scratch this call uses) must start at zero
    e = cudaMemsetAsync(ws, 0, need, (cudaStream_t)stream);
    if (e != cudaSuccess) return qk::fail(QK_ERR_CUDA, "qk_mmvq_static_ws: clearing scratch: %s", cudaGetErrorString(e));
    return qk_mmvq(img, img_row_blocks, T, n_proj, projs, d_live_rows, ws, QK_MMVQ_STATIC_WS_BYTES, stream);
}
